"""GPU parity of nc_sample (temperature, top-k, top-p, inverse-CDF draw)
against the sampling oracle, through the C ABI.

Each row's token and its kept counts (after top-k, after top-p) must equal
the oracle's. The only tolerated differences are where fp32 rounding decides
them: the device's expf and the host's float32 exp may differ by a few ulp,
so (a) a top-p running sum within TOPP_TOL(n) of 1 - p, or (b) u * total
within DRAW_TOL * total of a cumulative boundary, may fall on either side;
then the device's answer must still be one of those the bound allows.
"""
import math

import numpy as np
import pytest
import torch

from helpers import guarded
from oracle import sampling
from transformer_decode_gb300 import nc

pytestmark = pytest.mark.gpu

V_MODEL = 151936
ULP = 2.0 ** -24


def TOPP_TOL(n):
    # Both sides fold the same n fp32 terms in the same order; their terms
    # differ by a few ulp, which moves a running sum by at most a few ulp per
    # term in a random walk: 8 + 4 sqrt(n) ulp of a sum <= 1.
    return ULP * (8 + 4 * math.sqrt(n))


DRAW_TOL = 8 * ULP  # fp32 weights a few ulp apart; fp64 sums: relative to the total


@pytest.fixture(scope="module", autouse=True)
def _lib():
    nc.load()


def _u(B, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.rand(B, generator=g, dtype=torch.float64)


def _rows(B, V, seed, std):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, V, generator=g) * std).float()


def _run(logits_cpu, T, k, p, u_cpu, scratch=True):
    B, V = logits_cpu.shape
    lg = logits_cpu.cuda()
    u = u_cpu.cuda()
    tok, chk_t = guarded(B, torch.int32)
    kept, chk_k = guarded(2 * B, torch.int32)
    sampler = nc.Sampler(B, V) if scratch else None
    if sampler is None:
        nc.sample(lg, T, k, p, u, tok, kept.view(B, 2), None)
    else:
        sampler(lg, T, k, p, u, tok, kept.view(B, 2))
    torch.cuda.synchronize()
    chk_t()
    chk_k()
    return tok.cpu().numpy(), kept.view(B, 2).cpu().numpy()


def _check_row(v, T, k, p, u, tok, nk, npp):
    """Compare one row with the oracle; returns 'exact' or 'boundary'."""
    if not sampling.valid(v, T):
        assert (tok, nk, npp) == (-1, 0, 0)
        return "exact"
    if T == 0.0:
        assert (tok, nk, npp) == (sampling.sample(v, 0.0, k, p, u), 1, 1)
        return "exact"
    s = sampling.scaled(v, T)
    km = sampling.top_k_mask(s, k)
    assert nk == int(km.sum()), "top-k count"  # keys compare exactly: no tolerance
    how = "exact"
    keep = km
    if p < 1.0 and nk > 1:
        order, tot, c, cut = sampling.top_p_trace(s, km, p, full=True)
        n = order.size
        keep = km.copy()
        keep[order[:cut]] = False
        jg = n - npp
        if jg != cut:
            thr = float(np.float32(1) - np.float32(p))
            lo, hi = min(jg, cut), max(jg, cut)
            assert 0 <= jg <= n - 1, f"device cut {jg} outside [0, {n - 1}]"
            disputed = c[lo:hi].astype(np.float64)
            assert np.all(np.abs(disputed - thr) <= TOPP_TOL(n)), \
                f"top-p count {npp} vs {n - cut}: running sums {disputed[:4]} vs 1-p {thr}"
            keep_g = km.copy()
            keep_g[order[:jg]] = False
            assert keep_g[tok], "drawn token outside the device's own kept set"
            return "boundary"
    t_o, idx, cum, r = sampling.draw_trace(s, keep, u)
    if tok != t_o:
        assert tok in set(idx.tolist()), "drawn token not kept"
        a, b = sorted((int(np.searchsorted(idx, tok)), int(np.searchsorted(idx, t_o))))
        bounds = cum[a:b]
        assert np.all(np.abs(bounds - r) <= DRAW_TOL * cum[-1]), \
            f"token {tok} vs {t_o}: u*total {r} vs boundaries {bounds[:4]}"
        how = "boundary"
    return how


def _check(logits_cpu, T, k, p, u_cpu):
    tok, kept = _run(logits_cpu, T, k, p, u_cpu)
    L = logits_cpu.numpy()
    U = u_cpu.numpy()
    hows = [_check_row(L[b], T, k, p, float(U[b]), int(tok[b]), int(kept[b, 0]), int(kept[b, 1]))
            for b in range(L.shape[0])]
    return tok, kept, hows


# ------------------------------------------------------------------ small and ragged rows
@pytest.mark.parametrize("V", [1, 7, 1000, 5003])
@pytest.mark.parametrize("T,k,p", [
    (0.7, 20, 0.8),     # the defaults the page reads from Qwen2.5's config
    (1.0, 0, 1.0),      # temperature only
    (0.5, 50, 1.0),     # top-k only
    (1.3, 0, 0.9),      # top-p only
    (0.9, 1, 0.5),      # top-k 1 = arg-max of the scores
    (0.0, 20, 0.8),     # greedy
])
def test_rows_match_oracle(V, T, k, p):
    B = 48
    lg = _rows(B, V, seed=V * 7 + int(T * 10) + k, std=2.0)
    lg[:, : V // 3] = lg[:, V // 3: 2 * (V // 3)]  # exact ties everywhere
    _, kept, hows = _check(lg, T, k, p, _u(B, seed=V + k))
    assert hows.count("boundary") <= B // 8
    if 0 < k < V and T > 0:
        assert (kept[:, 0] >= min(k, V)).all()


# ------------------------------------------------------------------ model-sized rows
@pytest.mark.parametrize("std", [0.6, 3.0])
def test_model_vocab_default_sampler(std):
    """Rows of 151,936 logits (std 0.6: the spread of this model's logits at
    random init, 0.02 * sqrt(896); 3.0: a peakier row) under temperature
    0.7, top-k 20, top-p 0.8; batch 16 as in the paged decode workload."""
    B = 16
    lg = _rows(B, V_MODEL, seed=31 + int(std * 10), std=std)
    lg[3, 1000:1040] = lg[3].max() + 1.0  # an exact 40-way tie at the top
    _, kept, hows = _check(lg, 0.7, 20, 0.8, _u(B, seed=5))
    assert kept[3, 0] >= 40
    assert hows.count("boundary") <= 1


def test_model_vocab_large_kept_sets():
    """Kept sets beyond the shared-memory sort: top-p alone over the whole
    vocabulary, and temperature alone (every token drawn from)."""
    B = 2
    lg = _rows(B, V_MODEL, seed=77, std=1.0)
    _, kept, hows = _check(lg, 1.0, 0, 0.8, _u(B, seed=6))
    assert (kept[:, 0] == V_MODEL).all() and (kept[:, 1] > 8192).all()
    assert hows.count("boundary") <= 1
    lg = _rows(3, V_MODEL, seed=78, std=1.0)
    _, kept, _ = _check(lg, 0.8, 0, 1.0, _u(3, seed=7))
    assert (kept == V_MODEL).all()


@pytest.mark.parametrize("k,p", [(3000, 0.95), (9000, 0.9), (9000, 1.0)])
def test_model_vocab_wide_top_k(k, p):
    """Top-k wide enough that the candidates of the first select pass may not
    fit shared memory (9000): the radix select then finishes over the keys."""
    lg = _rows(3, V_MODEL, seed=90 + k, std=1.0)
    _, kept, hows = _check(lg, 1.0, k, p, _u(3, seed=14))
    assert (kept[:, 0] >= k).all()
    assert hows.count("boundary") <= 1


def test_top_ties_beyond_the_candidate_buffer():
    """10,000 equal top logits at top-k 20: every one of them stays (ties at
    the k-th place), more than the shared-memory buffer holds."""
    lg = _rows(2, V_MODEL, seed=95, std=1.0)
    lg[:, 5000:15000] = 9.0
    tok, kept, hows = _check(lg, 1.0, 20, 0.5, _u(2, seed=15))
    assert (kept[:, 0] == 10000).all() and hows == ["exact", "exact"]
    assert ((tok >= 5000) & (tok < 15000)).all()
    tok, kept, _ = _check(lg, 1.0, 20, 1.0, _u(2, seed=16))
    assert (kept == 10000).all()


def test_ties_beyond_the_shared_sort_are_exact():
    """20,000 equal logits, top-p 0.5: every weight is exactly 1 on both
    sides, so the fp32 chain is identical and the kept half exact."""
    V = 20000
    lg = torch.zeros(2, V)
    lg[1, 123] = 0.5
    tok, kept, hows = _check(lg, 1.0, 0, 0.5, _u(2, seed=8))
    assert hows == ["exact", "exact"]
    assert kept[0, 1] == sampling.sample_counts(lg[0].numpy(), 1.0, 0, 0.5)[1]
    assert tok[0] >= V - kept[0, 1]  # the stable order keeps the highest indices


# ------------------------------------------------------------------ the page's facts
def test_page_tie_facts():
    # 100 equiprobable tokens at p = 0.5 keep 50, the upper half by index
    lg = torch.zeros(64, 100)
    u = _u(64, seed=9)
    tok, kept, hows = _check(lg, 1.0, 0, 0.5, u)
    assert (kept[:, 1] == 50).all() and (tok >= 50).all() and hows.count("exact") == 64
    # the stable order of [1, 1, 0, 0] keeps index 1 alone at a small p
    lg = torch.tensor([[1.0, 1.0, 0.0, 0.0]] * 8)
    tok, kept, _ = _check(lg, 1.0, 0, 0.01, _u(8, seed=10))
    assert (tok == 1).all() and (kept[:, 1] == 1).all()


# ------------------------------------------------------------------ edge rows
def test_invalid_and_masked_rows():
    V = 3000
    lg = _rows(8, V, seed=40, std=1.0)
    lg[0, 17] = float("nan")
    lg[1, 5] = float("inf")
    lg[2, :] = float("-inf")
    lg[3, ::2] = float("-inf")  # masked tokens
    lg[4, 100] = 1e30           # overflows at T = 1e-9: +inf score
    lg[5, :] = 0.0
    lg[5, ::3] = -0.0           # -0 and +0 are the same score
    for T, k, p in ((1e-9, 0, 1.0), (0.8, 10, 0.9), (1.0, 0, 1.0)):
        tok, kept, _ = _check(lg, T, k, p, _u(8, seed=11))
        assert tok[0] == -1 and tok[1] == -1 and tok[2] == -1
        assert (tok[4] == -1) == (T < 1e-6) and tok[4] == (100 if T >= 1e-6 else -1)
        assert tok[3] % 2 == 1
    tok, kept, _ = _check(lg, 0.0, 0, 1.0, _u(8, seed=12))  # greedy
    assert tok[0] == -1 and tok[1] == 5 and tok[2] == 0 and tok[5] == 0


def test_u_grid_reproduces_the_distribution():
    """One row, 4096 evenly spaced u: every device token equals the
    oracle's, so the drawn frequencies are the oracle's exactly."""
    V = 50
    row = _rows(1, V, seed=50, std=1.5)
    B = 4096
    lg = row.repeat(B, 1)
    u = (torch.arange(B, dtype=torch.float64) + 0.5) / B
    tok, _, hows = _check(lg, 0.8, 0, 1.0, u)
    assert hows.count("boundary") == 0
    assert len(set(tok.tolist())) > 10


def test_deterministic_and_temperature_zero_needs_no_scratch():
    lg = _rows(16, V_MODEL, seed=60, std=1.0)
    u = _u(16, seed=13)
    a, ka = _run(lg, 0.7, 20, 0.8, u)
    b, kb = _run(lg, 0.7, 20, 0.8, u)
    assert np.array_equal(a, b) and np.array_equal(ka, kb)
    g, kg = _run(lg, 0.0, 0, 1.0, u, scratch=False)
    assert np.array_equal(g, lg.numpy().argmax(1)) and (kg == 1).all()
