"""Pins of the sampling oracle (oracle/sampling.py) against facts the pages
print, the definitions of the warpers, and brute force. CPU only."""
import os

import numpy as np

from oracle import sampling

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sampling_ties.txt")


def _golden():
    out = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, *v = line.split()
            out[k] = v
    return out


def test_equiprobable_top_p_keeps_fifty():
    g = _golden()
    n, p = int(g["equiprobable_n"][0]), float(g["equiprobable_p"][0])
    # the page's fp32 running sum of fifty 0.01 probabilities
    c = np.float32(0)
    for _ in range(50):
        c = np.float32(c + np.float32(1) / np.float32(100))
    assert float(c) == float(g["equiprobable_fp32_sum_50"][0])
    keep = sampling.top_p_mask(np.zeros(n, np.float32), np.ones(n, bool), p)
    assert keep.sum() == int(g["equiprobable_kept"][0])
    assert keep[n // 2:].all() and not keep[:n // 2].any()  # ascending stable: the last 50 stay


def test_stable_sort_keeps_index_one():
    g = _golden()
    v = np.array([float(x) for x in g["stable_sort_input"]], np.float32)
    assert np.argsort(v, kind="stable").tolist() == [int(x) for x in g["stable_sort_order"]]
    keep = sampling.top_p_mask(v, np.ones(4, bool), 0.01)  # small enough to keep one token
    assert keep.tolist() == [False, True, False, False]
    for u in (0.0, 0.3, 0.999):
        assert sampling.sample(v, 1.0, 0, 0.01, u) == 1


def test_temperature_zero_is_lowest_index_argmax():
    v = np.array([0.5, 2.0, -1.0, 2.0], np.float32)
    for u in (0.0, 0.7):
        assert sampling.sample(v, 0.0, 20, 0.8, u) == 1


def test_top_k_one_is_argmax_and_ties_at_kth_stay():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(1000).astype(np.float32)
    for u in (0.0, 0.5, 0.999):
        assert sampling.sample(v, 0.7, 1, 1.0, u) == int(np.argmax(v))
    w = np.array([3, 2, 2, 2, 1], np.float32)
    assert sampling.top_k_mask(w, 2).tolist() == [True, True, True, True, False]
    assert sampling.top_k_mask(w, 1).tolist() == [True, False, False, False, False]
    assert sampling.top_k_mask(w, 0).all() and sampling.top_k_mask(w, 9).all()


def test_temperature_scaling_exact_for_powers_of_two():
    v = np.array([1.5, -3.25, 0.0, 7.0], np.float32)
    assert np.array_equal(sampling.scaled(v, 1.0), v)
    assert np.array_equal(sampling.scaled(v, 0.5), 2 * v)


def test_draw_frequencies_match_softmax():
    """Brute force over a fine grid of u: the draw's frequencies are the
    normalised kept weights (every token once per its share of [0, 1))."""
    rng = np.random.default_rng(11)
    v = rng.standard_normal(7).astype(np.float32)
    T = 0.8
    s = sampling.scaled(v, T).astype(np.float64)
    p = np.exp(s - s.max())
    p /= p.sum()
    n = 20000
    counts = np.zeros(7)
    for i in range(n):
        counts[sampling.sample(v, T, 0, 1.0, (i + 0.5) / n)] += 1
    assert np.abs(counts / n - p).max() < 2.0 / n


def test_top_p_matches_fp64_definition_away_from_the_boundary():
    """Kept sets equal the fp64 reading of the rule wherever no running sum is
    within 1e-5 of 1 - p (the fp32 rounding cannot decide those cases)."""
    rng = np.random.default_rng(5)
    checked = 0
    for trial in range(300):
        v = (rng.standard_normal(12) * 2).astype(np.float32)
        p = float(rng.uniform(0.1, 0.99))
        order = np.argsort(v, kind="stable")
        e = np.exp(v[order].astype(np.float64) - float(v.max()))
        cs = np.cumsum(e / e.sum())
        if np.abs(cs[:-1] - (1 - p)).min() < 1e-5:
            continue
        want = np.ones(12, bool)
        want[order[:-1][cs[:-1] <= 1 - p]] = False
        got = sampling.top_p_mask(v, np.ones(12, bool), p)
        assert np.array_equal(got, want), trial
        checked += 1
    assert checked > 250


def test_drawn_token_is_kept_and_extremes():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(300).astype(np.float32)
    for u in np.linspace(0, 0.999999, 50):
        t, keep = sampling.sample(v, 0.7, 20, 0.8, float(u), return_kept=True)
        assert keep[t]
        assert 1 <= keep.sum() <= 20
    t0, keep = sampling.sample(v, 0.7, 20, 0.8, 0.0, return_kept=True)
    assert t0 == int(np.nonzero(keep)[0][0])  # u = 0: the first kept index
    t1 = sampling.sample(v, 0.7, 20, 0.8, 0.9999999)
    assert t1 == int(np.nonzero(keep)[0][-1])  # u -> 1: the last kept index


def test_rows_without_a_distribution_give_minus_one():
    v = np.array([0.5, 1.0, -2.0], np.float32)
    for T in (0.0, 0.7):
        assert sampling.sample(np.array([0.5, np.nan, 1.0], np.float32), T, 0, 1.0, 0.3) == -1
    assert sampling.sample(np.array([0.5, np.inf, 1.0], np.float32), 0.7, 0, 1.0, 0.3) == -1
    assert sampling.sample(np.array([0.5, np.inf, 1.0], np.float32), 0.0, 0, 1.0, 0.3) == 1
    ninf = np.full(5, -np.inf, np.float32)
    assert sampling.sample(ninf, 0.9, 0, 0.8, 0.3) == -1
    assert sampling.sample(ninf, 0.0, 0, 0.8, 0.3) == 0  # all equal: lowest index
    # a large logit over a tiny temperature overflows to +inf in fp32
    assert sampling.sample(np.array([100.0, 1.0], np.float32), 1e-37, 0, 1.0, 0.3) == -1
    assert sampling.sample_counts(np.array([0.5, np.nan], np.float32), 0.7, 0, 1.0) == (0, 0)
    assert sampling.sample(v, 0.7, 0, 1.0, 0.3) >= 0


def test_minus_inf_is_a_masked_token():
    v = np.array([-np.inf, 0.3, -np.inf, 1.1, -0.4, -np.inf], np.float32)
    seen = set()
    for i in range(2000):
        t = sampling.sample(v, 0.8, 0, 1.0, (i + 0.5) / 2000)
        seen.add(t)
    assert seen == {1, 3, 4}
    # u -> 1: the last kept token of positive weight, never the trailing -inf
    assert sampling.sample(v, 0.8, 0, 1.0, 1.0) == 4
    assert sampling.sample_counts(v, 0.8, 0, 1.0) == (6, 6)
    assert sampling.sample_counts(v, 0.8, 4, 1.0) == (6, 6)  # ties at the 4th place: all stay
    assert sampling.sample_counts(v, 0.8, 3, 1.0) == (3, 3)


def test_counts_and_trace_agree_with_masks():
    rng = np.random.default_rng(9)
    for trial in range(40):
        v = (rng.standard_normal(300) * 3).astype(np.float32)
        v[rng.integers(0, 300, 40)] = v[rng.integers(0, 300, 40)]  # forced ties
        T, k, p = float(rng.uniform(0.3, 1.5)), int(rng.integers(0, 60)), float(rng.uniform(0.2, 1.0))
        s = sampling.scaled(v, T)
        km = sampling.top_k_mask(s, k)
        pm = sampling.top_p_mask(s, km, p)
        assert sampling.sample_counts(v, T, k, p) == (int(km.sum()), int(pm.sum()))
        order, tot, c, cut = sampling.top_p_trace(s, km, p)
        assert set(order[cut:].tolist()) == set(np.nonzero(pm)[0].tolist()) or p >= 1.0
        # the kept set after top-p is a suffix of the ascending (score, index) order
        keys = [(float(s[i]), int(i)) for i in order]
        assert keys == sorted(keys)


def test_brute_force_three_tokens():
    """Every kept set of a three-token row from the definitions written out by
    hand: the k largest (with ties), then the ascending cut."""
    vals = np.array([0.0, 1.0, 2.0], np.float32)
    e = np.exp(vals.astype(np.float64) - 2.0)
    for k in range(0, 4):
        for p in (0.05, 0.3, 0.6, 0.8, 0.95, 1.0):
            kept = [0, 1, 2] if k in (0, 3) else [2, 1, 0][:k]
            kept = sorted(kept)
            tot = e[kept].sum()
            c = 0.0
            out = list(kept)
            if p < 1.0:
                for j in kept[:-1]:  # ascending order == index order here
                    c += e[j] / tot
                    if c <= 1 - p:
                        out.remove(j)
                    else:
                        break
            _, keep = sampling.sample(vals, 1.0, k, p, 0.5, return_kept=True)
            assert sorted(np.nonzero(keep)[0].tolist()) == out, (k, p)
