"""Token sampling from one row of logits: the oracle of nc_sample.

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's CPU
baseline use this module. Plain numpy, one explicit loop wherever the order
of floating-point operations decides an integer.

The steps follow nanoinfer's sampling section (sampling.py: "temperature,
top-k, top-p, seeded draw"): temperature, then top-k, then top-p, then the
softmax of what is left, then an inverse-CDF draw; temperature 0 is the
arg-max (lowest index on ties). The truncations are the transformers logits
warpers the page checks itself against:

* top-k keeps every token whose scaled logit is at least the k-th largest
  (tied values at the k-th place all stay);
* top-p sorts the surviving tokens ascending with a stable sort (equal
  values in index order), takes their softmax, and drops every token whose
  ascending running sum is <= 1 - p; the largest always stays. The page
  reports the two facts this reading rests on: fifty tokens of probability
  0.01 sum to 0.4999997913837433 in fp32, so at p = 0.5 fifty of a hundred
  equiprobable tokens stay, and the stable order of [1, 1, 0, 0] is
  [2, 3, 0, 1], so the token kept alone is index 1.

Precision: the scaled logits, the top-p softmax and its running sum are fp32
(as in the page's implementation), each added in the stated order. The page
leaves the precision of the draw open; here its weights are the same fp32
values exp(s - max) that top-p thresholds, summed in fp64 in index order,
and the drawn token is the first kept one with a positive weight whose
running sum exceeds u times the total (so the weights need not sum to
exactly one, as the page notes; if rounding leaves none, the last kept token
of positive weight). u is the caller's uniform number in [0, 1).

Rows the distribution is undefined for give -1: a NaN logit (any
temperature), and at temperature > 0 a scaled logit of +inf or a row whose
scaled logits are all -inf. A logit of -inf is a valid masked token: its
weight is 0 and it is never drawn.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32


def _argmax_lowest(v: np.ndarray) -> int:
    best = 0
    for i in range(1, v.size):
        if v[i] > v[best]:
            best = i
    return best


def scaled(logits, temperature: float) -> np.ndarray:
    """logits / temperature, each quotient rounded to fp32 (overflow gives inf)."""
    with np.errstate(over="ignore"):
        return (np.asarray(logits, np.float32) / F32(temperature)).astype(np.float32)


def top_k_mask(s: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose score is at least the k-th largest (k <= 0 or k >= V: all)."""
    if k <= 0 or k >= s.size:
        return np.ones(s.size, bool)
    kth = np.sort(s)[::-1][k - 1]
    return s >= kth


def weights(s: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """fp32 exp(s_i - max) of the tokens idx (the max over the kept tokens is
    the row's max: the largest score always stays)."""
    m = F32(np.max(s[idx]))
    return np.array([np.exp(F32(s[i] - m), dtype=np.float32) for i in idx], np.float32)


def top_p_trace(s: np.ndarray, keep: np.ndarray, p: float, full: bool = False):
    """The steps of the top-p cut: the kept tokens in stable ascending order,
    their fp32 softmax total, the fp32 running sums c_j and the cut position
    (the first j < n - 1 with c_j > 1 - p, else n - 1; tokens before it drop).
    Returns (order, tot, c, cut); c has n - 1 entries, filled up to the cut
    (with full=True, all of them: the same chain continued past the cut)."""
    idx = np.nonzero(keep)[0]
    order = idx[np.argsort(s[idx], kind="stable")]  # ascending; equal scores by index
    e = weights(s, order)
    tot = F32(0)
    for x in e:
        tot = F32(tot + x)
    thr = F32(F32(1) - F32(p))
    c = np.full(max(order.size - 1, 0), np.nan, np.float32)
    run = F32(0)
    cut = order.size - 1
    for j in range(order.size - 1):  # the largest always stays
        run = F32(run + F32(e[j] / tot))
        c[j] = run
        if run > thr and cut == order.size - 1:
            cut = j
            if not full:
                break
    return order, tot, c, cut


def top_p_mask(s: np.ndarray, keep: np.ndarray, p: float) -> np.ndarray:
    """Drop, from the kept tokens in stable ascending order, those whose running
    softmax sum is <= 1 - p (p >= 1: nothing dropped)."""
    keep = keep.copy()
    if p >= 1.0:
        return keep
    order, _, _, cut = top_p_trace(s, keep, p)
    keep[order[:cut]] = False
    return keep


def draw_trace(s: np.ndarray, keep: np.ndarray, u: float):
    """Inverse-CDF draw over the kept tokens in index order: fp32 weights,
    fp64 running sums. Returns (token, idx, running sums, r)."""
    idx = np.nonzero(keep)[0]
    w = weights(s, idx)
    tot = 0.0
    for x in w:
        tot += float(x)
    r = float(u) * tot
    cum = np.empty(idx.size, np.float64)
    c = 0.0
    tok = -1
    for j, (i, x) in enumerate(zip(idx, w)):
        c += float(x)
        cum[j] = c
        if tok < 0 and x > 0 and c > r:
            tok = int(i)
    if tok < 0:
        tok = int(idx[np.nonzero(w > 0)[0][-1]])
    return tok, idx, cum, r


def draw(s: np.ndarray, keep: np.ndarray, u: float) -> int:
    return draw_trace(s, keep, u)[0]


def valid(logits, temperature: float) -> bool:
    """False for the rows the sampler answers with -1."""
    v = np.asarray(logits, np.float32)
    if np.isnan(v).any():
        return False
    if temperature == 0.0:
        return True
    s = scaled(v, temperature)
    return not (np.isposinf(s).any() or np.isneginf(s).all())


def sample_counts(logits, temperature: float, top_k: int, top_p: float):
    """(tokens kept after top-k, tokens kept after top-p): (1, 1) at
    temperature 0, (0, 0) for an invalid row."""
    if not valid(logits, temperature):
        return 0, 0
    if temperature == 0.0:
        return 1, 1
    s = scaled(logits, temperature)
    k = top_k_mask(s, top_k)
    return int(k.sum()), int(top_p_mask(s, k, top_p).sum())


def sample(logits, temperature: float, top_k: int, top_p: float, u: float,
           return_kept: bool = False):
    """The sampled token of one row (and, with return_kept, the kept set)."""
    v = np.asarray(logits, np.float32)
    if not valid(v, temperature):
        keep = np.zeros(v.size, bool)
        return (-1, keep) if return_kept else -1
    if temperature == 0.0:
        t = _argmax_lowest(v)
        keep = np.zeros(v.size, bool)
        keep[t] = True
        return (t, keep) if return_kept else t
    s = scaled(v, temperature)
    keep = top_p_mask(s, top_k_mask(s, top_k), top_p)
    t = draw(s, keep, u)
    return (t, keep) if return_kept else t
