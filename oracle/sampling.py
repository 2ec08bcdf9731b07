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
leaves the precision of the draw open; here it is fp64: the kept tokens'
weights exp(s - max), their running sum in index order, and the first token
whose running sum exceeds u times the total (so the weights need not sum to
exactly one, as the page notes). u is the caller's uniform number in [0, 1).
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
    """logits / temperature, each quotient rounded to fp32."""
    return (np.asarray(logits, np.float32) / F32(temperature)).astype(np.float32)


def top_k_mask(s: np.ndarray, k: int) -> np.ndarray:
    """Tokens whose score is at least the k-th largest (k <= 0 or k >= V: all)."""
    if k <= 0 or k >= s.size:
        return np.ones(s.size, bool)
    kth = np.sort(s)[::-1][k - 1]
    return s >= kth


def top_p_mask(s: np.ndarray, keep: np.ndarray, p: float) -> np.ndarray:
    """Drop, from the kept tokens in stable ascending order, those whose running
    softmax sum is <= 1 - p (p >= 1: nothing dropped)."""
    keep = keep.copy()
    if p >= 1.0:
        return keep
    idx = np.nonzero(keep)[0]
    order = idx[np.argsort(s[idx], kind="stable")]  # ascending; equal scores by index
    m = s[order[-1]]
    e = [np.exp(F32(s[i] - m), dtype=np.float32) for i in order]
    tot = F32(0)
    for x in e:
        tot = F32(tot + x)
    thr = F32(F32(1) - F32(p))
    c = F32(0)
    for j in range(order.size - 1):  # the largest always stays
        c = F32(c + F32(e[j] / tot))
        if c <= thr:
            keep[order[j]] = False
        else:
            break
    return keep


def draw(s: np.ndarray, keep: np.ndarray, u: float) -> int:
    """Inverse-CDF draw over the kept tokens in index order, fp64."""
    idx = np.nonzero(keep)[0]
    m = float(max(s[i] for i in idx))
    w = [np.exp(float(s[i]) - m) for i in idx]
    tot = 0.0
    for x in w:
        tot += x
    r = float(u) * tot
    c = 0.0
    for i, x in zip(idx, w):
        c += x
        if c > r:
            return int(i)
    return int(idx[-1])


def sample(logits, temperature: float, top_k: int, top_p: float, u: float,
           return_kept: bool = False):
    """The sampled token of one row (and, with return_kept, the kept set)."""
    v = np.asarray(logits, np.float32)
    if temperature == 0.0:
        t = _argmax_lowest(v)
        keep = np.zeros(v.size, bool)
        keep[t] = True
        return (t, keep) if return_kept else t
    s = scaled(v, temperature)
    keep = top_p_mask(s, top_k_mask(s, top_k), top_p)
    t = draw(s, keep, u)
    return (t, keep) if return_kept else t
