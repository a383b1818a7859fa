"""Parity tolerances, as numbers, with the reading each one takes.

* Index scores: "within 1e-5 relative".  Two checks.
  - Relative to the score itself: |g - o| <= 1e-5 * o at every visible
    position whose score is positive and whose condition number
    kappa = A / o is at most KAPPA_MAX, where A[t,s] = sum_h |w| sum_d
    |q_hat k_hat| is the sum of the absolute terms.  Any fp32 evaluation of a
    sum can only be held to a multiple of u * A (u = 2^-24), so where kappa is
    large (the heads' dot products cancel to a score near 0) the relative
    error of a correct fp32 evaluation exceeds 1e-5 * o; there
  - relative to the condition magnitude: |g - o| <= 1e-5 * A, which holds at
    every visible position (A >= |o|).
  Positions past n_vis must be -inf exactly.
* Top-k: "index sets identical, except for positions whose oracle score lies
  within 1e-5 relative of the k-th score".  Ambiguous = |S[s] - S_k| <=
  1e-5 * (A[s] + A_k), the band in which two scores each within tolerance can
  swap order.  Outside it the sets must agree; sizes must agree; the output
  must be ascending and -1 padded.
* Attention: "2e-3 max relative error (bf16 output)", per (token, head) row,
  relative to the row's largest |o| (o the unrounded float64 oracle).  The
  output is bf16, so what the kernel computed before its final rounding is
  only known to lie in the interval of reals that round (nearest, ties to
  even) to the bf16 value g it wrote.  The check: the distance from o to that
  interval is at most 2e-3 * max_d |o|, i.e. g is the correct rounding of some
  value within 2e-3 of the row max of the oracle.  (Comparing g with
  bf16(o) instead would charge a full bf16 step, up to 2^-7 of an element,
  whenever o lies near a rounding midpoint: more than 2e-3 of the row max at
  the row's larger elements, whatever the kernel's accuracy.)  The share of
  elements equal to bf16(o) and the worst |g - bf16(o)| are recorded too.

Every check records its worst observed error against its bound
(tests/margins.py); the test session prints the table at its end.
"""
import numpy as np

import margins

SCORE_RTOL = 1e-5
ATTN_RTOL = 2e-3
KAPPA_MAX = 64.0


def check_scores(g: np.ndarray, o: np.ndarray, A: np.ndarray):
    """g: GPU scores (fp32), o/A: oracle scores/magnitudes (f64), same shape."""
    g = g.astype(np.float64)
    masked = ~np.isfinite(o)
    assert np.all(np.isneginf(g[masked])), "positions past n_vis must be -inf"
    fin = ~masked
    err = np.abs(g[fin] - o[fin])
    a = A[fin]
    worst_a = float(np.max(err / np.maximum(a, 1e-300))) if err.size else 0.0
    margins.record("score |g-o|/A", worst_a, SCORE_RTOL)
    assert np.all(err <= SCORE_RTOL * a), f"score error {worst_a:.3g} x A exceeds {SCORE_RTOL}"
    s = o[fin]
    pos = s > 0
    rel = err[pos] / s[pos]
    kappa = a[pos] / s[pos]
    cond = kappa <= KAPPA_MAX
    worst_rel = float(np.max(rel[cond])) if np.any(cond) else 0.0
    margins.record("score |g-o|/o (kappa<=64)", worst_rel, SCORE_RTOL)
    margins.record("score |g-o|/o (all S>0)", float(np.max(rel)) if rel.size else 0.0, None)
    margins.record("score share kappa>64", float(np.mean(~cond)) if cond.size else 0.0, None)
    assert np.all(rel[cond] <= SCORE_RTOL), (
        f"score error {worst_rel:.3g} x |S| exceeds {SCORE_RTOL} at a position with A/S <= {KAPPA_MAX}")
    return worst_a


def check_topk_sets(g_idx: np.ndarray, o_idx: np.ndarray, S: np.ndarray, A: np.ndarray, nv: int, K: int):
    """One row: GPU indices vs oracle indices under the ambiguity band."""
    g = g_idx.tolist()
    o = o_idx.tolist()
    k_eff = min(K, nv)
    assert g[k_eff:] == [-1] * (K - k_eff), "tail must be -1"
    gs, os_ = g[:k_eff], o[:k_eff]
    assert gs == sorted(gs), "indices must be ascending"
    assert len(set(gs)) == k_eff and all(0 <= s < nv for s in gs), "indices must be distinct and visible"
    if k_eff == 0 or k_eff == nv:
        assert gs == os_
        return 0
    vals = S[:nv]
    order = np.lexsort((np.arange(nv), -vals))
    kth = order[k_eff - 1]
    amb = np.abs(vals - vals[kth]) <= SCORE_RTOL * (A[:nv] + A[kth])
    gset = {s for s in gs if not amb[s]}
    oset = {s for s in os_ if not amb[s]}
    assert gset == oset, f"top-k sets differ outside the ambiguity band: {sorted(gset ^ oset)[:10]}"
    diff = int(len(set(gs) ^ set(os_)))
    margins.record("top-k picks swapped inside the band", float(diff), None)
    return diff


def _bf16_bits_of_f32(x32: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of float32 values, as uint16 bits."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def _bf16_value(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_step(bits: np.ndarray, up: bool) -> np.ndarray:
    """The adjacent bfloat16 value above (up) or below each finite value."""
    mag = (bits & 0x7FFF).astype(np.int64)
    ordv = np.where(bits & 0x8000, -mag, mag) + (1 if up else -1)
    out = np.where(ordv < 0, 0x8000 | (-ordv), ordv).astype(np.uint16)
    return _bf16_value(out)


def bf16_round(o: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of float64 values, rounded once."""
    o = np.asarray(o, dtype=np.float64)
    c = _bf16_bits_of_f32(o.astype(np.float32))
    cand = np.stack([_bf16_step(c, False), _bf16_value(c), _bf16_step(c, True)])
    dist = np.abs(cand - o[None])
    best = np.argmin(dist, axis=0)
    val = np.take_along_axis(cand, best[None], axis=0)[0]
    # a tie between two neighbours goes to the one with an even last bit
    d_sorted = np.sort(dist, axis=0)
    tie = d_sorted[0] == d_sorted[1]
    if np.any(tie):
        for i in zip(*np.nonzero(tie)):
            opts = [cand[k][i] for k in range(3) if dist[k][i] == d_sorted[0][i]]
            even = [v for v in opts if (_bf16_bits_of_f32(np.float32(v)) & 1) == 0]
            val[i] = even[0]
    return val


def attn_rounding_interval(g: np.ndarray):
    """[lo, hi]: the reals that round to each bf16 value g (ends included)."""
    bits = _bf16_bits_of_f32(np.asarray(g, dtype=np.float64).astype(np.float32))
    v = _bf16_value(bits)
    return (v + _bf16_step(bits, False)) / 2, (v + _bf16_step(bits, True)) / 2


def check_attn(g: np.ndarray, o: np.ndarray):
    """g: GPU bf16 output decoded to f64, o: oracle f64; shape [..., D]."""
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    rowmax = np.max(np.abs(o), axis=-1, keepdims=True)
    lo, hi = attn_rounding_interval(g)
    pre = np.maximum(np.maximum(lo - o, o - hi), 0.0) / np.maximum(rowmax, 1e-300)
    worst = float(np.max(pre)) if pre.size else 0.0
    r = bf16_round(o)
    margins.record("attn pre-rounding error / row max", worst, ATTN_RTOL)
    margins.record("attn |g-bf16(o)| / row max", float(np.max(np.abs(g - r) / np.maximum(rowmax, 1e-300)))
                   if g.size else 0.0, None)
    margins.record("attn share g != bf16(o)", float(np.mean(g != r)) if g.size else 0.0, None)
    assert np.all(pre <= ATTN_RTOL), f"attention error {worst:.3g} x row max exceeds {ATTN_RTOL} before rounding"
    return worst
