"""Parity tolerances, as numbers, with the reading each one takes.

* Index scores: "within 1e-5 relative".  Read relative to the score's
  condition magnitude A[t,s] = sum_h |w| sum_d |q_hat k_hat| (A >= |S|): a
  finite-precision dot product can only be held to a fraction of the sum of
  its absolute terms.  Positions past n_vis must be -inf exactly.
* Top-k: "index sets identical, except for positions whose oracle score lies
  within 1e-5 relative of the k-th score".  Ambiguous = |S[s] - S_k| <=
  1e-5 * (A[s] + A_k), the band in which two scores each within tolerance can
  swap order.  Outside it the sets must agree; sizes must agree; the output
  must be ascending and -1 padded.
* Attention: "2e-3 max relative error (bf16 output)".  The output is rounded
  to bf16, whose own rounding error is up to 2^-8 of an element, so the bound
  is |g - o| <= 2^-8 |o| + 2e-3 * max_d |o| per (token, head) row, with o the
  unrounded float64 oracle.
"""
import numpy as np

SCORE_RTOL = 1e-5
ATTN_RTOL = 2e-3
BF16_HALF_ULP_REL = 2.0 ** -8


def check_scores(g: np.ndarray, o: np.ndarray, A: np.ndarray):
    """g: GPU scores (fp32), o/A: oracle scores/magnitudes (f64), same shape."""
    g = g.astype(np.float64)
    masked = ~np.isfinite(o)
    assert np.all(np.isneginf(g[masked])), "positions past n_vis must be -inf"
    fin = ~masked
    err = np.abs(g[fin] - o[fin])
    bound = SCORE_RTOL * A[fin]
    worst = float(np.max(err / np.maximum(A[fin], 1e-300))) if err.size else 0.0
    assert np.all(err <= bound), f"score error {worst:.3g} x A exceeds {SCORE_RTOL}"
    return worst


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
    return int(len(set(gs) ^ set(os_)))


def check_attn(g: np.ndarray, o: np.ndarray):
    """g: GPU bf16 output decoded to f64, o: oracle f64; shape [..., D]."""
    rowmax = np.max(np.abs(o), axis=-1, keepdims=True)
    err = np.abs(g - o)
    bound = BF16_HALF_ULP_REL * np.abs(o) + ATTN_RTOL * rowmax
    excess = float(np.max((err - BF16_HALF_ULP_REL * np.abs(o)) / np.maximum(rowmax, 1e-300)))
    assert np.all(err <= bound), f"attention error {excess:.3g} x row max exceeds {ATTN_RTOL} (+ bf16 rounding)"
    return excess
