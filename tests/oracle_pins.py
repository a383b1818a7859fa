"""Pins of the float64 oracle to facts other than itself.

Each pin raises AssertionError when it fails.  Every pin takes ``mutant``: 0
checks the real oracle; n > 0 checks a deliberately wrong build
(``-DORC_MUTANT=n``), which test_oracle_mutants.py expects to fail at least one
pin.

What the pins rest on:
  * the storage formats: exhaustive comparison with torch's own bf16 and
    float8_e4m3fn decoders, plus hand-worked values (tests/golden);
  * the visibility and window rules as the V4.1 page states them (prefill
    and decode forms), plus hand-worked cases (tests/golden);
  * scores: exact rational arithmetic on tiny inputs (Python fractions of the
    torch-decoded values), a closed form (q = k gives |k|^2) and the head
    permutation invariance;
  * top-k: brute force by Python sorting, with planted ties;
  * attention: a second, dense-masked formulation (the V3.2 page's
    index_mask form) in numpy, the identity that keeping every
    visible position equals dense attention over window + all visible
    compressed rows, V = 1 giving 1 (weights sum to one), W=1/K=0 giving the
    query's own V row, Q = 0 giving the plain mean of V.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import oracle
from helpers import bf16_to_f64, decode, e4m3_to_f64, problem
from indexer_selected_sparse_score_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- formats ---

def pin_bf16_exhaustive(mutant=0):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bf16_to_f64(bits)
    got = np.array([oracle.bf16_value(int(b), mutant) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got)), "bf16 decode differs from torch"
    assert np.array_equal(np.signbit(ref[~both_nan]), np.signbit(got[~both_nan]))


def pin_e4m3_exhaustive(mutant=0):
    bits = np.arange(256, dtype=np.uint32).astype(np.uint8)
    ref = e4m3_to_f64(bits)
    got = np.array([oracle.e4m3_value(int(b), mutant) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got)), "e4m3 decode differs from torch"


def pin_format_golden(mutant=0):
    with open(os.path.join(GOLDEN, "e4m3_bf16_values.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, hx, val = line.split()
            bits = int(hx, 16)
            got = oracle.e4m3_value(bits, mutant) if fmt == "e4m3" else oracle.bf16_value(bits, mutant)
            want = float(val)
            if np.isnan(want):
                assert np.isnan(got), line
            else:
                assert got == want and np.signbit(got) == np.signbit(want), (line, got)


# ------------------------------------------------------ visibility, window ---

def _parse_slots(text):
    out = []
    for part in text.split(","):
        if ".." in part:
            a, b = part.split("..")
            out.extend(range(int(a), int(b) + 1))
        else:
            out.append(int(part))
    return out


def pin_window_golden(mutant=0):
    with open(os.path.join(GOLDEN, "window_visibility.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, nv, slots = [x.strip() for x in line.split("|")]
            pos, W, R, r = map(int, head.split())
            assert oracle.n_vis(pos, r, mutant) == int(nv), line
            assert oracle.window_slots(pos, W, R, mutant) == _parse_slots(slots), line


def pin_visibility_forms(mutant=0):
    """Both forms the V4.1 page gives for the visible compressed count, and the
    per-entry form (j+1)*r <= t+1, for every t < 64 and r in 1..8."""
    for r in range(1, 9):
        seqlen = 64
        # prefill form: query i sees positions j < (i+1)//r among seqlen//r
        compress_lens = np.arange(1, seqlen + 1) // r
        for t in range(seqlen):
            visible_prefill = [j for j in range(seqlen // r) if not (j >= compress_lens[t])]
            nv = oracle.n_vis(t, r, mutant)
            assert list(range(min(nv, seqlen // r))) == visible_prefill, (r, t)
            # decode form: end_pos // ratio with end_pos = start_pos + 1
            assert nv == (t + 1) // r, (r, t)
            for j in range(70):
                assert ((j + 1) * r <= t + 1) == (j < nv), (r, t, j)


def pin_window_rule(mutant=0):
    """Decode ring (V4.1 get_window_topk_idxs): the set of filled slots is the
    last W positions ending at the query's own position, oldest first."""
    for W in (1, 3, 8, 16):
        for pos in range(0, 3 * W + 2):
            slots = oracle.window_slots(pos, W, W, mutant)
            oldest = pos % W + 1
            ring = list(range(oldest, W)) + list(range(oldest))
            ring = [s for s in ring if s <= pos]           # ring still filling
            assert slots == ring, (W, pos, slots, ring)


# ------------------------------------------------------------------ scores ---

def _tiny_index_problem(seed, q_dtype, k_dtype, q_scale, k_scale, H_I=3, D_I=8, N_c=11, B=2, T=3, r=2):
    spec = wl.Spec("tiny", B=B, T=T, r=r, N_c=N_c, H_I=H_I, D_I=D_I, K=4, H=2, D=8, W=4, R=4,
                   q_dtype=q_dtype, k_dtype=k_dtype, q_scale=q_scale, k_scale=k_scale,
                   pos_mode="uniform", pos_lo=5, pos_hi=2 * N_c - 1, w_div=1.0)
    return wl.generate(spec, seed)


def _exact_scores(w):
    """Exact rational S[t, s] from the torch-decoded values."""
    q = decode(w.q_I, w.q_dtype)
    k = decode(w.k_I, w.k_dtype)
    out = {}
    for t in range(w.T):
        b, nv = int(w.q_seq[t]), (int(w.q_pos[t]) + 1) // w.r
        for s in range(nv):
            ks = Fraction(float(w.k_scale[b, s])) if w.k_scale is not None else Fraction(1)
            total = Fraction(0)
            for h in range(w.H_I):
                qs = Fraction(float(w.q_scale[t, h])) if w.q_scale is not None else Fraction(1)
                dot = sum(Fraction(float(q[t, h, d])) * qs * Fraction(float(k[b, s, d])) * ks
                          for d in range(w.D_I))
                total += Fraction(float(w.w[t, h])) * max(dot, Fraction(0))
            out[(t, s)] = total
    return out


def pin_scores_exact(mutant=0):
    cases = [(1, wl.BF16, wl.BF16, False, False), (2, wl.BF16, wl.FP8_E4M3, False, True),
             (3, wl.FP8_E4M3, wl.FP8_E4M3, True, True)]
    for seed, qd, kd, qs, ks in cases:
        w = _tiny_index_problem(seed, qd, kd, qs, ks)
        p = problem(w)
        S, A = oracle.index_scores(p, with_magnitude=True, mutant=mutant)
        exact = _exact_scores(w)
        for t in range(w.T):
            nv = (int(w.q_pos[t]) + 1) // w.r
            for s in range(w.N_c):
                if s >= nv:
                    assert S[t, s] == -np.inf, (t, s)
                    continue
                e = float(exact[(t, s)])
                assert abs(S[t, s] - e) <= 1e-13 * A[t, s] + 1e-300, (seed, t, s, S[t, s], e)
                assert A[t, s] >= abs(e) * (1 - 1e-12)


def pin_scores_closed_form(mutant=0):
    """One head with w = 1 whose query equals the key: S = |k|^2."""
    w = _tiny_index_problem(7, wl.BF16, wl.BF16, False, False, H_I=2, D_I=16, N_c=6, B=1, T=1, r=1)
    w.q_pos[:] = 5
    w.w[:] = 0.0
    w.w[0, 0] = 1.0
    s = 4
    w.q_I[0, 0] = w.k_I[0, s]
    S = oracle.index_scores(problem(w), mutant=mutant)
    k = bf16_to_f64(w.k_I[0, s])
    assert S[0, s] == float(np.dot(k, k)), (S[0, s], float(np.dot(k, k)))


def pin_scores_head_permutation(mutant=0):
    """Permuting the index heads (queries and weights together) keeps S."""
    w = _tiny_index_problem(11, wl.BF16, wl.FP8_E4M3, False, True, H_I=5)
    S0 = oracle.index_scores(problem(w), mutant=mutant)
    perm = np.array([3, 0, 4, 1, 2])
    w.q_I = np.ascontiguousarray(w.q_I[:, perm])
    w.w = np.ascontiguousarray(w.w[:, perm])
    S1 = oracle.index_scores(problem(w), mutant=mutant)
    fin = np.isfinite(S0)
    assert np.array_equal(np.isfinite(S1), fin)
    assert np.allclose(S0[fin], S1[fin], rtol=1e-13, atol=0)


# ------------------------------------------------------------------- top-k ---

def _brute_topk(scores, nv, K):
    order = sorted(range(nv), key=lambda s: (-scores[s], s))
    keep = sorted(order[:min(K, nv)])
    return keep + [-1] * (K - len(keep))


def pin_topk_bruteforce(mutant=0):
    rng = np.random.default_rng(5)
    for trial in range(300):
        nv = int(rng.integers(0, 40))
        K = int(rng.integers(0, 45))
        # coarse values plant many ties
        sc = np.round(rng.normal(size=max(nv, 1)) * 3) / 3
        got = oracle.topk_row(sc, nv, K, mutant).tolist()
        assert got == _brute_topk(sc.tolist(), nv, K), (trial, nv, K)


# --------------------------------------------------------------- attention ---

def _tiny_attn(seed, r=2, W=4, R=None, N_c=12, T=4, B=2, H=3, D=8, sink=False, pos_lo=3):
    R = R or W
    spec = wl.Spec("tiny_attn", B=B, T=T, r=r, N_c=N_c, H_I=2, D_I=8, K=5, H=H, D=D, W=W, R=R,
                   pos_mode="uniform", pos_lo=pos_lo, pos_hi=r * N_c - 1, w_div=1.0, sink=sink)
    return wl.generate(spec, seed)


def _dense_masked(w, idx):
    """The V3.2 page's dense form: scores over every stored key of the sequence
    with an additive mask that is -inf except at the attended keys."""
    Q = bf16_to_f64(w.Q)
    Kw, Vw = bf16_to_f64(w.Kw), bf16_to_f64(w.Vw)
    Kc, Vc = bf16_to_f64(w.Kc), bf16_to_f64(w.Vc)
    out = np.zeros((w.T, w.H, w.D))
    for t in range(w.T):
        b, p = int(w.q_seq[t]), int(w.q_pos[t])
        keys = np.concatenate([Kw[b], Kc[b]])          # [R + N_c, D]
        vals = np.concatenate([Vw[b], Vc[b]])
        mask = np.full(w.R + w.N_c, -np.inf)
        for pp in range(max(0, p - w.W + 1), p + 1):
            mask[pp % w.R] = 0.0
        sel = [c for c in idx[t] if c >= 0]
        mask[w.R + np.array(sel, dtype=np.int64)] = 0.0
        logits = (Q[t] @ keys.T) * float(w.scale) + mask[None, :]   # [H, R + N_c]
        cols = logits
        if w.sink is not None:
            cols = np.concatenate([logits, w.sink.astype(np.float64)[:, None]], axis=1)
        m = cols.max(axis=1, keepdims=True)
        e = np.exp(cols - m)
        a = e / e.sum(axis=1, keepdims=True)
        out[t] = a[:, :logits.shape[1]] @ vals
    return out


def _random_unique_idx(w, K, rng):
    idx = np.full((w.T, K), -1, dtype=np.int32)
    for t in range(w.T):
        nv = (int(w.q_pos[t]) + 1) // w.r
        k = min(K, nv)
        sel = np.sort(rng.choice(nv, size=k, replace=False)) if k else np.array([], dtype=np.int64)
        idx[t, :k] = sel
    return idx


def pin_attn_dense_masked(mutant=0):
    rng = np.random.default_rng(3)
    for seed, r, W, R in [(21, 2, 4, 4), (22, 1, 3, 3), (23, 4, 8, 8), (24, 2, 1, 1), (25, 2, 4, 9)]:
        w = _tiny_attn(seed, r=r, W=W, R=R, pos_lo=0 if seed == 25 else 3)
        idx = _random_unique_idx(w, 5, rng)
        got = oracle.sparse_attn(problem(w), idx, mutant=mutant)
        ref = _dense_masked(w, idx)
        assert np.allclose(got, ref, rtol=0, atol=1e-12), (seed, np.abs(got - ref).max())


def pin_attn_sink_dense(mutant=0):
    rng = np.random.default_rng(4)
    w = _tiny_attn(31, sink=True)
    idx = _random_unique_idx(w, 5, rng)
    got = oracle.sparse_attn(problem(w), idx, mutant=mutant)
    assert np.allclose(got, _dense_masked(w, idx), rtol=0, atol=1e-12)


def pin_attn_sink_limits(mutant=0):
    """The sink joins the softmax denominator only, so for any sink value s a
    head's output is the sink-free output times Z / (Z + e^s), with Z the sum of
    e^l over the attended logits: O_s * (1 + e^(s - LSE)) = O_none (LSE =
    log Z).  Three limits follow: s -> -inf gives O_none exactly, s = LSE
    halves it, s -> +inf sends it to 0.  Z is taken here from the logits
    written out directly (numpy, one dot product per key)."""
    rng = np.random.default_rng(7)
    w = _tiny_attn(33, sink=True)
    idx = _random_unique_idx(w, 5, rng)
    none = _tiny_attn(33, sink=False)
    O0 = oracle.sparse_attn(problem(none), idx, mutant=mutant)
    Q, Kw, Kc = bf16_to_f64(w.Q), bf16_to_f64(w.Kw), bf16_to_f64(w.Kc)
    lse = np.zeros((w.T, w.H))
    for t in range(w.T):
        b, p = int(w.q_seq[t]), int(w.q_pos[t])
        keys = [Kw[b, pp % w.R] for pp in range(max(0, p - w.W + 1), p + 1)]
        keys += [Kc[b, c] for c in idx[t] if c >= 0]
        lg = (Q[t] @ np.array(keys).T) * float(w.scale)          # [H, n]
        mx = lg.max(axis=1)
        lse[t] = mx + np.log(np.exp(lg - mx[:, None]).sum(axis=1))
    # s -> -inf: the sink-free output, exactly
    w.sink = np.full(w.H, -1e30, dtype=np.float32)
    assert np.array_equal(oracle.sparse_attn(problem(w), idx, mutant=mutant), O0)
    # s -> +inf: nothing left of the output
    w.sink = np.full(w.H, 1e30, dtype=np.float32)
    assert np.array_equal(oracle.sparse_attn(problem(w), idx, mutant=mutant), np.zeros_like(O0))
    # s = LSE (one token's values, rounded to the sink's fp32): O_none / (1 + e^(s - LSE))
    for t in range(w.T):
        w.sink = lse[t].astype(np.float32)
        s = w.sink.astype(np.float64)
        Os = oracle.sparse_attn(problem(w), idx, rows=[t], mutant=mutant)[0]
        want = O0[t] / (1.0 + np.exp(s - lse[t]))[:, None]
        assert np.allclose(Os, want, rtol=1e-12, atol=1e-14), (t, np.abs(Os - want).max())
        assert np.allclose(Os, O0[t] / 2, rtol=1e-6, atol=1e-14)


def pin_attn_all_visible_identity(mutant=0):
    """With K >= n_vis the selected set is every visible
    position, so the step equals dense attention over the window plus all
    visible compressed rows."""
    w = _tiny_attn(41, r=2, W=4, N_c=8, pos_lo=3)
    K = 16
    idx, O = oracle.fused(problem(w), K, mutant=mutant)
    full = np.full((w.T, K), -1, dtype=np.int32)
    for t in range(w.T):
        nv = (int(w.q_pos[t]) + 1) // w.r
        full[t, :nv] = np.arange(nv)
    assert np.array_equal(idx, full)
    assert np.allclose(O, _dense_masked(w, full), rtol=0, atol=1e-12)


def pin_attn_weights_sum_to_one(mutant=0):
    """With every V row equal to 1 the output is exactly the
    sum of the softmax weights, which must be 1."""
    w = _tiny_attn(51)
    one = wl.to_bf16_bits(np.ones(1, dtype=np.float32))[0]
    w.Vw[:] = one
    w.Vc[:] = one
    idx = _random_unique_idx(w, 5, np.random.default_rng(1))
    O = oracle.sparse_attn(problem(w), idx, mutant=mutant)
    assert np.allclose(O, 1.0, rtol=0, atol=1e-12)


def pin_attn_special_cases(mutant=0):
    # W = 1, nothing selected: the output is the query's own V row.
    w = _tiny_attn(61, W=1, R=5)
    idx = np.full((w.T, 3), -1, dtype=np.int32)
    O = oracle.sparse_attn(problem(w), idx, mutant=mutant)
    Vw = bf16_to_f64(w.Vw)
    for t in range(w.T):
        b, p = int(w.q_seq[t]), int(w.q_pos[t])
        assert np.array_equal(O[t], np.broadcast_to(Vw[b, p % w.R], (w.H, w.D))), t
    # Q = 0: every logit is 0 and the output is the mean of the attended V rows.
    w = _tiny_attn(62, W=4)
    w.Q[:] = 0
    idx = _random_unique_idx(w, 5, np.random.default_rng(2))
    O = oracle.sparse_attn(problem(w), idx, mutant=mutant)
    Vw, Vc = bf16_to_f64(w.Vw), bf16_to_f64(w.Vc)
    for t in range(w.T):
        b, p = int(w.q_seq[t]), int(w.q_pos[t])
        rows = [Vw[b, pp % w.R] for pp in range(max(0, p - w.W + 1), p + 1)]
        rows += [Vc[b, c] for c in idx[t] if c >= 0]
        mean = np.mean(rows, axis=0)
        assert np.allclose(O[t], mean[None, :], rtol=0, atol=1e-13), t


ALL_PINS = [pin_bf16_exhaustive, pin_e4m3_exhaustive, pin_format_golden, pin_window_golden,
            pin_visibility_forms, pin_window_rule, pin_scores_exact, pin_scores_closed_form,
            pin_scores_head_permutation, pin_topk_bruteforce, pin_attn_dense_masked,
            pin_attn_sink_dense, pin_attn_sink_limits, pin_attn_all_visible_identity, pin_attn_weights_sum_to_one,
            pin_attn_special_cases]
