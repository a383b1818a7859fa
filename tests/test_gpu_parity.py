"""CUDA path vs the float64 oracle, element by element, on small seeded
workloads that span several tiles and a ragged tail (GPU only)."""
import numpy as np
import pytest

import oracle
from gpu_run import run_attn, run_fused, run_scores, run_topk, run_topk_rows
from helpers import n_vis, problem
from indexer_selected_sparse_score_gb300 import binding
from indexer_selected_sparse_score_gb300 import workloads as wl
from tolerances import check_attn, check_scores, check_topk_sets

pytestmark = pytest.mark.gpu

SMALL = {
    # index 16 x 64 (V4.1 defaults), fp8 keys with scales, r=2
    "i16x64_fp8k": wl.small("i16x64_fp8k"),
    # bf16 keys, no scales (V4.1 bf16-valued keys)
    "i16x64_bf16k": wl.small("i16x64_bf16k", k_dtype=wl.BF16, k_scale=False),
    # index 64 x 128, fp8 keys, r=4, topk 100, attention 64 heads
    "i64x128_fp8k": wl.small("i64x128_fp8k", H_I=64, D_I=128, r=4, N_c=700, K=100, H=64,
                             pos_lo=900, pos_hi=2799, w_div=64.0),
    # fp8 queries with per-token scale and fp8 keys (prefill-style dtypes)
    "i64x128_fp8qk": wl.small("i64x128_fp8qk", H_I=64, D_I=128, r=4, N_c=700, K=100, H=64,
                              q_dtype=wl.FP8_E4M3, q_scale=True, pos_lo=900, pos_hi=2799,
                              w_div=64.0),
    # r = 1 (no compression), one index head, sink present
    "r1_h1_sink": wl.small("r1_h1_sink", r=1, N_c=520, H_I=1, K=33, sink=True, pos_lo=100,
                           pos_hi=519),
    # 64 attention heads (tensor-core attention) with a sink and a window over 128
    "h64_sink_w200": wl.small("h64_sink_w200", H_I=64, D_I=128, r=4, N_c=700, K=300, H=64, W=200,
                              R=200, sink=True, pos_lo=900, pos_hi=2799, w_div=64.0),
    # positions below the window (ring still filling) and n_vis < K, = K
    "early": wl.small("early", B=4, T=4, r=2, N_c=64, K=40, W=32, R=32, pos_lo=0, pos_hi=100),
    # tensor-core index path with 32 and 128 index heads (V4.1 released: 32 x 128)
    "i32x128_fp8k": wl.small("i32x128_fp8k", H_I=32, D_I=128, r=2, N_c=900, K=128, H=32,
                             pos_lo=300, pos_hi=1799, w_div=32.0),
    "i128x128_fp8qk": wl.small("i128x128_fp8qk", H_I=128, D_I=128, r=4, N_c=700, K=100, H=128,
                               q_dtype=wl.FP8_E4M3, q_scale=True, pos_lo=900, pos_hi=2799,
                               w_div=128.0),
    # tensor-core path with tokens that see no compressed row between long ones
    "umma_early": wl.small("umma_early", B=6, T=6, H_I=64, D_I=128, r=4, N_c=700, K=100, H=64,
                           W=32, R=32, w_div=64.0),
    # many short decode tokens on the tensor-core index path: 0-3 key tiles each, so a
    # work-pool chunk spans several tokens and each plan thread takes two tokens
    "umma_many": wl.small("umma_many", B=300, T=300, H_I=64, D_I=128, r=4, N_c=300, K=64, H=64,
                          pos_lo=0, pos_hi=1199, w_div=64.0),
    # tensor-core attention with 9 tiles per token: 64 tokens (cluster pairs, each
    # merging two parts of 5 and 4 tiles) and 128 tokens with a sink (whole tokens)
    "pairs_9tiles": wl.small("pairs_9tiles", B=64, T=64, H_I=64, D_I=128, r=4, N_c=1200, K=1024, H=64,
                             W=128, R=128, pos_lo=4100, pos_hi=4799, w_div=64.0),
    "whole_9tiles_sink": wl.small("whole_9tiles_sink", B=128, T=128, H_I=64, D_I=128, r=4, N_c=1200, K=1024,
                                  H=64, W=128, R=128, sink=True, pos_lo=4100, pos_hi=4799, w_div=64.0),
    # prefill chunk: 96 causal tokens of one sequence, ring of T + W - 1 slots
    "prefill": wl.small("prefill", B=1, T=96, r=4, N_c=160, H_I=64, D_I=128, K=48, H=64, W=16,
                        R=112, q_dtype=wl.FP8_E4M3, q_scale=True, pos_mode="prefill",
                        pos_lo=540, pos_hi=635, w_div=64.0),
}


# fixed positions where the edge cases must appear: n_vis = 0 (position 0),
# n_vis < K, n_vis == K (79 -> 40 with r=2, K=40), window not yet full
POSITIONS = {"early": (np.arange(4, dtype=np.int32), np.array([0, 5, 79, 100], dtype=np.int32)),
             "umma_early": (np.arange(6, dtype=np.int32),
                            np.array([2, 2799, 0, 510, 3, 127], dtype=np.int32))}


@pytest.fixture(scope="module", params=sorted(SMALL))
def case(request):
    w = wl.generate(SMALL[request.param], seed=1000 + sorted(SMALL).index(request.param),
                    positions=POSITIONS.get(request.param))
    S, A = oracle.index_scores(problem(w), with_magnitude=True)
    return request.param, w, S, A


def test_scores(case):
    name, w, S, A = case
    g = run_scores(w)
    check_scores(g, S, A)


def test_topk_exact_on_gpu_scores(case):
    """Top-k is integer work: on the same fp32 scores it must equal the
    oracle's selection exactly."""
    name, w, S, A = case
    g_scores = run_scores(w)
    idx = run_topk(w, g_scores, w.K)
    for t in range(w.T):
        nv = n_vis(int(w.q_pos[t]), w.r)
        ref = oracle.topk_row(g_scores[t].astype(np.float64), nv, w.K)
        assert idx[t].tolist() == ref.tolist(), (name, t)


def test_attn_on_oracle_indices(case):
    name, w, S, A = case
    o_idx = oracle.topk(problem(w), S, w.K)
    g = run_attn(w, o_idx)
    o = oracle.sparse_attn(problem(w), o_idx)
    check_attn(g, o)


def test_fused(case):
    name, w, S, A = case
    g_idx, g_out = run_fused(w)
    o_idx = oracle.topk(problem(w), S, w.K)
    for t in range(w.T):
        check_topk_sets(g_idx[t], o_idx[t], S[t], A[t], n_vis(int(w.q_pos[t]), w.r), w.K)
    # attention parity on the GPU's own selection
    check_attn(g_out, oracle.sparse_attn(problem(w), g_idx))


def test_fused_without_idx_out(case):
    name, w, S, A = case
    _, g_out = run_fused(w, with_idx=False)
    g_idx, g_out2 = run_fused(w)
    assert np.array_equal(g_out, g_out2)


@pytest.mark.parametrize("N_c", [5000, 12000, 30000, 40000])
def test_topk_ties_and_sizes(N_c):
    """Planted ties across chunk boundaries, for rows held in registers (up to
    32768 scores, three block sizes) and rows streamed from memory: exact match
    with the oracle's lower-position tie rule."""
    spec = wl.small("ties", B=5, T=5, r=1, N_c=N_c, K=700, D=128, H=16, pos_mode="fixed", pos_lo=0, pos_hi=0)
    pos = np.array([N_c - 1, N_c // 2, 700, 699, 1500], dtype=np.int32)
    w = wl.generate(spec, seed=77, positions=(np.arange(5, dtype=np.int32), pos))
    rng = np.random.default_rng(8)
    scores = np.round(rng.normal(size=(5, N_c)) * 4).astype(np.float32) / 4
    scores[4, :] = 1.0  # a row of equal scores: the lowest positions win
    scores[3, 10:20] = -0.0
    idx = run_topk(w, scores, spec.K)
    for t in range(5):  # noqa: B007
        nv = n_vis(int(w.q_pos[t]), w.r)
        ref = oracle.topk_row(scores[t].astype(np.float64), nv, spec.K)
        assert idx[t].tolist() == ref.tolist(), t


@pytest.mark.parametrize("T", [6, 320])
@pytest.mark.parametrize("N_c", [5000, 12000, 30000])
def test_topk_threshold_at_the_row_minimum(N_c, T):
    """Rows whose k-th largest score is at or next to the row's minimum, so the
    selection meets the slots past the visible count (key 0, the smallest after
    the range shift), plus rows of two or three levels and a constant row: exact
    match with the oracle, for every register top-k shape (6 rows: 1024 threads
    per row; 320 rows: 512 threads).  Scores past the visible count are large,
    so reading any of them would show."""
    K = 700
    rng = np.random.default_rng(N_c + T)
    nv = np.empty(T, dtype=np.int64)
    scores = np.full((T, N_c), 100.0, dtype=np.float32)
    for t in range(T):
        kind = t % 6
        if kind == 0:    # one position left out: the k-th largest is the second smallest
            nv[t] = K + 1
            row = rng.normal(size=nv[t])
        elif kind == 1:  # the ten smallest tie at the row minimum; five of them are taken
            nv[t] = K + 5
            row = rng.normal(size=nv[t])
            row[rng.choice(nv[t], 10, replace=False)] = row.min() - 1.0
        elif kind == 2:  # three levels over the whole row
            nv[t] = N_c
            row = rng.integers(0, 3, size=nv[t]).astype(np.float64)
        elif kind == 3:  # quarter steps (ties everywhere) at a random visible count
            nv[t] = rng.integers(K + 1, N_c + 1)
            row = np.round(rng.normal(size=nv[t]) * 4) / 4
        elif kind == 4:  # a constant row
            nv[t] = rng.integers(K + 1, N_c + 1)
            row = np.full(nv[t], -1.0)
        else:            # two levels, the upper one held by fewer than K positions
            nv[t] = rng.integers(2 * K, N_c + 1)
            row = np.zeros(nv[t])
            row[rng.choice(nv[t], K // 3, replace=False)] = 2.0
        scores[t, :nv[t]] = row
    idx = run_topk_rows(scores, np.arange(T, dtype=np.int32), (nv - 1).astype(np.int32), T, 1, K)
    for t in range(T):
        ref = oracle.topk_row(scores[t].astype(np.float64), int(nv[t]), K)
        assert idx[t].tolist() == ref.tolist(), (t, t % 6, int(nv[t]))


@pytest.mark.parametrize("K", [1, 2, 31, 255, 256, 257, 4095, 9000])
def test_topk_k_sweep(K):
    """K from one pick to most of the row, around the 256-key bin that is ranked
    directly, on rows of normal scores, of ties (quarter steps) and of two
    levels: exact against the oracle (rows shorter than K keep all of theirs)."""
    T, N_c = 9, 12000
    rng = np.random.default_rng(K)
    nv = np.array([N_c, N_c - 1, 10000, 5000, max(1, K - 1), K, K + 1, 3, N_c], dtype=np.int64)
    nv = np.minimum(nv, N_c)
    scores = np.full((T, N_c), 50.0, dtype=np.float32)
    for t in range(T):
        row = rng.normal(size=N_c)
        if t % 3 == 1:
            row = np.round(row * 4) / 4
        elif t % 3 == 2:
            row = (rng.random(N_c) < 0.3).astype(np.float64)
        scores[t, :nv[t]] = row[:nv[t]]
    idx = run_topk_rows(scores, np.arange(T, dtype=np.int32), (nv - 1).astype(np.int32), T, 1, K)
    for t in range(T):
        ref = oracle.topk_row(scores[t].astype(np.float64), int(nv[t]), K)
        assert idx[t].tolist() == ref.tolist(), (K, t, int(nv[t]))


@pytest.mark.parametrize("H", [16, 64])
def test_k_zero_is_window_only(H):
    w = wl.generate(wl.small("k0", K=0, H=H, W=130, R=130), seed=5)
    _, g = run_fused(w, K=0)
    o = oracle.sparse_attn(problem(w), np.zeros((w.T, 0), dtype=np.int32))
    check_attn(g, o)


def test_shared_kv_tensor():
    """K and V given as one tensor (the V4.1 page's single kv): pointers equal."""
    w = wl.generate(wl.small("kv_same"), seed=6)
    w.Vw = w.Kw
    w.Vc = w.Kc
    S, A = oracle.index_scores(problem(w), with_magnitude=True)
    o_idx = oracle.topk(problem(w), S, w.K)
    dp = binding.upload(w)
    dp.tensors["Vw"], dp.tensors["Vc"] = dp.tensors["Kw"], dp.tensors["Kc"]
    dp.aa.Vw, dp.aa.Vc = dp.aa.Kw, dp.aa.Kc
    g_idx, g = run_fused(w, dp=dp)
    check_attn(g, oracle.sparse_attn(problem(w), g_idx))


def test_empty_batch():
    w = wl.generate(wl.small("empty", T=0, B=1), seed=9, positions=(np.zeros(0, np.int32), np.zeros(0, np.int32)))
    idx, out = run_fused(w)
    assert idx.shape == (0, w.K) and out.shape == (0, w.H, w.D)


def test_bad_device_indices_are_skipped_and_flagged():
    w = wl.generate(wl.small("badidx"), seed=10)
    S = oracle.index_scores(problem(w))
    o_idx = oracle.topk(problem(w), S, w.K)
    bad = o_idx.copy()
    bad[0, 3] = n_vis(int(w.q_pos[0]), w.r) + 5   # past n_vis
    bad[1, 0] = -9                                  # not -1
    g = run_attn(w, bad, expect_status=binding.SA_ERR_DEVICE_DATA)
    clean = bad.copy()
    clean[0, 3] = -1
    clean[1, 0] = -1
    check_attn(g, oracle.sparse_attn(problem(w), clean))


def test_bad_sequence_id_tensor_core_path():
    """A token with an out-of-range sequence id among valid ones on the
    tensor-core index path: flagged, its row fully masked, every other row
    as the oracle computes it."""
    w = wl.generate(wl.small("badseq_umma", B=8, T=8, H_I=64, D_I=128, r=4, N_c=700, K=100, H=64,
                             pos_lo=900, pos_hi=2799, w_div=64.0), seed=12)
    bad = 3
    ref_w = wl.generate(wl.small("badseq_umma", B=8, T=8, H_I=64, D_I=128, r=4, N_c=700, K=100, H=64,
                                 pos_lo=900, pos_hi=2799, w_div=64.0), seed=12)
    S, A = oracle.index_scores(problem(ref_w), with_magnitude=True)
    w.q_seq = w.q_seq.copy()
    w.q_seq[bad] = 99
    dp = binding.upload(w)
    ws = binding.new_workspace(dp)
    import torch
    scores = torch.empty((w.T, w.N_c), dtype=torch.float32, device="cuda")
    binding.sa_indexer_scores(dp.ia, scores, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_ERR_DEVICE_DATA
    g = scores.cpu().numpy()
    assert np.all(np.isneginf(g[bad]))
    keep = [t for t in range(w.T) if t != bad]
    check_scores(g[keep], S[keep], A[keep])


def test_bad_sequence_id_is_flagged():
    w = wl.generate(wl.small("badseq"), seed=11)
    w.q_seq = w.q_seq.copy()
    w.q_seq[1] = 99
    dp = binding.upload(w)
    ws = binding.new_workspace(dp)
    import torch
    scores = torch.empty((w.T, w.N_c), dtype=torch.float32, device="cuda")
    binding.sa_indexer_scores(dp.ia, scores, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_ERR_DEVICE_DATA
    assert binding.sa_check_device_status(ws) == binding.SA_OK  # read-and-clear
