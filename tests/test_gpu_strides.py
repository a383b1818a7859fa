"""Caches kept in larger allocations, as a model holds them, and padded score
rows (GPU only).

"DeepSeek-V4.1-Flash-NVFP4 inference/model.py" allocates the index key cache
and the compressed KV cache for max_seq_len / ratio rows per sequence and
uses the first end_pos // ratio of them (Indexer.__init__, Indexer.forward;
Attention.__init__); the window ring likewise lives in a per-layer buffer.
Here every cache sits in an allocation with more rows per sequence than are
in use (the extra rows hold a byte pattern that must never be read as data),
the sequence strides are passed in the argument structs, and the score
matrix has a row stride above N_c.  Results are compared element by element
with the oracle on the dense arrays.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_run import config_workload, ensure_built
from helpers import n_vis, problem
from indexer_selected_sparse_score_gb300 import binding
from indexer_selected_sparse_score_gb300 import workloads as wl
from tolerances import check_attn, check_scores, check_topk_sets

pytestmark = pytest.mark.gpu

CASES = {
    # decode, batch 4, index 16 x 64 fp8 keys, attention 16 x 128 (CUDA-core paths)
    "c1": lambda: config_workload("c1"),
    # decode, batch 64, index 64 x 128 fp8 keys, 64 heads x 128 (tensor-core paths)
    "c2": lambda: config_workload("c2"),
    # bf16 index keys of dim 64 (CUDA-core scorer) and a sink
    "bf16k_sink": lambda: wl.generate(wl.small("bf16k_sink", k_dtype=wl.BF16, k_scale=False, sink=True)),
    # head dim 512 over one kv tensor is covered by the released-shape tests; here
    # head dim 512 with separate K and V, 16 heads
    "d512": lambda: wl.generate(wl.small("d512", H_I=32, D_I=128, r=2, N_c=600, K=96, H=16, D=512,
                                         pos_lo=300, pos_hi=1199, w_div=32.0)),
}


def pads(w):
    return {"k": w.N_c + 77, "w": w.R + 5, "c": w.N_c + 131}


def sample_rows(w):
    if w.T <= 8:
        return list(range(w.T))
    rng = np.random.default_rng(5)
    return sorted({0, w.T - 1} | set(rng.choice(w.T, size=6, replace=False).tolist()))


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    ensure_built()
    w = CASES[request.param]()
    rows = sample_rows(w)
    S, A = oracle.index_scores(problem(w), rows=rows, with_magnitude=True)
    return request.param, w, rows, S, A


def test_padded_caches_and_score_rows(case):
    name, w, rows, S, A = case
    dp = binding.upload(w, pad=pads(w))
    assert dp.ia.k_seq_stride == (w.N_c + 77) * w.D_I and dp.aa.c_seq_stride == (w.N_c + 131) * w.D
    ws = binding.new_workspace(dp)
    ld = w.N_c + 36
    scores = torch.full((w.T, ld), float("nan"), dtype=torch.float32, device="cuda")
    binding.sa_indexer_scores(dp.ia, scores, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    g = scores.cpu().numpy()
    assert np.isnan(g[:, w.N_c:]).all(), "columns past N_c must be left alone"
    check_scores(g[rows, :w.N_c], S, A)
    # top-k on the padded score rows: exactly the oracle's selection on the same fp32 scores
    idx = torch.full((w.T, w.K), -7, dtype=torch.int32, device="cuda")
    binding.sa_topk(scores, dp.ia, w.K, idx, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    gi = idx.cpu().numpy()
    for t in rows:
        ref = oracle.topk_row(g[t, :w.N_c].astype(np.float64), n_vis(int(w.q_pos[t]), w.r), w.K)
        assert gi[t].tolist() == ref.tolist(), (name, t)
    # attention on the oracle's own indices, read from the padded caches
    o_idx = oracle.topk(problem(w), S, w.K, rows=rows)
    full = gi.copy()
    full[rows] = o_idx
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    binding.sa_sparse_attn(dp.ia, dp.aa, torch.from_numpy(full).cuda(), w.K, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    check_attn(out.float().cpu().numpy().astype(np.float64)[rows], oracle.sparse_attn(problem(w), full, rows=rows))


def test_padded_fused_step(case):
    name, w, rows, S, A = case
    dp = binding.upload(w, pad=pads(w))
    ws = binding.new_workspace(dp)
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((w.T, w.K), -7, dtype=torch.int32, device="cuda")
    binding.sa_fused_decode(dp.ia, dp.aa, w.K, idx, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    g_idx = idx.cpu().numpy()
    o_idx = oracle.topk(problem(w), S, w.K, rows=rows)
    for i, t in enumerate(rows):
        check_topk_sets(g_idx[t], o_idx[i], S[i], A[i], n_vis(int(w.q_pos[t]), w.r), w.K)
    check_attn(out.float().cpu().numpy().astype(np.float64)[rows], oracle.sparse_attn(problem(w), g_idx, rows=rows))
    # the same step on dense caches gives the same indices and outputs
    dd = binding.upload(w)
    ws2 = binding.new_workspace(dd)
    out2 = torch.empty_like(out)
    idx2 = torch.empty_like(idx)
    binding.sa_fused_decode(dd.ia, dd.aa, w.K, idx2, out2, ws2)
    assert torch.equal(idx, idx2) and torch.equal(out, out2)
