"""The five workloads at full size (GPU only).

c0 and c1 are compared on every query token; c2 (decode, batch 64), c3
(prefill chunk of 4096 tokens) and c4 (ragged decode, batch 128) on sampled
tokens that the oracle evaluates one by one, including the longest and
shortest contexts and the chunk ends.  The fused path runs exactly as the
benchmark launches it (sa_fused_decode over the whole batch).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_run import config_workload, ensure_built, run_scores, run_topk
from helpers import n_vis, problem
from indexer_selected_sparse_score_gb300 import binding
from tolerances import check_attn, check_scores, check_topk_sets

pytestmark = pytest.mark.gpu


def sample_rows(w, n_random=4):
    if w.T <= 8:
        return list(range(w.T))
    nv = (w.q_pos.astype(np.int64) + 1) // w.r
    rng = np.random.default_rng(w.seed)
    rows = {0, w.T - 1, int(np.argmax(nv)), int(np.argmin(nv))}
    rows |= set(rng.choice(w.T, size=n_random, replace=False).tolist())
    return sorted(rows)


@pytest.fixture(scope="module", params=["c0", "c1", "c2", "c3", "c4"])
def cfg(request):
    ensure_built()
    oracle.set_threads(max(1, min(16, __import__("os").cpu_count() or 1)))
    w = config_workload(request.param)
    rows = sample_rows(w)
    S, A = oracle.index_scores(problem(w), rows=rows, with_magnitude=True)
    return request.param, w, rows, S, A


def test_config_scores(cfg):
    name, w, rows, S, A = cfg
    g = run_scores(w)
    check_scores(g[rows], S, A)


def test_config_topk_exact(cfg):
    name, w, rows, S, A = cfg
    g = run_scores(w)
    idx = run_topk(w, g, w.K)
    for t in rows:
        ref = oracle.topk_row(g[t].astype(np.float64), n_vis(int(w.q_pos[t]), w.r), w.K)
        assert idx[t].tolist() == ref.tolist(), (name, t)


def test_config_fused(cfg):
    name, w, rows, S, A = cfg
    dp = binding.upload(w)
    ws = binding.new_workspace(dp)
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((w.T, w.K), dtype=torch.int32, device="cuda")
    binding.sa_fused_decode(dp.ia, dp.aa, w.K, idx, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    g_idx = idx.cpu().numpy()
    g_out = out.float().cpu().numpy().astype(np.float64)
    o_idx = oracle.topk(problem(w), S, w.K, rows=rows)
    for i, t in enumerate(rows):
        check_topk_sets(g_idx[t], o_idx[i], S[i], A[i], n_vis(int(w.q_pos[t]), w.r), w.K)
    o_out = oracle.sparse_attn(problem(w), g_idx, rows=rows)
    check_attn(g_out[rows], o_out)


def test_config_attn_on_oracle_indices(cfg):
    name, w, rows, S, A = cfg
    o_idx = oracle.topk(problem(w), S, w.K, rows=rows)
    # every token needs valid indices; unsampled tokens take the GPU's own
    g_scores = run_scores(w)
    full = run_topk(w, g_scores, w.K)
    full[rows] = o_idx
    dp = binding.upload(w)
    ws = binding.new_workspace(dp)
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    binding.sa_sparse_attn(dp.ia, dp.aa, torch.from_numpy(full).cuda(), w.K, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    g = out.float().cpu().numpy().astype(np.float64)
    check_attn(g[rows], oracle.sparse_attn(problem(w), full, rows=rows))


@pytest.mark.parametrize("topk_blocks", [2048, 256])
def test_config_two_level_topk(cfg, topk_blocks):
    """Two-level top-k at full size on the indexer's own scores: level one
    (blocks of 8, as the pages' configuration) exact on every token, level two
    exact on the sampled tokens.  With 256 blocks the selection is active on
    every config; with 2048 it is on c4's longer rows."""
    from gpu_run import run_candidates, run_topk_candidates, unpack_blocks
    name, w, rows, S, A = cfg
    g = run_scores(w)
    bs = 8
    nb = (w.N_c + bs - 1) // bs
    cand = run_candidates(g, w.q_seq, w.q_pos, w.B, w.r, bs, topk_blocks)
    got = unpack_blocks(cand, nb)
    idx = run_topk_candidates(g, w.q_seq, w.q_pos, w.B, w.r, w.K, cand, bs)
    for t in range(w.T):
        nv = n_vis(int(w.q_pos[t]), w.r)
        keep = oracle.candidate_blocks_row(g[t].astype(np.float64), nv, bs, topk_blocks)
        assert np.array_equal(got[t], keep), (name, t)
        if t in rows:
            ref = oracle.candidate_topk_row(g[t].astype(np.float64), nv, w.K, keep, bs)
            assert idx[t].tolist() == ref.tolist(), (name, t)
