"""The released V4.1 attention shape on the GPU against the oracle
("DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Attention.forward, with the
released config of the atlas page "DeepSeek V4.1 ... compressed-kv": 64 query
heads of dim 512, one kv tensor serving as K and V, the attention sink,
index 32 x 128, window 128, ratio 2).  Also 32 and 16 heads (the shapes one
rank holds under 2- and 4-way head parallelism) and separate K and V."""
import numpy as np
import pytest

import oracle
from gpu_run import run_attn, run_fused
from helpers import n_vis, problem
from indexer_selected_sparse_score_gb300 import binding
from indexer_selected_sparse_score_gb300 import workloads as wl
from tolerances import check_attn, check_topk_sets

pytestmark = pytest.mark.gpu


def v41(name, H=64, same=True, **kw):
    base = dict(B=4, T=4, H_I=32, D_I=128, r=2, N_c=700, K=96, H=H, D=512, W=128, R=128, sink=True,
                pos_lo=300, pos_hi=1399, w_div=32.0)
    base.update(kw)
    return wl.small(name, **base), same


CASES = {
    "h64_kv_sink": v41("h64_kv_sink"),                              # the released shape (K scaled down)
    "h32_kv": v41("h32_kv", H=32, sink=False),
    "h16_kv": v41("h16_kv", H=16),
    "h64_sep": v41("h64_sep", same=False),                          # separate K and V: 16-key tiles
    "h16_sep": v41("h16_sep", H=16, same=False, sink=False),
    # ring still filling, n_vis below K, one split per token (many tokens)
    "h64_kv_early": v41("h64_kv_early", B=40, T=40, N_c=200, K=64, pos_lo=0, pos_hi=399),
    "h64_kv_many": v41("h64_kv_many", B=320, T=320, N_c=200, K=64, pos_lo=200, pos_hi=399),
}


def share_kv(w, dp=None):
    """K and V as one tensor: the same host arrays and the same device pointers."""
    w.Vw, w.Vc = w.Kw, w.Kc
    if dp is not None:
        dp.tensors["Vw"], dp.tensors["Vc"] = dp.tensors["Kw"], dp.tensors["Kc"]
        dp.aa.Vw, dp.aa.Vc = dp.aa.Kw, dp.aa.Kc
    return dp


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    spec, same = CASES[request.param]
    w = wl.generate(spec, seed=500 + sorted(CASES).index(request.param))
    if same:
        share_kv(w)
    S, A = oracle.index_scores(problem(w), with_magnitude=True)
    return request.param, w, same, S, A


def test_attn_dim512_on_oracle_indices(case):
    """sa_sparse_attn on the oracle's indices (run_attn uploads K and V as two device
    copies, so this runs the separate-K/V kernel; the fused test shares the pointers)."""
    name, w, same, S, A = case
    o_idx = oracle.topk(problem(w), S, w.K)
    g = run_attn(w, o_idx)
    check_attn(g, oracle.sparse_attn(problem(w), o_idx))


def test_fused_dim512(case):
    name, w, same, S, A = case
    dp = binding.upload(w)
    if same:
        share_kv(w, dp)
    g_idx, g_out = run_fused(w, dp=dp)
    o_idx = oracle.topk(problem(w), S, w.K)
    for t in range(w.T):
        check_topk_sets(g_idx[t], o_idx[t], S[t], A[t], n_vis(int(w.q_pos[t]), w.r), w.K)
    check_attn(g_out, oracle.sparse_attn(problem(w), g_idx))


def test_attn_dim512_one_kv_on_oracle_indices(case):
    """sa_sparse_attn on the oracle's indices with K and V as one device tensor:
    at 64 heads this is the tensor-core (tcgen05) kernel of the released shape."""
    import torch
    name, w, same, S, A = case
    if not same:
        pytest.skip("K and V are separate tensors in this case")
    o_idx = oracle.topk(problem(w), S, w.K)
    dp = share_kv(w, binding.upload(w))
    ws = binding.new_workspace(dp)
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    binding.sa_sparse_attn(dp.ia, dp.aa, torch.from_numpy(o_idx).cuda(), w.K, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    check_attn(out.float().cpu().numpy().astype(np.float64), oracle.sparse_attn(problem(w), o_idx))
