"""The timeout path of the tensor-core attention kernels (GPU only).

sa_set_wait_budget cuts the bound on every wait between a kernel's own stages
to a few dozen SM cycles, which no copy from HBM meets: each launch gives up,
sets the timeout flag of the status word, waits for the copies and products it
already started (those waits keep the full bound) and returns.  The test reads
SA_ERR_TIMEOUT from the status word, restores the default bound, and checks in
the same CUDA context that the attention and the whole decode step then match
the oracle: nothing was left running, hung or corrupted.  Covered: heads of dim
128 split over 2-CTA clusters (config c2's shape) and heads of dim 512 over one
kv tensor, split (4 tokens) and whole tokens (320 tokens).
"""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_run import config_workload, ensure_built
from helpers import problem
from indexer_selected_sparse_score_gb300 import binding
from indexer_selected_sparse_score_gb300 import workloads as wl
from tolerances import check_attn

pytestmark = pytest.mark.gpu

TINY_BUDGET = 64  # SM cycles: far below one HBM round trip


def v41(name, **kw):
    base = dict(B=4, T=4, H_I=32, D_I=128, r=2, N_c=700, K=96, H=64, D=512, W=128, R=128, sink=True,
                pos_lo=300, pos_hi=1399, w_div=32.0)
    base.update(kw)
    return wl.generate(wl.small(name, **base), seed=77)


CASES = {
    "d128_split": lambda: config_workload("c2"),
    "d512_split": lambda: v41("d512_split"),
    "d512_whole": lambda: v41("d512_whole", B=320, T=320, N_c=200, K=64, pos_lo=200, pos_hi=399),
}


def share_kv(w, dp):
    w.Vw, w.Vc = w.Kw, w.Kc
    dp.tensors["Vw"], dp.tensors["Vc"] = dp.tensors["Kw"], dp.tensors["Kc"]
    dp.aa.Vw, dp.aa.Vc = dp.aa.Kw, dp.aa.Kc


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    ensure_built()
    w = CASES[request.param]()
    dp = binding.upload(w)
    if w.D == 512:
        share_kv(w, dp)
    return request.param, w, dp


def test_wait_budget_rejects_negative():
    ensure_built()
    with pytest.raises(binding.SAError):
        binding.sa_set_wait_budget(-1)
    binding.sa_set_wait_budget(0)


def test_timeout_flags_and_context_recovers(case):
    name, w, dp = case
    ws = binding.new_workspace(dp)
    rows = [0, w.T // 2, w.T - 1]
    # valid indices for every token, from a first step at the default bound
    idx = torch.empty((w.T, w.K), dtype=torch.int32, device="cuda")
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    binding.sa_fused_decode(dp.ia, dp.aa, w.K, idx, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    g_idx = idx.cpu().numpy()
    o = oracle.sparse_attn(problem(w), g_idx, rows=rows)
    check_attn(out.float().cpu().numpy().astype(np.float64)[rows], o)
    # every launch gives up at the tiny bound and says so
    binding.sa_set_wait_budget(TINY_BUDGET)
    try:
        t0 = time.perf_counter()
        binding.sa_sparse_attn(dp.ia, dp.aa, idx, w.K, out, ws)
        st = binding.sa_check_device_status(ws)
        elapsed = time.perf_counter() - t0
    finally:
        binding.sa_set_wait_budget(0)
    assert st == binding.SA_ERR_TIMEOUT, (name, st)
    # the drains (copies and products already started) keep the full bound of
    # about a second: a launch that gives up promptly never ran one out
    assert elapsed < 0.5, (name, elapsed)
    # the same context at the default bound: the attention and the whole step are right again
    out.zero_()
    binding.sa_sparse_attn(dp.ia, dp.aa, idx, w.K, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    check_attn(out.float().cpu().numpy().astype(np.float64)[rows], o)
    idx2 = torch.empty_like(idx)
    out2 = torch.empty_like(out)
    binding.sa_fused_decode(dp.ia, dp.aa, w.K, idx2, out2, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    assert torch.equal(idx2, idx) and torch.equal(out2, out)
