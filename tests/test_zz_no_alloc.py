"""sa_fused_decode_noalloc: the fused step for callers that cannot allocate
device memory (a plugin host that passes no workspace, a serving loop that
forbids allocation after start-up).  It must give the same results as
sa_fused_decode with a caller workspace, call after call, although every call
reuses the same library-owned scratch array.  This file is collected last so
that a run stopping at its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_run import ensure_built
from indexer_selected_sparse_score_gb300 import binding
from indexer_selected_sparse_score_gb300 import workloads as wl
from tolerances import check_attn

pytestmark = pytest.mark.gpu


def _outputs_close(g, ref):
    """g within the parity tests' attention tolerance of ref (two bf16 outputs)."""
    check_attn(g.float().cpu().numpy().astype(np.float64), ref.float().cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("name", ["c1", "c2", "c4"])
def test_noalloc_matches_workspace_path_twice(name):
    ensure_built()
    w = wl.generate(wl.CONFIGS[name])
    dp = binding.upload(w)
    ws = binding.new_workspace(dp)
    out_ref = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    idx_ref = torch.empty((w.T, w.K), dtype=torch.int32, device="cuda")
    binding.sa_fused_decode(dp.ia, dp.aa, w.K, idx_ref, out_ref, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK

    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((w.T, w.H, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        idx = torch.full((w.T, w.K), -7, dtype=torch.int32, device="cuda")
        binding.sa_fused_decode_noalloc(dp.ia, dp.aa, w.K, idx, out, status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, call
        assert torch.equal(idx, idx_ref), call          # integer work: identical
        _outputs_close(out, out_ref)                    # attention tolerance of the parity tests
    # without an index output the indices stay in the scratch; the output is unchanged
    out = torch.empty_like(out_ref)
    binding.sa_fused_decode_noalloc(dp.ia, dp.aa, w.K, None, out, None)
    torch.cuda.synchronize()
    _outputs_close(out, out_ref)
    if name == "c1":  # small enough to check every token against the oracle as well
        import oracle
        from helpers import n_vis, problem
        from tolerances import check_topk_sets
        S, A = oracle.index_scores(problem(w), with_magnitude=True)
        o_idx = oracle.topk(problem(w), S, w.K)
        g_idx = idx.cpu().numpy()
        for t in range(w.T):
            check_topk_sets(g_idx[t], o_idx[t], S[t], A[t], n_vis(int(w.q_pos[t]), w.r), w.K)
        check_attn(out.float().cpu().numpy().astype(np.float64), oracle.sparse_attn(problem(w), g_idx))


def test_noalloc_rejects_problems_beyond_its_scratch():
    ensure_built()
    lib = binding.load()
    s = wl.CONFIGS["c3"]  # 4096 tokens x 8192 scores alone exceed the fixed scratch
    ia = binding.IndexArgs(s.B, s.T, s.H_I, s.D_I, s.N_c, s.r, 256, 256, 256, s.q_dtype, 256, 256,
                           256, s.k_dtype, 256)
    aa = binding.AttnArgs(s.H, s.D, s.W, s.R, 256, 256, 256, 256, 256, None, 0.088)
    need = binding.sa_workspace_size(ia, aa, s.K)
    assert need > lib_scratch_bytes()
    st = lib.sa_fused_decode_noalloc(ctypes.byref(ia), ctypes.byref(aa), s.K, None, 256, None, None)
    assert st == binding.SA_ERR_UNSUPPORTED
    assert b"scratch" in lib.sa_last_error_detail()


def lib_scratch_bytes():
    return binding.sa_noalloc_scratch_bytes()


def test_scratch_size_matches_the_header():
    """The compiled size equals SA_NOALLOC_SCRATCH_BYTES as include/sa.h states it."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "sa.h")).read()
    m = re.search(r"#define SA_NOALLOC_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", hdr)
    assert m, "SA_NOALLOC_SCRATCH_BYTES not found in include/sa.h"
    ensure_built()
    assert lib_scratch_bytes() == int(m.group(1)) << int(m.group(2))
