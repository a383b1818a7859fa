"""Runs the CUDA library through its C ABI on host workloads (GPU tests only)."""
import functools

import numpy as np
import torch

from indexer_selected_sparse_score_gb300 import binding, build
from indexer_selected_sparse_score_gb300 import workloads as wl


@functools.lru_cache(maxsize=1)
def ensure_built() -> str:
    path = build.build()
    binding.load()
    return path


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def run_scores(w, K=None):
    ensure_built()
    dp = binding.upload(w, K=K)
    ws = binding.new_workspace(dp)
    scores = torch.empty((w.T, w.N_c), dtype=torch.float32, device="cuda")
    binding.sa_indexer_scores(dp.ia, scores, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    return scores.cpu().numpy()


def run_topk(w, scores: np.ndarray, K: int):
    ensure_built()
    dp = binding.upload(w, K=K)
    ws = binding.new_workspace(dp)
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    idx = torch.full((w.T, max(K, 1)), -7, dtype=torch.int32, device="cuda")
    binding.sa_topk(s, dp.ia, K, idx, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    return idx[:, :K].cpu().numpy()


def run_attn(w, idx: np.ndarray, expect_status=binding.SA_OK):
    ensure_built()
    K = idx.shape[1]
    dp = binding.upload(w, K=K)
    ws = binding.new_workspace(dp)
    d_idx = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    binding.sa_sparse_attn(dp.ia, dp.aa, d_idx if K > 0 else None, K, out, ws)
    assert binding.sa_check_device_status(ws) == expect_status
    return bf16_tensor_to_f64(out)


def run_fused(w, K=None, with_idx=True, dp=None):
    ensure_built()
    K = w.K if K is None else K
    dp = dp or binding.upload(w, K=K)
    ws = binding.new_workspace(dp)
    out = torch.empty((w.T, w.H, w.D), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((w.T, max(K, 1)), -7, dtype=torch.int32, device="cuda") if with_idx else None
    binding.sa_fused_decode(dp.ia, dp.aa, K, idx, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    return (idx[:, :K].cpu().numpy() if with_idx else None), bf16_tensor_to_f64(out)


@functools.lru_cache(maxsize=2)
def config_workload(name: str):
    return wl.generate(wl.CONFIGS[name])
