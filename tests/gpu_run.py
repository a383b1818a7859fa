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


def _token_args(B: int, N_c: int, r: int, q_seq: np.ndarray, q_pos: np.ndarray):
    """IndexArgs carrying only the token arrays (all the top-k entry points
    read), plus the device tensors that must outlive the call."""
    d_seq = torch.from_numpy(np.ascontiguousarray(q_seq, dtype=np.int32)).cuda()
    d_pos = torch.from_numpy(np.ascontiguousarray(q_pos, dtype=np.int32)).cuda()
    ia = binding.IndexArgs(B, len(q_seq), 16, 64, N_c, r, d_seq.data_ptr(), d_pos.data_ptr(), None, 0, None,
                           None, None, 0, None)
    return ia, (d_seq, d_pos)


def _small_ws() -> torch.Tensor:
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    return ws


def run_candidates(scores: np.ndarray, q_seq, q_pos, B: int, r: int, block_size: int, topk_blocks: int):
    """Level one on the GPU: the [T, words] uint32 block mask."""
    ensure_built()
    T, N_c = scores.shape
    ia, keep = _token_args(B, N_c, r, q_seq, q_pos)
    ws = _small_ws()
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    words = binding.sa_candidate_words(N_c, block_size)
    cand = torch.full((T, words), -1, dtype=torch.int32, device="cuda")  # every bit set beforehand
    binding.sa_candidate_blocks(s, ia, block_size, topk_blocks, cand, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    del keep
    return cand.cpu().numpy().view(np.uint32)


def run_topk_rows(scores: np.ndarray, q_seq, q_pos, B: int, r: int, K: int):
    """sa_topk on given score rows and token arrays alone: [T, K] indices."""
    ensure_built()
    T, N_c = scores.shape
    ia, keep = _token_args(B, N_c, r, q_seq, q_pos)
    ws = _small_ws()
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    idx = torch.full((T, max(K, 1)), -7, dtype=torch.int32, device="cuda")
    binding.sa_topk(s, ia, K, idx, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    del keep
    return idx[:, :K].cpu().numpy()


def run_topk_candidates(scores: np.ndarray, q_seq, q_pos, B: int, r: int, K: int, cand: np.ndarray,
                        block_size: int):
    """Level two on the GPU: [T, K] indices."""
    ensure_built()
    T, N_c = scores.shape
    ia, keep = _token_args(B, N_c, r, q_seq, q_pos)
    ws = _small_ws()
    s = torch.from_numpy(np.ascontiguousarray(scores, dtype=np.float32)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(cand).view(np.int32)).cuda()
    idx = torch.full((T, max(K, 1)), -7, dtype=torch.int32, device="cuda")
    binding.sa_topk_candidates(s, ia, K, c, block_size, idx, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    del keep
    return idx[:, :K].cpu().numpy()


def unpack_blocks(cand: np.ndarray, nb: int) -> np.ndarray:
    """[T, words] uint32 block masks -> [T, nb] bool; bits past nb must be 0."""
    bits = np.unpackbits(np.ascontiguousarray(cand).view(np.uint8), axis=1, bitorder="little")
    assert not bits[:, nb:].any(), "bits past the last block are set"
    return bits[:, :nb].astype(bool)


def pack_blocks(keep: np.ndarray) -> np.ndarray:
    """[T, nb] bool -> [T, ceil(nb / 32)] uint32 (bit b % 32 of word b / 32)."""
    T, nb = keep.shape
    words = (nb + 31) // 32
    padded = np.zeros((T, words * 32), dtype=np.uint8)
    padded[:, :nb] = keep
    return np.packbits(padded, axis=1, bitorder="little").view(np.uint32)
