"""ctypes binding of libsa.so (include/sa.h), with the same entry-point names.

Argument marshalling only: every step of the computation runs in the CUDA
library.  Tensors are passed as raw device pointers (``tensor.data_ptr()``)
and streams as ``torch.cuda.Stream.cuda_stream`` handles; torch provides device
memory and streams, nothing else.  If libsa.so is missing the first call
raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from .build import LIB

SA_OK = 0
SA_ERR_INVALID_ARG = 1
SA_ERR_UNSUPPORTED = 2
SA_ERR_WORKSPACE = 3
SA_ERR_CUDA = 4
SA_ERR_TIMEOUT = 5
SA_ERR_DEVICE_DATA = 6

SA_BF16 = 0
SA_FP8_E4M3 = 1


class SAError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"sa status {status}: {detail}")
        self.status = status
        self.detail = detail


class IndexArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H_I", ctypes.c_int32), ("D_I", ctypes.c_int32),
        ("N_c", ctypes.c_int32), ("r", ctypes.c_int32),
        ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
        ("q_I", ctypes.c_void_p), ("q_dtype", ctypes.c_int32), ("q_scale", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("k_I", ctypes.c_void_p), ("k_dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p),
        ("k_seq_stride", ctypes.c_int64),
    ]


class AttnArgs(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("W", ctypes.c_int32), ("R", ctypes.c_int32),
        ("Q", ctypes.c_void_p), ("Kw", ctypes.c_void_p), ("Vw", ctypes.c_void_p),
        ("Kc", ctypes.c_void_p), ("Vc", ctypes.c_void_p),
        ("sink", ctypes.c_void_p), ("scale", ctypes.c_float),
        ("w_seq_stride", ctypes.c_int64), ("c_seq_stride", ctypes.c_int64),
    ]


class RopeArgs(ctypes.Structure):
    _fields_ = [
        ("dim", ctypes.c_int32), ("base", ctypes.c_double), ("factor", ctypes.c_double),
        ("original_seq_len", ctypes.c_int32), ("beta_fast", ctypes.c_double), ("beta_slow", ctypes.c_double),
    ]


EXPORTED = ("sa_workspace_size", "sa_workspace_init", "sa_indexer_scores", "sa_topk",
            "sa_candidate_blocks", "sa_candidate_words", "sa_topk_candidates", "sa_rotate_quant",
            "sa_compress_prefill", "sa_compress_decode", "sa_index_key_publish",
            "sa_sparse_attn", "sa_fused_decode", "sa_fused_decode_staged",
            "sa_fused_decode_launch_count", "sa_check_device_status", "sa_status_string",
            "sa_last_error_detail", "sa_fused_decode_noalloc", "sa_noalloc_scratch_bytes", "sa_set_wait_budget")

_LIB = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libsa.so (built by ``build.build()``); raises if it is absent."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run indexer_selected_sparse_score_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    IA, AA = ctypes.POINTER(IndexArgs), ctypes.POINTER(AttnArgs)
    lib.sa_workspace_size.argtypes = [IA, AA, i32]
    lib.sa_workspace_size.restype = sz
    lib.sa_workspace_init.argtypes = [vp, sz, vp]
    i64 = ctypes.c_int64
    lib.sa_indexer_scores.argtypes = [IA, vp, i64, vp, sz, vp]
    lib.sa_topk.argtypes = [vp, i64, IA, i32, vp, vp, sz, vp]
    lib.sa_candidate_blocks.argtypes = [vp, i64, IA, i32, i32, vp, vp, sz, vp]
    lib.sa_candidate_words.argtypes = [i32, i32]
    lib.sa_candidate_words.restype = i32
    lib.sa_topk_candidates.argtypes = [vp, i64, IA, i32, vp, i32, vp, vp, sz, vp]
    lib.sa_rotate_quant.argtypes = [vp, i32, i32, vp, ctypes.c_int64, vp, vp, vp, sz, vp]
    lib.sa_compress_prefill.argtypes = [vp, vp, i32, i32, i32, i32, vp, ctypes.c_float, vp, vp, vp, vp]
    lib.sa_compress_decode.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp, ctypes.c_float, vp, vp, sz, vp]
    lib.sa_index_key_publish.argtypes = [vp, i32, i32, vp, vp, i32, vp, ctypes.c_float, ctypes.POINTER(RopeArgs),
                                         vp, vp, i32, i32, i64, vp, sz, vp]
    lib.sa_sparse_attn.argtypes = [IA, AA, vp, i32, vp, vp, sz, vp]
    lib.sa_fused_decode.argtypes = [IA, AA, i32, vp, vp, vp, sz, vp]
    lib.sa_fused_decode_staged.argtypes = [IA, AA, i32, vp, vp, vp, sz, vp, ctypes.POINTER(vp)]
    lib.sa_fused_decode_launch_count.argtypes = [IA, AA, i32]
    lib.sa_fused_decode_launch_count.restype = i32
    lib.sa_fused_decode_noalloc.argtypes = [IA, AA, i32, vp, vp, vp, vp]
    lib.sa_fused_decode_noalloc.restype = i32
    lib.sa_noalloc_scratch_bytes.argtypes = []
    lib.sa_noalloc_scratch_bytes.restype = sz
    lib.sa_check_device_status.argtypes = [vp, vp]
    lib.sa_set_wait_budget.argtypes = [i64]
    lib.sa_set_wait_budget.restype = i32
    lib.sa_status_string.argtypes = [i32]
    lib.sa_status_string.restype = ctypes.c_char_p
    lib.sa_last_error_detail.restype = ctypes.c_char_p
    for name in ("sa_workspace_init", "sa_indexer_scores", "sa_topk", "sa_candidate_blocks",
                 "sa_topk_candidates", "sa_rotate_quant", "sa_compress_prefill", "sa_compress_decode",
                 "sa_index_key_publish", "sa_sparse_attn",
                 "sa_fused_decode", "sa_fused_decode_staged", "sa_check_device_status"):
        getattr(lib, name).restype = i32
    if path == LIB:
        _LIB = lib
    return lib


def _p(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int) -> None:
    if status != SA_OK:
        raise SAError(status, load().sa_last_error_detail().decode())


def _ws(ws):
    return _p(ws), (ws.numel() * ws.element_size() if ws is not None else 0)


# ----------------------------------------------------------- entry points ---

def sa_workspace_size(ia: IndexArgs, aa: Optional[AttnArgs], K: int) -> int:
    return int(load().sa_workspace_size(ctypes.byref(ia), ctypes.byref(aa) if aa is not None else None, K))


def sa_workspace_init(ws, stream=None) -> None:
    p, n = _ws(ws)
    _check(load().sa_workspace_init(p, n, _s(stream)))


def _ld(scores, ld, ia) -> int:
    """Row stride of a score matrix: as given, else that of a 2-D tensor, else N_c."""
    if ld is not None:
        return int(ld)
    if isinstance(scores, torch.Tensor) and scores.dim() == 2:
        return int(scores.stride(0))
    return int(ia.N_c)


def sa_indexer_scores(ia: IndexArgs, scores, ws, stream=None, ld=None) -> None:
    p, n = _ws(ws)
    _check(load().sa_indexer_scores(ctypes.byref(ia), _p(scores), _ld(scores, ld, ia), p, n, _s(stream)))


def sa_topk(scores, ia: IndexArgs, K: int, idx, ws, stream=None, ld=None) -> None:
    p, n = _ws(ws)
    _check(load().sa_topk(_p(scores), _ld(scores, ld, ia), ctypes.byref(ia), K, _p(idx), p, n, _s(stream)))


def sa_candidate_words(N_c: int, block_size: int) -> int:
    return int(load().sa_candidate_words(N_c, block_size))


def sa_candidate_blocks(scores, ia: IndexArgs, block_size: int, topk_blocks: int, cand, ws,
                        stream=None, ld=None) -> None:
    """Level one of the two-level top-k: ``cand`` ([T, sa_candidate_words] int32
    or uint32) receives one bit per kept block."""
    p, n = _ws(ws)
    _check(load().sa_candidate_blocks(_p(scores), _ld(scores, ld, ia), ctypes.byref(ia), block_size, topk_blocks,
                                      _p(cand), p, n, _s(stream)))


def sa_topk_candidates(scores, ia: IndexArgs, K: int, cand, block_size: int, idx, ws, stream=None,
                       ld=None) -> None:
    """Level two: sa_topk with the scores outside the kept blocks of ``cand`` at -inf."""
    p, n = _ws(ws)
    _check(load().sa_topk_candidates(_p(scores), _ld(scores, ld, ia), ctypes.byref(ia), K, _p(cand), block_size,
                                     _p(idx), p, n, _s(stream)))


def sa_rotate_quant(x, rows: int, codes, scales, ws, dst=None, dst_rows: int = 0, dim: int = 128,
                    stream=None) -> None:
    """V3.2 index producer: Hadamard rotation and e4m3 block quantisation of
    ``rows`` rows of 128 bf16 values; row r lands at row ``dst[r]`` when given."""
    p, n = _ws(ws)
    _check(load().sa_rotate_quant(_p(x), rows, dim, _p(dst), dst_rows, _p(codes), _p(scales), p, n, _s(stream)))


def sa_compress_prefill(kv, score, B: int, S: int, D: int, r: int, weight, eps: float, out, stream=None,
                        kv_state=None, score_state=None) -> None:
    """V4.1 compressor from position 0: [B, S // r, D] bf16 pooled, normalised
    rows; the trailing S % r tokens go to the states when given."""
    _check(load().sa_compress_prefill(_p(kv), _p(score), B, S, D, r, _p(weight), eps, _p(out), _p(kv_state),
                                      _p(score_state), _s(stream)))


def sa_compress_decode(kv, score, pos, B: int, D: int, r: int, kv_state, score_state, weight, eps: float, out, ws,
                       stream=None) -> None:
    """One V4.1 compressor decode step: row b of ``out`` is written when the
    group of sequence b completes at position pos[b]."""
    p, n = _ws(ws)
    _check(load().sa_compress_decode(_p(kv), _p(score), _p(pos), B, D, r, _p(kv_state), _p(score_state), _p(weight),
                                     eps, _p(out), p, n, _s(stream)))


def sa_index_key_publish(kproj, n: int, seq, grp, r: int, weight, eps: float, rope: "RopeArgs", k_I, k_scale,
                         B: int, N_rows: int, ws, k_seq_stride: int = 0, D_I: int = 128, stream=None) -> None:
    """V4.1 index keys: k_norm, rotary embedding at the group start, e4m3 codes
    and a scale per position, written into the key cache."""
    p, nb = _ws(ws)
    _check(load().sa_index_key_publish(_p(kproj), n, D_I, _p(seq), _p(grp), r, _p(weight), eps, ctypes.byref(rope),
                                       _p(k_I), _p(k_scale), B, N_rows, k_seq_stride, p, nb, _s(stream)))


def sa_sparse_attn(ia: IndexArgs, aa: AttnArgs, idx, K: int, out, ws, stream=None) -> None:
    p, n = _ws(ws)
    _check(load().sa_sparse_attn(ctypes.byref(ia), ctypes.byref(aa), _p(idx), K, _p(out), p, n, _s(stream)))


def sa_fused_decode(ia: IndexArgs, aa: AttnArgs, K: int, idx_out, out, ws, stream=None) -> None:
    p, n = _ws(ws)
    _check(load().sa_fused_decode(ctypes.byref(ia), ctypes.byref(aa), K, _p(idx_out), _p(out), p, n,
                                  _s(stream)))


def sa_fused_decode_staged(ia: IndexArgs, aa: AttnArgs, K: int, idx_out, out, ws, events,
                           stream=None) -> None:
    """``events``: four raw cudaEvent_t handles (ints) recorded between stages."""
    p, n = _ws(ws)
    arr = (ctypes.c_void_p * 4)(*events)
    _check(load().sa_fused_decode_staged(ctypes.byref(ia), ctypes.byref(aa), K, _p(idx_out), _p(out),
                                         p, n, _s(stream), arr))


def sa_fused_decode_launch_count(ia: IndexArgs, aa: AttnArgs, K: int) -> int:
    return int(load().sa_fused_decode_launch_count(ctypes.byref(ia), ctypes.byref(aa), K))


def sa_fused_decode_noalloc(ia: IndexArgs, aa: AttnArgs, K: int, idx_out, out, device_status=None,
                            stream=None) -> None:
    """The fused step on the library's fixed device scratch (no workspace, no
    allocation); see include/sa.h for its size limit and sharing rules."""
    _check(load().sa_fused_decode_noalloc(ctypes.byref(ia), ctypes.byref(aa), K, _p(idx_out), _p(out),
                                          _p(device_status), _s(stream)))


def sa_noalloc_scratch_bytes() -> int:
    """Bytes of the fixed scratch behind sa_fused_decode_noalloc."""
    return int(load().sa_noalloc_scratch_bytes())


def sa_check_device_status(ws, stream=None) -> int:
    """Synchronise, read and clear the sticky device status; returns the sa status."""
    return int(load().sa_check_device_status(_p(ws), _s(stream)))


def sa_set_wait_budget(cycles: int) -> None:
    """Bound (SM cycles, 0 = default) on each pipeline wait of the tensor-core attention kernels."""
    _check(load().sa_set_wait_budget(int(cycles)))


# ------------------------------------------------------ device marshalling ---

def _dev(a: Optional[np.ndarray], device) -> Optional[torch.Tensor]:
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


@dataclass
class DeviceProblem:
    """Device copies of a workload's arrays plus the C argument structs."""
    tensors: dict
    ia: IndexArgs
    aa: AttnArgs
    K: int
    T: int
    H: int
    D: int


def _padded(a: Optional[np.ndarray], rows: int, device, fill: int = 0x55):
    """[B, n, ...] host array into a device tensor of [B, rows, ...] (rows >= n),
    the extra rows filled with a byte pattern; returns (tensor, view of the used rows)."""
    if a is None:
        return None, None
    src = torch.from_numpy(np.ascontiguousarray(a))
    full = torch.empty((a.shape[0], rows) + tuple(a.shape[2:]), dtype=src.dtype, device=device)
    full.view(torch.uint8).fill_(fill)
    full[:, :a.shape[1]].copy_(src.to(device))
    return full, full[:, :a.shape[1]]


def upload(w, device="cuda", K: Optional[int] = None, pad: Optional[dict] = None) -> DeviceProblem:
    """Copy a workload (host numpy arrays in storage formats) to the device.

    ``pad`` places caches in larger allocations, as a model keeps them:
    {"k": rows, "w": rows, "c": rows} allocates that many rows per sequence for
    the index keys (and their scales), the raw ring and the compressed cache,
    and passes the matching sequence strides."""
    pad = pad or {}
    names = ("q_seq", "q_pos", "q_I", "q_scale", "w", "Q", "sink")
    t = {n: _dev(getattr(w, n), device) for n in names}
    kr, wr, cr = pad.get("k", w.N_c), pad.get("w", w.R), pad.get("c", w.N_c)
    t["k_I"], _ = _padded(w.k_I, kr, device)
    t["k_scale"], _ = _padded(w.k_scale, kr, device)
    for n in ("Kw", "Vw"):
        t[n], _ = _padded(getattr(w, n), wr, device)
    for n in ("Kc", "Vc"):
        t[n], _ = _padded(getattr(w, n), cr, device)
    ia = IndexArgs(w.B, w.T, w.H_I, w.D_I, w.N_c, w.r, _p(t["q_seq"]), _p(t["q_pos"]),
                   _p(t["q_I"]), w.q_dtype, _p(t["q_scale"]), _p(t["w"]),
                   _p(t["k_I"]), w.k_dtype, _p(t["k_scale"]), kr * w.D_I if "k" in pad else 0)
    aa = AttnArgs(w.H, w.D, w.W, w.R, _p(t["Q"]), _p(t["Kw"]), _p(t["Vw"]), _p(t["Kc"]), _p(t["Vc"]),
                  _p(t["sink"]), float(w.scale), wr * w.D if "w" in pad else 0, cr * w.D if "c" in pad else 0)
    return DeviceProblem(t, ia, aa, w.K if K is None else K, w.T, w.H, w.D)


def new_workspace(dp: DeviceProblem, device="cuda", stream=None) -> torch.Tensor:
    n = sa_workspace_size(dp.ia, dp.aa, dp.K)
    if n == 0:
        raise SAError(SA_ERR_INVALID_ARG, "workspace size query rejected the arguments")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    sa_workspace_init(ws, stream)
    return ws
