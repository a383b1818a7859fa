"""Float64 CPU oracle for the indexer-selected sparse attention step.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers; the product package
never imports this module.  The arithmetic lives in ``oracle.c`` (plain C,
IEEE double); this file compiles it with gcc and marshals numpy arrays.

Pages followed (title, section): "DeepSeek-V4.1-Flash-NVFP4 inference/model.py"
(Indexer.forward, get_window_topk_idxs, Attention._window_kv,
Attention.forward, select_candidate_blocks, Compressor.forward, RMSNorm.forward)
and "DeepSeek-V3.2-Exp inference/model.py" (Indexer.forward with fp8 keys and
per-position scales; rotate_activation and act_quant).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SRC = os.path.join(_HERE, "oracle.c")

BF16 = 0
FP8_E4M3 = 1


def build(mutant: int = 0, out_dir: Optional[str] = None) -> str:
    """Compile oracle.c into a shared library and return its path.

    ``mutant`` > 0 compiles one of the deliberately wrong variants used by the
    pin tests (``-DORC_MUTANT=n``) into ``out_dir``.
    """
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so"
    out = os.path.join(out_dir, name)
    if os.path.exists(out) and os.path.getmtime(out) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", f"-DORC_MUTANT={mutant}", "-o", out + ".tmp", _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("T", ctypes.c_int32), ("r", ctypes.c_int32), ("N_c", ctypes.c_int32),
        ("q_seq", ctypes.c_void_p), ("q_pos", ctypes.c_void_p),
        ("H_I", ctypes.c_int32), ("D_I", ctypes.c_int32),
        ("q_I", ctypes.c_void_p), ("q_dtype", ctypes.c_int32), ("q_scale", ctypes.c_void_p),
        ("w", ctypes.c_void_p),
        ("k_I", ctypes.c_void_p), ("k_dtype", ctypes.c_int32), ("k_scale", ctypes.c_void_p),
        ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("W", ctypes.c_int32), ("R", ctypes.c_int32),
        ("Q", ctypes.c_void_p), ("Kw", ctypes.c_void_p), ("Vw", ctypes.c_void_p),
        ("Kc", ctypes.c_void_p), ("Vc", ctypes.c_void_p),
        ("sink", ctypes.c_void_p), ("scale", ctypes.c_float),
    ]


_LIBS: dict = {}


def _lib(mutant: int = 0, path: Optional[str] = None):
    key = path or mutant
    if key not in _LIBS:
        lib = ctypes.CDLL(path or build(mutant))
        P = ctypes.POINTER(_Problem)
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_value.restype = ctypes.c_double
        lib.orc_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_value.restype = ctypes.c_double
        lib.orc_n_vis.argtypes = [i32, i32]
        lib.orc_n_vis.restype = i32
        lib.orc_window_slots.argtypes = [i32, i32, i32, vp]
        lib.orc_window_slots.restype = i32
        lib.orc_index_scores.argtypes = [P, vp, i32, vp, vp]
        lib.orc_index_scores.restype = i32
        lib.orc_topk_row.argtypes = [vp, i32, i32, vp]
        lib.orc_topk_row.restype = i32
        lib.orc_candidate_blocks.argtypes = [vp, i32, i32, i32, i32, vp]
        lib.orc_hadamard_bf16.argtypes = [vp, i32, vp]
        lib.orc_hadamard_bf16.restype = i32
        lib.orc_hadamard_f64.argtypes = [vp, i32, vp]
        lib.orc_hadamard_f64.restype = i32
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_act_quant_row.argtypes = [vp, i32, vp, vp]
        lib.orc_act_quant_row.restype = i32
        lib.orc_compress_prefill.argtypes = [vp, vp, i32, i32, i32, vp, ctypes.c_double, vp, vp, vp]
        lib.orc_compress_prefill.restype = i32
        lib.orc_compress_decode.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, ctypes.c_double, vp]
        lib.orc_compress_decode.restype = i32
        lib.orc_rope_angle.argtypes = [i32, i32, ctypes.c_int64, ctypes.c_double, ctypes.c_double, i32,
                                       ctypes.c_double, ctypes.c_double]
        lib.orc_rope_angle.restype = ctypes.c_double
        lib.orc_apply_rope.argtypes = [vp, i32, ctypes.c_int64, ctypes.c_double, ctypes.c_double, i32,
                                       ctypes.c_double, ctypes.c_double, i32]
        lib.orc_candidate_blocks.restype = i32
        lib.orc_index_key.argtypes = [vp, i32, vp, ctypes.c_double, ctypes.c_int64, i32, ctypes.c_double,
                                      ctypes.c_double, i32, ctypes.c_double, ctypes.c_double, vp, vp, vp]
        lib.orc_index_key.restype = i32
        lib.orc_sparse_attn.argtypes = [P, vp, i32, vp, i32, vp]
        lib.orc_sparse_attn.restype = i32
        lib.orc_fused.argtypes = [P, i32, vp, i32, vp, vp]
        lib.orc_fused.restype = i32
        lib.orc_set_threads.argtypes = [i32]
        lib.orc_get_threads.restype = i32
        _LIBS[key] = lib
    return _LIBS[key]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


@dataclass
class Problem:
    """Host arrays of one problem, in the library's storage formats.

    bf16 arrays are uint16 bit patterns, fp8-e4m3fn arrays are uint8 bit
    patterns; scales and weights are float32; q_seq/q_pos are int32.
    """
    B: int
    T: int
    r: int
    N_c: int
    q_seq: np.ndarray
    q_pos: np.ndarray
    H_I: int
    D_I: int
    q_I: np.ndarray
    q_dtype: int
    q_scale: Optional[np.ndarray]
    w: np.ndarray
    k_I: np.ndarray
    k_dtype: int
    k_scale: Optional[np.ndarray]
    H: int
    D: int
    W: int
    R: int
    Q: np.ndarray
    Kw: np.ndarray
    Vw: np.ndarray
    Kc: np.ndarray
    Vc: np.ndarray
    sink: Optional[np.ndarray]
    scale: float

    def _struct(self) -> _Problem:
        def c(a, dt):
            if a is None:
                return None
            assert a.dtype == dt and a.flags.c_contiguous, (a.dtype, dt)
            return a

        qd = np.uint16 if self.q_dtype == BF16 else np.uint8
        kd = np.uint16 if self.k_dtype == BF16 else np.uint8
        self._keep = [c(self.q_seq, np.int32), c(self.q_pos, np.int32), c(self.q_I, qd),
                      c(self.q_scale, np.float32), c(self.w, np.float32), c(self.k_I, kd),
                      c(self.k_scale, np.float32), c(self.Q, np.uint16), c(self.Kw, np.uint16),
                      c(self.Vw, np.uint16), c(self.Kc, np.uint16), c(self.Vc, np.uint16),
                      c(self.sink, np.float32)]
        return _Problem(self.B, self.T, self.r, self.N_c, _ptr(self.q_seq), _ptr(self.q_pos),
                        self.H_I, self.D_I, _ptr(self.q_I), self.q_dtype, _ptr(self.q_scale),
                        _ptr(self.w), _ptr(self.k_I), self.k_dtype, _ptr(self.k_scale),
                        self.H, self.D, self.W, self.R, _ptr(self.Q), _ptr(self.Kw), _ptr(self.Vw),
                        _ptr(self.Kc), _ptr(self.Vc), _ptr(self.sink), float(self.scale))


def _rows(rows: Optional[Sequence[int]], T: int) -> np.ndarray:
    if rows is None:
        rows = range(T)
    return np.ascontiguousarray(np.asarray(list(rows), dtype=np.int32))


def bf16_value(bits: int, mutant: int = 0) -> float:
    return _lib(mutant).orc_bf16_value(bits)


def e4m3_value(bits: int, mutant: int = 0) -> float:
    return _lib(mutant).orc_e4m3_value(bits)


def n_vis(pos: int, r: int, mutant: int = 0) -> int:
    return _lib(mutant).orc_n_vis(pos, r)


def window_slots(pos: int, W: int, R: int, mutant: int = 0) -> list:
    out = np.zeros(max(W, 1), dtype=np.int32)
    n = _lib(mutant).orc_window_slots(pos, W, R, out.ctypes.data)
    return out[:n].tolist()


def index_scores(p: Problem, rows=None, with_magnitude: bool = False, mutant: int = 0):
    """Scores [n_rows, N_c] (float64, -inf past n_vis) and, optionally, the
    condition magnitudes A [n_rows, N_c]."""
    rr = _rows(rows, p.T)
    S = np.empty((len(rr), p.N_c), dtype=np.float64)
    A = np.empty((len(rr), p.N_c), dtype=np.float64) if with_magnitude else None
    st = p._struct()
    if _lib(mutant).orc_index_scores(ctypes.byref(st), rr.ctypes.data, len(rr), S.ctypes.data, _ptr(A)) != 0:
        raise ValueError("oracle: invalid problem")
    return (S, A) if with_magnitude else S


def topk_row(scores: np.ndarray, nv: int, K: int, mutant: int = 0) -> np.ndarray:
    s = np.ascontiguousarray(scores, dtype=np.float64)
    out = np.empty(max(K, 1), dtype=np.int32)
    if _lib(mutant).orc_topk_row(s.ctypes.data, nv, K, out.ctypes.data) < 0:
        raise ValueError("oracle: invalid top-k arguments")
    return out[:K]


def topk(p: Problem, scores: np.ndarray, K: int, rows=None, mutant: int = 0) -> np.ndarray:
    """Top-k indices [n_rows, K] from score rows (one per entry of ``rows``)."""
    rr = _rows(rows, p.T)
    out = np.empty((len(rr), K), dtype=np.int32)
    for i, t in enumerate(rr):
        out[i] = topk_row(scores[i], n_vis(int(p.q_pos[t]), p.r, mutant), K, mutant)
    return out


def candidate_blocks_row(scores: np.ndarray, nv: int, block_size: int, topk_blocks: int,
                         mutant: int = 0) -> np.ndarray:
    """Level one of the two-level top-k ("DeepSeek-V4.1-Flash-NVFP4
    inference/model.py", select_candidate_blocks) on one score row of N_c
    positions: a bool per block of ``block_size`` positions, True if kept."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    nb = (s.size + block_size - 1) // block_size
    keep = np.zeros(max(nb, 1), dtype=np.uint8)
    if _lib(mutant).orc_candidate_blocks(s.ctypes.data, nv, s.size, block_size, topk_blocks, keep.ctypes.data) < 0:
        raise ValueError("oracle: invalid candidate-block arguments")
    return keep[:nb].astype(bool)


def candidate_topk_row(scores: np.ndarray, nv: int, K: int, keep: np.ndarray, block_size: int,
                       mutant: int = 0) -> np.ndarray:
    """Level two ("DeepSeek-V4.1-Flash-NVFP4 inference/model.py",
    Indexer.forward in a layer that uses candidates): the row's positions
    outside the kept blocks are set to -inf, then the same top-k as topk_row
    (K_eff = min(K, n_vis), ties to the lower position, ascending, -1 padded)."""
    s = np.array(scores, dtype=np.float64)
    blocks = np.arange(s.size) // block_size
    s[~keep[blocks]] = -np.inf
    return topk_row(s, nv, K, mutant)


def hadamard_bf16(x_bits: np.ndarray, mutant: int = 0) -> np.ndarray:
    """V3.2 rotate_activation ("DeepSeek-V3.2-Exp inference/model.py"): each row
    of bf16 bits times the Sylvester-Hadamard matrix, scaled by n^-1/2, the
    exact value rounded once to bf16 (nearest, ties to even)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows = x.reshape(-1, x.shape[-1])
    out = np.empty_like(rows)
    for i in range(rows.shape[0]):
        rc = _lib(mutant).orc_hadamard_bf16(rows[i].ctypes.data, rows.shape[1], out[i].ctypes.data)
        if rc == -1:
            raise ValueError("oracle: row length is not a power of two")
        if rc != 0:
            raise ValueError("oracle: the row's dynamic range is beyond the exact evaluation (2^46)")
    return out.reshape(x.shape)


def hadamard_f64(x_bits: np.ndarray) -> np.ndarray:
    """The same rotation before its rounding to bf16 (float64)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows = x.reshape(-1, x.shape[-1])
    out = np.empty(rows.shape, dtype=np.float64)
    for i in range(rows.shape[0]):
        if _lib().orc_hadamard_f64(rows[i].ctypes.data, rows.shape[1], out[i].ctypes.data) != 0:
            raise ValueError("oracle: row length is not a power of two")
    return out.reshape(x.shape)


def e4m3_encode(v: np.ndarray, mutant: int = 0) -> np.ndarray:
    """Nearest float8 e4m3fn codes (ties to even, saturating at +-448)."""
    f = np.ascontiguousarray(v, dtype=np.float32).reshape(-1)
    lib = _lib(mutant)
    return np.array([lib.orc_e4m3_encode(float(x)) for x in f], dtype=np.uint8).reshape(np.shape(v))


def act_quant_rows(y_bits: np.ndarray, mutant: int = 0):
    """act_quant with one block per row (V3.2 Indexer.forward): (codes uint8, scales float32)."""
    y = np.ascontiguousarray(y_bits, dtype=np.uint16)
    rows = y.reshape(-1, y.shape[-1])
    codes = np.empty(rows.shape, dtype=np.uint8)
    scales = np.empty(rows.shape[0], dtype=np.float32)
    for i in range(rows.shape[0]):
        if _lib(mutant).orc_act_quant_row(rows[i].ctypes.data, rows.shape[1], codes[i].ctypes.data,
                                          scales[i:i + 1].ctypes.data) != 0:
            raise ValueError("oracle: empty row")
    return codes.reshape(y.shape), scales.reshape(y.shape[:-1])


def rotate_quant_rows(x_bits: np.ndarray, mutant: int = 0):
    """The V3.2 index producer on rows of bf16 bits: rotation, then act_quant."""
    return act_quant_rows(hadamard_bf16(x_bits, mutant), mutant)


@dataclass
class Rope:
    """Rotary parameters of "DeepSeek-V4.1-Flash-NVFP4 inference/model.py"
    (precompute_freqs_cis); the defaults are the released config's index and
    compressor settings on the atlas page (rope_head_dim 64, compress_rope_theta
    160000, rope_factor 16, original_seq_len 65536, beta_fast 32, beta_slow 1)."""
    dim: int = 64
    base: float = 160000.0
    factor: float = 16.0
    original_seq_len: int = 65536
    beta_fast: float = 32.0
    beta_slow: float = 1.0


def rope_angles(rope: Rope, pos: int, mutant: int = 0) -> np.ndarray:
    lib = _lib(mutant)
    return np.array([lib.orc_rope_angle(rope.dim, i, pos, rope.base, rope.factor, rope.original_seq_len,
                                        rope.beta_fast, rope.beta_slow) for i in range(rope.dim // 2)])


def apply_rope(x: np.ndarray, rope: Rope, pos: int, inverse: bool = False, mutant: int = 0) -> np.ndarray:
    """apply_rotary_emb on one row of rope.dim values (float64, a new array)."""
    v = np.array(x, dtype=np.float64).reshape(-1).copy()
    assert v.size == rope.dim
    _lib(mutant).orc_apply_rope(v.ctypes.data, rope.dim, pos, rope.base, rope.factor, rope.original_seq_len,
                                rope.beta_fast, rope.beta_slow, int(inverse))
    return v


class CompressorState:
    """The partial group a compressor carries across decode steps (kv_state,
    score_state of "DeepSeek-V4.1-Flash-NVFP4 inference/model.py", Compressor)."""

    def __init__(self, r: int, D: int):
        self.kv = np.zeros((r, D), dtype=np.float32)
        self.score = np.full((r, D), -np.inf, dtype=np.float32)


def compress_prefill(kv: np.ndarray, score: np.ndarray, r: int, weight: np.ndarray, eps: float,
                     state: Optional[CompressorState] = None, mutant: int = 0) -> np.ndarray:
    """Compressor.forward from position 0 on one sequence: kv, score [S, D] fp32;
    returns the S // r pooled, normalised rows [S // r, D] (float64, before the
    cast); the trailing S % r tokens go to ``state``."""
    kv = np.ascontiguousarray(kv, dtype=np.float32)
    score = np.ascontiguousarray(score, dtype=np.float32)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    S, D = kv.shape
    out = np.empty((max(S // r, 1), D), dtype=np.float64)
    ks = state.kv.ctypes.data if state is not None else None
    ss = state.score.ctypes.data if state is not None else None
    g = _lib(mutant).orc_compress_prefill(kv.ctypes.data, score.ctypes.data, S, D, r, w.ctypes.data, eps,
                                          out.ctypes.data, ks, ss)
    if g < 0:
        raise ValueError("oracle: invalid compressor arguments")
    return out[:g]


def compress_decode(kv_tok: np.ndarray, score_tok: np.ndarray, pos: int, r: int, weight: np.ndarray, eps: float,
                    state: CompressorState, mutant: int = 0) -> Optional[np.ndarray]:
    """One Compressor.forward decode step at position ``pos``: the pooled row [D]
    when the group completes, else None."""
    kv_tok = np.ascontiguousarray(kv_tok, dtype=np.float32)
    score_tok = np.ascontiguousarray(score_tok, dtype=np.float32)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    D = kv_tok.shape[0]
    out = np.empty(D, dtype=np.float64)
    rc = _lib(mutant).orc_compress_decode(kv_tok.ctypes.data, score_tok.ctypes.data, pos, D, r, state.kv.ctypes.data,
                                          state.score.ctypes.data, w.ctypes.data, eps, out.ctypes.data)
    if rc < 0:
        raise ValueError("oracle: invalid compressor arguments")
    return out if rc == 1 else None


def index_key(x_bits: np.ndarray, weight: np.ndarray, eps: float, pos: int, rope: Rope, mutant: int = 0):
    """The index key of one compressed row ("DeepSeek-V4.1-Flash-NVFP4
    inference/model.py", Indexer.forward, the key-owning layer): x_bits is a row
    of wk(latent) as bf16 bits; returns (codes uint8 [D], scale float32, the
    bf16 key before quantisation as bits [D]).  The rotation takes `pos`, the
    position of the group's first token."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16).reshape(-1)
    w = np.ascontiguousarray(weight, dtype=np.float32)
    D = x.size
    codes = np.empty(D, dtype=np.uint8)
    scale = np.empty(1, dtype=np.float32)
    k = np.empty(D, dtype=np.uint16)
    if _lib(mutant).orc_index_key(x.ctypes.data, D, w.ctypes.data, eps, pos, rope.dim, rope.base, rope.factor,
                                  rope.original_seq_len, rope.beta_fast, rope.beta_slow, codes.ctypes.data,
                                  scale.ctypes.data, k.ctypes.data) != 0:
        raise ValueError("oracle: invalid index-key arguments")
    return codes, scale[0], k


def sparse_attn(p: Problem, idx: np.ndarray, rows=None, mutant: int = 0) -> np.ndarray:
    """Attention output [n_rows, H, D] (float64) for idx [T, K]."""
    rr = _rows(rows, p.T)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    assert idx.ndim == 2 and idx.shape[0] == p.T
    K = idx.shape[1]
    O = np.empty((len(rr), p.H, p.D), dtype=np.float64)
    st = p._struct()
    if _lib(mutant).orc_sparse_attn(ctypes.byref(st), idx.ctypes.data, K, rr.ctypes.data, len(rr), O.ctypes.data) != 0:
        raise ValueError("oracle: invalid problem or indices")
    return O


def fused(p: Problem, K: int, rows=None, mutant: int = 0):
    """(idx [n_rows, K], O [n_rows, H, D]) of the whole step."""
    rr = _rows(rows, p.T)
    idx = np.empty((len(rr), K), dtype=np.int32)
    O = np.empty((len(rr), p.H, p.D), dtype=np.float64)
    st = p._struct()
    if _lib(mutant).orc_fused(ctypes.byref(st), K, rr.ctypes.data, len(rr), idx.ctypes.data, O.ctypes.data) != 0:
        raise ValueError("oracle: invalid problem")
    return idx, O


def set_threads(n: int) -> None:
    _lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_lib().orc_get_threads())


def mutant_build(mutant: int) -> str:
    """Build a deliberately wrong variant in a scratch directory (pin tests)."""
    d = os.path.join(tempfile.gettempdir(), "sa_oracle_mutants")
    return build(mutant, d)
