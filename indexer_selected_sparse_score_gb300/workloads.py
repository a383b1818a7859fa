"""Seeded synthetic inputs for the sparse attention step.

This module only draws random inputs in the library's storage formats; it
holds none of the method's arithmetic.  Both the CUDA path (tests, benchmark)
and the float64 oracle consume the same host bytes it produces.

Storage formats: bf16 tensors are uint16 bit patterns, fp8-e4m3fn tensors are
uint8 bit patterns (round-to-nearest-even from float32 draws, done by torch's
CPU dtype conversion), scales and head weights are float32, positions and
sequence ids are int32.

Workload shapes follow the model pages' settings: "DeepSeek-V4.1-Flash-NVFP4
inference/model.py" ModelArgs defaults (index 16 x 64, topk 64, 16 heads of
128, window 128, ratio 2) for the small decode cases and "DeepSeek-V3.2-Exp
inference/model.py" ModelArgs (index 64 x 128, topk 2048, fp8 keys with one
fp32 scale per position) for the long-context cases.

Rows of a cache that a sequence has not reached yet (compressed rows at or past
its visible count) are left at zero, as freshly allocated caches are.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

BF16 = 0
FP8_E4M3 = 1


@dataclass(frozen=True)
class Spec:
    """Shape and distribution of one synthetic workload."""
    name: str
    B: int                      # sequences
    T: int                      # query tokens
    r: int                      # compression ratio
    N_c: int                    # compressed rows stored per sequence
    H_I: int                    # index heads
    D_I: int                    # index head dim
    K: int                      # index_topk
    H: int                      # attention heads
    D: int                      # attention head dim
    W: int                      # window length
    R: int                      # raw ring slots per sequence
    q_dtype: int = BF16
    k_dtype: int = BF16
    q_scale: bool = False       # per-token scale for fp8 queries
    k_scale: bool = False       # per-position scale for fp8 keys
    pos_mode: str = "fixed"     # fixed | uniform | prefill | length
    pos_lo: int = 0
    pos_hi: int = 0
    w_div: float = 1.0          # w ~ U(0,1) / w_div
    sink: bool = False
    description: str = ""


CONFIGS = {
    "c0": Spec("c0", B=1, T=1, r=2, N_c=500, H_I=16, D_I=64, K=64, H=16, D=128, W=128, R=128,
               pos_mode="fixed", pos_lo=999, pos_hi=999, w_div=16.0,
               description="decode, batch 1, one query at position 999; r=2; index 16x64 bf16; "
                           "topk 64; attention 16x128; window 128"),
    "c1": Spec("c1", B=4, T=4, r=2, N_c=2048, H_I=16, D_I=64, K=64, H=16, D=128, W=128, R=128,
               k_dtype=FP8_E4M3, k_scale=True, pos_mode="uniform", pos_lo=2048, pos_hi=4095,
               w_div=16.0,
               description="decode, batch 4, positions U[2048,4095]; r=2; index 16x64, fp8 keys "
                           "+ per-position scale; topk 64; attention 16x128; window 128"),
    "c2": Spec("c2", B=64, T=64, r=4, N_c=16384, H_I=64, D_I=128, K=2048, H=64, D=128, W=128,
               R=128, k_dtype=FP8_E4M3, k_scale=True, pos_mode="uniform", pos_lo=32768,
               pos_hi=65535, w_div=64.0,
               description="decode, batch 64, positions U[32768,65535]; r=4; index 64x128, fp8 "
                           "keys + per-position scale; topk 2048; attention 64x128; window 128"),
    "c3": Spec("c3", B=1, T=4096, r=4, N_c=8192, H_I=64, D_I=128, K=2048, H=64, D=128, W=128,
               R=4224, q_dtype=FP8_E4M3, k_dtype=FP8_E4M3, q_scale=True, k_scale=True,
               pos_mode="prefill", pos_lo=28672, pos_hi=32767, w_div=64.0,
               description="prefill chunk of 4096 causal query tokens at positions "
                           "28672..32767; r=4; index 64x128 fp8 q (per-token scale) and fp8 "
                           "keys; topk 2048; attention 64x128; window 128"),
    "c4": Spec("c4", B=128, T=128, r=4, N_c=32768, H_I=64, D_I=128, K=2048, H=64, D=128, W=128,
               R=128, k_dtype=FP8_E4M3, k_scale=True, pos_mode="length", pos_lo=8192,
               pos_hi=131072, w_div=64.0,
               description="ragged long-context decode, batch 128, lengths U[8192,131072] "
                           "(query at L-1); r=4; index 64x128 fp8 keys + per-position scale; "
                           "topk 2048; attention 64x128; window 128"),
}

SEEDS = {"c0": 20260, "c1": 20261, "c2": 20262, "c3": 20263, "c4": 20264}


@dataclass
class Workload:
    """Host arrays of one problem (field names match the C ABI)."""
    spec: Spec
    seed: int
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
    K: int

    def problem_fields(self) -> dict:
        """The arrays and sizes, without the spec/seed/K bookkeeping."""
        skip = {"spec", "seed", "K"}
        return {k: v for k, v in self.__dict__.items() if k not in skip}


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([seed, *stream]))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (round to nearest even, torch CPU cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def to_e4m3_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> fp8-e4m3fn bit patterns (round to nearest even, torch CPU cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _normal_bits(rng: np.random.Generator, shape, dtype: int) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return to_bf16_bits(x) if dtype == BF16 else to_e4m3_bits(x)


def draw_positions(spec: Spec, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """(q_seq, q_pos) of the T query tokens."""
    rng = _rng(seed, 1)
    if spec.pos_mode == "fixed":
        pos = np.full(spec.T, spec.pos_lo, dtype=np.int64)
        seq = np.arange(spec.T) % spec.B
    elif spec.pos_mode == "uniform":
        pos = rng.integers(spec.pos_lo, spec.pos_hi, size=spec.T, endpoint=True)
        seq = np.arange(spec.T) % spec.B
    elif spec.pos_mode == "length":
        L = rng.integers(spec.pos_lo, spec.pos_hi, size=spec.T, endpoint=True)
        pos = L - 1
        seq = np.arange(spec.T) % spec.B
    elif spec.pos_mode == "prefill":
        # one causal chunk per sequence: tokens pos_lo .. pos_lo + T/B - 1
        per = spec.T // spec.B
        seq = np.repeat(np.arange(spec.B), per)
        pos = spec.pos_lo + np.tile(np.arange(per), spec.B)
    else:
        raise ValueError(spec.pos_mode)
    return seq.astype(np.int32), pos.astype(np.int32)


def generate(spec: Spec, seed: Optional[int] = None, positions=None) -> Workload:
    """Draw one workload.  ``positions`` = (q_seq, q_pos) overrides the draw."""
    if seed is None:
        seed = SEEDS.get(spec.name, 12345)
    q_seq, q_pos = positions if positions is not None else draw_positions(spec, seed)
    q_seq = np.ascontiguousarray(q_seq, dtype=np.int32)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int32)
    B, T, N_c = spec.B, spec.T, spec.N_c

    # highest visible compressed row of each sequence (rows past it stay zero)
    reach = np.zeros(B, dtype=np.int64)
    for b, p in zip(q_seq.tolist(), q_pos.tolist()):
        reach[b] = max(reach[b], min(N_c, (p + 1) // spec.r))

    q_I = _normal_bits(_rng(seed, 2), (T, spec.H_I, spec.D_I), spec.q_dtype)
    q_scale = None
    if spec.q_scale:
        per_tok = _rng(seed, 3).uniform(0.5, 2.0, size=T).astype(np.float32)
        q_scale = np.ascontiguousarray(np.repeat(per_tok[:, None], spec.H_I, axis=1))
    w = (_rng(seed, 4).uniform(0.0, 1.0, size=(T, spec.H_I)) / spec.w_div).astype(np.float32)

    kbytes = np.uint16 if spec.k_dtype == BF16 else np.uint8
    k_I = np.zeros((B, N_c, spec.D_I), dtype=kbytes)
    k_scale = np.zeros((B, N_c), dtype=np.float32) if spec.k_scale else None
    Kc = np.zeros((B, N_c, spec.D), dtype=np.uint16)
    Vc = np.zeros((B, N_c, spec.D), dtype=np.uint16)
    for b in range(B):
        n = int(reach[b])
        if n == 0:
            continue
        k_I[b, :n] = _normal_bits(_rng(seed, 5, b), (n, spec.D_I), spec.k_dtype)
        if k_scale is not None:
            k_scale[b, :n] = _rng(seed, 6, b).uniform(0.5, 2.0, size=n).astype(np.float32)
        Kc[b, :n] = _normal_bits(_rng(seed, 7, b), (n, spec.D), BF16)
        Vc[b, :n] = _normal_bits(_rng(seed, 8, b), (n, spec.D), BF16)

    Q = _normal_bits(_rng(seed, 9), (T, spec.H, spec.D), BF16)
    Kw = _normal_bits(_rng(seed, 10), (B, spec.R, spec.D), BF16)
    Vw = _normal_bits(_rng(seed, 11), (B, spec.R, spec.D), BF16)
    sink = _rng(seed, 12).normal(size=spec.H).astype(np.float32) if spec.sink else None

    return Workload(spec=spec, seed=seed, B=B, T=T, r=spec.r, N_c=N_c, q_seq=q_seq, q_pos=q_pos,
                    H_I=spec.H_I, D_I=spec.D_I, q_I=q_I, q_dtype=spec.q_dtype, q_scale=q_scale,
                    w=w, k_I=k_I, k_dtype=spec.k_dtype, k_scale=k_scale, H=spec.H, D=spec.D,
                    W=spec.W, R=spec.R, Q=Q, Kw=Kw, Vw=Vw, Kc=Kc, Vc=Vc, sink=sink,
                    scale=float(np.float32(1.0 / math.sqrt(spec.D))), K=spec.K)


def small(name: str = "small", **kw) -> Spec:
    """A small spec for parity tests (defaults span several tiles and a tail)."""
    base = dict(B=3, T=3, r=2, N_c=300, H_I=16, D_I=64, K=64, H=16, D=128, W=16, R=16,
                k_dtype=FP8_E4M3, k_scale=True, pos_mode="uniform", pos_lo=200, pos_hi=599,
                w_div=16.0)
    base.update(kw)
    return Spec(name, **base)
