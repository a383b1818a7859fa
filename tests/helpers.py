"""Shared test helpers: format decoding through torch (a library routine that
is independent of the oracle's own decoders) and workload -> oracle problem."""
import numpy as np
import torch

import oracle
from indexer_selected_sparse_score_gb300 import workloads as wl


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.double().numpy()


def e4m3_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8)).view(torch.float8_e4m3fn)
    return t.double().numpy()


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    return bf16_to_f64(bits) if dtype == wl.BF16 else e4m3_to_f64(bits)


def problem(w: "wl.Workload") -> oracle.Problem:
    return oracle.Problem(**w.problem_fields())


def n_vis(pos: int, r: int) -> int:
    return (pos + 1) // r
