"""GB300-native sparse attention step: index scores -> per-query top-k ->
windowed + sparse MQA with a split-KV combine, as hand-written sm_103a CUDA
behind the C ABI of include/sa.h.

The Python surface is the ctypes binding in ``binding`` (same names as the C
entry points).  Importing the package does not load the CUDA library; the
first call does, and raises if libsa.so has not been built.
"""
from .binding import (  # noqa: F401
    AttnArgs,
    DeviceProblem,
    IndexArgs,
    SAError,
    SA_BF16,
    SA_FP8_E4M3,
    new_workspace,
    sa_check_device_status,
    sa_fused_decode,
    sa_indexer_scores,
    sa_sparse_attn,
    sa_topk,
    sa_workspace_init,
    sa_workspace_size,
    upload,
)
