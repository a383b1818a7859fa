"""The V4.1 compressor on the GPU against the oracle ("DeepSeek-V4.1-Flash-NVFP4
inference/model.py", Compressor.forward from position 0 and RMSNorm.forward)
(GPU only)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_run import ensure_built
from indexer_selected_sparse_score_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,S,D,r", [(3, 37, 64, 4), (2, 64, 512, 2), (1, 9, 1024, 8), (4, 3, 128, 4)])
def test_compress_prefill(B, S, D, r):
    ensure_built()
    rng = np.random.default_rng(S * D + r)
    kv = rng.normal(size=(B, S, D)).astype(np.float32)
    score = (rng.normal(size=(B, S, D)) * 2).astype(np.float32)
    w = rng.uniform(0.5, 2.0, size=D).astype(np.float32)
    G = S // r
    out = torch.full((B, max(G, 1), D), float("nan"), dtype=torch.bfloat16, device="cuda")
    binding.sa_compress_prefill(torch.from_numpy(kv).cuda(), torch.from_numpy(score).cuda(), B, S, D, r,
                                torch.from_numpy(w).cuda(), 1e-6, out)
    torch.cuda.synchronize()
    g = out[:, :G].float().cpu().numpy().astype(np.float64)
    for b in range(B):
        o = oracle.compress_prefill(kv[b], score[b], r, w, 1e-6)
        # bf16 output rounding on both sides, plus one bf16 step of the pooled value
        # where fp32 and float64 pooling round to different neighbours before the norm
        assert np.all(np.abs(g[b] - o) <= 2.0 ** -7 * np.abs(o) + 1e-6), b
    if G == 0:
        assert torch.isnan(out).all()
