"""The V3.2 index producer on the GPU (Hadamard rotation and e4m3 block
quantisation, "DeepSeek-V3.2-Exp inference/model.py", Indexer.forward): codes
and scales equal the oracle's bit for bit -- the oracle rounds the exact
rotation once to bf16 -- except on rows where the exact rotation lies within
2^-40 of its own size of a bf16 rounding midpoint, where the kernel's exact
fallback (64-bit integer sums, one double product) may round either way;
such rows are counted and must be rare.  Rows scatter to their cache rows,
and bad destinations are skipped and flagged (GPU only)."""
import numpy as np
import pytest
import torch

import margins
import oracle
from gpu_run import ensure_built
from indexer_selected_sparse_score_gb300 import binding

pytestmark = pytest.mark.gpu


def bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)


def ws256():
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    return ws


def run(x_bits, dst=None, dst_rows=0, fill=0x55):
    ensure_built()
    rows = x_bits.shape[0]
    n_out = dst_rows if dst is not None else rows
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    codes = torch.full((max(n_out, 1), 128), fill, dtype=torch.uint8, device="cuda")
    scales = torch.full((max(n_out, 1),), float("nan"), dtype=torch.float32, device="cuda")
    d = torch.from_numpy(np.asarray(dst, dtype=np.int32)).cuda() if dst is not None else None
    ws = ws256()
    binding.sa_rotate_quant(x, rows, codes, scales, ws, dst=d, dst_rows=dst_rows)
    st = binding.sa_check_device_status(ws)
    return codes[:n_out].cpu().numpy(), scales[:n_out].cpu().numpy(), st


def special_rows():
    rng = np.random.default_rng(99)
    tiny = rng.normal(size=128)
    tiny[::9] *= 2.0 ** -30          # elements far below the row's largest
    rows = [np.zeros(128), np.full(128, -0.0), np.eye(128)[5], np.full(128, 0.75), -np.eye(128)[127] * 3e4,
            np.linspace(-1e-20, 1e-20, 128), np.where(np.arange(128) % 2, 1e30, -1e30),
            rng.normal(size=128) * 1e33, rng.normal(size=128) * 1e-33, tiny,
            np.round(rng.normal(size=128) * 8) / 8]
    return bf16_bits(np.stack(rows))


N_SPECIAL = 11


def near_midpoint_rows(xb):
    """Rows whose exact rotation has an element within 2^-40 of its size of a
    bf16 rounding midpoint (where a rounding decision taken from a value with
    relative error below 2^-40 may go either way)."""
    y = oracle.hadamard_f64(xb)
    yr = oracle.hadamard_bf16(xb).astype(np.uint32)
    val = (yr << 16).view(np.float32).astype(np.float64)
    mag = (yr & 0x7FFF).astype(np.int64)
    neighbour = []
    for step in (-1, 1):
        o = np.where(yr & 0x8000, -mag, mag) + step
        b = np.where(o < 0, 0x8000 | (-o), o).astype(np.uint32)
        neighbour.append((b << 16).view(np.float32).astype(np.float64))
    dist = np.minimum(np.abs(y - (val + neighbour[0]) / 2), np.abs(y - (val + neighbour[1]) / 2))
    return np.any(dist <= 2.0 ** -40 * np.abs(y), axis=1)


@pytest.mark.parametrize("rows", [1, 7, 8, 33, 1000, 4103])
def test_codes_and_scales_exact(rows):
    rng = np.random.default_rng(rows)
    x = rng.normal(size=(rows, 128)) * np.exp(rng.uniform(-8, 8, size=(rows, 1)))
    xb = bf16_bits(x)
    if rows >= N_SPECIAL:
        xb[:N_SPECIAL] = special_rows()
    codes, scales, st = run(xb)
    assert st == binding.SA_OK
    want_c, want_s = oracle.rotate_quant_rows(xb)
    near = near_midpoint_rows(xb)
    margins.record("producer rows near a bf16 midpoint (share)", float(near.mean()), 0.01)
    assert near.mean() <= 0.01
    ok = ~near
    assert np.array_equal(scales[ok].view(np.uint32), want_s[ok].view(np.uint32))
    assert np.array_equal(codes[ok], want_c[ok])


def test_scatter_to_cache_rows():
    """r = 1 cache append: token t's key lands at row q_seq[t] * N_c + q_pos[t];
    the other rows are untouched."""
    rng = np.random.default_rng(4)
    B, N_c, T = 3, 50, 20
    q_seq = rng.integers(0, B, size=T)
    q_pos = rng.choice(N_c, size=T, replace=False)
    dst = (q_seq * N_c + q_pos).astype(np.int32)
    xb = bf16_bits(rng.normal(size=(T, 128)))
    codes, scales, st = run(xb, dst=dst, dst_rows=B * N_c)
    assert st == binding.SA_OK
    want_c, want_s = oracle.rotate_quant_rows(xb)
    assert np.array_equal(codes[dst], want_c) and np.array_equal(scales[dst], want_s)
    others = np.setdiff1d(np.arange(B * N_c), dst)
    assert (codes[others] == 0x55).all() and np.isnan(scales[others]).all()


def test_bad_destinations_are_skipped_and_flagged():
    xb = bf16_bits(np.random.default_rng(6).normal(size=(4, 128)))
    codes, scales, st = run(xb, dst=[0, -1, 9, 3], dst_rows=4)
    assert st == binding.SA_ERR_DEVICE_DATA
    want_c, want_s = oracle.rotate_quant_rows(xb)
    assert np.array_equal(codes[[0, 3]], want_c[[0, 3]])
    assert (codes[[1, 2]] == 0x55).all()


def test_no_rows():
    codes, scales, st = run(np.zeros((0, 128), dtype=np.uint16))
    assert st == binding.SA_OK


def test_produced_keys_feed_the_scorer():
    """Rotated fp8 queries (q_scale) and keys (k_scale) from the producer, scored by
    sa_indexer_scores with r = 1, match the oracle's score on the same codes."""
    from gpu_run import run_scores
    from helpers import problem
    from indexer_selected_sparse_score_gb300 import workloads as wl
    spec = wl.small("v32", B=2, T=2, r=1, N_c=300, H_I=64, D_I=128, K=64, H=16,
                    q_dtype=wl.FP8_E4M3, k_dtype=wl.FP8_E4M3, q_scale=True, k_scale=True,
                    pos_mode="fixed", pos_lo=299, pos_hi=299, w_div=64.0)
    w = wl.generate(spec, seed=8)
    rng = np.random.default_rng(8)
    q = bf16_bits(rng.normal(size=(2 * 64, 128)))
    k = bf16_bits(rng.normal(size=(2 * 300, 128)))
    qc, qs, st1 = run(q)
    kc, ks, st2 = run(k)
    assert st1 == binding.SA_OK and st2 == binding.SA_OK
    w.q_I = qc.reshape(2, 64, 128)
    w.q_scale = qs.reshape(2, 64)
    w.k_I = kc.reshape(2, 300, 128)
    w.k_scale = ks.reshape(2, 300)
    from tolerances import check_scores
    g = run_scores(w)
    S, A = oracle.index_scores(problem(w), with_magnitude=True)
    check_scores(g, S, A)
