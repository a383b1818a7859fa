"""The V4.1 compressor and index-key producer on the GPU against the oracle
("DeepSeek-V4.1-Flash-NVFP4 inference/model.py": Compressor.forward from
position 0 and in decode steps, RMSNorm.forward; Indexer.forward's key
publication in the layer that owns the index keys) (GPU only)."""
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
        _close_after_cast(g[b], o, "prefill", kv[b, :G * r].reshape(G, r, D), score[b, :G * r].reshape(G, r, D), w)
    if G == 0:
        assert torch.isnan(out).all()


def _close_after_cast(g, o, what, kv, score, w, eps=1e-6):
    """g (bf16 from the GPU) is the correct rounding of a value within
    2^-7 |o| + 1e-5 (w / rms) A of the oracle's o, per element.  kv, score:
    [G, r, D] the groups' inputs, w the norm weight.  The pooled row c is cast
    to bf16 before the norm: where fp32 and float64 pooling fall on either side
    of a bf16 midpoint that cast differs by one bf16 step: 2^-7 of the element
    at the bottom of a binade, 2^-8 at its top.  The fp32 pooling itself errs by a few units of 2^-24 of
    A = sum_j p_j |kv_j| (p the softmax weights), which the norm scales by
    w / rms(c); 1e-5 covers it many times over."""
    from tolerances import attn_rounding_interval
    import margins
    sc = score.astype(np.float64)
    p = np.exp(sc - sc.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    A = (p * np.abs(kv.astype(np.float64))).sum(axis=1)          # [G, D]
    c = (p * kv.astype(np.float64)).sum(axis=1)
    rms = np.sqrt((c * c).mean(axis=1, keepdims=True) + eps)
    bound = 2.0 ** -7 * np.abs(o) + 1e-5 * np.abs(w)[None, :] / rms * A
    lo, hi = attn_rounding_interval(g)
    dist = np.maximum(np.maximum(lo - o, o - hi), 0.0)
    margins.record(f"compressor {what}: distance / bound", float((dist / bound).max()) if dist.size else 0.0, 1.0)
    assert np.all(dist <= bound), what


@pytest.mark.parametrize("B,S0,steps,D,r", [(3, 10, 13, 128, 4), (2, 0, 9, 512, 2), (4, 7, 17, 64, 8), (128, 64, 8, 512, 4)])
def test_prefill_then_decode(B, S0, steps, D, r):
    """sa_compress_prefill on the first S0 tokens (partial group into the
    states), then one sa_compress_decode per token, against the oracle's
    prefill and decode with its own state (Compressor.forward)."""
    ensure_built()
    rng = np.random.default_rng(B * 1000 + S0 * 10 + r)
    S = S0 + steps
    kv = rng.normal(size=(B, S, D)).astype(np.float32)
    score = (rng.normal(size=(B, S, D)) * 2).astype(np.float32)
    w = rng.uniform(0.5, 2.0, size=D).astype(np.float32)
    eps = 1e-6
    d_kv, d_sc = torch.from_numpy(kv).cuda(), torch.from_numpy(score).cuda()
    d_w = torch.from_numpy(w).cuda()
    kvs = torch.zeros((B, r, D), dtype=torch.float32, device="cuda")
    scs = torch.full((B, r, D), float("-inf"), dtype=torch.float32, device="cuda")
    G0 = S0 // r
    pre = torch.full((B, max(G0, 1), D), float("nan"), dtype=torch.bfloat16, device="cuda")
    if S0 > 0:
        binding.sa_compress_prefill(d_kv[:, :S0].contiguous(), d_sc[:, :S0].contiguous(), B, S0, D, r, d_w, eps,
                                    pre, kv_state=kvs, score_state=scs)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    got = {}
    for t in range(S0, S):
        out = torch.full((B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        binding.sa_compress_decode(d_kv[:, t].contiguous(), d_sc[:, t].contiguous(), pos, B, D, r, kvs, scs, d_w, eps,
                                   out, ws)
        o = out.float().cpu().numpy().astype(np.float64)
        if (t + 1) % r == 0:
            got[t] = o
        else:
            assert np.isnan(o).all(), "rows are written only when a group completes"
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    for b in range(B):
        st = oracle.CompressorState(r, D)
        o_pre = oracle.compress_prefill(kv[b, :S0], score[b, :S0], r, w, eps, state=st)
        if G0:
            _close_after_cast(pre[b, :G0].float().cpu().numpy().astype(np.float64), o_pre, "prefill",
                              kv[b, :G0 * r].reshape(G0, r, D), score[b, :G0 * r].reshape(G0, r, D), w)
        for t in range(S0, S):
            o = oracle.compress_decode(kv[b, t], score[b, t], t, r, w, eps, st)
            assert (o is not None) == (t in got)
            if o is not None:
                g0 = t + 1 - r  # the group's tokens
                _close_after_cast(got[t][b][None], o[None], "decode", kv[b, g0:t + 1][None], score[b, g0:t + 1][None], w)


def test_decode_flags_negative_positions():
    ensure_built()
    B, D, r = 2, 64, 4
    z = torch.zeros((B, D), dtype=torch.float32, device="cuda")
    kvs = torch.zeros((B, r, D), dtype=torch.float32, device="cuda")
    scs = torch.zeros((B, r, D), dtype=torch.float32, device="cuda")
    out = torch.full((B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    pos = torch.tensor([3, -1], dtype=torch.int32, device="cuda")
    binding.sa_compress_decode(z, z, pos, B, D, r, kvs, scs, torch.ones(D, device="cuda"), 1e-6, out, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_ERR_DEVICE_DATA
    assert not torch.isnan(out[0]).any() and torch.isnan(out[1]).all()


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)


def test_index_key_publish_codes_exact():
    """Keys of compressed rows (V4.1 Indexer.forward, owning layer): codes and
    scales equal the oracle's bit for bit (norm and rotation in double on both
    sides, each bf16 result one rounding), written to their rows of a padded
    cache; other rows untouched; bad sequence ids and rows flagged and skipped."""
    ensure_built()
    rng = np.random.default_rng(17)
    B, N_rows, pad, n, r = 5, 300, 40, 400, 4
    rope = oracle.Rope()
    seq = rng.integers(0, B, size=n).astype(np.int32)
    grp = np.zeros(n, dtype=np.int32)
    for b in range(B):  # distinct rows per sequence, up to the cache's end (positions up to 1196)
        idx = np.nonzero(seq == b)[0]
        grp[idx] = rng.choice(N_rows, size=idx.size, replace=False)
    x = _bf16_bits(rng.normal(size=(n, 128)) * rng.choice([1e-3, 1.0, 30.0], size=(n, 1)))
    w = rng.uniform(0.5, 2.0, size=128).astype(np.float32)
    eps = float(np.float32(1e-6))
    kI = torch.full((B, N_rows + pad, 128), 0x55, dtype=torch.uint8, device="cuda")
    ks = torch.full((B, N_rows + pad), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    ra = binding.RopeArgs(rope.dim, rope.base, rope.factor, rope.original_seq_len, rope.beta_fast, rope.beta_slow)
    binding.sa_index_key_publish(torch.from_numpy(x.view(np.int16)).cuda(), n, torch.from_numpy(seq).cuda(),
                                 torch.from_numpy(grp).cuda(), r, torch.from_numpy(w).cuda(), eps, ra, kI, ks, B,
                                 N_rows, ws, k_seq_stride=(N_rows + pad) * 128)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    gc, gs = kI.cpu().numpy(), ks.cpu().numpy()
    written = np.zeros((B, N_rows + pad), dtype=bool)
    for i in range(n):
        codes, scale, _ = oracle.index_key(x[i], w, eps, int(grp[i]) * r, rope)
        assert np.array_equal(gc[seq[i], grp[i]], codes), i
        assert np.float32(gs[seq[i], grp[i]]).view(np.uint32) == np.float32(scale).view(np.uint32), i
        written[seq[i], grp[i]] = True
    assert (gc[~written] == 0x55).all() and np.isnan(gs[~written]).all()
    # a bad sequence id and a row past the cache are skipped and flagged
    bad_seq = torch.tensor([0, B], dtype=torch.int32, device="cuda")
    bad_grp = torch.tensor([N_rows, 1], dtype=torch.int32, device="cuda")
    binding.sa_index_key_publish(torch.from_numpy(x[:2].view(np.int16)).cuda(), 2, bad_seq, bad_grp, r,
                                 torch.from_numpy(w).cuda(), eps, ra, kI, ks, B, N_rows, ws,
                                 k_seq_stride=(N_rows + pad) * 128)
    assert binding.sa_check_device_status(ws) == binding.SA_ERR_DEVICE_DATA
    assert np.array_equal(kI.cpu().numpy(), gc)


def test_index_key_publish_codes_exact_long_positions():
    """4096 rows at positions up to 131068 (angles of up to ~1.3e5 radians for
    the fastest pair, where the argument reduction of the rotation matters):
    codes and scales equal the oracle's bit for bit."""
    ensure_built()
    rng = np.random.default_rng(29)
    B, N_rows, n, r = 1, 32768, 4096, 4
    rope = oracle.Rope()
    seq = np.zeros(n, dtype=np.int32)
    grp = rng.choice(N_rows, size=n, replace=False).astype(np.int32)
    x = _bf16_bits(rng.normal(size=(n, 128)) * rng.choice([1e-2, 1.0, 7.0], size=(n, 1)))
    w = rng.uniform(0.5, 2.0, size=128).astype(np.float32)
    eps = float(np.float32(1e-6))
    kI = torch.zeros((B, N_rows, 128), dtype=torch.uint8, device="cuda")
    ks = torch.zeros((B, N_rows), dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    ra = binding.RopeArgs(rope.dim, rope.base, rope.factor, rope.original_seq_len, rope.beta_fast, rope.beta_slow)
    binding.sa_index_key_publish(torch.from_numpy(x.view(np.int16)).cuda(), n, torch.from_numpy(seq).cuda(),
                                 torch.from_numpy(grp).cuda(), r, torch.from_numpy(w).cuda(), eps, ra, kI, ks, B,
                                 N_rows, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    gc, gs = kI.cpu().numpy(), ks.cpu().numpy()
    for i in range(n):
        codes, scale, _ = oracle.index_key(x[i], w, eps, int(grp[i]) * r, rope)
        assert np.array_equal(gc[0, grp[i]], codes), i
        assert np.float32(gs[0, grp[i]]).view(np.uint32) == np.float32(scale).view(np.uint32), i


def test_compressed_keys_feed_the_scorer():
    """The f3 path end to end on the GPU: compressor prefill of one sequence,
    the caller's key projection (a random bf16 matrix here), the key publisher
    into the cache, then sa_indexer_scores on those fp8 keys, against the
    oracle's scores on the same codes."""
    ensure_built()
    from gpu_run import run_scores
    from helpers import problem
    from indexer_selected_sparse_score_gb300 import workloads as wl
    from tolerances import check_scores
    rng = np.random.default_rng(23)
    r, S, D = 4, 1024, 512
    G = S // r
    kv = rng.normal(size=(1, S, D)).astype(np.float32)
    score = rng.normal(size=(1, S, D)).astype(np.float32)
    w = rng.uniform(0.5, 2.0, size=D).astype(np.float32)
    latent = torch.empty((1, G, D), dtype=torch.bfloat16, device="cuda")
    binding.sa_compress_prefill(torch.from_numpy(kv).cuda(), torch.from_numpy(score).cuda(), 1, S, D, r,
                                torch.from_numpy(w).cuda(), 1e-6, latent)
    wk = torch.from_numpy((rng.normal(size=(D, 128)) / np.sqrt(D)).astype(np.float32)).cuda().bfloat16()
    kproj = (latent[0].float() @ wk.float()).bfloat16().contiguous()  # the caller's projection
    kI = torch.zeros((1, G, 128), dtype=torch.uint8, device="cuda")
    ks = torch.zeros((1, G), dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    binding.sa_workspace_init(ws)
    rope = oracle.Rope()
    ra = binding.RopeArgs(rope.dim, rope.base, rope.factor, rope.original_seq_len, rope.beta_fast, rope.beta_slow)
    kn = torch.from_numpy(rng.uniform(0.5, 2.0, size=128).astype(np.float32)).cuda()
    binding.sa_index_key_publish(kproj, G, torch.zeros(G, dtype=torch.int32, device="cuda"),
                                 torch.arange(G, dtype=torch.int32, device="cuda"), r, kn, float(np.float32(1e-6)), ra,
                                 kI, ks, 1, G, ws)
    assert binding.sa_check_device_status(ws) == binding.SA_OK
    spec = wl.small("f3", B=1, T=3, r=r, N_c=G, H_I=64, D_I=128, K=32, H=16, pos_mode="uniform", pos_lo=100,
                    pos_hi=S - 1, w_div=64.0)
    wkl = wl.generate(spec, seed=23)
    wkl.k_I = kI.cpu().numpy()
    wkl.k_scale = ks.cpu().numpy()
    g = run_scores(wkl)
    S_, A = oracle.index_scores(problem(wkl), with_magnitude=True)
    check_scores(g, S_, A)
