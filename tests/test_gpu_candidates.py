"""Two-level top-k on the GPU against the oracle ("DeepSeek-V4.1-Flash-NVFP4
inference/model.py", select_candidate_blocks and Indexer.forward): level one
(the kept candidate blocks) must match bit for bit and level two (the top-k
inside them) index for index, on the same fp32 scores (GPU only)."""
import numpy as np
import pytest

import oracle
from gpu_run import (pack_blocks, run_candidates, run_scores, run_topk_candidates, unpack_blocks)
from helpers import n_vis
from indexer_selected_sparse_score_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

R = 2  # compression ratio of the planted rows: position p sees (p + 1) // 2 entries


def planted(T, N_c, seed, quant=2.0):
    """Scores on a coarse grid (many equal block maxima), with rows of equal
    scores, planted -inf, +inf and -0."""
    rng = np.random.default_rng(seed)
    s = (np.round(rng.normal(size=(T, N_c)) * quant) / quant).astype(np.float32)
    if T > 3:
        s[1, :] = 0.5                       # every block ties
        s[2, 5:N_c:7] = -np.inf             # planted -inf positions
        s[2, 3] = np.inf                    # a block that ties the pinned newest block
        s[3, : N_c // 2] = -0.0             # -0 and +0 compare equal
        s[3, N_c // 2:] = 0.0
    return s


def visible_counts(T, N_c, bs, seed):
    """n_vis per row: 0, 1, block edges, the full row, then random."""
    fixed = [0, 1, bs, bs + 1, N_c, N_c - 1, max(1, N_c - bs)]
    rng = np.random.default_rng(seed + 1)
    nv = [min(N_c, v) for v in fixed] + rng.integers(0, N_c + 1, size=max(0, T - len(fixed))).tolist()
    return np.array(nv[:T], dtype=np.int64)


def tokens_for(nv):
    """q_seq / q_pos with n_vis = nv at r = 2 (each token its own sequence)."""
    T = len(nv)
    q_pos = np.where(nv > 0, 2 * nv, 0).astype(np.int32)  # (2 nv + 1) // 2 = nv; position 0 sees none
    return np.arange(T, dtype=np.int32), q_pos


def check_level_one(scores, nv, bs, tb):
    T, N_c = scores.shape
    nb = (N_c + bs - 1) // bs
    q_seq, q_pos = tokens_for(nv)
    assert all(n_vis(int(p), R) == v for p, v in zip(q_pos, nv))
    cand = run_candidates(scores, q_seq, q_pos, T, R, bs, tb)
    got = unpack_blocks(cand, nb)
    keep = np.zeros((T, nb), dtype=bool)
    for t in range(T):
        keep[t] = oracle.candidate_blocks_row(scores[t].astype(np.float64), int(nv[t]), bs, tb)
        assert np.array_equal(got[t], keep[t]), (t, int(nv[t]), np.flatnonzero(got[t] != keep[t])[:8])
    return cand, keep, q_seq, q_pos


def check_level_two(scores, nv, K, keep, bs, q_seq, q_pos, cand=None):
    T = scores.shape[0]
    cand = pack_blocks(keep) if cand is None else cand
    idx = run_topk_candidates(scores, q_seq, q_pos, T, R, K, cand, bs)
    for t in range(T):
        ref = oracle.candidate_topk_row(scores[t].astype(np.float64), int(nv[t]), K, keep[t], bs)
        assert idx[t].tolist() == ref.tolist(), (t, int(nv[t]))


@pytest.mark.parametrize("N_c,bs,tb", [
    (300, 8, 4),            # few blocks taken, ties at the threshold
    (300, 8, 1000),         # more blocks asked for than there are
    (1000, 3, 50),          # a block size that does not divide the row
    (1000, 1, 100),         # one position per block
    (4099, 64, 7),          # long blocks, short last block
    (5000, 8, 0),           # no block taken
    (32768, 8, 2048),       # the pages' 2048 blocks of 8 over a long row
    (262144, 8, 2048),      # 32768 blocks, the most one row may hold
])
def test_level_one_planted(N_c, bs, tb):
    T = 12
    scores = planted(T, N_c, seed=N_c + bs)
    nv = visible_counts(T, N_c, bs, seed=N_c)
    check_level_one(scores, nv, bs, tb)


@pytest.mark.parametrize("T,N_c,K", [
    (12, 5000, 64), (12, 12000, 300), (12, 30000, 700),   # register top-k, 1024 threads
    (320, 5000, 64), (320, 12000, 300), (320, 30000, 700),  # 512 threads (rows outnumber the SMs)
    (6, 40000, 500),                                      # rows streamed from memory
])
def test_level_two_every_topk_kernel(T, N_c, K):
    """Both levels over each top-k kernel shape; with 40 blocks of 8 the kept
    positions run short of K on most rows, so the -inf fill (lowest visible
    positions outside the kept blocks) is exercised too."""
    bs = 8
    scores = planted(T, N_c, seed=T + N_c)
    nv = visible_counts(T, N_c, bs, seed=T * N_c)
    for tb in (40, 2048):
        cand, keep, q_seq, q_pos = check_level_one(scores, nv, bs, tb)
        check_level_two(scores, nv, K, keep, bs, q_seq, q_pos, cand=cand)


def test_level_two_arbitrary_mask():
    """A mask need not come from level one: random blocks, including blocks
    past a token's visible end (they hold no visible position)."""
    T, N_c, bs, K = 10, 3000, 5, 200
    scores = planted(T, N_c, seed=3)
    nv = visible_counts(T, N_c, bs, seed=4)
    q_seq, q_pos = tokens_for(nv)
    keep = np.random.default_rng(5).random((T, (N_c + bs - 1) // bs)) < 0.2
    check_level_two(scores, nv, K, keep, bs, q_seq, q_pos)


@pytest.mark.parametrize("bs", [1, 2, 3, 4])
@pytest.mark.parametrize("T,N_c,K", [(12, 5000, 300), (12, 30000, 700), (320, 12000, 300)])
def test_level_two_block_sizes_around_compaction(T, N_c, K, bs):
    """Blocks of 1-3 positions take the masked register kernel and blocks of 4
    the compacting one: both exact against the oracle, with level one's masks
    (few and many blocks kept) and with random masks (about a tenth and half of
    the blocks), at 1024 and 512 threads per row."""
    scores = planted(T, N_c, seed=T + N_c + bs)
    nv = visible_counts(T, N_c, bs, seed=T * N_c + bs)
    q_seq, q_pos = tokens_for(nv)
    nb = (N_c + bs - 1) // bs
    for tb in (K // bs // 4 + 1, nb // 2):
        cand, keep, q_seq1, q_pos1 = check_level_one(scores, nv, bs, tb)
        check_level_two(scores, nv, K, keep, bs, q_seq1, q_pos1, cand=cand)
    rng = np.random.default_rng(bs)
    for frac in (0.1, 0.5):
        keep = rng.random((T, nb)) < frac
        check_level_two(scores, nv, K, keep, bs, q_seq, q_pos)


@pytest.mark.parametrize("name", ["i64x128_fp8k", "umma_many"])
def test_two_level_on_indexer_scores(name):
    """Index scores from the GPU's indexer, then level one (blocks of 8) and
    level two, each exact against the oracle on those scores."""
    specs = {
        "i64x128_fp8k": wl.small("i64x128_fp8k", H_I=64, D_I=128, r=4, N_c=700, K=100, H=64,
                                 pos_lo=900, pos_hi=2799, w_div=64.0),
        "umma_many": wl.small("umma_many", B=300, T=300, H_I=64, D_I=128, r=4, N_c=300, K=64, H=64,
                              pos_lo=0, pos_hi=1199, w_div=64.0),
    }
    w = wl.generate(specs[name], seed=41)
    g = run_scores(w)
    bs, tb = 8, 12
    nb = (w.N_c + bs - 1) // bs
    cand = run_candidates(g, w.q_seq, w.q_pos, w.B, w.r, bs, tb)
    got = unpack_blocks(cand, nb)
    idx = run_topk_candidates(g, w.q_seq, w.q_pos, w.B, w.r, w.K, cand, bs)
    for t in range(w.T):
        nv = n_vis(int(w.q_pos[t]), w.r)
        keep = oracle.candidate_blocks_row(g[t].astype(np.float64), nv, bs, tb)
        assert np.array_equal(got[t], keep), t
        ref = oracle.candidate_topk_row(g[t].astype(np.float64), nv, w.K, keep, bs)
        assert idx[t].tolist() == ref.tolist(), t
