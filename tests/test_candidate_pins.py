"""Pins of the two-level top-k oracle (candidate blocks, then top-k inside
them): hand-worked cases and invariants that follow from the definition."""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "candidate_blocks.txt")


def _golden():
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, scores, kept, idx = [f.strip() for f in line.split("|")]
        N_c, bs, tb, nv, K = map(int, head.split())
        yield (N_c, bs, tb, nv, K, np.array([float(x) for x in scores.split(",")]),
               [] if kept == "-" else [int(x) for x in kept.split(",")], [int(x) for x in idx.split(",")])


@pytest.mark.parametrize("case", list(_golden()))
def test_golden(case):
    N_c, bs, tb, nv, K, S, kept, idx = case
    assert S.size == N_c
    keep = oracle.candidate_blocks_row(S, nv, bs, tb)
    assert np.flatnonzero(keep).tolist() == kept
    assert oracle.candidate_topk_row(S, nv, K, keep, bs).tolist() == idx


def _rows(seed, n=40):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        N_c = int(rng.integers(1, 400))
        bs = int(rng.choice([1, 2, 4, 8, 16]))
        nv = int(rng.integers(0, N_c + 1))
        tb = int(rng.integers(0, 60))
        # coarse values so that ties between blocks occur
        S = rng.integers(0, 12, size=N_c).astype(np.float64)
        yield N_c, bs, nv, tb, S


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_invariants(seed):
    for N_c, bs, nv, tb, S in _rows(seed):
        keep = oracle.candidate_blocks_row(S, nv, bs, tb)
        nb = (N_c + bs - 1) // bs
        reach = (nv + bs - 1) // bs  # blocks with a visible position (finite scores)
        assert keep.size == nb
        assert not keep[reach:].any(), "an unreachable block was kept"
        assert keep.sum() == min(tb, reach)
        if nv >= 1 and tb >= 1:
            assert keep[(nv - 1) // bs], "the newest block must be kept"
        # a kept block (other than the pinned one) scores at least as high as
        # every dropped reachable block, and wins ties only by a lower index
        bscore = np.array([S[b * bs:min((b + 1) * bs, nv)].max() if b < reach else -np.inf for b in range(nb)])
        pinned = (nv - 1) // bs if nv >= 1 else -1
        for k in np.flatnonzero(keep):
            if k == pinned:
                continue
            for d in range(reach):
                if keep[d] or d == pinned:
                    continue
                assert bscore[k] > bscore[d] or (bscore[k] == bscore[d] and k < d)


@pytest.mark.parametrize("seed", [4, 5])
def test_all_blocks_kept_is_plain_topk(seed):
    """With at least as many blocks requested as exist, every reachable block
    is a candidate and level two is the plain top-k."""
    for N_c, bs, nv, _, S in _rows(seed):
        nb = (N_c + bs - 1) // bs
        keep = oracle.candidate_blocks_row(S, nv, bs, nb)
        for K in (1, 7, 64):
            assert oracle.candidate_topk_row(S, nv, K, keep, bs).tolist() == oracle.topk_row(S, nv, K).tolist()


def test_block_size_one_keeps_top_positions():
    """Block size 1: the kept set is the newest position plus the
    (topk_blocks - 1) best of the others (ties to the lower position)."""
    rng = np.random.default_rng(6)
    for _ in range(20):
        N_c = int(rng.integers(2, 300))
        nv = int(rng.integers(1, N_c + 1))
        tb = int(rng.integers(1, nv + 1))
        S = rng.integers(0, 50, size=N_c).astype(np.float64)
        keep = oracle.candidate_blocks_row(S, nv, 1, tb)
        others = sorted(range(nv - 1), key=lambda s: (-S[s], s))[:tb - 1]
        assert np.flatnonzero(keep).tolist() == sorted(others + [nv - 1])
