"""Host-side accounting of bench.py (no GPU): the roofline numerator of the two
HBM-bound workloads against the per-query formula (index keys of the visible
positions plus the gathered window and top-k K/V rows), on the seeded positions."""
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from indexer_selected_sparse_score_gb300 import workloads as wl  # noqa: E402


def light_workload(name):
    spec = wl.CONFIGS[name]
    q_seq, q_pos = wl.draw_positions(spec, wl.SEEDS[name])
    return SimpleNamespace(q_pos=q_pos, r=spec.r, N_c=spec.N_c, k_dtype=spec.k_dtype, D_I=spec.D_I,
                           k_scale=object() if spec.k_scale else None, W=spec.W, K=spec.K, D=spec.D, T=spec.T)


@pytest.mark.parametrize("name,mean_mb", [("c2", 175.1), ("c4", 436.7)])
def test_step_bytes_match_the_per_query_formula(name, mean_mb):
    w = light_workload(name)
    nb = bench.algorithmic_bytes(w)
    nv = np.minimum((w.q_pos.astype(np.int64) + 1) // w.r, w.N_c)
    per_query = nv * (w.D_I + 4) + (np.minimum(w.W, w.q_pos + 1) + np.minimum(w.K, nv)) * w.D * 2 * 2
    assert nb["step"] == int(per_query.sum())
    assert nb["step"] == nb["idx_score"] + nb["sparse_mqa"]
    # the seeded draw lands near the analytic mean of the position distribution
    assert abs(nb["step"] / 1e6 - mean_mb) / mean_mb < 0.05


def test_peak_source():
    peak, src = bench.peaks()
    assert peak > 1000 and src in ("measured", "fallback")


def test_recorded_traffic_survives_comment_edits_only():
    """A capture stays attached to a kernel while only its comments change:
    the source hash ignores comments and blank lines but not code."""
    src = "int f(int x) {  // doubles x\n  /* a block\n     comment */\n  return 2 * x;\n}\n"
    same = "int f(int x) {  // twice x\n\n  return 2 * x;  // result\n}\n"
    other = "int f(int x) {  // doubles x\n  return 3 * x;\n}\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
    for stage in bench.STAGE_SOURCES:
        assert len(bench.kernel_source_hash(stage)) == 16
