"""The parity checks themselves: bf16 rounding helpers against torch's cast
and hand-worked values, and the attention check's acceptance region."""
import numpy as np
import torch

import margins
from tolerances import attn_rounding_interval, bf16_round, check_attn


def test_bf16_round_matches_torch_on_float32():
    rng = np.random.default_rng(0)
    x = (rng.normal(size=20000) * np.exp(rng.uniform(-20, 20, size=20000))).astype(np.float32)
    want = torch.from_numpy(x).bfloat16().double().numpy()
    assert np.array_equal(bf16_round(x.astype(np.float64)), want)


def test_bf16_round_is_a_single_rounding():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: ties go to the even value 1;
    # a hair above it must go up even though float32 rounding would first land
    # on the midpoint (double rounding)
    assert bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert bf16_round(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1 + 2.0 ** -7
    assert bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6   # tie, odd below -> up
    assert bf16_round(np.array([-(1 + 2.0 ** -8 + 2.0 ** -40)]))[0] == -(1 + 2.0 ** -7)


def test_rounding_interval():
    lo, hi = attn_rounding_interval(np.array([1.0, 1 + 2.0 ** -7, -2.0, 0.0]))
    assert lo[0] == 1 - 2.0 ** -9 and hi[0] == 1 + 2.0 ** -8     # below 1 the step halves
    assert lo[1] == 1 + 2.0 ** -8 and hi[1] == 1 + 3 * 2.0 ** -8
    assert lo[2] == -2 - 2.0 ** -7 and hi[2] == -2 + 2.0 ** -8
    assert lo[3] < 0 < hi[3] and hi[3] == 2.0 ** -134


def test_attention_check_accepts_correct_roundings_and_rejects_errors():
    with margins.suspended():
        _attention_check_cases()


def _attention_check_cases():
    rng = np.random.default_rng(1)
    o = rng.normal(size=(50, 128))
    # the correctly rounded oracle passes with zero pre-rounding error
    assert check_attn(bf16_round(o), o) == 0.0
    # a value 1e-3 of the row max away, then rounded, passes
    rowmax = np.abs(o).max(axis=-1, keepdims=True)
    assert check_attn(bf16_round(o + 1e-3 * rowmax), o) <= 2e-3
    # 3e-3 of the row max on one element fails
    bad = o.copy()
    bad[7, 5] += 3e-3 * rowmax[7, 0] + 2.0 ** -8 * abs(o[7, 5])
    try:
        check_attn(bf16_round(bad), o)
    except AssertionError:
        return
    raise AssertionError("an error of 3e-3 of the row max passed")
