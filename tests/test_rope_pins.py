"""Pins for the rotary-embedding oracle ("DeepSeek-V4.1-Flash-NVFP4
inference/model.py", precompute_freqs_cis with YaRN and apply_rotary_emb), the
rotation the compressor's index keys take at their group's start position:
closed-form frequencies, the YaRN band's endpoints, and the algebra of
rotations (norm kept, inverse undoes, angles add)."""
import math

import numpy as np
import pytest

import oracle

PLAIN = oracle.Rope(dim=64, base=10000.0, factor=1.0, original_seq_len=0)
YARN = oracle.Rope()  # the released config's index / compressor settings


def yarn_band(r):
    def corrected(rot):
        return r.dim * math.log(r.original_seq_len / (rot * 2 * math.pi)) / (2 * math.log(r.base))
    return max(math.floor(corrected(r.beta_fast)), 0), min(math.ceil(corrected(r.beta_slow)), r.dim - 1)


def pin_plain_frequencies(mutant=0):
    a = oracle.rope_angles(PLAIN, 1, mutant)
    assert a[0] == 1.0                                   # base^0
    assert abs(a[16] - 0.01) < 1e-15                     # 10000^(-1/2)
    assert np.all(np.diff(a) < 0)                        # strictly falling with the pair index


def pin_yarn_band(mutant=0):
    low, high = yarn_band(YARN)
    a = oracle.rope_angles(YARN, 1, mutant)
    base = oracle.rope_angles(oracle.Rope(dim=YARN.dim, base=YARN.base, factor=1.0, original_seq_len=0), 1, mutant)
    assert np.allclose(a[:low + 1], base[:low + 1], rtol=1e-15)                  # inside the context: kept
    assert np.allclose(a[high:], base[high:] / YARN.factor, rtol=1e-15)         # far beyond it: divided
    mid = a[low + 1:high] / base[low + 1:high]
    assert np.all((mid < 1.0) & (mid > 1.0 / YARN.factor)) and np.all(np.diff(mid) < 0)  # the fade


def pin_rotation_algebra(mutant=0):
    rng = np.random.default_rng(7)
    x = rng.normal(size=YARN.dim)
    y = oracle.apply_rope(x, YARN, 1234, mutant=mutant)
    assert np.allclose(np.hypot(y[0::2], y[1::2]), np.hypot(x[0::2], x[1::2]), rtol=1e-14)
    assert np.allclose(oracle.apply_rope(y, YARN, 1234, inverse=True, mutant=mutant), x, atol=1e-13)
    two = oracle.apply_rope(oracle.apply_rope(x, YARN, 1000, mutant=mutant), YARN, 234, mutant=mutant)
    assert np.allclose(two, y, atol=1e-10)               # angles add: pos 1000 then 234 = pos 1234
    unit = np.zeros(YARN.dim)
    unit[0::2] = 1.0                                     # (1, 0) pairs land on (cos a, sin a)
    z = oracle.apply_rope(unit, YARN, 77, mutant=mutant)
    ang = oracle.rope_angles(YARN, 77, mutant)
    assert np.allclose(z[0::2], np.cos(ang), atol=1e-15) and np.allclose(z[1::2], np.sin(ang), atol=1e-15)


PINS = (pin_plain_frequencies, pin_yarn_band, pin_rotation_algebra)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_position_zero_is_the_identity():
    x = np.random.default_rng(1).normal(size=YARN.dim)
    assert np.array_equal(oracle.apply_rope(x, YARN, 0), x)


def test_reversed_ramp_is_caught():
    path = oracle.mutant_build(18)
    oracle._lib(18, path)
    oracle._LIBS[18] = oracle._LIBS[path]
    failed = []
    for pin in PINS:
        try:
            pin(mutant=18)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed
