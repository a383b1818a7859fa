"""Pins for the oracle of the V3.2 index producer ("DeepSeek-V3.2-Exp
inference/model.py", rotate_activation and act_quant in Indexer.forward):
the Hadamard rotation against scipy's Sylvester matrix and closed forms, the
e4m3 encoder exhaustively against the format's decoder and torch's cast, and
the block quantisation against its defining properties."""
import numpy as np
import pytest
import torch

import oracle

scipy_linalg = pytest.importorskip("scipy.linalg")


def to_bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def e4m3_values(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def pin_hadamard_matrix(n=128, mutant=0):
    rng = np.random.default_rng(n)
    x = to_bf16_bits(rng.normal(size=(20, n)) * rng.choice([1e-3, 1.0, 50.0], size=(20, 1)))
    xv = bf16_values(x)
    exact = xv @ scipy_linalg.hadamard(n).T.astype(np.float64) / np.sqrt(n)
    got = bf16_values(oracle.hadamard_bf16(x, mutant))
    # bf16 rounding of the result plus the fp32 butterfly's rounding (log2 n stages)
    bound = 2.0 ** -8 * np.abs(exact) + 2.0 ** -21 * np.abs(xv).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - exact) <= bound)


@pytest.mark.parametrize("n", [2, 8, 128])
def test_hadamard_matches_sylvester_matrix(n):
    pin_hadamard_matrix(n)


def test_hadamard_closed_forms():
    n = 128
    sc = np.float32(1.0 / np.sqrt(n))
    # a unit vector e_j maps to column j of H times n^-1/2
    for j in (0, 1, 77, 127):
        x = np.zeros(n, dtype=np.float32)
        x[j] = 1.0
        got = bf16_values(oracle.hadamard_bf16(to_bf16_bits(x)[None])[0])
        want = bf16_values(to_bf16_bits(scipy_linalg.hadamard(n)[:, j] * sc))
        assert np.array_equal(got, want)
    # a constant vector maps to sqrt(n) c e_0 (the sums are exact in fp32 here)
    got = bf16_values(oracle.hadamard_bf16(to_bf16_bits(np.full(n, 0.75))[None])[0])
    assert got[0] == bf16_values(to_bf16_bits(np.float32(0.75 * n) * sc)) and not got[1:].any()


def test_hadamard_is_an_involution():
    rng = np.random.default_rng(3)
    x = to_bf16_bits(rng.normal(size=(16, 128)))
    twice = bf16_values(oracle.hadamard_bf16(oracle.hadamard_bf16(x)))
    xv = bf16_values(x)
    assert np.all(np.abs(twice - xv) <= 2.0 ** -7 * np.abs(xv).max(axis=1, keepdims=True))


def test_e4m3_encoder_round_trips_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = e4m3_values(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def pin_e4m3_ties(mutant=0):
    pos = np.array([c for c in range(0x7F)], dtype=np.uint8)
    v = e4m3_values(pos)
    mid = ((v[:-1] + v[1:]) / 2).astype(np.float32)  # exactly representable in fp32
    got = oracle.e4m3_encode(mid, mutant)
    even = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(got, even)


def test_e4m3_encoder_ties_and_saturation():
    pin_e4m3_ties()
    assert np.array_equal(oracle.e4m3_encode(np.array([448.0, 449.0, 1e6, -500.0], dtype=np.float32)),
                          np.array([0x7E, 0x7E, 0x7E, 0xFE], dtype=np.uint8))
    assert oracle.e4m3_encode(np.array([-0.0], dtype=np.float32))[0] == 0x80


def test_e4m3_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(5)
    v = (rng.normal(size=20000) * np.exp(rng.uniform(-12, 6, size=20000))).astype(np.float32)
    v = v[np.abs(v) < 448.0]
    ours = oracle.e4m3_encode(v)
    theirs = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def pin_act_quant(mutant=0):
    rng = np.random.default_rng(9)
    y = to_bf16_bits(rng.normal(size=(50, 128)) * rng.uniform(1e-3, 1e3, size=(50, 1)))
    codes, scales = oracle.act_quant_rows(y, mutant)
    yv = bf16_values(y)
    amax = np.abs(yv).max(axis=1)
    assert np.array_equal(scales, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32))
    # the largest element takes the largest code; dequantised values sit within half a code step
    big = np.abs(yv).argmax(axis=1)
    assert np.all(codes[np.arange(50), big] & 0x7F == 0x7E)
    deq = e4m3_values(codes) * scales[:, None].astype(np.float64)
    assert np.all(np.abs(deq - yv) <= 2.0 ** -4 * np.abs(yv) + 2.0 ** -10 * scales[:, None])


def test_act_quant_properties():
    pin_act_quant()
    # an all-zero row: scale 1, zero codes
    c0, s0 = oracle.act_quant_rows(np.zeros((1, 128), dtype=np.uint16))
    assert s0[0] == 1.0 and not c0.any()


PRODUCER_MUTANTS = {12: "butterfly difference reversed", 13: "ties away from zero", 14: "scale for a max of 240"}


@pytest.mark.parametrize("mutant", sorted(PRODUCER_MUTANTS), ids=lambda m: PRODUCER_MUTANTS[m].replace(" ", "_"))
def test_producer_mutant_is_caught(mutant):
    """Each planted mistake in the producer's oracle fails at least one pin."""
    path = oracle.mutant_build(mutant)
    oracle._lib(mutant, path)
    oracle._LIBS[mutant] = oracle._LIBS[path]
    failed = []
    for pin in (pin_hadamard_matrix, pin_e4m3_ties, pin_act_quant):
        try:
            pin(mutant=mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({PRODUCER_MUTANTS[mutant]}) passed every pin"
