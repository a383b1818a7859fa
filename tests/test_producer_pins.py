"""Pins for the oracle of the V3.2 index producer ("DeepSeek-V3.2-Exp
inference/model.py", rotate_activation and act_quant in Indexer.forward):
the Hadamard rotation against scipy's Sylvester matrix, an exact evaluation in
Python integers rounded in decimal arithmetic, and closed forms, the
e4m3 encoder exhaustively against the format's decoder and torch's cast, and
the block quantisation against its defining properties."""
from decimal import Decimal, getcontext
from fractions import Fraction

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
    # one rounding to bf16: within half a bf16 step, at most 2^-8 of the value
    # (plus the float64 evaluation of `exact` here)
    bound = 2.0 ** -8 * np.abs(exact) + 2.0 ** -40 * np.abs(xv).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - exact) <= bound)


def _exact_bf16(num: int, den_pow2: int, n: int) -> float:
    """The bfloat16 nearest (ties to even) to num * 2^-den_pow2 * n^-1/2,
    decided in 80-digit decimal arithmetic against the neighbouring bf16
    values (an evaluation independent of the oracle's integer rounding)."""
    if num == 0:
        return 0.0
    getcontext().prec = 80
    y = Decimal(num) / (Decimal(2) ** den_pow2) / Decimal(n).sqrt()
    c = int(to_bf16_bits(np.array([float(y)], dtype=np.float32))[0])
    cand = [float(bf16_values(np.array([b], dtype=np.uint16))[0]) for b in (c - 1, c, c + 1) if 0 <= b <= 0xFFFF]
    cand = [v for v in cand if np.isfinite(v) and np.sign(v) == np.sign(float(y))]
    dist = sorted((abs(Decimal(v) - y), v) for v in cand)
    if dist[0][0] == dist[1][0]:   # a tie: the value with the even last bit
        return [v for d, v in dist[:2] if int(to_bf16_bits(np.array([v], dtype=np.float32))[0]) % 2 == 0][0]
    return dist[0][1]


def pin_hadamard_exact_rounding(mutant=0):
    """Each output is the exact sum H x (in Python integers) times n^-1/2,
    rounded once to the nearest bf16 (ties to even): for odd and even log2 n,
    on rows of several scales and with exact ties (n = 64: y = S / 8)."""
    rng = np.random.default_rng(11)
    for n in (2, 8, 64, 128, 256):
        H = scipy_linalg.hadamard(n).astype(np.int64)
        rows = rng.normal(size=(6, n)) * rng.choice([1e-30, 1e-3, 1.0, 3e4], size=(6, 1))
        rows[0] = np.round(rng.normal(size=n) * 4) / 4   # coarse values: ties when n = 64
        x = to_bf16_bits(rows)
        got = bf16_values(oracle.hadamard_bf16(x, mutant))
        xv = bf16_values(x)
        for i in range(x.shape[0]):
            xi = [int(Fraction(float(v)) * 2 ** 140) for v in xv[i]]   # every bf16 value is k * 2^-140
            for o in range(n):
                S = sum(int(H[o, j]) * xi[j] for j in range(n))
                want = _exact_bf16(S, 140, n)
                assert got[i, o] == want and (want != 0.0 or not np.signbit(got[i, o])), (n, i, o, got[i, o], want)


def test_hadamard_exact_rounding():
    pin_hadamard_exact_rounding()


@pytest.mark.parametrize("n", [2, 8, 128])
def test_hadamard_matches_sylvester_matrix(n):
    pin_hadamard_matrix(n)


def test_hadamard_closed_forms():
    n = 128
    # a unit vector e_j maps to column j of H times n^-1/2: +-bf16(128^-1/2)
    one = _exact_bf16(1, 0, n)
    assert one == 0.08837890625           # 128^-1/2 = 0.0883883..., nearest bf16 181 * 2^-11
    for j in (0, 1, 77, 127):
        x = np.zeros(n, dtype=np.float32)
        x[j] = 1.0
        got = bf16_values(oracle.hadamard_bf16(to_bf16_bits(x)[None])[0])
        assert np.array_equal(got, scipy_linalg.hadamard(n)[:, j] * one)
    # a constant vector c maps to sqrt(n) c e_0: 0.75 * 128^1/2 = 8.485..., nearest bf16 8.5
    got = bf16_values(oracle.hadamard_bf16(to_bf16_bits(np.full(n, 0.75))[None])[0])
    assert got[0] == 8.5 and not got[1:].any() and not np.signbit(got[1:]).any()


def test_hadamard_rejects_rows_beyond_its_exact_range():
    x = np.zeros(128, dtype=np.float32)
    x[0], x[1] = 1e30, 1e-30
    with pytest.raises(ValueError):
        oracle.hadamard_bf16(to_bf16_bits(x)[None])


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


PRODUCER_MUTANTS = {12: "Hadamard sign from popcount(i ^ j)", 13: "ties away from zero", 14: "scale for a max of 240"}


@pytest.mark.parametrize("mutant", sorted(PRODUCER_MUTANTS), ids=lambda m: PRODUCER_MUTANTS[m].replace(" ", "_"))
def test_producer_mutant_is_caught(mutant):
    """Each planted mistake in the producer's oracle fails at least one pin."""
    path = oracle.mutant_build(mutant)
    oracle._lib(mutant, path)
    oracle._LIBS[mutant] = oracle._LIBS[path]
    failed = []
    for pin in (pin_hadamard_matrix, pin_hadamard_exact_rounding, pin_e4m3_ties, pin_act_quant):
        try:
            pin(mutant=mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({PRODUCER_MUTANTS[mutant]}) passed every pin"
