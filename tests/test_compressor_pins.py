"""Pins for the oracle of the V4.1 compressor ("DeepSeek-V4.1-Flash-NVFP4
inference/model.py", Compressor.forward and RMSNorm.forward): per channel, the
softmax over a group's r tokens of their gate scores weights their kv values;
the pooled row is RMS-normalised.  Checked against closed forms, the norm's
defining property, and the agreement of the prefill and decode forms."""
import numpy as np
import pytest
import torch

import oracle

EPS = 1e-6


def rows(rng, S, D, scale=1.0):
    return (rng.normal(size=(S, D)) * scale).astype(np.float32)


def rms(v):
    return np.sqrt(np.mean(v * v, axis=-1))


def to_bf16(v):
    """The cast to the activation dtype: fp32 then bf16, nearest even (torch's cast)."""
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).bfloat16().double().numpy()


def pin_equal_scores_give_the_mean(mutant=0):
    rng = np.random.default_rng(1)
    r, D = 4, 64
    kv = rows(rng, 3 * r, D)
    score = np.zeros_like(kv)  # equal gates: the plain mean of the group, then the norm
    out = oracle.compress_prefill(kv, score, r, np.ones(D, np.float32), EPS, mutant=mutant)
    mean = to_bf16(kv.astype(np.float64).reshape(3, r, D).mean(axis=1))
    want = mean / np.sqrt((mean * mean).mean(axis=1, keepdims=True) + EPS)
    assert np.allclose(out, want, rtol=1e-12, atol=1e-12)


def pin_dominant_gate_selects_a_token(mutant=0):
    rng = np.random.default_rng(2)
    r, D = 4, 32
    kv = rows(rng, r, D)
    score = np.full((r, D), -np.inf, dtype=np.float32)
    pick = rng.integers(0, r, size=D)
    score[pick, np.arange(D)] = 0.0  # channel d takes token pick[d] alone
    out = oracle.compress_prefill(kv, score, r, np.ones(D, np.float32), EPS, mutant=mutant)[0]
    c = to_bf16(kv[pick, np.arange(D)])
    assert np.allclose(out, c / np.sqrt(np.mean(c * c) + EPS), rtol=1e-12, atol=1e-12)


def pin_norm_property(mutant=0):
    rng = np.random.default_rng(3)
    r, D = 2, 128
    kv, score = rows(rng, 8, D, 5.0), rows(rng, 8, D, 3.0)
    w = rng.uniform(0.5, 2.0, size=D).astype(np.float32)
    out = oracle.compress_prefill(kv, score, r, w, 0.0, mutant=mutant)
    assert np.allclose(rms(out / w), 1.0, rtol=1e-12)  # unit RMS before the weight


def pin_decode_matches_prefill(mutant=0):
    """The token stream compressed by one prefill equals a shorter prefill
    followed by decode steps (the partial group carried in the state)."""
    rng = np.random.default_rng(4)
    r, D, S = 4, 16, 23
    kv, score = rows(rng, S, D), rows(rng, S, D)
    w = rng.uniform(0.5, 2.0, size=D).astype(np.float32)
    whole = oracle.compress_prefill(kv, score, r, w, EPS, mutant=mutant)
    for split in (1, 6, 8, 13):
        st = oracle.CompressorState(r, D)
        got = list(oracle.compress_prefill(kv[:split], score[:split], r, w, EPS, st, mutant=mutant))
        for pos in range(split, S):
            o = oracle.compress_decode(kv[pos], score[pos], pos, r, w, EPS, st, mutant=mutant)
            if o is not None:
                got.append(o)
        assert len(got) == len(whole)
        assert np.allclose(np.array(got), whole, rtol=1e-12, atol=1e-12), split


PINS = (pin_equal_scores_give_the_mean, pin_dominant_gate_selects_a_token, pin_norm_property,
        pin_decode_matches_prefill)


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


def test_weights_sum_to_one():
    """A constant kv row pools to itself whatever the gates (then the norm)."""
    rng = np.random.default_rng(5)
    r, D = 8, 32
    kv = np.tile(rng.normal(size=(1, D)).astype(np.float32), (r, 1))
    out = oracle.compress_prefill(kv, rows(rng, r, D, 10.0), r, np.ones(D, np.float32), EPS)[0]
    c = to_bf16(kv[0])
    assert np.allclose(out, c / np.sqrt(np.mean(c * c) + EPS), rtol=1e-10)


def test_incomplete_groups_yield_nothing():
    rng = np.random.default_rng(6)
    st = oracle.CompressorState(4, 8)
    assert oracle.compress_prefill(rows(rng, 3, 8), rows(rng, 3, 8), 4, np.ones(8, np.float32), EPS, st).shape == (0, 8)
    assert oracle.compress_decode(rows(rng, 1, 8)[0], rows(rng, 1, 8)[0], 3, 4, np.ones(8, np.float32), EPS, st) is not None
    assert oracle.compress_decode(rows(rng, 1, 8)[0], rows(rng, 1, 8)[0], 4, 4, np.ones(8, np.float32), EPS, st) is None


COMPRESSOR_MUTANTS = {15: "softmax over channels", 16: "norm by the sum", 17: "decode slot off by one"}


@pytest.mark.parametrize("mutant", sorted(COMPRESSOR_MUTANTS), ids=lambda m: COMPRESSOR_MUTANTS[m].replace(" ", "_"))
def test_compressor_mutant_is_caught(mutant):
    """Each planted mistake in the compressor's oracle fails at least one pin."""
    path = oracle.mutant_build(mutant)
    oracle._lib(mutant, path)
    oracle._LIBS[mutant] = oracle._LIBS[path]
    failed = []
    for pin in PINS:
        try:
            pin(mutant=mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({COMPRESSOR_MUTANTS[mutant]}) passed every pin"
