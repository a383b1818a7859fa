"""Pins for the oracle of the V4.1 index-key producer ("DeepSeek-V4.1-Flash-NVFP4
inference/model.py", Indexer.forward in the layer that owns the index keys:
k_norm(wk(latent)), apply_rotary_emb on the last rope_head_dim values at the
group's first position, the key quantisation, the cache write).  The pins
rest on the norm's definition evaluated here in numpy with an independent
single rounding to bf16, on the already pinned rotation (test_rope_pins) and
quantiser (test_producer_pins) composed by hand, and on invariants: position
0 rotates nothing, the rotation touches only the last rope_head_dim values
and keeps each pair's length."""
import numpy as np
import pytest
import torch

import oracle
from tolerances import bf16_round

EPS = 1e-6
D = 128
ROPE = oracle.Rope()  # released config: 64 rotated dims, theta 160000, YaRN factor 16 over 65536


def bf16_bits(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double().numpy()


def f64_to_bits(v):
    return bf16_bits(bf16_round(np.asarray(v, dtype=np.float64)).astype(np.float32))


def rows(seed, n, scale=1.0):
    rng = np.random.default_rng(seed)
    return bf16_bits(rng.normal(size=(n, D)) * scale), rng.uniform(0.5, 2.0, size=D).astype(np.float32)


def pin_position_zero_is_the_normalised_row(mutant=0):
    """At position 0 every angle is 0: the key is bf16(weight * x / sqrt(mean x^2 + eps)),
    and its codes and scale are act_quant of that key (rows at three scales,
    one small enough for eps to matter)."""
    for scale in (1.0, 3e-4, 40.0):
        xs, w = rows(1, 6, scale)
        for x in xs:
            codes, s, k = oracle.index_key(x, w, EPS, 0, ROPE, mutant)
            xv = bits_to_f64(x)
            want = f64_to_bits(w.astype(np.float64) * xv / np.sqrt(np.mean(xv * xv) + EPS))
            assert np.array_equal(k, want), scale
            wc, ws_ = oracle.act_quant_rows(k[None])
            assert np.array_equal(codes, wc[0]) and s == ws_[0]


def pin_rotation_is_the_pinned_rope_on_the_last_dims(mutant=0):
    """At position p the key is the position-0 key with its last 64 values
    rotated by the (separately pinned) rotary embedding at p and rounded to
    bf16 again; the first 64 values are untouched."""
    xs, w = rows(2, 5)
    for p in (1, 4, 4096, 131068):
        for x in xs:
            _, _, k0 = oracle.index_key(x, w, EPS, 0, ROPE, mutant)
            _, _, kp = oracle.index_key(x, w, EPS, p, ROPE, mutant)
            assert np.array_equal(kp[:D - ROPE.dim], k0[:D - ROPE.dim]), p
            rot = oracle.apply_rope(bits_to_f64(k0[D - ROPE.dim:]), ROPE, p)
            assert np.array_equal(kp[D - ROPE.dim:], f64_to_bits(rot)), p


def pin_rotation_keeps_pair_lengths(mutant=0):
    xs, w = rows(3, 4)
    for x in xs:
        _, _, k0 = oracle.index_key(x, w, EPS, 0, ROPE, mutant)
        _, _, kp = oracle.index_key(x, w, EPS, 777, ROPE, mutant)
        a = bits_to_f64(k0[D - ROPE.dim:]).reshape(-1, 2)
        b = bits_to_f64(kp[D - ROPE.dim:]).reshape(-1, 2)
        la, lb = np.hypot(a[:, 0], a[:, 1]), np.hypot(b[:, 0], b[:, 1])
        assert np.all(np.abs(la - lb) <= 2.0 ** -7 * la + 1e-30)


ALL = [pin_position_zero_is_the_normalised_row, pin_rotation_is_the_pinned_rope_on_the_last_dims,
       pin_rotation_keeps_pair_lengths]


@pytest.mark.parametrize("pin", ALL, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_unit_norm_and_weight():
    """With weight 1 the normalised key has unit RMS up to its bf16 rounding."""
    xs, _ = rows(4, 8)
    for x in xs:
        _, _, k = oracle.index_key(x, np.ones(D, np.float32), 0.0, 0, ROPE)
        kv = bits_to_f64(k)
        assert abs(np.sqrt(np.mean(kv * kv)) - 1.0) <= 2.0 ** -8


KEY_MUTANTS = {22: "rotation on the first dims", 23: "norm without eps"}


@pytest.mark.parametrize("mutant", sorted(KEY_MUTANTS), ids=lambda m: KEY_MUTANTS[m].replace(" ", "_"))
def test_index_key_mutant_is_caught(mutant):
    path = oracle.mutant_build(mutant)
    oracle._lib(mutant, path)
    oracle._LIBS[mutant] = oracle._LIBS[path]
    failed = []
    for pin in ALL:
        try:
            pin(mutant=mutant)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"mutant {mutant} ({KEY_MUTANTS[mutant]}) passed every pin"
