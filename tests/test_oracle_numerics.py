"""Pins for the oracle's exact conversions (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from oracle.numerics import bf16_bits_to_f32, bf16_rn_bits, f16_rn, round_half_away, ulp


def test_round_half_away_hand_values():
    v = np.array([0.5, -0.5, 1.5, 2.5, -2.5, 0.49999997, -0.49999997, 3.0, -7.5, 7.4999995],
                 dtype=np.float32)
    want = [1, -1, 2, 3, -3, 0, 0, 3, -8, 7]
    assert list(round_half_away(v)) == want


def test_round_half_away_matches_decimal_rounding():
    # brute force against Python's decimal ROUND_HALF_UP (which rounds ties
    # away from zero in magnitude) on exact float32 values
    from decimal import ROUND_HALF_UP, Decimal
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(4000) * 50).astype(np.float32)
    v[:100] = np.round(v[:100]) + np.float32(0.5)   # exact halves
    got = round_half_away(v)
    for a, g in zip(v, got):
        ref = Decimal(float(a)).quantize(Decimal(1), rounding=ROUND_HALF_UP)
        assert int(ref) == g


def test_f16_rn_hand_values():
    assert f16_rn(np.float32(1) / np.float32(127)).view(np.uint16) == 0x2008
    assert f16_rn(np.float32(2.0 ** -25)).view(np.uint16) == 0x0000      # tie -> even (0)
    assert f16_rn(np.float32(3 * 2.0 ** -25)).view(np.uint16) == 0x0002  # tie -> even (2 * 2^-24)
    assert f16_rn(np.float32(2.0 ** -24)).view(np.uint16) == 0x0001      # smallest subnormal kept
    assert f16_rn(np.float32(1 + 2.0 ** -11)).view(np.uint16) == 0x3C00  # tie -> even
    assert f16_rn(np.float32(1 + 3 * 2.0 ** -11)).view(np.uint16) == 0x3C02


def test_f16_rn_matches_torch():
    rng = np.random.default_rng(2)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 10, 100000))).astype(np.float32)
    v = v[np.abs(v) < 65000]
    t = torch.from_numpy(v).to(torch.float16).numpy()
    assert np.array_equal(f16_rn(v).view(np.uint16), t.view(np.uint16))


def test_bf16_hand_values():
    f = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -2.0, 0.0], dtype=np.float32)
    assert list(bf16_rn_bits(f)) == [0x3F80, 0x3F80, 0x3F82, 0xC000, 0x0000]
    assert np.array_equal(bf16_bits_to_f32(np.array([0x3F80, 0xBF00], np.uint16)),
                          np.array([1.0, -0.5], np.float32))


def test_bf16_matches_torch():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-40, 40, 100000))).astype(np.float32)
    t = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_rn_bits(v), t)


@pytest.mark.parametrize("fmt,npdt", [("f16", np.float16), ("f32", np.float32)])
def test_ulp_matches_numpy_spacing(fmt, npdt):
    rng = np.random.default_rng(4)
    v = np.abs(rng.standard_normal(20000) * np.exp(rng.uniform(-12, 9, 20000))).astype(npdt)
    v = v[np.isfinite(v) & (v > 0)]
    # np.spacing(x) is the gap to the next larger value, which is the ulp of
    # the binade containing x
    assert np.array_equal(ulp(v.astype(np.float64), fmt), np.spacing(v).astype(np.float64))


def test_ulp_hand_values():
    assert ulp(1.0, "f16") == 2.0 ** -10
    assert ulp(1.5, "bf16") == 2.0 ** -7
    assert ulp(0.0, "f16") == 2.0 ** -24
    assert ulp(2.0 ** -15, "f16") == 2.0 ** -24
    assert ulp(65504.0, "f16") == 32.0
    assert ulp(1.0, "f32") == 2.0 ** -23


def test_parity_bound_never_tighter_than_fp16_ulp():
    y = np.array([1.0, 1000.0, 1e-3])
    b = oracle.parity_bound(y, np.zeros(3), "f32")
    assert np.array_equal(b, ulp(y, "f16"))
    b = oracle.parity_bound(y, np.zeros(3), "bf16")
    assert np.array_equal(b, ulp(y, "bf16"))
    b = oracle.parity_bound(np.array([2.0]), np.array([10.0]), "f16")
    assert b[0] == pytest.approx(1e-2 + 2.0 ** -9)
