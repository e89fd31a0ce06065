"""Pins of the oracle's element codecs (e2m1, e4m3fn, e8m0, bf16 rounding).

Independent references: torch's own float8_e4m3fn / float8_e8m0fnu / bfloat16
casts (library routines, run only), a generic minifloat decoder that is first
checked against torch on e4m3fn and e5m2 and then applied to e2m1, and the
round-to-nearest-even tie table of the e2m1 grid.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def minifloat(code, ebits, mbits, bias):
    """Generic sign/exponent/mantissa decoder (no NaN/inf handling)."""
    s = (code >> (ebits + mbits)) & 1
    e = (code >> mbits) & ((1 << ebits) - 1)
    m = code & ((1 << mbits) - 1)
    if e == 0:
        v = m / (1 << mbits) * 2.0 ** (1 - bias)
    else:
        v = (1 + m / (1 << mbits)) * 2.0 ** (e - bias)
    return -v if s else v


def test_minifloat_reference_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    e4 = codes.view(torch.float8_e4m3fn).float().tolist()
    e5 = codes.view(torch.float8_e5m2).float().tolist()
    for c in range(256):
        if not math.isnan(e4[c]):
            assert minifloat(c, 4, 3, 7) == e4[c]
        if not (math.isnan(e5[c]) or math.isinf(e5[c])):
            assert minifloat(c, 5, 2, 15) == e5[c]


def test_e2m1_decode_table():
    got = [oracle.e2m1_decode(c) for c in range(16)]
    assert got == [minifloat(c, 2, 1, 1) for c in range(16)]
    # the e2m1 grid: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives
    assert got[:8] == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert all(got[8 + i] == -got[i] for i in range(8))
    assert math.copysign(1.0, got[8]) == -1.0


def test_e4m3_decode_all_codes_vs_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().tolist()
    for c in range(256):
        v = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c] and math.copysign(1, v) == math.copysign(1, ref[c]), c
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e8m0_decode_all_codes_vs_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().tolist()
    for c in range(256):
        v = oracle.e8m0_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(v)
        else:
            assert v == ref[c], c


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.normal(0, 50, 4000), rng.normal(0, 0.01, 2000), rng.uniform(-448, 448, 2000),
        np.array([0.0, 2.0 ** -10, 3 * 2.0 ** -11, 447.9, 448.0, 450.0, 463.9]),
    ]).astype(np.float32)
    # exact midpoints between neighbouring e4m3 values: ties go to the even code
    grid = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in vals], np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_saturates_and_keeps_sign():
    assert oracle.e4m3_encode(1e6) == 0x7E
    assert oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(465.0) == 0x7E  # torch gives NaN here; satfinite keeps 448
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-1e-9) == 0x80
    assert oracle.e4m3_encode(0.0) == 0x00


def test_e2m1_encode_tie_table():
    # round-to-nearest-even on the e2m1 grid: a midpoint goes to the even mantissa
    ties = {0.25: 0.0, 0.75: 1.0, 1.25: 1.0, 1.75: 2.0, 2.5: 2.0, 3.5: 4.0, 5.0: 4.0}
    for v, want in ties.items():
        assert oracle.e2m1_decode(oracle.e2m1_encode(v)) == want
        assert oracle.e2m1_decode(oracle.e2m1_encode(-v)) == -want
    assert oracle.e2m1_encode(7.0) == 7 and oracle.e2m1_encode(1e9) == 7  # saturate at 6
    assert oracle.e2m1_encode(-0.0) == 8


def test_e2m1_encode_roundtrip_and_monotone():
    for c in range(16):
        v = oracle.e2m1_decode(c)
        if v == 0.0:
            continue
        assert oracle.e2m1_encode(v) == c
    xs = np.linspace(-8, 8, 4001)
    vals = [oracle.e2m1_decode(oracle.e2m1_encode(float(x))) for x in xs]
    assert all(a <= b for a, b in zip(vals, vals[1:]))
    # nearest-value property: no grid point is strictly closer than the chosen one
    grid = [oracle.e2m1_decode(c) for c in range(16)]
    for x, v in zip(xs, vals):
        if abs(x) <= 6:
            assert abs(x - v) <= min(abs(x - g) for g in grid) + 1e-12


def test_round_bf16_matches_torch_on_fp32_inputs():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-3, 1000),
                           rng.normal(0, 1e30, 500)]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.bfloat16).double().numpy()
    got = np.array([oracle.round_bf16(float(v)) for v in vals])
    np.testing.assert_array_equal(got, ref)
    bits = oracle.bf16_bits(vals.astype(np.float64))
    np.testing.assert_array_equal(oracle.bf16_values(bits), ref)


def test_round_bf16_ties_to_even_from_fp64():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to even (1.0)
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    # a value just above the tie rounds up, even when fp32 would first round it onto the tie
    assert oracle.round_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40) == 1.0 + 2.0 ** -7
