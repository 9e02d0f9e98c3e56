"""Pins of the oracle's element codecs against format definitions, hand-worked
cases (tests/golden) and an independent library routine (torch's float8/bf16
conversions)."""
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_constants_match_pages():
    consts = {r[0]: float(r[1]) for r in _rows("nvfp4_constants.txt")}
    assert F.E2M1_MAX == consts["FLOAT4_E2M1_MAX"]
    assert F.E4M3_MAX == consts["FLOAT8_E4M3_MAX"]
    assert F.E2M1_MAGNITUDES.max() == consts["FLOAT4_E2M1_MAX"]
    assert np.nanmax(F.E4M3_TABLE) == consts["FLOAT8_E4M3_MAX"]


def test_e2m1_table():
    for code, val in _rows("e2m1_values.txt"):
        v = F.e2m1_decode(np.array([int(code)]))[0]
        assert v == float(val)
        assert np.signbit(v) == val.startswith("-")


def test_e2m1_roundtrip_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    vals = F.e2m1_decode(codes).astype(np.float32)
    assert np.array_equal(F.e2m1_encode(vals), codes)


def test_e2m1_round_cases():
    for x, code in _rows("e2m1_round_cases.txt"):
        got = F.e2m1_encode(np.array([np.float32(x)]))[0]
        assert got == int(code), (x, got, code)


def test_e2m1_nearest_brute_force():
    # every code is the nearest grid point (by brute force over all 16 codes)
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(20000) * 3).astype(np.float32)
    codes = F.e2m1_encode(x)
    allv = F.e2m1_decode(np.arange(16, dtype=np.uint8))
    d = np.abs(x.astype(np.float64)[:, None] - allv[None, :])
    best = d.min(axis=1)
    got = np.abs(x.astype(np.float64) - F.e2m1_decode(codes))
    sat = np.abs(x) > 6
    assert np.all(got[~sat] == best[~sat])
    assert np.all((codes[sat] & 7) == 7)
    assert np.all(np.signbit(F.e2m1_decode(codes)) == np.signbit(x))


def test_e4m3_golden_cases():
    for x, hexcode in _rows("e4m3_cases.txt"):
        got = F.e4m3_encode(np.array([np.float32(x)]))[0]
        assert got == int(hexcode, 16), (x, hex(got), hexcode)


def test_e4m3_table_against_torch():
    b = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    ours = F.E4M3_TABLE
    nan = np.isnan(b)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(b[~nan].astype(np.float64), ours[~nan])


def test_e4m3_roundtrip_all_bytes():
    codes = np.arange(256, dtype=np.uint8)
    ok = ~np.isnan(F.E4M3_TABLE)
    vals = F.E4M3_TABLE[ok].astype(np.float32)
    assert np.array_equal(F.e4m3_encode(vals), codes[ok])


def test_e4m3_rne_against_torch():
    # torch's float32 -> float8_e4m3fn conversion rounds to nearest even; within
    # the finite range it must agree with the oracle everywhere
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.uniform(0, 448, 50000), np.exp(rng.uniform(np.log(2e-4), np.log(448), 50000)),
        # exact midpoints between neighbouring E4M3 values
        (F.E4M3_POSITIVE[:-1] + F.E4M3_POSITIVE[1:]) / 2,
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(x), ref)
    assert np.array_equal(F.e4m3_encode(-x), ref | 0x80)


def test_e4m3_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, np.inf], dtype=np.float32)
    assert np.all(F.e4m3_encode(x) == 0x7E)
    assert np.all(F.e4m3_encode(-x) == 0xFE)


def test_bf16_round_against_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
                        [0.0, -0.0, 1.0, 3.0e38]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(F.bf16_round(x.astype(np.float64)), ref)
    assert np.array_equal(F.bits_to_bf16(F.bf16_to_bits(ref)), ref)


def test_bf16_round_ties_even():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: ties to the even mantissa (1.0)
    assert F.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert F.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2 * 2.0 ** -7
    # from float64 directly: a hair above the midpoint rounds up
    assert F.bf16_round(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1.0 + 2.0 ** -7


def test_pack_nibble_order():
    codes = np.array([[1, 2, 3, 4]], dtype=np.uint8)
    packed = F.pack_e2m1(codes)
    # even logical element in the low nibble (FlashInfer alphamoe_nvfp4_aligned_moe)
    assert packed.tolist() == [[0x21, 0x43]]
    assert np.array_equal(F.unpack_e2m1(packed), codes)


def test_nan_rejected():
    with pytest.raises(ValueError):
        F.e2m1_encode(np.array([np.nan], dtype=np.float32))
