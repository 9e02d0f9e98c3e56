"""Element codecs: E2M1 (FP4), E4M3 (float8_e4m3fn) and BF16.

Sources:
* Megatron-Core ``core.inference.moe.flashinfer_nvfp4`` (Data):
  ``FLOAT4_E2M1_MAX = 6.0`` and ``FLOAT8_E4M3_MAX = 448.0``.
* FlashInfer ``fused_moe.alphamoe_nvfp4_aligned_moe`` (description): two E2M1
  values per uint8 byte, the even logical value in the low nibble; scales are
  ``torch.float8_e4m3fn``.
* The bit layouts themselves (E2M1: 1 sign, 2 exponent, 1 mantissa bit, bias 1;
  E4M3 "fn": 1-4-3, bias 7, no infinities, S.1111.111 = NaN) follow the OCP
  Microscaling formats definition; the pages name the types but not the bits.

Rounding readings (the pages are silent): every encoder rounds to nearest,
ties to the even code, and saturates at the format's largest finite value.
The sign of an input that rounds to zero is kept (-0 encodes as code 8 in
E2M1).
"""
from __future__ import annotations

import numpy as np

# E2M1 magnitudes of codes 0..7: exponent field e (2 bits), mantissa m (1 bit);
# e == 0 -> subnormal m * 0.5, else (1 + m/2) * 2**(e-1).
E2M1_MAGNITUDES = np.array(
    [(m * 0.5) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
     for e in range(4) for m in range(2)], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0


def _e4m3_value(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
# non-negative finite values, ascending; position == code for codes 0x00..0x7E
E4M3_POSITIVE = E4M3_TABLE[:0x7F].copy()


def _round_to_grid(a: np.ndarray, grid: np.ndarray) -> np.ndarray:
    """Index of the nearest grid value to each a >= 0 (ties to the even index).

    ``grid`` is ascending and starts at 0; values at or above its last entry
    saturate to the last index. Distances are taken in float64, where they are
    exact for the float32 inputs used here.
    """
    a = np.asarray(a, dtype=np.float64)
    top = grid.size - 1
    lo = np.clip(np.searchsorted(grid, a, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0) & (hi != lo))
    idx = np.where(pick_hi, hi, lo)
    return np.where(a >= grid[top], top, idx)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """float32 values -> E2M1 codes (uint8, 0..15), RNE, saturating at +-6."""
    x = np.asarray(x, dtype=np.float32)
    if np.isnan(x).any():
        raise ValueError("NaN has no E2M1 encoding")
    mag = _round_to_grid(np.abs(x), E2M1_MAGNITUDES).astype(np.uint8)
    return (mag | (np.signbit(x).astype(np.uint8) << 3)).astype(np.uint8)


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    v = E2M1_MAGNITUDES[codes & 7]
    return np.where(codes & 8, -v, v)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """float32 values -> float8_e4m3fn bytes, RNE, saturating at +-448."""
    x = np.asarray(x, dtype=np.float32)
    mag = _round_to_grid(np.abs(x), E4M3_POSITIVE).astype(np.uint8)
    out = mag | (np.signbit(x).astype(np.uint8) << 7)
    return np.where(np.isnan(x), np.uint8(0x7F), out).astype(np.uint8)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """[..., K] codes -> [..., K/2] bytes; element 2i in the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 (or float32) values to the nearest BF16 value, ties to even.

    A BF16 value has 8 significant bits and the float32 exponent range; the
    result is returned as float64 holding that value exactly.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    m, e = np.frexp(x[nz])                 # x = m * 2**e, 0.5 <= |m| < 1
    e = np.maximum(e, -125)                # below 2**-126 the quantum is fixed
    q = np.ldexp(1.0, e - 8)
    out[nz] = np.rint(x[nz] / q) * q       # rint rounds half to even
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    big = np.abs(out) > 3.3895313892515355e38
    out[big] = np.copysign(np.inf, out[big])
    return np.where(x == 0, x, out)


def bf16_to_bits(v: np.ndarray) -> np.ndarray:
    """Exact BF16 values (float64) -> uint16 bit patterns."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def bits_to_bf16(b: np.ndarray) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
