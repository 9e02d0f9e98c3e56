"""NVFP4 16-wide block quantiser.

Sources:
* Megatron-Core ``core.inference.moe.flashinfer_nvfp4`` (Data):
  ``NVFP4_BLOCK_SIZE = 16``, ``FLOAT4_E2M1_MAX = 6.0``,
  ``FLOAT8_E4M3_MAX = 448.0``; ``_global_encode_scale`` returns "the
  one-element NVFP4 global encode scale for a weight matrix";
  ``quantize_routed_nvfp4_input`` returns packed E2M1 ``[tokens, H/2]``, linear
  block scales ``[tokens, H/16]`` and FP32 per-token scales ``[tokens]``.
* FlashInfer ``fused_moe.CudnnGroupedGemmNvfp4Config`` (Activations): the
  activation pack with token-major E4M3 block scales and a global scale of one.
* vLLM ``flashinfer_utils.quantize_nvfp4_per_token_input``: "one FP32 decode
  scale per token", linear scale-factor layout.

Readings (the pages name the scales but print no formula):
* global encode scale ``g_enc = (448 * 6) / amax`` and decode scale
  ``g_dec = amax / (448 * 6)``, both single IEEE float32 divisions; ``amax == 0``
  gives ``g_enc = g_dec = 1``. For weights amax runs over the whole expert
  matrix and ``alpha = g_dec``; per token it runs over the token's row and the
  per-token scale is ``g_dec``; with "a global scale of one" both are 1.
* per 16-block, in float32 and in this order:
  ``s = (max|x| / 6) * g_enc``; ``q = e4m3(s)``;
  ``inv = 0 if q == 0 else g_enc / q``; ``code_i = e2m1(x_i * inv)``.
  The dequantised value is ``e2m1(code) * e4m3(q) * g_dec``.
"""
from __future__ import annotations

import numpy as np

from .formats import (E2M1_MAX, E4M3_MAX, e2m1_decode, e2m1_encode, e4m3_decode,
                      e4m3_encode, pack_e2m1, unpack_e2m1)

BLOCK = 16
F32 = np.float32
GLOBAL_NUMERATOR = F32(E4M3_MAX * E2M1_MAX)   # 2688


def global_scales(amax: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(g_enc, g_dec) float32 from float32 amax; amax == 0 -> (1, 1)."""
    amax = np.asarray(amax, dtype=F32)
    safe = np.where(amax > 0, amax, F32(1))
    g_enc = np.where(amax > 0, GLOBAL_NUMERATOR / safe, F32(1)).astype(F32)
    g_dec = np.where(amax > 0, safe / GLOBAL_NUMERATOR, F32(1)).astype(F32)
    return g_enc, g_dec


def quantize_blocks(x: np.ndarray, g_enc) -> tuple[np.ndarray, np.ndarray]:
    """float32 x [rows, K] (K % 16 == 0), g_enc scalar or [rows] float32.

    Returns (codes uint8 [rows, K], scales uint8 [rows, K/16]).
    """
    x = np.asarray(x, dtype=F32)
    rows, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    g = np.broadcast_to(np.asarray(g_enc, dtype=F32).reshape(-1, 1), (rows, 1))
    xb = x.reshape(rows, K // BLOCK, BLOCK)
    bamax = np.abs(xb).max(axis=2).astype(F32)                  # [rows, K/16]
    s = ((bamax / F32(E2M1_MAX)).astype(F32) * g).astype(F32)
    q = e4m3_encode(s)
    qf = e4m3_decode(q).astype(F32)
    safe = np.where(qf == 0, F32(1), qf)
    inv = np.where(qf == 0, F32(0), (g / safe).astype(F32)).astype(F32)
    v = (xb * inv[:, :, None]).astype(F32)
    codes = e2m1_encode(v).reshape(rows, K)
    return codes, q


def quantize_rows(x: np.ndarray, g_enc) -> tuple[np.ndarray, np.ndarray]:
    """Block-quantise and pack: (data uint8 [rows, K/2], scales uint8 [rows, K/16])."""
    codes, q = quantize_blocks(x, g_enc)
    return pack_e2m1(codes), q


def quantize_activations(x_bf16: np.ndarray, mode: str):
    """Activation pack of BF16 hidden states (given as their float32 values).

    mode "global_one": global scale one, per-token scale array of ones.
    mode "per_token":  one FP32 decode scale per token.
    Returns (xq uint8 [M, H/2], xsf uint8 [M, H/16], xs float32 [M]).
    """
    x = np.asarray(x_bf16, dtype=F32)
    M = x.shape[0]
    if mode == "global_one":
        g_enc = np.ones(M, dtype=F32)
        xs = np.ones(M, dtype=F32)
    elif mode == "per_token":
        amax = np.abs(x).max(axis=1).astype(F32) if x.shape[1] else np.zeros(M, F32)
        g_enc, xs = global_scales(amax)
    else:
        raise ValueError(mode)
    xq, xsf = quantize_rows(x, g_enc)
    return xq, xsf, xs


def quantize_weight(w_bf16: np.ndarray):
    """One expert matrix [rows, cols] -> (data [rows, cols/2], sf [rows, cols/16], alpha)."""
    w = np.asarray(w_bf16, dtype=F32)
    amax = F32(np.abs(w).max()) if w.size else F32(0)
    g_enc, g_dec = global_scales(np.array([amax], dtype=F32))
    data, sf = quantize_rows(w, g_enc[0])
    return data, sf, F32(g_dec[0])


def dequantize_rows(data: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """float64 e2m1(code) * e4m3(scale) for every element (global scale not applied)."""
    codes = unpack_e2m1(data)
    rows, K = codes.shape
    vals = e2m1_decode(codes).reshape(rows, K // BLOCK, BLOCK)
    return (vals * e4m3_decode(sf)[:, :, None]).reshape(rows, K)
