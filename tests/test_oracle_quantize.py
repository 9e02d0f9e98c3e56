"""Pins of the oracle's NVFP4 block quantiser: exact round trips on exactly
representable inputs, brute-force nearest-code checks, special blocks, and the
relation between the global-one and per-token modes."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import quantize as Q


def _exact_row(rng, nblocks, exps, sign=True):
    """Blocks of E2M1 grid values times 2**e, each block containing a +-6."""
    codes = rng.integers(0, 8, size=(nblocks, 16))
    codes[:, 0] = 7
    vals = F.E2M1_MAGNITUDES[codes]
    if sign:
        vals = vals * np.where(rng.random((nblocks, 16)) < 0.5, -1.0, 1.0)
    return (vals * (2.0 ** exps)[:, None]).reshape(-1).astype(np.float32)


def test_global_one_roundtrip_exact():
    # block max 6 * 2^e with 2^e an E4M3 value: scale encodes exactly, codes too
    rng = np.random.default_rng(0)
    exps = rng.integers(-6, 8, size=32).astype(np.float64)
    x = _exact_row(rng, 32, exps)[None, :]
    xq, xsf, xs = Q.quantize_activations(x, "global_one")
    assert xs.tolist() == [1.0]
    assert np.array_equal(F.e4m3_decode(xsf[0]), 2.0 ** exps)
    deq = Q.dequantize_rows(xq, xsf) * xs[:, None]
    assert np.array_equal(deq, x.astype(np.float64))


def test_per_token_roundtrip_exact():
    # one block holds the row max 6 * 2^emax; g_enc = 448 * 2^-emax exactly, so
    # every block scale 448 * 2^(e - emax) is an E4M3 value for e - emax >= -14
    rng = np.random.default_rng(1)
    rows, rel_exps = [], []
    for r in range(6):
        emax = int(rng.integers(-4, 6))
        exps = emax - rng.integers(0, 14, size=24).astype(np.float64)
        exps[3] = emax
        rows.append(_exact_row(rng, 24, exps))
        rel_exps.append(exps - emax)
    x = np.stack(rows)
    xq, xsf, xs = Q.quantize_activations(x, "per_token")
    # block scales are exactly 448 * 2^(e - emax) and the codes reproduce the grid values
    assert np.array_equal(F.e4m3_decode(xsf), 448.0 * 2.0 ** np.stack(rel_exps))
    grid_vals = Q.dequantize_rows(xq, xsf) / np.repeat(F.e4m3_decode(xsf), 16, axis=1)
    want = x.astype(np.float64) / np.repeat(2.0 ** (np.stack(rel_exps)
                                                    + np.log2(np.abs(x).max(1) / 6)[:, None]),
                                            16, axis=1)
    assert np.array_equal(grid_vals, want)
    # the decoded values equal x up to the rounding of xs = amax / 2688 (2^-24 relative)
    deq = Q.dequantize_rows(xq, xsf) * xs.astype(np.float64)[:, None]
    assert np.all(np.abs(deq - x) <= np.abs(x) * 2.0 ** -23)
    # per-token decode scale = amax / (448*6)
    assert np.array_equal(xs, (np.abs(x).max(1) / np.float32(2688)).astype(np.float32))


def test_zero_block_and_zero_row():
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, 16:32] = 3.0
    for mode in ("global_one", "per_token"):
        xq, xsf, xs = Q.quantize_activations(x, mode)
        assert xsf[0].tolist() == [0, 0, 0, 0]
        assert xq[0].tolist() == [0] * 32
        assert xsf[1, 0] == 0 and xsf[1, 2] == 0
    _, _, xs = Q.quantize_activations(x, "per_token")
    assert xs[0] == 1.0          # amax == 0 -> unit scales


def test_constant_block_maps_to_six():
    # a block of equal values c: s = c/6 * g, q ~= s, c * g / q ~= 6 -> code 7
    for c in [0.1, 1.0, 3.3, 100.0]:
        x = np.full((1, 16), c, dtype=np.float32)
        codes, q = Q.quantize_blocks(x, np.float32(1))
        qv = F.e4m3_decode(q)[0, 0]
        ratio = c / qv
        expect = F.e2m1_encode(np.array([np.float32(c) * np.float32(np.float32(1) / np.float32(qv))]))[0]
        assert np.all(codes == expect)
        if abs(ratio - 6.0) < 0.5:
            assert np.all(codes == 7)


def test_codes_are_nearest_after_scaling():
    # brute force: every code is the E2M1 value nearest to x * inv, where inv
    # comes from the block's decoded scale; the scale is e4m3(max/6 * g)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 256)).astype(np.float32) * 3
    g = np.float32(0.37)
    codes, q = Q.quantize_blocks(x, g)
    bamax = np.abs(x.reshape(8, 16, 16)).max(2)
    s_ref = ((bamax / np.float32(6)).astype(np.float32) * g).astype(np.float32)
    assert np.array_equal(q, F.e4m3_encode(s_ref))
    qv = F.e4m3_decode(q).astype(np.float32)
    inv = (g / qv).astype(np.float32)
    v = (x.reshape(8, 16, 16) * inv[:, :, None]).astype(np.float64)
    allv = F.e2m1_decode(np.arange(16, dtype=np.uint8))
    d = np.abs(v[..., None] - allv)
    got = np.abs(v - F.e2m1_decode(codes.reshape(8, 16, 16)))
    assert np.all((got == d.min(-1)) | (np.abs(v) > 6))


def test_global_vs_per_token_same_values():
    # both modes approximate the same row; with the per-token scale the
    # element error is at most half an E2M1 step of the block, ie
    # |x - deq| <= max|block|/6 * 1 (step near 6 is 2) * (1 + e4m3 rounding)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((16, 512)).astype(np.float32)
    for mode in ("global_one", "per_token"):
        xq, xsf, xs = Q.quantize_activations(x, mode)
        deq = Q.dequantize_rows(xq, xsf) * xs.astype(np.float64)[:, None]
        bamax = np.abs(x.reshape(16, 32, 16)).max(2)
        bound = np.repeat(bamax / 6.0 * 1.0 * (1 + 2 ** -3), 16, axis=1) + 1e-30
        assert np.all(np.abs(deq - x) <= bound)
    a = Q.quantize_activations(x, "global_one")
    b = Q.quantize_activations(x, "per_token")
    da = Q.dequantize_rows(a[0], a[1]) * a[2][:, None]
    db = Q.dequantize_rows(b[0], b[1]) * b[2][:, None]
    rel = np.linalg.norm(da - db) / np.linalg.norm(x)
    assert rel < 0.15


def test_weight_alpha_and_shapes():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((32, 64)) * 0.02).astype(np.float32)
    data, sf, alpha = Q.quantize_weight(w)
    assert data.shape == (32, 32) and sf.shape == (32, 4)
    assert alpha == np.float32(np.float32(np.abs(w).max()) / np.float32(2688))
    deq = Q.dequantize_rows(data, sf) * np.float64(alpha)
    assert np.linalg.norm(deq - w) / np.linalg.norm(w) < 0.12
    # the block holding the matrix max gets scale 448 (max|w| maps to 6 * 448)
    r, c = np.unravel_index(np.abs(w).argmax(), w.shape)
    assert F.e4m3_decode(sf[r, c // 16]) == 448.0


def test_k_not_multiple_of_16_rejected():
    with pytest.raises(ValueError):
        Q.quantize_blocks(np.zeros((1, 8), np.float32), np.float32(1))


def test_global_scales_zero_amax():
    ge, gd = Q.global_scales(np.array([0.0, 2688.0], dtype=np.float32))
    assert ge.tolist() == [1.0, 1.0] and gd.tolist() == [1.0, 1.0]
