"""Pins of the oracle's expert chain: brute-force GEMMs from independent decoders
(the golden E2M1 table, torch's float8_e4m3fn), activation identities, the
gate/up row order, and end-to-end invariants of the finalize."""
import math
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import formats as F
from oracle import moe as O
from oracle import plan as P
from oracle import quantize as Q

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _e2m1_table():
    with open(os.path.join(GOLD, "e2m1_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    return {int(c): float(v) for c, v in rows}


E2M1 = _e2m1_table()


def _e4m3(b):
    return float(torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])


def _val(packed_row, sf_row, h):
    byte = int(packed_row[h // 2])
    code = (byte >> 4) if h % 2 else (byte & 0xF)
    return E2M1[code] * _e4m3(sf_row[h // 16])


def _rand_pack(rng, rows, cols, pow2_scales=True):
    codes = rng.integers(0, 16, size=(rows, cols)).astype(np.uint8)
    if pow2_scales:
        # E4M3 bytes of 2^-3 .. 2^3 (mantissa 0): exact dyadic products
        sf = (((rng.integers(4, 11, size=(rows, cols // 16))) << 3)).astype(np.uint8)
    else:
        sf = rng.integers(0x08, 0x7E, size=(rows, cols // 16)).astype(np.uint8)
    return F.pack_e2m1(codes), sf


def _small_problem(seed, act="swiglu", M=3, H=32, I=16, E=3, k=2):
    rng = np.random.default_rng(seed)
    N1 = 2 * I if act == "swiglu" else I
    xq, xsf = _rand_pack(rng, M, H)
    xs = (2.0 ** rng.integers(-2, 3, size=M)).astype(np.float32)
    w1 = [(*_rand_pack(rng, N1, H), np.float32(2.0 ** int(rng.integers(-3, 1)))) for _ in range(E)]
    w2 = [(*_rand_pack(rng, H, I), np.float32(2.0 ** int(rng.integers(-3, 1)))) for _ in range(E)]
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    tw = rng.random((M, k)).astype(np.float32)
    W = O.ExpertWeights.from_packs(w1, w2, gated=(act == "swiglu"))
    return xq, xsf, xs, ids, tw, W, w1, w2


@pytest.mark.parametrize("act", ["swiglu", "relu2"])
def test_gemm1_brute_force_exact(act):
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(0, act)
    res = O.forward(xq, xsf, xs, ids, tw, W, act)
    M, k = ids.shape
    H = W.hidden
    N1 = w1[0][0].shape[0]
    t2r = res["plan"]["token_to_row"]
    for t in range(M):
        for j in range(k):
            l = int(ids[t, j])
            d1, s1, a1 = w1[l]
            row = t2r[t, j]
            for n in range(N1):
                acc = sum(_val(xq[t], xsf[t], h) * _val(d1[n], s1[n], h) for h in range(H))
                # dyadic operands: the sum, and y, are exact in float64
                assert res["preact"][row, n] == acc * float(xs[t]) * float(a1)


def test_gemm2_and_finalize_brute_force():
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(1, "swiglu")
    res = O.forward(xq, xsf, xs, ids, tw, W, "swiglu")
    M, k = ids.shape
    H, I = W.hidden, W.inter
    t2r = res["plan"]["token_to_row"]
    for t in range(M):
        acc = np.zeros(H, dtype=np.float32)
        for j in range(k):
            l = int(ids[t, j])
            row = t2r[t, j]
            ipacked = F.pack_e2m1(res["icodes"][row])
            d2, s2, a2 = w2[l]
            ref = np.array([
                sum(_val(ipacked, res["isf"][row], i) * _val(d2[h], s2[h], i) for i in range(I))
                for h in range(H)]) * float(a2)
            got = res["rows"][row]
            # the expert row is the BF16 rounding of the exact value
            bf = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16).double().numpy()
            assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 2.0 ** -133)
            assert np.mean(got == bf) > 0.95
            acc = (acc + (np.float32(tw[t, j]) * got.astype(np.float32)).astype(np.float32)).astype(np.float32)
        exp = torch.from_numpy(acc).to(torch.bfloat16).double().numpy()
        assert np.array_equal(res["out"][t], exp)


def test_requant_is_block_quantiser_of_bf16_intermediate():
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(2, "swiglu")
    for g2 in (1.0, 0.25, 3.0):
        res = O.forward(xq, xsf, xs, ids, tw, W, "swiglu", fc2_input_scale=g2)
        real = res["plan"]["row_to_slot"] >= 0
        h = res["act_bf16"][real]
        # h is exactly BF16 and is silu(g) * u of the pre-activations
        assert np.array_equal(F.bf16_round(h), h)
        y = res["preact"][real]
        I = W.inter
        with np.errstate(over="ignore"):
            ref = y[:, :I] / (1 + np.exp(-y[:, :I])) * y[:, I:]
        assert np.all(np.abs(h - ref) <= np.abs(ref) * 2.0 ** -8 + 2.0 ** -133)
        codes, sf = Q.quantize_blocks(h.astype(np.float32), np.float32(g2))
        assert np.array_equal(codes, res["icodes"][real])
        assert np.array_equal(sf, res["isf"][real])


def test_silu_identities():
    x = np.linspace(-30, 30, 1001)
    s = O.silu(x)
    assert O.silu(np.array([0.0]))[0] == 0.0
    # x*sigma(x) - (-x)*sigma(-x) = x*(sigma(x)+sigma(-x)) = x
    assert np.allclose(s - O.silu(-x), x, rtol=0, atol=1e-12)
    assert np.all(np.abs(O.silu(np.array([40.0, -40.0])) - [40.0, 0.0]) < 1e-15)
    # derivative at 0 is 1/2: silu(eps)/eps -> 1/2
    assert abs(O.silu(np.array([1e-8]))[0] / 1e-8 - 0.5) < 1e-7


def test_relu2_and_gate_zero():
    y = np.array([[-3.0, 2.0, 0.0, -0.5]])
    assert O.activation(y, "relu2", 4).tolist() == [[0.0, 4.0, 0.0, 0.0]]
    y = np.array([[0.0, 0.0, 5.0, -7.0]])    # gate 0 => 0 regardless of up
    assert O.activation(y, "swiglu", 2).tolist() == [[0.0, 0.0]]


def test_gate_up_row_order():
    # gate rows all 6.0, up rows all 1.0, activations all 1.0, alpha 1/16:
    # g = 16*6/16 = 6, u = 1 -> h = silu(6) * 1 (swapped halves give silu(1) * 6)
    H, I = 16, 16
    xq = F.pack_e2m1(np.full((1, H), 2, np.uint8))          # 1.0
    xsf = np.full((1, 1), 0x38, np.uint8)                    # scale 1.0
    gate = np.full((I, H), 7, np.uint8)                      # 6.0
    up = np.full((I, H), 2, np.uint8)                        # 1.0
    d1 = F.pack_e2m1(np.concatenate([gate, up]))
    s1 = np.full((2 * I, 1), 0x38, np.uint8)
    d2 = F.pack_e2m1(np.full((H, I), 2, np.uint8))
    s2 = np.full((H, 1), 0x38, np.uint8)
    W = O.ExpertWeights.from_packs([(d1, s1, np.float32(1 / 16))], [(d2, s2, np.float32(1))], True)
    res = O.forward(xq, xsf, np.ones(1, np.float32), np.zeros((1, 1), np.int32),
                    np.ones((1, 1), np.float32), W, "swiglu")
    h = res["act_bf16"][0]
    want = 6.0 / (1.0 + math.exp(-6.0))
    assert np.all(np.abs(h - want) < want * 2 ** -8)
    assert np.all(np.abs(h - 6.0 / (1.0 + math.exp(-1.0))) > 1.0)


def _cfg_problem(cfg):
    x = mi.hidden_bf16(cfg).float().numpy()
    ids, tw = mi.routing(cfg)
    xq, xsf, xs = Q.quantize_activations(x, cfg.scale_mode)
    w1 = [mi.expert_w1_bf16(cfg, l).float().numpy() for l in range(cfg.El)]
    w2 = [mi.expert_w2_bf16(cfg, l).float().numpy() for l in range(cfg.El)]
    W = O.ExpertWeights.from_bf16(w1, w2, cfg.gated)
    return x, ids, tw, xq, xsf, xs, W


def test_zero_weights_zero_output():
    cfg = mi.CONFIGS["tiny"]
    x, ids, tw, xq, xsf, xs, W = _cfg_problem(cfg)
    Z = O.ExpertWeights.from_bf16([np.zeros((cfg.N1, cfg.H), np.float32)] * cfg.El,
                                  [np.zeros((cfg.H, cfg.I), np.float32)] * cfg.El, True)
    res = O.forward(xq, xsf, xs, ids, tw, Z, "swiglu")
    assert np.all(res["out"] == 0)


def test_single_expert_weight_one_is_the_row():
    cfg = mi.CONFIGS["tiny"].with_(top_k=1)
    x, ids, tw, xq, xsf, xs, W = _cfg_problem(cfg)
    tw = np.ones_like(tw)
    res = O.forward(xq, xsf, xs, ids, tw, W, "swiglu")
    t2r = res["plan"]["token_to_row"][:, 0]
    assert np.array_equal(res["out"], res["rows"][t2r])


def test_tiny_end_to_end_close_to_bf16_math():
    # the NVFP4 path approximates the unquantised BF16 MoE within a few percent
    cfg = mi.CONFIGS["tiny"]
    x, ids, tw, xq, xsf, xs, W = _cfg_problem(cfg)
    res = O.forward(xq, xsf, xs, ids, tw, W, "swiglu")
    w1 = [mi.expert_w1_bf16(cfg, l).double().numpy() for l in range(cfg.El)]
    w2 = [mi.expert_w2_bf16(cfg, l).double().numpy() for l in range(cfg.El)]
    ref = np.zeros((cfg.M, cfg.H))
    for t in range(cfg.M):
        for j in range(cfg.top_k):
            l = ids[t, j]
            y = w1[l] @ x[t].astype(np.float64)
            h = O.silu(y[:cfg.I]) * y[cfg.I:]
            ref[t] += tw[t, j] * (w2[l] @ h)
    rel = np.linalg.norm(res["out"] - ref) / np.linalg.norm(ref)
    assert rel < 0.25, rel


def test_expert_parallel_shards_sum_to_full():
    cfg = mi.CONFIGS["decode_t4"].with_(H=256, I=128, E=16, top_k=4)
    x, ids, tw, xq, xsf, xs, W = _cfg_problem(cfg)
    full = O.forward(xq, xsf, xs, ids, tw, W, "swiglu")
    halves = []
    for off in (0, 8):
        Wh = O.ExpertWeights(8, W.hidden, W.inter, True, lambda l, o=off: W.get(l + o))
        halves.append(O.forward(xq, xsf, xs, ids, tw, Wh, "swiglu", local_expert_offset=off))
    s = halves[0]["out"] + halves[1]["out"]
    # each shard rounds its partial sum to BF16 once
    tol = (np.abs(halves[0]["out"]) + np.abs(halves[1]["out"]) + np.abs(full["out"])) * 2.0 ** -8
    assert np.all(np.abs(s - full["out"]) <= tol + 1e-30)


def test_unrouted_slots_contribute_nothing():
    cfg = mi.CONFIGS["decode_t4"].with_(H=256, I=128, E=16, top_k=4)
    x, ids, tw, xq, xsf, xs, W = _cfg_problem(cfg)
    ids2 = mi.with_unrouted(ids, 0.3, 3, cfg.E)
    tw2 = tw.copy()
    tw2[(ids2 < 0) | (ids2 >= cfg.E)] = np.nan     # scores of unrouted slots are ignored
    a = O.forward(xq, xsf, xs, ids2, tw2, W, "swiglu")
    keep = ~((ids2 < 0) | (ids2 >= cfg.E))
    tw3 = np.where(keep, tw, 0).astype(np.float32)
    b = O.forward(xq, xsf, xs, ids, tw3, W, "swiglu")
    assert np.all(np.isfinite(a["out"]))
    assert np.array_equal(a["out"], b["out"])


def test_forward_tokens_matches_forward():
    cfg = mi.CONFIGS["decode_t8"].with_(H=256, I=128, E=32, top_k=4)
    x, ids, tw, xq, xsf, xs, W = _cfg_problem(cfg)
    full = O.forward(xq, xsf, xs, ids, tw, W, "swiglu")
    sub = O.forward_tokens([1, 6], xq, xsf, xs, ids, tw, W, "swiglu")
    assert np.array_equal(sub["out"], full["out"][[1, 6]])


def test_plan_capacity_matches_plan_module():
    assert P.plan_capacity(4096, 8, 256) == 32768 + 127 * 256  # already a multiple of 128


def test_gelu_closed_forms():
    x = np.linspace(-8, 8, 401)
    g = O.gelu(x)
    # x*Phi(x) - (-x)*Phi(-x) = x, Phi(0) = 1/2, GELU(x) -> x and -> 0 in the tails
    assert np.allclose(g - O.gelu(-x), x, rtol=0, atol=1e-14)
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert abs(O.gelu(np.array([1e-9]))[0] / 1e-9 - 0.5) < 1e-8
    assert abs(O.gelu(np.array([10.0]))[0] - 10.0) < 1e-20 + 10.0 * 1e-15
    # Phi(1) = 0.841344746068543 (standard normal table)
    assert abs(O.gelu(np.array([1.0]))[0] - 0.841344746068543) < 1e-12


@pytest.mark.parametrize("act", ["relu", "silu", "identity", "gelu"])
def test_nongated_activations_elementwise(act):
    y = np.array([[-2.0, -0.5, 0.0, 0.5, 3.0]])
    h = O.activation(y, act, 5)
    if act == "relu":
        assert h.tolist() == [[0.0, 0.0, 0.0, 0.5, 3.0]]
    elif act == "identity":
        assert h.tolist() == y.tolist()
    elif act == "silu":
        assert np.array_equal(h, O.silu(y))
    else:
        assert np.array_equal(h, O.gelu(y))


def test_geglu_uses_gate_half():
    # gate rows give g, up rows give u: geglu = gelu(g) * u, swapping halves differs
    y = np.array([[2.0, -1.0, 0.5, 4.0]])      # I = 2: g = [2, -1], u = [0.5, 4]
    h = O.activation(y, "geglu", 2)
    assert np.allclose(h, O.gelu(np.array([[2.0, -1.0]])) * np.array([[0.5, 4.0]]), rtol=0, atol=0)
    assert not np.allclose(h, O.gelu(np.array([[0.5, 4.0]])) * np.array([[2.0, -1.0]]))


def test_activation_names_cover_cudnn_page():
    assert set(O.ACTIVATIONS) == {"swiglu", "relu2", "geglu", "gelu", "relu", "silu", "identity"}
    with pytest.raises(ValueError):
        O.activation(np.zeros((1, 2)), "tanh", 1)


def test_routed_scaling_factor_scales_route_weights():
    rows = np.array([[1.0, -2.0], [0.5, 4.0]])
    t2r = np.array([[0, 1]], np.int32)
    w = np.array([[0.25, 0.5]], np.float32)
    a = O.finalize(rows, w, t2r, routed_scaling_factor=2.0)
    b = O.finalize(rows, (w * 2).astype(np.float32), t2r)
    assert np.array_equal(a, b)
    # 0.5*1 + 1.0*0.5 = 1.0 ; 0.5*-2 + 1.0*4 = 3.0 (exact)
    assert a.tolist() == [[1.0, 3.0]]
    assert np.array_equal(O.finalize(rows, w, t2r, 1.0), O.finalize(rows, w, t2r))
