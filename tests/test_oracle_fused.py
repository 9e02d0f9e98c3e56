"""Pins of the oracle's fused-variant pieces (FlashInfer alphamoe_nvfp4_aligned_moe page):
separate gate and up scalars, the accumulated FP32 output, and packed routing slots
(CudnnGroupedGemmNvfp4Config, "Routing weights")."""
import os
from fractions import Fraction

import numpy as np
import torch

from oracle import formats as F
from oracle import moe as O
from oracle import plan as P

from test_oracle_moe import _small_problem, _val

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _packed_cases():
    with open(os.path.join(GOLD, "packed_topk.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    return [(int(w, 16), int(i), float(v)) for w, i, v in rows]


def test_unpack_topk_golden():
    cases = _packed_cases()
    words = np.array([w for w, _, _ in cases], dtype=np.uint32).view(np.int32).reshape(1, -1)
    ids, scores = P.unpack_topk(words)
    assert ids.tolist() == [[i for _, i, _ in cases]]
    assert scores.tolist() == [[v for _, _, v in cases]]


def test_unpack_topk_matches_torch_bf16():
    np.seterr(invalid="ignore")  # NaN score patterns
    # every BF16 bit pattern of the score field decodes to torch's bfloat16 value
    hi = np.arange(1 << 16, dtype=np.uint32)
    words = ((hi << 16) | (hi & 0xFFFF) ^ 0x5A5A).view(np.int32)
    ids, scores = P.unpack_topk(words)
    ref = torch.from_numpy(hi.astype(np.int32).astype(np.int16)).view(torch.bfloat16).double().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(scores[fin], ref[fin])
    assert np.all(np.isnan(scores[np.isnan(ref)]))
    assert np.array_equal(ids, (hi & 0xFFFF) ^ 0x5A5A)


def test_packed_plan_masks_ids_beyond_range():
    # a packed id of 0xFFFF (or any id past the local range) is an unrouted slot
    ids = np.array([[3, 0xFFFF], [1, 2]], np.int64)
    plan = P.make_plan(ids, 0, 4)
    assert plan["token_to_row"][0, 1] == -1 and plan["counts"].sum() == 3


def _double_gate_scales(pack, inter):
    d, s, a = pack
    s2 = s.copy()
    # +1 in the E4M3 exponent field doubles a normal scale exactly
    assert np.all((s2[:inter] & 0x78) != 0) and np.all((s2[:inter] & 0x78) != 0x78)
    s2[:inter] = s2[:inter] + 8
    return d, s2, a


def test_gate_scalar_equals_doubled_gate_scales():
    # gate_alpha = 2 * alpha1 must equal the same weights with every gate-row block scale
    # doubled (an independent route through the dequantiser); the up rows keep alpha1
    for act in ("swiglu", "geglu"):
        xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(5, "swiglu")
        I = W.inter
        w1d = [_double_gate_scales(p, I) for p in w1]
        Wd = O.ExpertWeights.from_packs(w1d, w2, True)
        ga = np.array([2.0 * float(p[2]) for p in w1])
        a = O.forward(xq, xsf, xs, ids, tw, W, act, gate_alpha=ga)
        b = O.forward(xq, xsf, xs, ids, tw, Wd, act)
        for key in ("preact", "act_bf16", "rows"):
            assert np.array_equal(a[key], b[key], equal_nan=True), key
        # and differs from scaling the up rows instead
        c = O.forward(xq, xsf, xs, ids, tw, W, act)
        assert not np.array_equal(a["preact"], c["preact"], equal_nan=True)
        real = a["plan"]["row_to_slot"] >= 0
        assert np.array_equal(a["preact"][real][:, I:], c["preact"][real][:, I:])


def test_gate_scalar_equal_to_alpha_changes_nothing():
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(6, "swiglu")
    ga = np.array([float(p[2]) for p in w1])
    a = O.forward(xq, xsf, xs, ids, tw, W, "swiglu", gate_alpha=ga)
    b = O.forward(xq, xsf, xs, ids, tw, W, "swiglu")
    assert np.array_equal(a["out"], b["out"])
    # non-gated activations ignore it
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(6, "relu2")
    a = O.forward(xq, xsf, xs, ids, tw, W, "relu2", gate_alpha=np.full(len(w1), 7.0))
    b = O.forward(xq, xsf, xs, ids, tw, W, "relu2")
    assert np.array_equal(a["out"], b["out"])


def _bf16_of(fr: Fraction) -> float:
    return float(F.bf16_round(np.array([float(fr)]))[0])


def test_accumulate_brute_force():
    # out = bf16(out_prev + sum_j w'[t,j] * y2), y2 from independent decoders, summed exactly
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(7, "swiglu")
    M, k = ids.shape
    H, I = W.hidden, W.inter
    rng = np.random.default_rng(7)
    prev = F.bf16_round(rng.standard_normal((M, H)))
    for rsf in (1.0, 2.5):
        res = O.forward(xq, xsf, xs, ids, tw, W, "swiglu", out_prev=prev, routed_scaling_factor=rsf)
        t2r = res["plan"]["token_to_row"]
        for t in range(M):
            for h in range(H):
                acc = Fraction(float(prev[t, h]))
                for j in range(k):
                    row = t2r[t, j]
                    d2, s2, a2 = w2[int(ids[t, j])]
                    ip = F.pack_e2m1(res["icodes"][row])
                    y2 = sum(Fraction(_val(ip, res["isf"][row], i)) * Fraction(_val(d2[h], s2[h], i))
                             for i in range(I)) * Fraction(float(a2))
                    wj = Fraction(float(np.float32(np.float32(tw[t, j]) * np.float32(rsf))))
                    acc += wj * y2
                assert res["out_acc"][t, h] == _bf16_of(acc), (t, h)


def test_accumulate_special_cases():
    xq, xsf, xs, ids, tw, W, w1, w2 = _small_problem(8, "swiglu", k=1)
    M = ids.shape[0]
    H = W.hidden
    # out_prev = 0, one slot of weight one: the expert row itself
    res = O.forward(xq, xsf, xs, ids, np.ones_like(tw), W, "swiglu", out_prev=np.zeros((M, H)))
    t2r = res["plan"]["token_to_row"][:, 0]
    assert np.array_equal(res["out_acc"], res["rows"][t2r])
    # every slot masked: out_prev comes back unchanged
    prev = F.bf16_round(np.random.default_rng(1).standard_normal((M, H)))
    res = O.forward(xq, xsf, xs, np.full_like(ids, -1), tw, W, "swiglu", out_prev=prev)
    assert np.array_equal(res["out_acc"], prev)
