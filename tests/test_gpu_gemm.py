"""GPU parity of the tcgen05 grouped GEMMs and the whole forward against the oracle.

* GEMM1 pre-activations (test hook, FP32) within the FP32 accumulation bound;
* the fused requantiser bit-exact on the kernel's own BF16 intermediate;
* the forward (both do_finalize modes) within the path's output tolerance, on sizes
  that span several tiles with ragged tails, plus edge cases."""
import numpy as np
import pytest
import torch

from gpu_harness import (DEV, O, Problem, Q, assert_close_output, bf16_np, mi, oracle_weights, pkg,
                         sf_tiles_to_linear, to_np)
from oracle.formats import pack_e2m1

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": mi.CONFIGS["tiny"],
    # several m-tiles per expert, ragged last tile, two column tiles
    "swiglu_ragged": mi.MoEConfig("swiglu_ragged", M=300, H=512, I=256, E=8, top_k=2, seed=11, weight_seed=11),
    # skewed routing: one expert takes most rows; K tail (H % 256 == 128)
    "swiglu_skew": mi.MoEConfig("swiglu_skew", M=400, H=384, I=128, E=16, top_k=3, seed=12, weight_seed=12,
                                skew=1.2),
    # squared-ReLU with EP masking; I % 256 == 128 (column and K tails)
    "relu2_ep_small": mi.MoEConfig("relu2_ep_small", M=513, H=256, I=384, E=12, top_k=3, act="relu2",
                                   seed=13, weight_seed=13, local_offset=4, num_local=6),
    "decode_t8": mi.CONFIGS["decode_t8"],
    # decode-shaped GEMMs (at most 16 tokens): experts with many rows (up to 16), K tails
    "decode_dense": mi.MoEConfig("decode_dense", M=16, H=384, I=256, E=4, top_k=3, seed=14, weight_seed=14),
    "relu2_decode": mi.MoEConfig("relu2_decode", M=13, H=512, I=384, E=10, top_k=4, act="relu2", seed=15,
                                 weight_seed=15, local_offset=2, num_local=6),
    # decode-shaped, GEMM2 with more K chunks (I = 1536: six) than pipeline stages, so its
    # tiles wait for the expert's GEMM1 tiles before loading; GEMM1 one K chunk (H = 256)
    "decode_long_k2": mi.MoEConfig("decode_long_k2", M=6, H=256, I=1536, E=6, top_k=2, seed=16, weight_seed=16),
}


def _gpu_debug(p: Problem, mode: int):
    cfg = p.cfg
    b = p.bufs(True)
    p.run(True)
    cap = b["capacity"]
    ncols = cfg.N1 if mode == 0 else cfg.I
    dbg = torch.full((cap, ncols), float("nan"), dtype=torch.float32 if mode == 0 else torch.bfloat16,
                     device=DEV)
    pkg.moe_test_gemm1(b["padded_offsets"], b["row_to_slot"], cfg.M, cfg.top_k, b["xq"], b["xsf"], b["xs"],
                        p.layer.w, p.layer.prepared, mode, dbg, b["ws"], b["dev_status"])
    torch.cuda.synchronize()
    return dbg


@pytest.mark.parametrize("name", list(SMALL))
def test_gemm1_preact_within_fp32_bound(name):
    p = Problem(SMALL[name])
    cfg = p.cfg
    dbg = _gpu_debug(p, 0)
    ref = p.oracle_forward()
    r2s = ref["plan"]["row_to_slot"]
    real = r2s >= 0
    got = to_np(dbg)[real].astype(np.float64)
    want = ref["preact"][real]
    # bound: |sum of K FP32 products, any order - exact| <= K * 2^-23 * sum|terms|
    xq, xsf, xs = p.oracle_inputs()
    W = oracle_weights(cfg)
    A = np.abs(Q.dequantize_rows(xq, xsf))
    tok = r2s[real] // cfg.top_k
    bound = np.zeros_like(want)
    rows = np.nonzero(real)[0]
    padded = ref["plan"]["padded_offsets"]
    for i, prow in enumerate(rows):
        l = np.searchsorted(padded, prow, side="right") - 1
        d1, s1, a1 = W.w1(l)
        absw = np.abs(Q.dequantize_rows(d1, s1))
        bound[i] = (A[tok[i]] @ absw.T) * xs[tok[i]] * a1 * cfg.H * 2.0 ** -23
    err = np.abs(got - want)
    assert np.all(err <= bound + 1e-30), (err.max(), (err - bound).max())
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-5


@pytest.mark.parametrize("name", list(SMALL))
def test_requant_bitexact_on_kernel_intermediate(name):
    p = Problem(SMALL[name])
    cfg = p.cfg
    h = _gpu_debug(p, 1)                       # BF16 intermediate of the same GEMM1
    p.run(True)                                # product path: fused requant into the workspace
    b = p.bufs(True)
    offs = pkg.moe_forward_workspace_layout(cfg.M, cfg.top_k, p.layer.w, 1)
    ws = to_np(b["ws"])
    cap = b["capacity"]
    r2s = to_np(b["row_to_slot"])[:cap]
    real = r2s >= 0
    iq = ws[offs[2]:offs[2] + cap * cfg.I // 2].reshape(cap, cfg.I // 2)[real]
    isf = sf_tiles_to_linear(ws[offs[3]:offs[4] if offs[4] else offs[5]], cap, cfg.I // 16)[real]
    hv = bf16_np(h)[real].astype(np.float32)
    codes, sf = Q.quantize_blocks(hv, np.float32(cfg.fc2_input_scale))
    assert np.array_equal(isf, sf)
    assert np.array_equal(iq, pack_e2m1(codes))
    # the kernel's intermediate is the activation of its own FP32 pre-activations,
    # within one BF16 rounding of the oracle's float64 activation of the same values
    y = _gpu_debug(p, 0)
    yv = to_np(y)[real].astype(np.float64)
    act = O.activation(yv, cfg.act, cfg.I)
    assert np.all(np.abs(hv - act) <= np.abs(act) * 2.0 ** -7 + 2.0 ** -126)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("do_finalize", [True, False])
def test_forward_matches_oracle(name, do_finalize):
    p = Problem(SMALL[name])
    cfg = p.cfg
    res = p.run(do_finalize)
    ref = p.oracle_forward()
    assert int(p.bufs(do_finalize)["dev_status"][0]) == 0
    if do_finalize:
        assert_close_output(bf16_np(res), ref["out"], name)
    else:
        g2, tw, t2r = res
        assert np.array_equal(to_np(t2r), ref["plan"]["token_to_row"])
        assert tw.data_ptr() == p.tw_t.data_ptr()
        real = ref["plan"]["row_to_slot"] >= 0
        assert_close_output(bf16_np(g2)[real], ref["rows"][real], name + " rows")


@pytest.mark.parametrize("name", ["swiglu_ragged", "relu2_ep_small", "decode_t8", "decode_dense", "relu2_decode", "decode_long_k2"])
def test_finalize_of_unfinalized_equals_finalized(name):
    # decode-sized batches combine inside the GEMM launch; the standalone combine of their
    # unfinalized rows must give the same bytes
    p = Problem(SMALL[name])
    cfg = p.cfg
    fin = bf16_np(p.run(True)).copy()
    g2, tw, t2r = p.run(False)
    out = torch.empty(cfg.M, cfg.H, dtype=torch.bfloat16, device=DEV)
    pkg.moe_finalize(g2, tw, t2r, out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_np(out), fin)


def test_unrouted_and_masked_slots():
    cfg = SMALL["swiglu_ragged"]
    ids, tw = mi.routing(cfg)
    ids = mi.with_unrouted(ids, 0.25, 4, cfg.E)
    ids[3, :] = -1                                   # a token with no routed slot -> zero row
    tw = tw.copy()
    tw[(ids < 0) | (ids >= cfg.E)] = np.nan
    p = Problem(cfg, ids, tw)
    out = bf16_np(p.run(True))
    ref = p.oracle_forward()["out"]
    assert np.all(out[3] == 0)
    assert_close_output(out, ref, "unrouted")


def test_single_token_single_expert():
    cfg = mi.MoEConfig("one", M=1, H=256, I=128, E=1, top_k=1, seed=3, weight_seed=3)
    p = Problem(cfg)
    assert_close_output(bf16_np(p.run(True)), p.oracle_forward()["out"], "one")


def test_fc2_input_scale():
    cfg = SMALL["swiglu_ragged"].with_(fc2_input_scale=0.125)
    p = Problem(cfg)
    assert_close_output(bf16_np(p.run(True)), p.oracle_forward()["out"], "g2")


def test_zero_tokens_is_noop():
    cfg = mi.CONFIGS["tiny"]
    p = Problem(cfg)
    empty_ids = torch.empty(0, cfg.top_k, dtype=torch.int32, device=DEV)
    empty_w = torch.empty(0, cfg.top_k, dtype=torch.float32, device=DEV)
    x = torch.empty(0, cfg.H, dtype=torch.bfloat16, device=DEV)
    out = p.layer.forward(x, empty_ids, empty_w)
    torch.cuda.synchronize()
    assert out.shape == (0, cfg.H)


def test_repeat_calls_are_deterministic():
    p = Problem(SMALL["swiglu_skew"])
    a = bf16_np(p.run(True)).copy()
    b = bf16_np(p.run(True)).copy()
    assert np.array_equal(a, b)


def test_step_events_recorded():
    p = Problem(SMALL["swiglu_ragged"])
    cfg = p.cfg
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in evs:
        e.record()
    b = p.bufs(True)
    p.layer.quantize(p.x, b)
    p.layer.plan(p.ids_t, b)
    p.layer.experts(p.tw_t, b, True, step_events=evs)
    torch.cuda.synchronize()
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(4)]
    assert all(t >= 0 for t in times)
    assert_close_output(bf16_np(b["out"]), p.oracle_forward()["out"], "events")


def test_cuda_graph_replay_with_new_routing():
    # capture once; refill hidden states and routing in place; replay == eager forward
    cfg = SMALL["swiglu_skew"]
    p = Problem(cfg)
    x = p.x.clone()
    ids = p.ids_t.clone()
    tw = p.tw_t.clone()
    g = p.layer.capture(x, ids, tw, True)
    cfg2 = cfg.with_(seed=99, skew=0.0)
    ids2, tw2 = mi.routing(cfg2)
    x.copy_(mi.hidden_bf16(cfg2, DEV))
    ids.copy_(torch.from_numpy(ids2))
    tw.copy_(torch.from_numpy(tw2))
    g.replay()
    torch.cuda.synchronize()
    got = bf16_np(p.layer.routed_buffers(cfg.M, cfg.top_k, True)["out"]).copy()
    ref = bf16_np(p.layer.forward(x.clone(), ids.clone(), tw.clone()))
    torch.cuda.synchronize()
    assert np.array_equal(got, ref)
    p2 = Problem(cfg2)
    assert_close_output(got, p2.oracle_forward()["out"], "graph")


@pytest.mark.parametrize("act", ["geglu", "gelu", "relu", "silu", "identity"])
def test_forward_other_activations(act):
    # the typed activations of the cuDNN backend page beyond SwiGLU / squared-ReLU
    gated = act == "geglu"
    cfg = mi.MoEConfig(f"act_{act}", M=300, H=384, I=384 if not gated else 256, E=8, top_k=2, act=act,
                       seed=21, weight_seed=21)
    p = Problem(cfg)
    ref = p.oracle_forward()
    assert_close_output(bf16_np(p.run(True)), ref["out"], act)
    # the fused requantiser stays bit-exact on the kernel's own intermediate
    h = _gpu_debug(p, 1)
    p.run(True)
    b = p.bufs(True)
    offs = pkg.moe_forward_workspace_layout(cfg.M, cfg.top_k, p.layer.w, 1)
    ws = to_np(b["ws"])
    cap = b["capacity"]
    real = to_np(b["row_to_slot"])[:cap] >= 0
    iq = ws[offs[2]:offs[2] + cap * cfg.I // 2].reshape(cap, cfg.I // 2)[real]
    codes, _ = Q.quantize_blocks(bf16_np(h)[real].astype(np.float32), np.float32(1.0))
    assert np.array_equal(iq, pack_e2m1(codes))


def test_forward_routed_scaling_factor_and_bf16_weights():
    cfg = SMALL["swiglu_ragged"].with_(routed_scaling_factor=2.5)
    p = Problem(cfg)
    assert_close_output(bf16_np(p.run(True)), p.oracle_forward()["out"], "rsf")
    # BF16 route weights: the same result as FP32 weights holding the same (BF16) values
    tw16 = p.tw_t.to(torch.bfloat16)
    out16 = bf16_np(p.layer.forward(p.x, p.ids_t, tw16)).copy()
    out32 = bf16_np(p.layer.forward(p.x, p.ids_t, tw16.float())).copy()
    torch.cuda.synchronize()
    assert np.array_equal(out16, out32)
