"""The one-call path (moe_routed_forward, the small-batch fused prologue and the large-batch
chain of separate kernels) against the separate calls, bit for bit, and against the oracle."""
import numpy as np
import pytest
import torch

from gpu_harness import DEV, Problem, assert_close_output, bf16_np, mi, pkg, to_np

pytestmark = pytest.mark.gpu

CASES = {
    # fused prologue (M * top_k <= 2048 and M * H <= 2^17)
    "tiny": mi.CONFIGS["tiny"],
    "decode_t8": mi.CONFIGS["decode_t8"],
    "decode_ep": mi.MoEConfig("decode_ep", M=12, H=1024, I=256, E=32, top_k=6, seed=31, weight_seed=31,
                              local_offset=8, num_local=16),
    "relu2_small": mi.MoEConfig("relu2_small", M=64, H=512, I=384, E=12, top_k=3, act="relu2", seed=32,
                                weight_seed=32, local_offset=4, num_local=6),
    "geglu_small": mi.MoEConfig("geglu_small", M=40, H=768, I=256, E=16, top_k=4, act="geglu", seed=33,
                                weight_seed=33),
    # separate kernels (too large for the prologue)
    "swiglu_ragged": mi.MoEConfig("swiglu_ragged", M=300, H=512, I=256, E=8, top_k=2, seed=11, weight_seed=11),
    # the plan's three kernels and the quantiser storing into the plan rows, with K tails in
    # both GEMMs (H and I = 128 mod 256: zero scale groups on the K padding)
    "ktail_large": mi.MoEConfig("ktail_large", M=400, H=384, I=384, E=12, top_k=6, seed=34, weight_seed=34,
                                local_offset=2, num_local=8),
    # size limits: exactly 2048 slots and M*H = 2^17 (the largest fused-prologue batch); 2051
    # slots (the separate kernels, a two-block plan); 17 tokens (just past the decode-shaped
    # GEMMs); the largest local expert count (512) with expert-parallel masking
    "slots_2048": mi.MoEConfig("slots_2048", M=256, H=512, I=256, E=16, top_k=8, seed=35, weight_seed=35),
    "slots_2051": mi.MoEConfig("slots_2051", M=293, H=256, I=256, E=16, top_k=7, seed=36, weight_seed=36),
    "decode_m17": mi.MoEConfig("decode_m17", M=17, H=512, I=256, E=8, top_k=4, seed=37, weight_seed=37),
    "experts_512": mi.MoEConfig("experts_512", M=40, H=256, I=128, E=600, top_k=3, seed=38, weight_seed=38,
                                local_offset=50, num_local=512),
    # a very wide row: 2048 blocks per token, more than the prologue stages in shared memory
    # (it quantises after placing the rows instead); GEMM1 with 128 K chunks
    "wide_h": mi.MoEConfig("wide_h", M=3, H=32768, I=128, E=4, top_k=2, seed=39, weight_seed=39),
}


def _unrouted(cfg):
    ids, tw = mi.routing(cfg)
    ids = mi.with_unrouted(ids, 0.15, 7, cfg.E)
    tw = tw.copy()
    tw[(ids < 0) | (ids >= cfg.E)] = np.nan
    return ids, tw


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("do_finalize", [True, False])
def test_routed_equals_separate_calls(name, do_finalize):
    cfg = CASES[name]
    ids, tw = _unrouted(cfg) if name in ("decode_ep", "relu2_small", "ktail_large") else (None, None)
    p = Problem(cfg, ids, tw)
    if do_finalize:
        a = bf16_np(p.run_routed(True)).copy()
        b = bf16_np(p.run(True))
        assert np.array_equal(a, b)
        assert_close_output(a, p.oracle_forward()["out"], name)
    else:
        g2, tw_r, t2r = p.run_routed(False)
        g2 = bf16_np(g2).copy()
        t2r = to_np(t2r).copy()
        g2s, _, t2rs = p.run(False)
        assert np.array_equal(t2r, to_np(t2rs))
        real = t2r[t2r >= 0]
        assert np.array_equal(g2[real], bf16_np(g2s)[real])
        assert tw_r.data_ptr() == p.tw_t.data_ptr()
    assert p.layer.device_status(cfg.M, cfg.top_k, do_finalize) == 0


@pytest.mark.parametrize("name", ["tiny", "decode_t8", "decode_ep"])
@pytest.mark.parametrize("hooks", [1, 2, 3])
def test_decode_scheduling_fallbacks(name, hooks):
    """The decode GEMM loads each CTA's first unit's weights before the plan exists, guessing
    the expert from the routing ids, and offers that unit to the CTA through an ownership
    flag. Wrong guesses (bit 0: the stages are reloaded) and first units left to other CTAs
    (bit 1: taken by the sweep before any GEMM2 unit), forced through the test build's
    options, give the same bytes as the normal schedule, finalized and unfinalized."""
    cfg = CASES[name]
    ids, tw = _unrouted(cfg) if name == "decode_ep" else (None, None)
    p = Problem(cfg, ids, tw)
    ref = bf16_np(p.run_routed(True)).copy()
    g2r, _, t2r = p.run_routed(False)
    g2r, t2r = bf16_np(g2r).copy(), to_np(t2r).copy()
    opts = pkg.test_options(decode_hooks=hooks)

    def hooked(mode):
        b = p.layer.routed_buffers(cfg.M, cfg.top_k, mode)
        p.layer.routed(p.x, p.ids_t, p.tw_t, b, mode, test_options=opts)
        torch.cuda.synchronize()
        return b

    got = bf16_np(hooked(True)["out"]).copy()
    b = hooked(False)
    g2, t2 = bf16_np(b["gemm2_out"]).copy(), to_np(b["token_to_row"]).copy()
    assert np.array_equal(got, ref)
    assert np.array_equal(t2, t2r)
    real = t2r[t2r >= 0]
    assert np.array_equal(g2[real], g2r[real])
    for mode in (True, False):
        assert p.layer.device_status(cfg.M, cfg.top_k, mode) == 0


def test_routed_row_stride_and_packed_routing():
    cfg = CASES["decode_ep"]
    p = Problem(cfg)
    wide = torch.zeros(cfg.M, cfg.H + 64, dtype=torch.bfloat16, device=DEV)
    wide[:, :cfg.H] = p.x
    x = wide[:, :cfg.H]                                   # ld_x = H + 64
    a = bf16_np(p.layer.forward(x, p.ids_t, p.tw_t)).copy()
    assert np.array_equal(a, bf16_np(p.run(True)))
    hi = p.tw_t.to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
    packed = ((hi << 16) | (p.ids_t & 0xFFFF)).contiguous()
    b = bf16_np(p.layer.forward(p.x, packed, None)).copy()
    c = bf16_np(p.layer.forward(p.x, p.ids_t, p.tw_t.to(torch.bfloat16)))
    assert np.array_equal(b, c)


@pytest.mark.parametrize("name", ["decode_t8", "swiglu_ragged"])
def test_routed_accumulate(name):
    cfg = CASES[name].with_(routed_scaling_factor=0.5)
    p = Problem(cfg)
    rng = np.random.default_rng(2)
    prev = torch.from_numpy(rng.standard_normal((cfg.M, cfg.H)).astype(np.float32) * 0.01).to(torch.bfloat16).to(DEV)
    out = prev.clone()
    p.layer.forward(p.x, p.ids_t, p.tw_t, do_finalize=2, out=out)
    torch.cuda.synchronize()
    ref = p.oracle_forward(out_prev=bf16_np(prev))["out_acc"]
    assert_close_output(bf16_np(out), ref, "routed accumulate")


def test_routed_graph_replay_new_routing_small_batch():
    cfg = CASES["decode_t8"]
    p = Problem(cfg)
    x, ids, tw = p.x.clone(), p.ids_t.clone(), p.tw_t.clone()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in evs:
        e.record()
    g = p.layer.capture(x, ids, tw, True, step_events=evs)
    cfg2 = cfg.with_(seed=77)
    ids2, tw2 = mi.routing(cfg2)
    x.copy_(mi.hidden_bf16(cfg2, DEV))
    ids.copy_(torch.from_numpy(ids2))
    tw.copy_(torch.from_numpy(tw2))
    g.replay()
    torch.cuda.synchronize()
    got = bf16_np(p.layer.routed_buffers(cfg.M, cfg.top_k, True)["out"]).copy()
    assert all(evs[i].elapsed_time(evs[i + 1]) >= 0 for i in range(4))
    p2 = Problem(cfg2)
    assert np.array_equal(got, bf16_np(p2.run(True)))


@pytest.mark.parametrize("name", ["decode_t8", "swiglu_ragged"])
def test_refresh_in_place_under_captured_graph(name):
    """In-place weight refresh at stable addresses (Megatron-Core prepare_routed_nvfp4_weights
    with out=...): a graph captured before the refresh computes with the new weights after it.
    The layer's linear NVFP4 weights are overwritten with a second seeded set, refresh()
    re-prepares them into the same buffer, and one replay of the old graph must equal the
    oracle on the new weights (and the new weights' own layer, bit for bit)."""
    cfg = CASES[name]
    p = Problem(cfg)
    x, ids, tw = p.x.clone(), p.ids_t.clone(), p.tw_t.clone()
    g = p.layer.capture(x, ids, tw, True)
    g.replay()
    torch.cuda.synchronize()
    out_buf = p.layer.routed_buffers(cfg.M, cfg.top_k, True)["out"]
    before = bf16_np(out_buf).copy()
    assert np.array_equal(before, bf16_np(p.run_routed(True)))
    prepared_ptr = p.layer.prepared.data_ptr()
    cfg2 = cfg.with_(weight_seed=cfg.weight_seed + 1000)
    p2 = Problem(cfg2)                       # same tokens and routing, new weights
    for dst, src in zip(p.q1 + p.q2, p2.q1 + p2.q2):
        dst.copy_(src)
    p.layer.refresh()
    g.replay()
    torch.cuda.synchronize()
    got = bf16_np(out_buf).copy()
    assert p.layer.prepared.data_ptr() == prepared_ptr
    assert not np.array_equal(got, before)
    assert np.array_equal(got, bf16_np(p2.run_routed(True)))
    assert_close_output(got, p2.oracle_forward()["out"], f"{name} after refresh")
    assert p.layer.device_status(cfg.M, cfg.top_k, True) == 0


@pytest.mark.parametrize("direct", [False, True])
@pytest.mark.parametrize("name", ["decode_t8", "swiglu_ragged"])
def test_capture_host_matches_device_path(name, direct):
    """capture_host: one graph copies the pinned inputs in, runs the forward and copies the
    output out (direct: the kernels read the pinned inputs and write the pinned output in
    place). Its host output equals the device path's bit for bit, and stays so after the
    staging buffer is refilled with new hidden states and a new routing."""
    cfg = CASES[name]
    p = Problem(cfg)
    M, k, H = cfg.M, cfg.top_k, cfg.H
    staging = pkg.HostStaging(M, H, k, DEV)
    hout = torch.empty(M, H, dtype=torch.bfloat16).pin_memory()
    staging.x.copy_(p.x.cpu())
    staging.ids.copy_(torch.from_numpy(np.ascontiguousarray(p.ids, dtype=np.int32)))
    staging.weights.copy_(torch.from_numpy(np.ascontiguousarray(p.tw, dtype=np.float32)))
    g = p.layer.capture_host(staging, hout, direct=direct)
    for rep in range(2):
        if rep == 1:
            # a second step: other tokens (the rows reversed) and another routing
            cfg2 = cfg.with_(seed=cfg.seed + 100)
            ids2, tw2 = mi.routing(cfg2)
            staging.x.copy_(p.x.cpu().flip(0))
            staging.ids.copy_(torch.from_numpy(np.ascontiguousarray(ids2, dtype=np.int32)))
            staging.weights.copy_(torch.from_numpy(np.ascontiguousarray(tw2, dtype=np.float32)))
        g.replay()
        torch.cuda.synchronize()
        got = bf16_np(hout).copy()
        x_dev = staging.x.to(DEV)
        ref = p.layer.forward(x_dev, staging.ids.to(DEV), staging.weights.to(DEV), do_finalize=True)
        torch.cuda.synchronize()
        assert np.array_equal(got, bf16_np(ref)), f"step {rep}"
        assert p.layer.device_status(M, k, True) == 0
