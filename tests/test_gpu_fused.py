"""GPU parity of the fused-variant features (FlashInfer alphamoe_nvfp4_aligned_moe page):
separate gate / up scalars, the accumulated FP32 output, packed routing slots
(CudnnGroupedGemmNvfp4Config, "Routing weights"), and the token-capacity prefix
(Megatron-Core flashinfer_routed_nvfp4_moe token_capacity)."""
import numpy as np
import pytest
import torch

from gpu_harness import DEV, O, Problem, assert_close_output, bf16_np, mi, pkg, to_np
from oracle.plan import make_plan, unpack_topk

pytestmark = pytest.mark.gpu

RAGGED = mi.MoEConfig("swiglu_ragged", M=300, H=512, I=256, E=8, top_k=2, seed=11, weight_seed=11)
EP = mi.MoEConfig("relu2_ep_small", M=513, H=256, I=384, E=12, top_k=3, act="relu2", seed=13, weight_seed=13,
                  local_offset=4, num_local=6)


def _pack_np(ids: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Packed slots from ids and scores (scores rounded to BF16 by torch), as int32."""
    hi = torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    word = (hi.astype(np.int64) & 0xFFFF) << 16 | (ids.astype(np.int64) & 0xFFFF)
    return word.astype(np.uint32).view(np.int32)


@pytest.mark.parametrize("M,E,k", [(300, 8, 2), (3000, 64, 6)])
def test_plan_packed_ids_bitexact(M, E, k):
    cfg = mi.MoEConfig("pk", M=M, H=128, I=128, E=E, top_k=k, seed=M + E)
    ids, tw = mi.routing(cfg)
    ids = mi.with_unrouted(ids, 0.1, 5, E)
    ids = np.where(ids < 0, 0xFFFF, ids)                  # unrouted: an id past every expert
    packed = _pack_np(ids, tw)
    uid, _ = unpack_topk(packed)
    off, El = 2, E - 3
    ref = make_plan(uid, off, El)
    cap = pkg.moe_plan_capacity(M, k, El)
    counts = torch.empty(El, dtype=torch.int32, device=DEV)
    padded = torch.empty(El + 1, dtype=torch.int32, device=DEV)
    r2s = torch.full((cap,), 7, dtype=torch.int32, device=DEV)
    t2r = torch.empty(M, k, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(pkg.moe_plan_workspace_bytes(M, k, El), 16), dtype=torch.uint8, device=DEV)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    pt = torch.from_numpy(packed).to(DEV)
    pkg.moe_plan(pt, E, off, El, counts, padded, r2s, t2r, ws, st, packed=True)
    torch.cuda.synchronize()
    assert np.array_equal(to_np(counts), ref["counts"])
    assert np.array_equal(to_np(padded), ref["padded_offsets"])
    assert np.array_equal(to_np(r2s), ref["row_to_slot"])
    assert np.array_equal(to_np(t2r), ref["token_to_row"])
    assert int(to_np(st)[0]) == 0


def test_finalize_packed_weights_bitexact():
    M, k, H, R = 40, 6, 512, 150
    rng = np.random.default_rng(3)
    rows = torch.from_numpy(rng.standard_normal((R, H)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    t2r = rng.integers(-1, R, size=(M, k)).astype(np.int32)
    packed = _pack_np(rng.integers(0, 64, size=(M, k)), rng.random((M, k)))
    _, scores = unpack_topk(packed)
    out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    pkg.moe_finalize(rows, torch.from_numpy(packed).to(DEV), torch.from_numpy(t2r).to(DEV), out,
                     routed_scaling_factor=1.5)
    torch.cuda.synchronize()
    ref = O.finalize(bf16_np(rows), scores.astype(np.float32), t2r, routed_scaling_factor=1.5)
    assert np.array_equal(bf16_np(out), ref)


def test_forward_packed_routing_equals_bf16_weights():
    p = Problem(RAGGED)
    packed = torch.from_numpy(_pack_np(p.ids, p.tw)).to(DEV)
    a = bf16_np(p.layer.forward(p.x, packed, None)).copy()
    b = bf16_np(p.layer.forward(p.x, p.ids_t, p.tw_t.to(torch.bfloat16))).copy()
    torch.cuda.synchronize()
    assert np.array_equal(a, b)


@pytest.mark.parametrize("act", ["swiglu", "geglu"])
def test_separate_gate_scalars(act):
    cfg = RAGGED.with_(act=act)
    factor = np.linspace(0.25, 3.0, cfg.El).astype(np.float32)
    p = Problem(cfg, gate_factor=factor)
    ref = p.oracle_forward()
    assert_close_output(bf16_np(p.run(True)), ref["out"], "gate scalars")
    # the separate scalars change the result (they are not ignored)
    plain = Problem(cfg).oracle_forward()["out"]
    assert np.linalg.norm(plain - ref["out"]) > 0.05 * np.linalg.norm(ref["out"])
    # pre-activations: gate columns carry the gate scalar, up columns alpha1
    b = p.bufs(True)
    cap = b["capacity"]
    dbg = torch.full((cap, cfg.N1), float("nan"), dtype=torch.float32, device=DEV)
    pkg.moe_test_gemm1(b["padded_offsets"], b["row_to_slot"], cfg.M, cfg.top_k, b["xq"], b["xsf"], b["xs"],
                        p.layer.w, p.layer.prepared, 0, dbg, b["ws"], b["dev_status"])
    torch.cuda.synchronize()
    real = ref["plan"]["row_to_slot"] >= 0
    got = to_np(dbg)[real].astype(np.float64)
    want = ref["preact"][real]
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 1e-5


@pytest.mark.parametrize("cfg", [RAGGED, EP], ids=["swiglu_ragged", "relu2_ep_small"])
def test_accumulate_into_out(cfg):
    ids, tw = mi.routing(cfg)
    ids = mi.with_unrouted(ids, 0.1, 9, cfg.E)
    ids[5, :] = -1                                           # a token with no routed slot
    tw = tw.copy()
    tw[(ids < 0) | (ids >= cfg.E)] = np.nan
    cfg = cfg.with_(routed_scaling_factor=1.75)
    p = Problem(cfg, ids, tw)
    rng = np.random.default_rng(4)
    fin = bf16_np(p.run(True)).copy()
    scale = float(np.abs(fin).max())
    prev = torch.from_numpy((rng.standard_normal((cfg.M, cfg.H)) * scale * 0.3).astype(np.float32))
    prev = prev.to(torch.bfloat16).to(DEV)
    out = prev.clone()
    res = p.layer.forward(p.x, p.ids_t, p.tw_t, do_finalize=2, out=out)
    torch.cuda.synchronize()
    assert res.data_ptr() == out.data_ptr()
    ref = p.oracle_forward(out_prev=bf16_np(prev))
    got = bf16_np(out)
    assert_close_output(got, ref["out_acc"], "accumulate")
    # rows of tokens with no local slot keep the caller's values, bit for bit
    t2r = ref["plan"]["token_to_row"]
    none = np.all(t2r < 0, axis=1)
    assert none[5] and np.array_equal(got[none], bf16_np(prev)[none])
    # from a zero out, the accumulated output is the finalized output up to FP32 order and
    # the BF16 rounding of the expert rows
    z = torch.zeros(cfg.M, cfg.H, dtype=torch.bfloat16, device=DEV)
    p.layer.forward(p.x, p.ids_t, p.tw_t, do_finalize=2, out=z)
    torch.cuda.synchronize()
    assert_close_output(bf16_np(z), fin, "accumulate from zero")


def test_accumulate_graph_replays_add_up():
    cfg = RAGGED
    p = Problem(cfg)
    out = torch.zeros(cfg.M, cfg.H, dtype=torch.bfloat16, device=DEV)
    g = p.layer.capture(p.x, p.ids_t, p.tw_t, do_finalize=2, out=out)
    g.replay()
    torch.cuda.synchronize()
    once = bf16_np(out).copy()
    assert_close_output(once, p.oracle_forward(out_prev=np.zeros((cfg.M, cfg.H)))["out_acc"], "replay 1")
    g.replay()
    torch.cuda.synchronize()
    twice = bf16_np(out)
    assert_close_output(twice, 2.0 * once, "replay 2")


def test_token_capacity_prefix():
    cfg = RAGGED
    p = Problem(cfg)
    T = 137
    sentinel = torch.full((cfg.M, cfg.H), 3.0, dtype=torch.bfloat16, device=DEV)
    res = p.layer.forward(p.x, p.ids_t, p.tw_t, out=sentinel, token_capacity=T)
    torch.cuda.synchronize()
    got = bf16_np(sentinel).copy()
    assert res.shape == (T, cfg.H)
    assert np.all(got[T:] == 3.0)                             # rows past the prefix untouched
    sub = p.layer.forward(p.x[:T].contiguous(), p.ids_t[:T].contiguous(), p.tw_t[:T].contiguous())
    torch.cuda.synchronize()
    assert np.array_equal(got[:T], bf16_np(sub))
    full = p.oracle_forward()["out"]
    assert_close_output(got[:T], full[:T], "prefix")
