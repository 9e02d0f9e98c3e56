"""GPU parity of the integer / byte steps against the oracle, bit for bit:
the NVFP4 quantiser (activations and weights), the routing plan, the permutation
and the standalone finalize. All calls go through the C ABI."""
import numpy as np
import pytest
import torch

from gpu_harness import DEV, F, O, Q, bf16_np, mi, pkg, sf_tiles_to_linear, to_np

pytestmark = pytest.mark.gpu


def test_generator_identical_on_gpu_and_cpu():
    cfg = mi.CONFIGS["decode_t4"]
    a = mi.normal_f32(3, 77, 12345, 100000, "cpu")
    b = mi.normal_f32(3, 77, 12345, 100000, DEV).cpu()
    assert torch.equal(a, b)
    assert torch.equal(mi.expert_w2_bf16(cfg, 5, "cpu"), mi.expert_w2_bf16(cfg, 5, DEV).cpu())
    # counters above 2^32 (large expert matrices)
    big = (1 << 32) + 7
    assert torch.equal(mi.normal_f32(4, 1003, big, 4096, "cpu"), mi.normal_f32(4, 1003, big, 4096, DEV).cpu())


def _special_rows(H):
    rows = [np.zeros(H, np.float32),                                  # all-zero row
            np.full(H, 3.0, np.float32),                              # constant
            np.linspace(-1000, 1000, H).astype(np.float32),           # wide range
            (np.arange(H) % 17 - 8).astype(np.float32) * 1e-3]        # small values
    r = np.zeros(H, np.float32)
    r[5] = -2.5
    r[200 % H] = 1e-30                                                # subnormal-ish input
    rows.append(r)
    r = np.full(H, -0.0, np.float32)
    r[0] = 1.0
    rows.append(r)                                                    # negative zeros
    return np.stack(rows)


@pytest.mark.parametrize("mode", ["global_one", "per_token"])
@pytest.mark.parametrize("M,H", [(1, 128), (37, 512), (300, 2048), (8, 7168)])
def test_quantize_input_bitexact(mode, M, H):
    cfg = mi.MoEConfig("q", M=M, H=H, I=128, E=1, top_k=1, seed=M + H)
    x = mi.hidden_bf16(cfg, DEV)
    if M >= 6:
        x[:6] = torch.from_numpy(_special_rows(H)).to(DEV).to(torch.bfloat16)
    m = pkg.MOE_SCALE_PER_TOKEN if mode == "per_token" else pkg.MOE_SCALE_GLOBAL_ONE
    xq = torch.empty(M, H // 2, dtype=torch.uint8, device=DEV)
    xsf = torch.empty(M, H // 16, dtype=torch.uint8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    pkg.moe_quantize_input(x.view(torch.int16), m, xq, xsf, xs)
    torch.cuda.synchronize()
    rq, rsf, rxs = Q.quantize_activations(x.float().cpu().numpy(), mode)
    assert np.array_equal(to_np(xsf), rsf)
    assert np.array_equal(to_np(xq), rq)
    assert np.array_equal(to_np(xs), rxs)


def test_quantize_input_row_stride():
    M, H, ld = 16, 256, 384
    full = mi.hidden_bf16(mi.MoEConfig("q", M=M, H=ld, I=128, E=1, top_k=1, seed=5), DEV)
    x = full[:, :H]
    xq = torch.empty(M, H // 2, dtype=torch.uint8, device=DEV)
    xsf = torch.empty(M, H // 16, dtype=torch.uint8, device=DEV)
    xs = torch.empty(M, dtype=torch.float32, device=DEV)
    pkg.moe_quantize_input(x.view(torch.int16), pkg.MOE_SCALE_PER_TOKEN, xq, xsf, xs)
    torch.cuda.synchronize()
    rq, rsf, rxs = Q.quantize_activations(x.float().cpu().numpy(), "per_token")
    assert np.array_equal(to_np(xq), rq) and np.array_equal(to_np(xsf), rsf)


@pytest.mark.parametrize("E,R,C", [(3, 256, 128), (2, 128, 2048), (1, 384, 640)])
def test_quantize_weights_bitexact(E, R, C):
    cfg = mi.MoEConfig("w", M=1, H=C, I=R, E=E, top_k=1, act="relu2", weight_seed=E * 7)
    w = torch.stack([mi.expert_w2_bf16(cfg.with_(H=R, I=C), e, DEV) for e in range(E)])
    w[0, 0, :16] = 0
    data, sf, alpha = pkg.quantize_weights(w)
    torch.cuda.synchronize()
    for e in range(E):
        rd, rs, ra = Q.quantize_weight(w[e].float().cpu().numpy())
        assert np.array_equal(to_np(data[e]), rd)
        assert np.array_equal(to_np(sf[e]), rs)
        assert to_np(alpha[e]) == ra


def test_quantize_weights_zero_matrix():
    w = torch.zeros(2, 128, 128, dtype=torch.bfloat16, device=DEV)
    data, sf, alpha = pkg.quantize_weights(w)
    torch.cuda.synchronize()
    assert to_np(alpha).tolist() == [1.0, 1.0]
    assert not to_np(data).any() and not to_np(sf).any()


def _run_plan(ids, E, off, El):
    M, k = ids.shape
    cap = pkg.moe_plan_capacity(M, k, El)
    ids_t = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(DEV)
    counts = torch.full((El,), -7, dtype=torch.int32, device=DEV)
    padded = torch.full((El + 1,), -7, dtype=torch.int32, device=DEV)
    r2s = torch.full((max(cap, 1),), 12345, dtype=torch.int32, device=DEV)
    t2r = torch.full((M, k), 12345, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(pkg.moe_plan_workspace_bytes(M, k, El), 16), dtype=torch.uint8, device=DEV)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    pkg.moe_plan(ids_t, E, off, El, counts, padded, r2s, t2r, ws, st)
    torch.cuda.synchronize()
    return to_np(counts), to_np(padded), to_np(r2s)[:cap], to_np(t2r), int(to_np(st)[0])


def _check_plan(ids, E, off, El, allow_dup=False):
    from oracle.plan import make_plan
    ref = make_plan(ids, off, El, allow_duplicates=allow_dup)
    counts, padded, r2s, t2r, st = _run_plan(ids, E, off, El)
    assert np.array_equal(counts, ref["counts"])
    assert np.array_equal(padded, ref["padded_offsets"])
    assert np.array_equal(r2s, ref["row_to_slot"])
    assert np.array_equal(t2r, ref["token_to_row"])
    return st


@pytest.mark.parametrize("name", ["tiny", "decode_t4", "decode_t8", "wide_decode", "prefill_uniform",
                                  "prefill_skewed", "relu2_ep"])
def test_plan_bitexact_configs(name):
    cfg = mi.CONFIGS[name]
    ids, _ = mi.routing(cfg)
    assert _check_plan(ids, cfg.E, cfg.local_offset, cfg.El) == 0


@pytest.mark.parametrize("seed", range(6))
def test_plan_bitexact_random(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.choice([1, 3, 100, 257, 1000, 3000]))
    E = int(rng.choice([2, 9, 64, 200, 512]))
    k = int(rng.integers(1, min(E, 10) + 1))
    El = int(rng.integers(1, E + 1))
    off = int(rng.integers(0, E - El + 1))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    ids = mi.with_unrouted(ids, 0.1, seed, E)
    assert _check_plan(ids, E, off, El) == 0


def test_plan_empty_and_all_masked():
    ids = np.full((5, 3), -1, np.int32)
    assert _check_plan(ids, 8, 0, 8) == 0
    ids = np.full((3000, 2), 9, np.int32)                 # all outside the local range (multi-block)
    assert _check_plan(ids, 16, 0, 8) == 0


def test_plan_duplicate_sets_status():
    ids = np.array([[1, 1], [2, 3]], np.int32)
    assert _check_plan(ids, 4, 0, 4, allow_dup=True) & pkg.MOE_DEV_DUPLICATE_EXPERT
    ids = np.tile(np.array([[5, 6, 5]], np.int32), (4000, 1))   # multi-block path
    assert _check_plan(ids, 8, 0, 8, allow_dup=True) & pkg.MOE_DEV_DUPLICATE_EXPERT


# shift = 8 values places rows and out 16 bytes past a 32-byte boundary (the API asks for
# 16-byte alignment only); H = 384 leaves most threads of a token's block without columns
@pytest.mark.parametrize("M,k,H,R,shift", [(1, 1, 128, 4, 0), (7, 3, 256, 30, 0), (300, 8, 2048, 900, 0),
                                           (64, 6, 7168, 128, 0), (1000, 4, 384, 2000, 0), (1000, 4, 384, 2000, 8),
                                           (300, 8, 2048, 900, 8)])
def test_finalize_bitexact(M, k, H, R, shift):
    rng = np.random.default_rng(M * k)
    rows_all = torch.from_numpy(rng.standard_normal((R * H + shift,)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    rows = rows_all[shift:].view(R, H)
    t2r = rng.integers(-1, R, size=(M, k)).astype(np.int32)
    w = rng.random((M, k)).astype(np.float32)
    w[t2r < 0] = np.nan                                   # scores of masked slots are never read
    out = torch.empty(M * H + shift, dtype=torch.bfloat16, device=DEV)[shift:].view(M, H)
    assert rows.data_ptr() % 32 == out.data_ptr() % 32 == 2 * shift % 32
    pkg.moe_finalize(rows, torch.from_numpy(w).to(DEV), torch.from_numpy(t2r).to(DEV), out)
    torch.cuda.synchronize()
    ref = O.finalize(bf16_np(rows), w, t2r)
    assert np.array_equal(bf16_np(out), ref)


@pytest.mark.parametrize("name,overrides", [("tiny", {}), ("decode_t8", {"H": 512, "E": 16}),
                                            ("relu2_ep", {"M": 700, "H": 384, "I": 256})])
def test_permute_bitexact(name, overrides):
    from gpu_harness import Problem
    cfg = mi.CONFIGS[name].with_(**overrides)
    p = Problem(cfg)
    p.run(do_finalize=True)
    b = p.bufs(True)
    offs = pkg.moe_forward_workspace_layout(cfg.M, cfg.top_k, p.layer.w, 1)
    ws = to_np(b["ws"])
    cap = b["capacity"]
    aq = ws[offs[0]:offs[0] + cap * cfg.H // 2].reshape(cap, cfg.H // 2)
    asf = sf_tiles_to_linear(ws[offs[1]:offs[2]], cap, cfg.H // 16)
    r2s = to_np(b["row_to_slot"])[:cap]
    xq, xsf, xs = p.oracle_inputs()
    real = r2s >= 0
    tok = r2s[real] // cfg.top_k
    assert np.array_equal(aq[real], xq[tok])
    assert np.array_equal(asf[real], xsf[tok])
    # scale columns of the K padding are zero in real rows
    kp = (cfg.H + 255) // 256 * 256
    if kp != cfg.H:
        pad = sf_tiles_to_linear(ws[offs[1]:offs[2]], cap, kp // 16)[real][:, cfg.H // 16:]
        assert not pad.any()


@pytest.mark.parametrize("rsf", [1.0, 0.75, 3.0])
def test_finalize_bf16_weights_and_scaling_bitexact(rsf):
    M, k, H, R = 50, 6, 512, 200
    rng = np.random.default_rng(11)
    rows = torch.from_numpy(rng.standard_normal((R, H)).astype(np.float32)).to(torch.bfloat16).to(DEV)
    t2r = rng.integers(-1, R, size=(M, k)).astype(np.int32)
    w16 = torch.from_numpy(rng.random((M, k)).astype(np.float32)).to(torch.bfloat16)
    out = torch.empty(M, H, dtype=torch.bfloat16, device=DEV)
    pkg.moe_finalize(rows, w16.to(DEV), torch.from_numpy(t2r).to(DEV), out, routed_scaling_factor=rsf)
    torch.cuda.synchronize()
    ref = O.finalize(bf16_np(rows), w16.float().numpy(), t2r, routed_scaling_factor=rsf)
    assert np.array_equal(bf16_np(out), ref)
