"""Full-size workloads, in the launch configuration the benchmark times (one
moe_routed_forward call).

* The plan and the activation quantiser are bit-exact over the whole batch, and the one-call
  path equals the separate calls bit for bit.
* Expert rows (the unfinalized gemm2_out) are compared with the oracle on a stratified sample
  that reaches every active local expert: its first row, its last real row (the ragged end of
  its segment) and one row of each further 128-row tile, so every expert index, every row
  tile count and both tile kinds (dense and ragged) of the persistent scheduler are covered.
  Decode-sized batches compare every row and every token's finalized output.
* Every local expert's weight encoding (codes, scales, alpha of W1 and W2) equals the
  oracle's own encoding of the same BF16 weights, compared through a digest.

The oracle's per-expert work runs in a spawn-started process pool (tests/oracle_pool.py).
"""
import numpy as np
import pytest
import torch

from gpu_harness import DEV, Problem, assert_close_output, bf16_np, mi, to_np
from oracle import moe as O
from oracle import quantize as Q
from oracle.plan import make_plan
from oracle_pool import pack_digest, run_experts

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

PER_EXPERT_SCREEN = 0.1   # relative Frobenius error of one expert's sampled rows


@pytest.mark.parametrize("name", ["decode_t4", "decode_t8", "wide_decode", "prefill_uniform", "prefill_skewed",
                                  "relu2_ep"])
def test_full_size_plan_and_quantiser(name):
    cfg = mi.CONFIGS[name]
    p = Problem(cfg)
    out = bf16_np(p.run_routed(True)).copy()
    assert p.layer.device_status(cfg.M, cfg.top_k, True) == 0
    # the benchmark's path (one call) equals the separate calls, whose intermediates are kept
    assert np.array_equal(bf16_np(p.run(True)), out)
    b = p.bufs(True)
    assert int(to_np(b["dev_status"])[0]) == 0
    ref_plan = make_plan(p.ids, cfg.local_offset, cfg.El)
    cap = b["capacity"]
    assert np.array_equal(to_np(b["counts"]), ref_plan["counts"])
    assert np.array_equal(to_np(b["padded_offsets"]), ref_plan["padded_offsets"])
    assert np.array_equal(to_np(b["row_to_slot"])[:cap], ref_plan["row_to_slot"])
    assert np.array_equal(to_np(b["token_to_row"]), ref_plan["token_to_row"])
    xq, xsf, xs = p.oracle_inputs()
    assert np.array_equal(to_np(b["xq"]), xq)
    assert np.array_equal(to_np(b["xsf"]), xsf)
    assert np.array_equal(to_np(b["xs"]), xs)


def stratified_rows(plan) -> np.ndarray:
    """Per local expert with routed rows: the first row of its segment, its last real row,
    and one row of each further 128-row tile (position inside the tile varied by expert)."""
    sel = []
    for l, c in enumerate(plan["counts"]):
        c = int(c)
        if c == 0:
            continue
        p0 = int(plan["padded_offsets"][l])
        rows = {p0, p0 + c - 1}
        for i in range(1, (c + 127) // 128):
            span = min(128, c - 128 * i)
            rows.add(p0 + 128 * i + (l * 37 + i * 11) % span)
        sel += sorted(rows)
    return np.array(sel, dtype=np.int64)


class Case:
    """One workload on a shared layer: GPU results of the one-call path and the plan rows to check."""

    def __init__(self, cfg, layer, all_rows: bool, full_tokens=()):
        self.cfg = cfg
        x = mi.hidden_bf16(cfg, DEV)
        self.ids, self.tw = mi.routing(cfg)
        ids_t = torch.from_numpy(np.ascontiguousarray(self.ids)).to(DEV)
        tw_t = torch.from_numpy(np.ascontiguousarray(self.tw)).to(DEV)
        self.plan = make_plan(self.ids, cfg.local_offset, cfg.El)
        k = cfg.top_k
        r2s = self.plan["row_to_slot"]
        real = np.nonzero(r2s >= 0)[0]
        rows = real if all_rows else stratified_rows(self.plan)
        # every slot of the fully checked tokens, for their finalized output
        self.full_tokens = list(full_tokens)
        t2r = self.plan["token_to_row"]
        extra = [int(t2r[t, j]) for t in self.full_tokens for j in range(k) if t2r[t, j] >= 0]
        self.rows = np.unique(np.concatenate([rows, np.array(extra, dtype=np.int64)]))
        g2, _, t2r_gpu = layer.forward(x, ids_t, tw_t, do_finalize=False)
        torch.cuda.synchronize()
        assert np.array_equal(to_np(t2r_gpu), t2r)
        self.gpu_rows = bf16_np(g2[torch.from_numpy(self.rows).to(DEV)])
        out = layer.forward(x, ids_t, tw_t, do_finalize=True)
        torch.cuda.synchronize()
        self.gpu_out = bf16_np(out)[self.full_tokens] if self.full_tokens else None
        assert layer.device_status(cfg.M, k, False) == 0 and layer.device_status(cfg.M, k, True) == 0
        self.xq, self.xsf, self.xs = Q.quantize_activations(x.float().cpu().numpy(), cfg.scale_mode)
        slots = r2s[self.rows]
        self.tok = slots // k
        self.expert = self.ids.reshape(-1)[slots].astype(np.int64) - cfg.local_offset
        self.ref_rows = np.full(self.gpu_rows.shape, np.nan)


def check_weight_set(p: Problem, cases):
    """Oracle rows for every case's sampled plan rows (one pool task per local expert, shared by
    the cases that use the same weights), every expert's weight encoding, and the comparisons."""
    cfg0 = p.cfg

    def tasks():
        for l in range(cfg0.El):
            picks = [(ci, np.nonzero(c.expert == l)[0]) for ci, c in enumerate(cases)]
            xq = np.concatenate([c.xq[c.tok[ix]] for (ci, ix), c in zip(picks, cases)])
            xsf = np.concatenate([c.xsf[c.tok[ix]] for (ci, ix), c in zip(picks, cases)])
            xs = np.concatenate([c.xs[c.tok[ix]] for (ci, ix), c in zip(picks, cases)])
            yield {"l": l, "picks": picks, "w1_bits": p.w1_bf16[l].view(torch.int16).cpu().numpy(),
                   "w2_bits": p.w2_bf16[l].view(torch.int16).cpu().numpy(), "xq": xq, "xsf": xsf, "xs": xs,
                   "act": cfg0.act, "inter": cfg0.I, "fc2_input_scale": cfg0.fc2_input_scale}

    picks_of = {}

    def tagged():
        for t in tasks():
            picks_of[t["l"]] = t.pop("picks")
            yield t

    mismatched = []
    for res in run_experts(tagged()):
        l = res["l"]
        gpu_digest = pack_digest(to_np(p.q1[0][l]), to_np(p.q1[1][l]), to_np(p.q1[2][l]), to_np(p.q2[0][l]),
                                 to_np(p.q2[1][l]), to_np(p.q2[2][l]))
        if gpu_digest != res["digest"]:
            mismatched.append(l)
        at = 0
        for ci, ix in picks_of.pop(l):
            if len(ix):
                cases[ci].ref_rows[ix] = res["rows"][at:at + len(ix)]
                at += len(ix)
    assert not mismatched, f"weight encodings differ from the oracle's for experts {mismatched[:10]}"
    for c in cases:
        name = c.cfg.name
        assert not np.isnan(c.ref_rows).any(), name
        # the required output tolerance over all sampled expert rows of the workload
        assert_close_output(c.gpu_rows, c.ref_rows, f"{name} all sampled rows")
        # and a per-expert screen: a row of the wrong expert, token or tile, stale operands or a
        # wrong scale give errors of the order of the rows themselves (relative error ~1), while
        # one requantised intermediate value landing on the other side of an E2M1 or E4M3
        # rounding boundary (FP32 accumulation order moves a BF16 intermediate by one ulp) moves
        # a decode-sized row (I = 512) by 1-3 %
        worst = (-1.0, -1)
        for l in np.unique(c.expert):
            m = c.expert == l
            err = np.linalg.norm(c.gpu_rows[m] - c.ref_rows[m]) / max(np.linalg.norm(c.ref_rows[m]), 1e-30)
            worst = max(worst, (err, int(l)))
        assert worst[0] <= PER_EXPERT_SCREEN, f"{name}: expert {worst[1]} rows off by {worst[0]:.3e}"
        print(f"{name}: {len(c.rows)} rows of {len(np.unique(c.expert))} experts, worst expert rel {worst[0]:.2e}")
        if c.full_tokens:
            # finalized output of the fully checked tokens from the oracle's rows
            k = c.cfg.top_k
            pos = {int(r): i for i, r in enumerate(c.rows)}
            t2r = c.plan["token_to_row"]
            sub = np.full((len(c.full_tokens), k), -1, dtype=np.int64)
            for i, t in enumerate(c.full_tokens):
                for j in range(k):
                    if t2r[t, j] >= 0:
                        sub[i, j] = pos[int(t2r[t, j])]
            ref = O.finalize(c.ref_rows, c.tw[c.full_tokens], sub)
            assert_close_output(c.gpu_out, ref, f"{name} finalized tokens")


def test_full_size_rows_h7168_i2048():
    """Prefill 4k uniform and Zipf-skewed (stratified rows of all 256 experts, tokens 0 and
    M-1 in full) and wide decode T=8 (every row and token), one weight set."""
    base = mi.CONFIGS["prefill_uniform"]
    p = Problem(base)
    cases = [Case(base, p.layer, False, (0, base.M - 1)),
             Case(mi.CONFIGS["prefill_skewed"], p.layer, False, (0, base.M - 1)),
             Case(mi.CONFIGS["wide_decode"], p.layer, True, range(mi.CONFIGS["wide_decode"].M))]
    check_weight_set(p, cases)


def test_full_size_rows_relu2_ep():
    """Squared-ReLU with experts 0-63 local of 128, 16k tokens: stratified rows of every local
    expert (about 6 row tiles each), tokens 0 and M-1 in full."""
    cfg = mi.CONFIGS["relu2_ep"]
    p = Problem(cfg)
    check_weight_set(p, [Case(cfg, p.layer, False, (0, cfg.M - 1))])


def test_full_size_rows_decode():
    """Decode T=4 and T=8 (H=2048, I=512, 128 experts, top-10): every row and every token."""
    base = mi.CONFIGS["decode_t8"]
    p = Problem(base)
    cases = [Case(mi.CONFIGS[n], p.layer, True, range(mi.CONFIGS[n].M)) for n in ("decode_t4", "decode_t8")]
    check_weight_set(p, cases)
