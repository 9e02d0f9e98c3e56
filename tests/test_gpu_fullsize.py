"""Full-size workloads, in the launch configuration the benchmark times: the plan and
the activation quantiser bit-exact over the whole batch, the weight encodings of the
sampled tokens' experts bit-exact, and the outputs of sampled tokens (computed one by
one by the oracle) within the path's tolerance."""
import numpy as np
import pytest
from gpu_harness import (Problem, assert_close_output, bf16_np, cfg_key, mi, oracle_expert, oracle_weights,
                         to_np)
from oracle import moe as O
from oracle.plan import make_plan

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _sample_tokens(cfg, ids, n):
    # first token, last token (ragged end), and tokens of the most-loaded local expert
    l = ids.astype(np.int64) - cfg.local_offset
    valid = (l >= 0) & (l < cfg.El)
    counts = np.bincount(l[valid], minlength=cfg.El)
    heavy = int(np.argmax(counts))
    heavy_tok = int(np.nonzero((l == heavy).any(axis=1))[0][0])
    cand = [0, cfg.M - 1, heavy_tok]
    out = []
    for t in cand:
        if t not in out:
            out.append(t)
    return out[:n]


@pytest.mark.parametrize("name,ntok", [("decode_t4", 2), ("decode_t8", 3), ("wide_decode", 1),
                                       ("prefill_uniform", 1), ("prefill_skewed", 1), ("relu2_ep", 2)])
def test_full_size_sampled(name, ntok):
    cfg = mi.CONFIGS[name]
    p = Problem(cfg)
    # the benchmark's path: one moe_routed_forward call; it equals the separate calls (whose
    # intermediates are checked below) bit for bit
    out = bf16_np(p.run_routed(True)).copy()
    assert p.layer.device_status(cfg.M, cfg.top_k, True) == 0
    assert np.array_equal(bf16_np(p.run(True)), out)
    b = p.bufs(True)
    assert int(to_np(b["dev_status"])[0]) == 0
    # plan, bit-exact over the whole batch
    ref_plan = make_plan(p.ids, cfg.local_offset, cfg.El)
    cap = b["capacity"]
    assert np.array_equal(to_np(b["padded_offsets"]), ref_plan["padded_offsets"])
    assert np.array_equal(to_np(b["row_to_slot"])[:cap], ref_plan["row_to_slot"])
    assert np.array_equal(to_np(b["token_to_row"]), ref_plan["token_to_row"])
    # activation quantiser, bit-exact over the whole batch
    xq, xsf, xs = p.oracle_inputs()
    assert np.array_equal(to_np(b["xq"]), xq)
    assert np.array_equal(to_np(b["xsf"]), xsf)
    assert np.array_equal(to_np(b["xs"]), xs)
    tokens = _sample_tokens(cfg, p.ids, ntok)
    # weight encodings of every expert the sampled tokens use
    key = cfg_key(cfg)
    for t in tokens:
        for j in range(cfg.top_k):
            l = int(p.ids[t, j]) - cfg.local_offset
            if 0 <= l < cfg.El:
                (d1, s1, a1), (d2, s2, a2) = oracle_expert(key, l)
                assert np.array_equal(to_np(p.q1[0][l]), d1) and np.array_equal(to_np(p.q1[1][l]), s1)
                assert np.array_equal(to_np(p.q2[0][l]), d2) and np.array_equal(to_np(p.q2[1][l]), s2)
                assert to_np(p.q1[2][l]) == a1 and to_np(p.q2[2][l]) == a2
    ref = O.forward_tokens(tokens, xq, xsf, xs, p.ids, p.tw, oracle_weights(cfg), cfg.act,
                           local_expert_offset=cfg.local_offset, fc2_input_scale=cfg.fc2_input_scale)
    assert_close_output(out[tokens], ref["out"], name)
    if name == "relu2_ep":
        # unfinalized mode at full size: the sampled tokens' expert rows
        g2, tw, t2r = p.run(False)
        g2n = bf16_np(g2)
        t2rn = to_np(t2r)
        for (t, j), row in ref["rows"].items():
            assert_close_output(g2n[t2rn[t, j]][None], row[None], f"{name} row {(t, j)}")
