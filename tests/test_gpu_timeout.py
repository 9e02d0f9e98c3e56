"""The GEMM kernels' bounded waits running out, through the test build (libmoe_nvfp4_test.so).

Every wait in the GEMM kernels gives up after a limit, sets MOE_DEV_TIMEOUT in the caller's
status word and lets the kernel drain its in-flight copies, release its tensor memory and
return. Normal inputs never reach that path; the test build's options do, without any fault:
the GEMM1 tiles of the first row tile (chained GEMMs) or of the first active expert (decode
GEMMs) withhold their completion release, so the GEMM2 tiles that read them wait on a counter
that nothing raises, and the wait limit is cut to 2 ms. The call must return, report the
timeout, and leave the context usable: the next normal call is bit-exact.
"""
import numpy as np
import pytest
import torch

from gpu_harness import Problem, bf16_np, mi, pkg

pytestmark = pytest.mark.gpu

CASES = {
    # 4 tokens: the decode-shaped GEMMs (weights as the 128-row MMA operand)
    "tiny": mi.CONFIGS["tiny"],
    # 300 tokens, 8 experts: the chained GEMM1 -> GEMM2 launch with per-row-tile counters
    "swiglu_ragged": mi.MoEConfig("swiglu_ragged", M=300, H=512, I=256, E=8, top_k=2, seed=11, weight_seed=11),
}


@pytest.mark.parametrize("do_finalize", [True, False])
@pytest.mark.parametrize("name", list(CASES))
def test_withheld_release_times_out_and_the_next_call_is_exact(name, do_finalize):
    cfg = CASES[name]
    p = Problem(cfg)
    mode = 1 if do_finalize else 0
    b = p.layer.routed_buffers(cfg.M, cfg.top_k, mode)
    key = "out" if do_finalize else "gemm2_out"

    def call(opts=None):
        b["dev_status"].zero_()
        p.layer.routed(p.x, p.ids_t, p.tw_t, b, mode, test_options=opts)
        torch.cuda.synchronize()
        return int(b["dev_status"][0].item()), bf16_np(b[key]).copy(), b["token_to_row"].cpu().numpy().copy()

    st, ref, t2r = call(pkg.test_options())          # the test build with default options
    assert st == 0
    real = t2r[t2r >= 0] if not do_finalize else slice(None)
    st, _, _ = call(pkg.test_options(withhold_release=True, wait_limit_ns=2_000_000))
    assert st & pkg.MOE_DEV_TIMEOUT, f"status {st}: the withheld counter's wait did not run out"
    st, got, t2r2 = call()                             # the product path, right after
    assert st == 0
    assert np.array_equal(t2r2, t2r)
    assert np.array_equal(got[real], ref[real])
