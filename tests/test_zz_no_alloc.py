"""moe_plan_noalloc: the routing plan for callers that cannot allocate device memory.

Some users of this library run where device allocation is not allowed after start-up
(serving runtimes with one pre-reserved memory pool, C hosts without a device allocator,
code that must not let cudaMalloc synchronise the device). moe_plan_noalloc gives them the
plan with no workspace argument: its scratch is a fixed array inside the library. These
tests call it through the C ABI twice in a row, on problems of different shapes (so the
second call runs over what the first left in the shared array), and require the result to
equal moe_plan's exactly. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import nvfp4_routed_moe_sort_gb300 as pkg
from nvfp4_routed_moe_sort_gb300.build import build

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _plan_both(ids, E, off, El):
    M, k = ids.shape
    cap = pkg.moe_plan_capacity(M, k, El)
    ids_t = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(DEV)

    def bufs():
        return (torch.full((El,), -7, dtype=torch.int32, device=DEV),
                torch.full((El + 1,), -7, dtype=torch.int32, device=DEV),
                torch.full((max(cap, 1),), 999, dtype=torch.int32, device=DEV),
                torch.full((M, k), 999, dtype=torch.int32, device=DEV),
                torch.zeros(4, dtype=torch.int32, device=DEV))

    a = bufs()
    ws = torch.empty(max(pkg.moe_plan_workspace_bytes(M, k, El), 16), dtype=torch.uint8, device=DEV)
    pkg.moe_plan(ids_t, E, off, El, a[0], a[1], a[2], a[3], ws, a[4])
    b = bufs()
    pkg.moe_plan_noalloc(ids_t, E, off, El, b[0], b[1], b[2], b[3], b[4])
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in a], [t.cpu().numpy() for t in b], cap


def _assert_same(a, b, cap):
    names = ["counts", "padded_offsets", "row_to_slot", "token_to_row", "dev_status"]
    for n, x, y in zip(names, a, b):
        if n == "row_to_slot":
            x, y = x[:cap], y[:cap]
        assert np.array_equal(x, y), n


def test_plan_noalloc_matches_plan_on_two_calls_in_a_row():
    build()
    # call 1: prefill routing, 256 experts, 16 slot blocks (multi-block path, scratch used)
    cfg1 = mi.CONFIGS["prefill_skewed"]
    ids1, _ = mi.routing(cfg1)
    a, b, cap = _plan_both(ids1, cfg1.E, 0, cfg1.El)
    _assert_same(a, b, cap)
    # call 2: a different shape and expert-parallel masking over what call 1 left behind
    cfg2 = mi.CONFIGS["relu2_ep"].with_(M=5000)
    ids2, _ = mi.routing(cfg2)
    ids2 = mi.with_unrouted(ids2, 0.05, 2, cfg2.E)
    a, b, cap = _plan_both(ids2, cfg2.E, cfg2.local_offset, cfg2.El)
    _assert_same(a, b, cap)


def test_plan_noalloc_small_input_and_size_limit():
    build()
    cfg = mi.CONFIGS["decode_t8"]
    ids, _ = mi.routing(cfg)
    a, b, cap = _plan_both(ids, cfg.E, 0, cfg.El)        # one block: no scratch needed
    _assert_same(a, b, cap)
    # more histogram entries than the fixed array holds: rejected on the host, nothing runs
    M, k, El = 1 << 20, 2, 512                           # 1024 blocks x 512 experts x 4 B > 1 MiB
    one = torch.zeros(16, dtype=torch.int32, device=DEV)
    st = pkg.lib().moe_plan_noalloc(one.data_ptr(), 0, M, k, El, 0, El, one.data_ptr(), one.data_ptr(),
                                    one.data_ptr(), one.data_ptr(), one.data_ptr(), None)
    assert st == 2                                       # MOE_ERR_UNSUPPORTED_SHAPE
