"""The C-ABI library loads, exports every entry point the header declares, and
validates arguments on the host (no GPU is touched by these calls)."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import nvfp4_routed_moe_sort_gb300 as pkg
from nvfp4_routed_moe_sort_gb300 import _lib as L
from nvfp4_routed_moe_sort_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_nvfp4.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return pkg.lib()


TEST_HEADER = os.path.join(ROOT, "include", "moe_nvfp4_test.h")


def _declared(header=HEADER):
    with open(header) as f:
        src = f.read()
    return sorted(set(re.findall(r"^MOE_API [^(]*?\b(moe_\w+)\(", src, flags=re.M)))


def test_header_declares_binding_names():
    assert _declared() == sorted(L.EXPORTED)
    assert _declared(TEST_HEADER) == sorted(L.TEST_EXPORTED)


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert pkg.moe_abi_version() == 3


def test_test_build_exports_product_and_test_symbols(lib):
    tl = pkg.test_lib()
    for name in _declared() + _declared(TEST_HEADER):
        assert hasattr(tl, name), name
    o = pkg.test_options()
    assert (o.decode_hooks, o.withhold_release, o.wait_limit_ns) == (0, 0, 2_000_000_000)


def test_product_library_exports_no_test_hooks(lib):
    """The test hooks (standalone GEMM1, decode scheduling fallbacks, shortened waits) live in
    the test build only: the product library exports no moe_test_* or moe_debug_* symbol."""
    for name in _declared(TEST_HEADER) + ["moe_debug_gemm1", "moe_debug_set_decode_hooks"]:
        assert not hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", pkg.LIB_PATH], capture_output=True, text=True)
    if out.returncode == 0:
        exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
        assert sorted(n for n in exported if n.startswith("moe_")) == sorted(L.EXPORTED)


def test_status_strings(lib):
    assert pkg.status_string(0) == "MOE_OK"
    assert pkg.status_string(4) == "MOE_ERR_WORKSPACE_TOO_SMALL"
    assert pkg.status_string(99) == "MOE_ERR_UNKNOWN"


def test_capacity_matches_oracle(lib):
    from oracle.plan import plan_capacity
    for M, k, El in [(0, 2, 4), (4, 2, 4), (8, 10, 128), (4096, 8, 256), (16384, 6, 64), (1, 1, 1)]:
        assert pkg.moe_plan_capacity(M, k, El) == plan_capacity(M, k, El)


# The checks below pass made-up device addresses that every call must reject on the
# host before launching anything; they run only where no GPU could execute a launch.
host_only = pytest.mark.skipif(torch.cuda.is_available(), reason="fake device pointers: host-only check")


def _w(El=4, H=128, I=128, act=0):
    return L.make_weights(El, H, I, act)


def test_size_queries(lib):
    w = _w()
    assert pkg.moe_prepared_weights_bytes(w) > 0
    assert pkg.moe_forward_workspace_bytes(4, 2, w, 1) > pkg.moe_forward_workspace_bytes(4, 2, w, 0)
    off = pkg.moe_forward_workspace_layout(4, 2, w, 1)
    assert off[0] >= 0 and all(o % 256 == 0 for o in off) and off[5] == pkg.moe_forward_workspace_bytes(4, 2, w, 1)
    # accumulated output: an FP32 [M, H] accumulator instead of BF16 rows [capacity, H]
    acc = pkg.moe_forward_workspace_layout(4, 2, w, 2)
    assert acc[5] - acc[4] >= 4 * 4 * 128 and acc[5] < off[5]
    assert pkg.moe_forward_workspace_bytes(4, 2, w, 3) == 0      # unknown output mode
    assert pkg.moe_plan_workspace_bytes(4, 2, 4) == 0            # one block: no scratch
    assert pkg.moe_plan_workspace_bytes(4096, 8, 256) > 0


@host_only
def test_shape_validation(lib):
    # H or I not a multiple of 128, too many experts, bad enums -> size 0 / error status
    assert pkg.moe_prepared_weights_bytes(_w(H=192)) == 0
    assert pkg.moe_prepared_weights_bytes(_w(I=64)) == 0
    assert pkg.moe_prepared_weights_bytes(_w(El=513)) == 0
    assert pkg.moe_prepared_weights_bytes(_w(act=7)) == 0
    f = lib.moe_quantize_input
    assert f(None, 4, 96, 96, 0, None, None, None, None) == 2      # H % 128
    assert f(None, 4, 128, 128, 5, None, None, None, None) == 1    # bad mode
    assert f(None, 4, 128, 64, 0, None, None, None, None) == 1     # ld_x < H
    assert f(None, 0, 128, 128, 0, None, None, None, None) == 0    # M == 0 is a no-op
    assert f(None, 4, 128, 128, 0, None, None, None, None) == 1    # null pointers


@host_only
def test_plan_validation(lib):
    f = lib.moe_plan
    # local range outside the global expert count
    assert f(None, 0, 4, 2, 8, 6, 4, None, None, None, None, None, 0, None, None) == 1
    # too many local experts
    assert f(None, 0, 4, 2, 1024, 0, 600, None, None, None, None, None, 0, None, None) == 2
    # misaligned counts pointer
    assert f(16, 0, 4, 2, 8, 0, 4, 8, 32, 48, 64, None, 0, 96, None) == 3
    # workspace too small for the multi-block path (plain and packed ids)
    assert f(16, 0, 4096, 8, 256, 0, 256, 16, 32, 48, 64, None, 0, 96, None) == 4
    assert f(16, 1, 4096, 8, 256, 0, 256, 16, 32, 48, 64, None, 0, 96, None) == 4
    # unknown id format
    assert f(16, 2, 4, 2, 8, 0, 4, 16, 32, 48, 64, None, 0, 96, None) == 1
    assert lib.moe_plan_noalloc(16, 7, 4, 2, 8, 0, 4, 16, 32, 48, 64, 96, None) == 1


@host_only
def test_forward_validation(lib):
    w = _w()
    f = lib.moe_grouped_fp4_forward
    null = None
    # missing prepared buffer
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), null, 0, 112, 0, 1.0, 1.0, 1, 128, null, 144, 1 << 30,
           160, null, 0, null)
    assert st == 1
    # workspace too small
    pb = pkg.moe_prepared_weights_bytes(w)
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 0, 1.0, 1.0, 1, 128, null, 144, 16,
           160, null, 0, null)
    assert st == 4
    # bad fc2_input_scale
    ws = pkg.moe_forward_workspace_bytes(4, 2, w, 1)
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 0, 1.0, 0.0, 1, 1 << 40, null, 1 << 36, ws,
           160, null, 0, null)
    assert st == 1
    # out overlapping the workspace
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 0, 1.0, 1.0, 1, 1 << 36, null, 1 << 36, ws,
           160, null, 0, null)
    assert st == 6
    # step events: count must be 0 or 5
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 0, 1.0, 1.0, 1, 1 << 40, null, 1 << 36, ws,
           160, null, 3, null)
    assert st == 1
    # unknown output mode; unknown route-weight storage
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 0, 1.0, 1.0, 3, 1 << 40, null, 1 << 36, ws,
           160, null, 0, null)
    assert st == 1
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 3, 1.0, 1.0, 1, 1 << 40, null, 1 << 36, ws,
           160, null, 0, null)
    assert st == 1
    # accumulated output needs out, and out must not overlap the workspace
    wsa = pkg.moe_forward_workspace_bytes(4, 2, w, 2)
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 2, 1.0, 1.0, 2, null, null, 1 << 36, wsa,
           160, null, 0, null)
    assert st == 1
    st = f(16, 32, 48, 4, 2, 64, 80, 96, ctypes.byref(w), 4096, pb, 112, 2, 1.0, 1.0, 2, 1 << 36, null, 1 << 36, wsa,
           160, null, 0, null)
    assert st == 6


@host_only
def test_routed_forward_validation(lib):
    w = _w()
    f = lib.moe_routed_forward
    pb = pkg.moe_prepared_weights_bytes(w)
    ws = pkg.moe_routed_forward_workspace_bytes(4, 2, w, 1)
    assert ws > pkg.moe_forward_workspace_bytes(4, 2, w, 1)
    assert pkg.moe_routed_forward_workspace_bytes(4, 2, w, 5) == 0

    def call(x=1 << 20, ld=128, mode=1, ids=2 << 20, fmt=0, E=4, off=0, wt=3 << 20, dt=0, g2=1.0, fin=1,
             out=4 << 20, t2r=5 << 20, wsp=1 << 36, wsb=ws, nev=0):
        return f(x, 4, ld, mode, ids, fmt, 2, E, off, wt, dt, 1.0, ctypes.byref(w), 6 << 20, pb, g2, fin, out, None,
                 t2r, wsp, wsb, 7 << 20, None, nev, None)
    assert call(ld=120) == 1                 # ld_x < H
    assert call(mode=3) == 1                 # bad activation-scale mode
    assert call(fmt=4) == 1                  # bad id format
    assert call(E=3) == 1                    # local range past the expert count
    assert call(g2=0.0) == 1                 # fc2_input_scale must be positive
    assert call(nev=2) == 1                  # step events: 0 or 5
    assert call(wsb=ws - 1) == 4             # workspace too small
    assert call(x=(1 << 20) + 8) == 3        # misaligned hidden states
    assert call(out=1 << 20) == 6            # out overlaps the hidden states
    assert call(t2r=(4 << 20) + 64) == 6     # token_to_row overlaps out


@host_only
def test_finalize_validation(lib):
    f = lib.moe_finalize
    assert f(16, 32, 0, 1.0, 48, 4, 2, 100, 64, None) == 2         # H % 128
    assert f(16, 32, 0, 1.0, 48, 4, 0, 128, 64, None) == 1         # top_k == 0
    assert f(16, 32, 0, 1.0, 48, 4, 2, 128, 24, None) == 3         # misaligned out
    assert f(16, 32, 0, 1.0, 48, 0, 2, 128, 64, None) == 0         # M == 0 no-op
    assert f(16, 32, 5, 1.0, 48, 4, 2, 128, 64, None) == 1         # bad weights dtype
    assert f(16, 32, 2, 1.0, 48, 0, 2, 128, 64, None) == 0         # packed weights accepted
    assert f(16, 32, 0, float("inf"), 48, 4, 2, 128, 64, None) == 1  # non-finite scaling factor


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(pkg.MoEError):
        L.lib()
