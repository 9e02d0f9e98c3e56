"""ctypes binding of libmoe_nvfp4.so (the C ABI in include/moe_nvfp4.h) and of the test
build libmoe_nvfp4_test.so (include/moe_nvfp4_test.h, loaded only by test_lib()).

Argument marshalling only: every function here turns torch tensors into device
pointers, passes torch's current CUDA stream and raises on a non-OK status. All of
the path runs in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_int64, c_size_t, c_void_p

from .build import LIB as LIB_PATH
from .build import TEST_LIB as TEST_LIB_PATH

_lib = None
_test_lib = None

MOE_OK = 0
MOE_ACT_SWIGLU, MOE_ACT_RELU2, MOE_ACT_GEGLU, MOE_ACT_GELU, MOE_ACT_RELU, MOE_ACT_SILU, MOE_ACT_IDENTITY = range(7)
ACTIVATIONS = {"swiglu": MOE_ACT_SWIGLU, "relu2": MOE_ACT_RELU2, "geglu": MOE_ACT_GEGLU, "gelu": MOE_ACT_GELU,
               "relu": MOE_ACT_RELU, "silu": MOE_ACT_SILU, "identity": MOE_ACT_IDENTITY}
MOE_SCALE_GLOBAL_ONE, MOE_SCALE_PER_TOKEN = 0, 1
MOE_DEV_DUPLICATE_EXPERT, MOE_DEV_TIMEOUT = 1, 2
MOE_WEIGHTS_F32, MOE_WEIGHTS_BF16, MOE_WEIGHTS_PACKED = 0, 1, 2
MOE_IDS_INT32, MOE_IDS_PACKED = 0, 1
MOE_OUTPUT_UNFINALIZED, MOE_OUTPUT_FINALIZED, MOE_OUTPUT_ACCUMULATE = 0, 1, 2

EXPORTED = [
    "moe_status_string", "moe_abi_version", "moe_quantize_input", "moe_plan_capacity",
    "moe_plan_workspace_bytes", "moe_plan", "moe_quantize_weights", "moe_prepared_weights_bytes",
    "moe_prepare_weights", "moe_forward_workspace_bytes", "moe_forward_workspace_layout",
    "moe_grouped_fp4_forward", "moe_finalize", "moe_plan_noalloc",
    "moe_routed_forward_workspace_bytes", "moe_routed_forward",
]
# the test build's extra entry points (include/moe_nvfp4_test.h)
TEST_EXPORTED = ["moe_test_default_options", "moe_test_routed_forward", "moe_test_gemm1"]
MOE_PLAN_NOALLOC_SCRATCH_BYTES = 1 << 20


class MoEError(RuntimeError):
    pass


class WeightsT(ctypes.Structure):
    """moe_nvfp4_weights_t"""
    _fields_ = [
        ("w1", c_void_p), ("w1_sf", c_void_p), ("w1_alpha", c_void_p),
        ("w2", c_void_p), ("w2_sf", c_void_p), ("w2_alpha", c_void_p),
        ("num_local_experts", c_int32), ("hidden", c_int32), ("inter", c_int32),
        ("activation", c_int32), ("w1_gate_alpha", c_void_p),
    ]


class TestOptionsT(ctypes.Structure):
    """moe_test_options_t"""
    _fields_ = [("decode_hooks", c_int32), ("withhold_release", c_int32), ("wait_limit_ns", ctypes.c_uint64)]


# moe_routed_forward's arguments up to (not including) the stream
_ROUTED_ARGS = [c_void_p, c_int32, c_int64, c_int32, c_void_p, c_int32, c_int32, c_int32, c_int32, c_void_p,
                c_int32, c_float, ctypes.POINTER(WeightsT), c_void_p, c_size_t, c_float, c_int32, c_void_p, c_void_p,
                c_void_p, c_void_p, c_size_t, c_void_p, ctypes.POINTER(c_void_p), c_int32]


def _declare(lib, test=False):
    P = c_void_p
    routed = list(_ROUTED_ARGS)
    sig = {
        "moe_status_string": (ctypes.c_char_p, [c_int32]),
        "moe_abi_version": (c_int32, []),
        "moe_quantize_input": (c_int32, [P, c_int32, c_int32, c_int64, c_int32, P, P, P, P]),
        "moe_plan_capacity": (c_size_t, [c_int32, c_int32, c_int32]),
        "moe_plan_workspace_bytes": (c_size_t, [c_int32, c_int32, c_int32]),
        "moe_plan": (c_int32, [P, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, P, P, P, P, P,
                               c_size_t, P, P]),
        "moe_plan_noalloc": (c_int32, [P, c_int32, c_int32, c_int32, c_int32, c_int32, c_int32, P, P, P, P,
                                       P, P]),
        "moe_quantize_weights": (c_int32, [P, c_int32, c_int32, c_int32, P, P, P, P, P]),
        "moe_prepared_weights_bytes": (c_size_t, [ctypes.POINTER(WeightsT)]),
        "moe_prepare_weights": (c_int32, [ctypes.POINTER(WeightsT), P, c_size_t, P]),
        "moe_forward_workspace_bytes": (c_size_t, [c_int32, c_int32, ctypes.POINTER(WeightsT), c_int32]),
        "moe_forward_workspace_layout": (c_int32, [c_int32, c_int32, ctypes.POINTER(WeightsT), c_int32,
                                                   ctypes.POINTER(c_size_t)]),
        "moe_grouped_fp4_forward": (c_int32, [P, P, P, c_int32, c_int32, P, P, P, ctypes.POINTER(WeightsT),
                                              P, c_size_t, P, c_int32, c_float, c_float, c_int32, P, P, P,
                                              c_size_t, P, ctypes.POINTER(c_void_p), c_int32, P]),
        "moe_finalize": (c_int32, [P, P, c_int32, c_float, P, c_int32, c_int32, c_int32, P, P]),
        "moe_routed_forward_workspace_bytes": (c_size_t, [c_int32, c_int32, ctypes.POINTER(WeightsT), c_int32]),
        "moe_routed_forward": (c_int32, routed + [P]),
    }
    if test:
        sig.update({
            "moe_test_default_options": (TestOptionsT, []),
            "moe_test_routed_forward": (c_int32, routed + [ctypes.POINTER(TestOptionsT), P]),
            "moe_test_gemm1": (c_int32, [P, P, c_int32, c_int32, P, P, P, ctypes.POINTER(WeightsT), P,
                                         c_size_t, c_int32, P, P, c_size_t, P, P]),
        })
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoEError(f"{LIB_PATH} is missing: build it first (nvfp4_routed_moe_sort_gb300.build, "
                           "nvcc for sm_103a); there is no fallback path")
        _lib = ctypes.CDLL(LIB_PATH)
        _declare(_lib)
    return _lib


def test_lib():
    """The test build (libmoe_nvfp4_test.so): every product entry point plus those of
    include/moe_nvfp4_test.h. Only tests load it."""
    global _test_lib
    if _test_lib is None:
        if not os.path.exists(TEST_LIB_PATH):
            raise MoEError(f"{TEST_LIB_PATH} is missing: build it first (nvfp4_routed_moe_sort_gb300.build)")
        _test_lib = ctypes.CDLL(TEST_LIB_PATH)
        _declare(_test_lib, test=True)
    return _test_lib


def test_options(decode_hooks: int = 0, withhold_release: bool = False, wait_limit_ns: int | None = None):
    """moe_test_options_t from the test build's defaults, with the given fields changed."""
    o = test_lib().moe_test_default_options()
    o.decode_hooks = int(decode_hooks)
    o.withhold_release = int(bool(withhold_release))
    if wait_limit_ns is not None:
        o.wait_limit_ns = int(wait_limit_ns)
    return o


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoEError(f"{what}: {status_string(code)}")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def make_weights(num_local_experts: int, hidden: int, inter: int, activation: int,
                 w1=None, w1_sf=None, w1_alpha=None, w2=None, w2_sf=None, w2_alpha=None,
                 w1_gate_alpha=None) -> WeightsT:
    return WeightsT(_ptr(w1), _ptr(w1_sf), _ptr(w1_alpha), _ptr(w2), _ptr(w2_sf), _ptr(w2_alpha),
                    num_local_experts, hidden, inter, activation, _ptr(w1_gate_alpha))


# ---------------------------------------------------------------- entry points
def moe_abi_version() -> int:
    return lib().moe_abi_version()


def moe_quantize_input(x, mode, xq, xsf, xs, stream=None):
    M, H = x.shape
    _check(lib().moe_quantize_input(_ptr(x), M, H, x.stride(0), mode, _ptr(xq), _ptr(xsf), _ptr(xs),
                                    _stream(stream)), "moe_quantize_input")


def moe_plan_capacity(M, top_k, num_local_experts) -> int:
    return lib().moe_plan_capacity(M, top_k, num_local_experts)


def moe_plan_workspace_bytes(M, top_k, num_local_experts) -> int:
    return lib().moe_plan_workspace_bytes(M, top_k, num_local_experts)


def moe_plan(topk_ids, num_experts, local_expert_offset, num_local_experts, counts, padded_offsets,
             row_to_slot, token_to_row, workspace, dev_status, stream=None, packed=False):
    """packed=True: topk_ids holds packed slots (BF16 score << 16 | expert id)."""
    M, k = topk_ids.shape
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fmt = MOE_IDS_PACKED if packed else MOE_IDS_INT32
    _check(lib().moe_plan(_ptr(topk_ids), fmt, M, k, num_experts, local_expert_offset, num_local_experts,
                          _ptr(counts), _ptr(padded_offsets), _ptr(row_to_slot), _ptr(token_to_row),
                          _ptr(workspace), wsb, _ptr(dev_status), _stream(stream)), "moe_plan")


def moe_plan_noalloc(topk_ids, num_experts, local_expert_offset, num_local_experts, counts, padded_offsets,
                     row_to_slot, token_to_row, dev_status, stream=None, packed=False):
    """moe_plan without a workspace, for callers that cannot allocate device memory (its
    histogram scratch is a fixed 1 MiB array inside the library; see the C header)."""
    M, k = topk_ids.shape
    fmt = MOE_IDS_PACKED if packed else MOE_IDS_INT32
    _check(lib().moe_plan_noalloc(_ptr(topk_ids), fmt, M, k, num_experts, local_expert_offset, num_local_experts,
                                  _ptr(counts), _ptr(padded_offsets), _ptr(row_to_slot), _ptr(token_to_row),
                                  _ptr(dev_status), _stream(stream)), "moe_plan_noalloc")


def moe_quantize_weights(w, data, sf, alpha, amax_scratch, stream=None):
    E, R, C = w.shape
    _check(lib().moe_quantize_weights(_ptr(w), E, R, C, _ptr(data), _ptr(sf), _ptr(alpha),
                                      _ptr(amax_scratch), _stream(stream)), "moe_quantize_weights")


def moe_prepared_weights_bytes(w: WeightsT) -> int:
    return lib().moe_prepared_weights_bytes(ctypes.byref(w))


def moe_prepare_weights(w: WeightsT, prepared, stream=None):
    _check(lib().moe_prepare_weights(ctypes.byref(w), _ptr(prepared), prepared.numel() * prepared.element_size(),
                                     _stream(stream)), "moe_prepare_weights")


def moe_forward_workspace_bytes(M, top_k, w: WeightsT, do_finalize) -> int:
    return lib().moe_forward_workspace_bytes(M, top_k, ctypes.byref(w), int(do_finalize))


def moe_forward_workspace_layout(M, top_k, w: WeightsT, do_finalize) -> list[int]:
    arr = (c_size_t * 6)()
    _check(lib().moe_forward_workspace_layout(M, top_k, ctypes.byref(w), int(do_finalize), arr),
           "moe_forward_workspace_layout")
    return list(arr)


def _weights_dtype(topk_weights) -> int:
    """float32 / bfloat16 route weights, or int32 packed slots (BF16 score in bits 31..16)."""
    import torch
    if topk_weights.dtype == torch.bfloat16:
        return MOE_WEIGHTS_BF16
    if topk_weights.dtype == torch.float32:
        return MOE_WEIGHTS_F32
    if topk_weights.dtype == torch.int32:
        return MOE_WEIGHTS_PACKED
    raise MoEError("topk_weights must be float32, bfloat16 or int32 (packed)")


def _events(step_events):
    if not step_events:
        return None, 0
    handles = [e.cuda_event for e in step_events]
    if not all(handles):
        raise MoEError("step_events: torch creates an event on its first record(); record each once first")
    return (c_void_p * len(step_events))(*handles), len(step_events)


def moe_routed_forward_workspace_bytes(M, top_k, w: WeightsT, do_finalize) -> int:
    return lib().moe_routed_forward_workspace_bytes(M, top_k, ctypes.byref(w), int(do_finalize))


def moe_routed_forward(x, act_scale_mode, topk_ids, num_experts, local_expert_offset, topk_weights, w: WeightsT,
                       prepared, fc2_input_scale, do_finalize, out, gemm2_out, token_to_row, workspace, dev_status,
                       step_events=None, stream=None, routed_scaling_factor=1.0, packed=False, test_options=None):
    """The whole layer from BF16 hidden states x [M, H] (one C call). packed=True: topk_ids holds
    packed slots (and topk_weights may be the same tensor). test_options (a TestOptionsT from
    test_options()): call the test build's moe_test_routed_forward instead."""
    M, k = topk_ids.shape
    ev, nev = _events(step_events)
    args = (_ptr(x), M, x.stride(0), act_scale_mode, _ptr(topk_ids), MOE_IDS_PACKED if packed else MOE_IDS_INT32, k,
            num_experts, local_expert_offset, _ptr(topk_weights), _weights_dtype(topk_weights),
            float(routed_scaling_factor), ctypes.byref(w), _ptr(prepared), prepared.numel() * prepared.element_size(),
            float(fc2_input_scale), int(do_finalize), _ptr(out), _ptr(gemm2_out), _ptr(token_to_row),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status), ev, nev)
    if test_options is None:
        _check(lib().moe_routed_forward(*args, _stream(stream)), "moe_routed_forward")
    else:
        _check(test_lib().moe_test_routed_forward(*args, ctypes.byref(test_options), _stream(stream)),
               "moe_test_routed_forward")


def moe_grouped_fp4_forward(padded_offsets, row_to_slot, token_to_row, xq, xsf, xs, w: WeightsT, prepared,
                            topk_weights, fc2_input_scale, do_finalize, out, gemm2_out, workspace,
                            dev_status, step_events=None, stream=None, routed_scaling_factor=1.0):
    """do_finalize: 0/False unfinalized rows, 1/True ordered finalize, 2 accumulate into out."""
    M, k = token_to_row.shape
    ev, nev = _events(step_events)
    _check(lib().moe_grouped_fp4_forward(
        _ptr(padded_offsets), _ptr(row_to_slot), _ptr(token_to_row), M, k, _ptr(xq), _ptr(xsf), _ptr(xs),
        ctypes.byref(w), _ptr(prepared), prepared.numel() * prepared.element_size(), _ptr(topk_weights),
        _weights_dtype(topk_weights), float(routed_scaling_factor), float(fc2_input_scale), int(do_finalize),
        _ptr(out), _ptr(gemm2_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), ev, nev, _stream(stream)),
        "moe_grouped_fp4_forward")


def moe_finalize(gemm2_out, topk_weights, token_to_row, out, stream=None, routed_scaling_factor=1.0):
    M, k = token_to_row.shape
    H = out.shape[1]
    _check(lib().moe_finalize(_ptr(gemm2_out), _ptr(topk_weights), _weights_dtype(topk_weights),
                              float(routed_scaling_factor), _ptr(token_to_row), M, k, H, _ptr(out),
                              _stream(stream)), "moe_finalize")


def moe_test_gemm1(padded_offsets, row_to_slot, M, top_k, xq, xsf, xs, w: WeightsT, prepared, mode,
                   dbg_out, workspace, dev_status, stream=None):
    """Test build: the forward's GEMM1 with a plain epilogue (mode 0 FP32 pre-activations,
    1 the BF16 intermediate) into dbg_out."""
    _check(test_lib().moe_test_gemm1(
        _ptr(padded_offsets), _ptr(row_to_slot), M, top_k, _ptr(xq), _ptr(xsf), _ptr(xs), ctypes.byref(w),
        _ptr(prepared), prepared.numel() * prepared.element_size(), mode, _ptr(dbg_out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)), "moe_test_gemm1")
