"""NVFP4 routed-MoE expert path for GB300 (sm_103a).

The compute runs in ``libmoe_nvfp4.so`` (C ABI: include/moe_nvfp4.h); this package
holds its build script, a ctypes binding with the same function names, and a small
buffer-owning wrapper. The test build ``libmoe_nvfp4_test.so`` (include/moe_nvfp4_test.h)
is loaded only through ``test_lib()``, by tests. Importing it never falls back to another implementation:
calls raise ``MoEError`` if the library is not built.
"""
from . import _lib
from ._lib import (  # noqa: F401
    ACTIVATIONS, EXPORTED, TEST_EXPORTED, MOE_ACT_GEGLU, MOE_ACT_GELU, MOE_ACT_IDENTITY, MOE_ACT_RELU, MOE_ACT_RELU2,
    MOE_ACT_SILU, MOE_ACT_SWIGLU, MOE_DEV_DUPLICATE_EXPERT, MOE_DEV_TIMEOUT,
    MOE_IDS_INT32, MOE_IDS_PACKED, MOE_OUTPUT_ACCUMULATE, MOE_OUTPUT_FINALIZED, MOE_OUTPUT_UNFINALIZED,
    MOE_SCALE_GLOBAL_ONE, MOE_SCALE_PER_TOKEN, MOE_WEIGHTS_BF16, MOE_WEIGHTS_F32, MOE_WEIGHTS_PACKED, MoEError,
    TestOptionsT, WeightsT, lib, make_weights, test_lib, test_options,
    moe_abi_version, moe_finalize, moe_forward_workspace_bytes,
    moe_forward_workspace_layout, moe_grouped_fp4_forward, moe_plan, moe_plan_capacity,
    moe_plan_workspace_bytes, moe_plan_noalloc, moe_prepare_weights, moe_prepared_weights_bytes, moe_quantize_input,
    moe_quantize_weights, moe_routed_forward, moe_routed_forward_workspace_bytes, moe_test_gemm1, status_string,
)
from .build import LIB as LIB_PATH  # noqa: F401
from .moe import HostStaging, NVFP4RoutedMoE, quantize_weights  # noqa: F401
