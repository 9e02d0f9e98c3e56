"""CPU oracle for the NVFP4 routed-MoE expert path.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import, call or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code, header, table or constant generator with the CUDA library
(``nvfp4_routed_moe_sort_gb300``); the two meet only in the seeded input
generator ``moe_inputs``, which holds none of the method's arithmetic.

The oracle restates, step by step and without blocking, fusion or reordering,
what the pages define:

* ``formats``  - E2M1 / E4M3 / BF16 codecs from the format definitions;
* ``quantize`` - the NVFP4 16-wide block quantiser (activations with global
  scale one or one FP32 scale per token; weights with one FP32 global scale per
  expert matrix);
* ``plan``     - the expert-sorted plan with segments padded to 128 rows;
* ``moe``      - block-scaled GEMM1, SwiGLU / squared-ReLU, requantisation of
  the intermediate, GEMM2, and the ordered FP32 finalize.

Precision: a floating-point step that decides an integer (a quantised code or
scale) runs in IEEE float32, the precision of the kernel; sums and
activations run in float64 unless the pages fix FP32 (the combine). Every
function is pinned by the ``-m "not gpu"`` tests under ``tests/`` against
closed forms, library routines, invariants or brute force.
"""
from . import formats, quantize, plan, moe  # noqa: F401
