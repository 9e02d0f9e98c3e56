"""Per-expert oracle work for the full-size parity tests, run in a process pool.

Test infrastructure. At full size (up to 256 experts of 7168 x 4096 weights) the oracle's
weight quantiser takes seconds per expert, so the tests hand each expert to a worker. The
pool is started with the spawn method, never forked from a process that has touched the GPU;
the workers import only numpy and the oracle.

Each task gets one expert's BF16 weights (as their 16-bit patterns) and the NVFP4 activation
packs of the plan rows sampled for that expert (quantised by the oracle in the parent), and
returns the oracle's BF16 expert rows for them plus a digest of the oracle's own weight
encoding, which the parent compares with the digest of the GPU's encoding.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import multiprocessing
import os

import numpy as np


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """BF16 16-bit patterns -> their exact float32 values."""
    return (np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def pack_digest(d1, s1, a1, d2, s2, a2) -> str:
    """sha256 over the bytes of two NVFP4 weight packs (codes, scales, FP32 alpha)."""
    h = hashlib.sha256()
    for part in (d1, s1, np.float32(a1), d2, s2, np.float32(a2)):
        h.update(np.ascontiguousarray(part).tobytes())
    return h.hexdigest()


def expert_task(task: dict) -> dict:
    """The oracle's weight encoding of one expert and its expert rows for the given activations."""
    from oracle import moe as O
    from oracle import quantize as Q
    p1 = Q.quantize_weight(bf16_bits_to_f32(task["w1_bits"]))
    p2 = Q.quantize_weight(bf16_bits_to_f32(task["w2_bits"]))
    out = {"l": task["l"], "digest": pack_digest(*p1, *p2), "rows": None}
    if task["xq"].shape[0]:
        A = Q.dequantize_rows(task["xq"], task["xsf"])
        r = O.expert_chain(A, task["xs"], p1, p2, task["act"], task["inter"], task["fc2_input_scale"])
        out["rows"] = r["rows"]
    return out


def run_experts(tasks, workers: int | None = None):
    """Runs expert_task over an iterable of tasks (drawn lazily, at most 2 x workers in flight)
    in a spawn-started pool; yields the results as they finish."""
    workers = workers or max(1, min(16, (os.cpu_count() or 2)))
    ctx = multiprocessing.get_context("spawn")
    env_threads = os.environ.get("OMP_NUM_THREADS")
    os.environ["OMP_NUM_THREADS"] = "1"   # one BLAS thread per worker (inherited at spawn)
    try:
        with concurrent.futures.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as ex:
            pending = set()
            it = iter(tasks)
            done = False
            while not done or pending:
                while not done and len(pending) < 2 * workers:
                    try:
                        pending.add(ex.submit(expert_task, next(it)))
                    except StopIteration:
                        done = True
                if pending:
                    fin, pending = concurrent.futures.wait(pending, return_when=concurrent.futures.FIRST_COMPLETED)
                    for f in fin:
                        yield f.result()
    finally:
        if env_threads is None:
            os.environ.pop("OMP_NUM_THREADS", None)
        else:
            os.environ["OMP_NUM_THREADS"] = env_threads
