"""Expert-sorted routing plan (moe_sort / moe_permute).

Sources:
* FlashInfer ``fused_moe.CudnnGroupedGemmNvfp4Config`` (Pipeline, Rows and
  scale rows, Expert parallelism, distinct topk_ids bullets): rows are permuted
  into expert order, each expert segment padded to a multiple of 128 rows;
  assignments to non-local experts are masked out; each token's topk_ids name
  distinct experts.
* Megatron-Core ``flashinfer_routed_nvfp4_moe``: routing entries of -1
  contribute zero output.
* FlashInfer ``fused_moe.FrostLowLatencyConfig`` (NVFP4 paragraph): expert ids
  outside ``[0, num_experts)`` mark unrouted slots.

Readings:
* local id ``l = id - local_expert_offset``; a slot is masked when
  ``l`` is outside ``[0, num_local_experts)`` (this covers -1 and ids >= E);
* rows inside a segment are in ascending slot order ``s = t * top_k + j``,
  which is ascending token order when the experts of a token are distinct
  (the plainest stable sort);
* ``padded_offsets[l+1] = padded_offsets[l] + roundup(count_l, 128)``, so an
  empty expert takes no rows;
* ``row_to_slot[p] = s`` for a real row and -1 for padding rows and for every
  row from the padded total up to the capacity; ``token_to_row[t, j]`` is the
  row of slot (t, j) or -1 when masked.
"""
from __future__ import annotations

import numpy as np

from .formats import bits_to_bf16

SEGMENT_ALIGN = 128


def roundup(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def plan_capacity(M: int, top_k: int, num_local_experts: int) -> int:
    """Largest padded row count any routing of M tokens can need.

    At most M*top_k routed slots, and every non-empty segment adds fewer than
    128 padding rows; at most min(E_local, M*top_k) segments are non-empty.
    """
    slots = M * top_k
    return roundup(slots + (SEGMENT_ALIGN - 1) * min(num_local_experts, slots), SEGMENT_ALIGN)


def unpack_topk(packed: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Packed routing slots -> (expert ids int64, scores float64).

    FlashInfer ``fused_moe.CudnnGroupedGemmNvfp4Config`` accepts routing weights
    "packed, or unpacked"; ``FrostLowLatencyConfig`` says packed scores keep their
    BF16 rounding. The bit layout is a reading (the pages do not print it): one
    32-bit word per slot, the BF16 score in bits 31..16 and the expert id, unsigned,
    in bits 15..0.
    """
    word = np.asarray(packed).astype(np.int64) & 0xFFFFFFFF
    ids = word & 0xFFFF
    scores = bits_to_bf16((word >> 16).astype(np.uint16))
    return ids, scores


def make_plan(topk_ids: np.ndarray, local_expert_offset: int, num_local_experts: int,
              allow_duplicates: bool = False) -> dict:
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, k = ids.shape
    El = num_local_experts
    loc = ids - local_expert_offset
    valid = (loc >= 0) & (loc < El)
    dup = False
    for t in range(M):
        ex = ids[t][valid[t]]
        if np.unique(ex).size != ex.size:
            dup = True
    if dup and not allow_duplicates:
        raise ValueError("a token names the same expert twice")
    flat_l = loc.ravel()
    flat_valid = valid.ravel()
    counts = np.bincount(flat_l[flat_valid], minlength=El).astype(np.int32)[:El]
    padded = np.zeros(El + 1, dtype=np.int32)
    for l in range(El):
        padded[l + 1] = padded[l] + roundup(int(counts[l]), SEGMENT_ALIGN)
    cap = plan_capacity(M, k, El)
    row_to_slot = np.full(cap, -1, dtype=np.int32)
    token_to_row = np.full(M * k, -1, dtype=np.int32)
    slots = np.nonzero(flat_valid)[0]
    # stable sort of the routed slots by local expert: slot order within a segment
    order = slots[np.argsort(flat_l[slots], kind="stable")]
    cursor = padded[:-1].astype(np.int64).copy()
    for s in order:
        l = flat_l[s]
        row = cursor[l]
        cursor[l] += 1
        row_to_slot[row] = s
        token_to_row[s] = row
    return {
        "counts": counts,
        "padded_offsets": padded,
        "row_to_slot": row_to_slot,
        "token_to_row": token_to_row.reshape(M, k),
        "num_rows": int(padded[El]),
        "capacity": cap,
        "duplicate": dup,
    }
