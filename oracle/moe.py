"""Routed-MoE expert forward: GEMM1, activation, requantisation, GEMM2, finalize.

Sources:
* FlashInfer ``fused_moe.CudnnGroupedGemmNvfp4Config``: GEMM1's output rows
  are multiplied by their expert's global dequant; the BF16 intermediate is
  quantised to NVFP4 with a global scale of one before GEMM2; GEMM2's global
  dequant is applied by the finalize or to the unfinalized rows;
  ``MoEFinalizeConfig(do_finalize=False)`` returns
  ``[gemm2_out, expert_weights, token_to_row]``; SwiGLU "with default scalars".
* Megatron-Core ``core.inference.moe.flashinfer_nvfp4``: squared-ReLU and
  SwiGLU experts; gated FC1 is stored ``[gate; up]``, non-gated FC1 is
  ``[experts, intermediate, hidden]``; one FP32 scale per token for the
  activations; ``fc2_input_scale`` is the recipe constant of the FC2 input.
* FlashInfer ``fused_moe.FrostLowLatencyConfig`` (NVFP4 paragraph): BF16
  activation and expert-output rounding, and a combine made of ordered,
  separate FP32 multiplications and additions; unrouted slots are ignored by
  the finalize and get zero rows in the raw output.

Readings:
* GEMM accumulation is exact-as-possible: float64 sums of the dequantised
  products (each product ``e2m1 * e4m3`` pair is exact in float64).
* GEMM1 output ``y = acc * xs[t] * alpha1[e]``; SwiGLU ``h = silu(g) * u``
  with ``silu(g) = g / (1 + exp(-g))``, gate = rows ``[0, I)`` and up = rows
  ``[I, 2I)`` of W1; squared-ReLU ``h = max(y, 0)**2``; the other typed
  activations of the cuDNN backend page (GeGLU, GELU, ReLU, SiLU, Identity) with
  GELU in its erf form; all in float64, then rounded to BF16 (the BF16
  intermediate).
* The intermediate is requantised by the block quantiser with the static
  encode scale ``fc2_input_scale`` (1.0 = "a global scale of one"); GEMM2 output
  ``y2 = acc2 / fc2_input_scale * alpha2[e]``, rounded to BF16 (the expert
  output); the finalize combines these BF16 rows.
* FlashInfer ``fused_moe.alphamoe_nvfp4_aligned_moe`` (the fused variant):
  separate per-expert scalars for the gate accumulators
  (``output1_scale_gate_scalar``, applied before the activation) and the up
  accumulators (``output1_scale_scalar``); each down accumulator times its
  expert's scalar, the route weight and ``routed_scaling_factor`` is added in FP32
  to an FP32 copy of the caller's BF16 ``out``, converted back once. The FP32
  reduction there is order-dependent; the oracle sums in float64 (the exact
  value up to the final BF16 rounding) and the GPU is held to a tolerance.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Callable, Dict, Optional, Sequence

import numpy as np

from .formats import bf16_round, e2m1_decode, e4m3_decode
from .plan import make_plan
from .quantize import F32, dequantize_rows, quantize_blocks, quantize_weight

ExpertPack = tuple  # (data uint8 [rows, cols/2], sf uint8 [rows, cols/16], alpha float32)


@dataclass
class ExpertWeights:
    """Per-local-expert NVFP4 weights in the linear (boundary) layout.

    ``w1(l)`` -> (data [N1, H/2], sf [N1, H/16], alpha1), rows [gate; up] when
    gated; ``w2(l)`` -> (data [H, I/2], sf [H, I/16], alpha2). Experts are
    produced lazily by ``loader`` and cached.
    """
    num_local: int
    hidden: int
    inter: int
    gated: bool
    loader: Callable[[int], tuple]       # l -> (w1 pack, w2 pack)
    _cache: Dict[int, tuple] = field(default_factory=dict)

    def get(self, l: int) -> tuple:
        if l not in self._cache:
            self._cache[l] = self.loader(l)
        return self._cache[l]

    def w1(self, l: int) -> ExpertPack:
        return self.get(l)[0]

    def w2(self, l: int) -> ExpertPack:
        return self.get(l)[1]

    @staticmethod
    def from_bf16(w1_bf16: Sequence[np.ndarray], w2_bf16: Sequence[np.ndarray],
                  gated: bool) -> "ExpertWeights":
        """Quantise canonical BF16 stacks (float32 values of BF16) with the oracle."""
        El = len(w1_bf16)
        H = w1_bf16[0].shape[1]
        I = w2_bf16[0].shape[1]

        def load(l):
            return quantize_weight(w1_bf16[l]), quantize_weight(w2_bf16[l])
        return ExpertWeights(El, H, I, gated, load)

    @staticmethod
    def from_packs(w1_packs: Sequence[ExpertPack], w2_packs: Sequence[ExpertPack],
                   gated: bool) -> "ExpertWeights":
        El = len(w1_packs)
        H = w1_packs[0][0].shape[1] * 2
        I = w2_packs[0][0].shape[1] * 2
        return ExpertWeights(El, H, I, gated, lambda l: (w1_packs[l], w2_packs[l]))


def silu(g: np.ndarray) -> np.ndarray:
    """g * sigmoid(g) = g / (1 + exp(-g)); exp overflow for g << 0 gives -0."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


GATED_ACTIVATIONS = ("swiglu", "geglu")
ACTIVATIONS = ("swiglu", "relu2", "geglu", "gelu", "relu", "silu", "identity")


def gelu(x: np.ndarray) -> np.ndarray:
    """GELU in its defining form x * Phi(x) = x/2 * (1 + erf(x / sqrt(2)))."""
    from scipy.special import erf
    return 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))


def activation(y: np.ndarray, act: str, inter: int) -> np.ndarray:
    """float64 pre-activations [rows, N1] -> float64 activations [rows, I].

    Gated (FC1 rows [gate; up], N1 = 2I): swiglu = silu(g) * u, geglu = gelu(g) * u.
    Non-gated (N1 = I): relu2 = max(y, 0)^2, gelu, relu = max(y, 0), silu, identity.
    """
    if act in GATED_ACTIVATIONS:
        g = y[:, :inter]
        u = y[:, inter:2 * inter]
        return (silu(g) if act == "swiglu" else gelu(g)) * u
    if act == "relu2":
        r = np.maximum(y, 0.0)
        return r * r
    if act == "gelu":
        return gelu(y)
    if act == "relu":
        return np.maximum(y, 0.0)
    if act == "silu":
        return silu(y)
    if act == "identity":
        return y.copy()
    raise ValueError(act)


def expert_chain(A_deq: np.ndarray, xs: np.ndarray, pack1: ExpertPack, pack2: ExpertPack,
                 act: str, inter: int, fc2_input_scale: float, alpha_gate=None) -> dict:
    """All steps for the rows routed to one expert.

    A_deq float64 [r, H] block-dequantised activations of those rows' tokens,
    xs float32 [r] their per-token scales. ``alpha_gate`` (gated activations only):
    the expert's separate scalar of the gate rows ``[0, I)``; W1's own alpha then
    scales the up rows ``[I, 2I)`` only.
    """
    d1, s1, a1 = pack1
    d2, s2, a2 = pack2
    W1 = dequantize_rows(d1, s1)                       # [N1, H]
    acc1 = A_deq @ W1.T                                # float64 sums
    y = acc1 * np.asarray(xs, np.float64)[:, None] * np.float64(a1)
    if alpha_gate is not None and act in GATED_ACTIVATIONS:
        y[:, :inter] = acc1[:, :inter] * np.asarray(xs, np.float64)[:, None] * np.float64(alpha_gate)
    h = bf16_round(activation(y, act, inter))          # BF16 intermediate
    codes, isf = quantize_blocks(h.astype(F32), F32(fc2_input_scale))
    I_deq = (e2m1_decode(codes).reshape(codes.shape[0], -1, 16)
             * e4m3_decode(isf)[:, :, None]).reshape(codes.shape)
    W2 = dequantize_rows(d2, s2)                       # [H, I]
    acc2 = I_deq @ W2.T
    y2 = acc2 / np.float64(F32(fc2_input_scale)) * np.float64(a2)
    return {"preact": y, "act_bf16": h, "icodes": codes, "isf": isf,
            "rows": bf16_round(y2), "y2": y2}


def finalize(rows: np.ndarray, topk_weights: np.ndarray, token_to_row: np.ndarray,
             routed_scaling_factor: float = 1.0) -> np.ndarray:
    """Ordered FP32 combine of BF16 expert rows -> BF16 [M, H] (as float64 values).

    ``acc = 0``; for j = 0..k-1 in order, skipping masked slots:
    ``acc = acc + w'[t, j] * row`` with a separate FP32 multiply and add;
    ``out = bf16(acc)``. A token whose slots are all masked gets a zero row.
    ``w' = fp32(w * routed_scaling_factor)`` (the AlphaMoE page's scalar applied to each
    routed contribution, read as scaling the route weight); BF16 weights enter as their
    exact FP32 values.
    """
    w = np.asarray(topk_weights, dtype=F32)
    if routed_scaling_factor != 1.0:
        w = (w * F32(routed_scaling_factor)).astype(F32)
    t2r = np.asarray(token_to_row)
    M, k = t2r.shape
    H = rows.shape[1]
    acc = np.zeros((M, H), dtype=F32)
    for j in range(k):
        r = t2r[:, j]
        m = r >= 0
        if not m.any():
            continue
        prod = (w[m, j][:, None] * rows[r[m]].astype(F32)).astype(F32)
        acc[m] = (acc[m] + prod).astype(F32)
    return bf16_round(acc.astype(np.float64))


def combine_accumulate(out_prev: np.ndarray, y2_rows: np.ndarray, topk_weights: np.ndarray,
                       token_to_row: np.ndarray, routed_scaling_factor: float = 1.0) -> np.ndarray:
    """Accumulated output of the fused variant: ``bf16(out_prev + sum_j y2[row(t,j)] * w')``.

    ``y2_rows`` are the unrounded GEMM2 rows, ``w' = fp32(w * routed_scaling_factor)``,
    masked slots skipped; the sum is taken in float64 (exact up to the final BF16
    rounding); a token with no routed local slot keeps its ``out_prev`` row.
    """
    w = np.asarray(topk_weights, dtype=F32)
    if routed_scaling_factor != 1.0:
        w = (w * F32(routed_scaling_factor)).astype(F32)
    t2r = np.asarray(token_to_row)
    acc = np.asarray(out_prev, dtype=np.float64).copy()
    for j in range(t2r.shape[1]):
        r = t2r[:, j]
        m = r >= 0
        if m.any():
            acc[m] += w[m, j][:, None].astype(np.float64) * y2_rows[r[m]]
    return bf16_round(acc)


def forward(xq: np.ndarray, xsf: np.ndarray, xs: np.ndarray, topk_ids: np.ndarray,
            topk_weights: np.ndarray, weights: ExpertWeights, act: str,
            local_expert_offset: int = 0, fc2_input_scale: float = 1.0,
            plan: Optional[dict] = None, allow_duplicates: bool = False,
            routed_scaling_factor: float = 1.0, gate_alpha: Optional[np.ndarray] = None,
            out_prev: Optional[np.ndarray] = None) -> dict:
    """The whole path on quantised activations, in plan row order.

    Returns the plan and, per row of the padded plan (NaN in padding rows):
    ``preact`` float64 [P_cap, N1], ``act_bf16`` [P_cap, I], ``icodes`` uint8
    [P_cap, I], ``isf`` uint8 [P_cap, I/16], ``rows`` (= gemm2_out) [P_cap, H],
    ``y2`` (unrounded rows); ``out`` = finalize(rows) [M, H]; and, when ``out_prev``
    [M, H] is given, ``out_acc`` = combine_accumulate(out_prev, y2). ``gate_alpha``
    [E_local]: separate gate-row scalars of a gated W1.
    """
    if plan is None:
        plan = make_plan(topk_ids, local_expert_offset, weights.num_local, allow_duplicates)
    M, k = np.asarray(topk_ids).shape
    H, I = weights.hidden, weights.inter
    N1 = 2 * I if weights.gated else I
    cap = plan["capacity"]
    res = {
        "preact": np.full((cap, N1), np.nan),
        "act_bf16": np.full((cap, I), np.nan),
        "icodes": np.zeros((cap, I), dtype=np.uint8),
        "isf": np.zeros((cap, I // 16), dtype=np.uint8),
        "rows": np.full((cap, H), np.nan),
        "y2": np.full((cap, H), np.nan),
    }
    A_all = dequantize_rows(xq, xsf)
    padded, counts = plan["padded_offsets"], plan["counts"]
    for l in range(weights.num_local):
        c = int(counts[l])
        if c == 0:
            continue
        prow = np.arange(padded[l], padded[l] + c)
        tok = plan["row_to_slot"][prow] // k
        r = expert_chain(A_all[tok], xs[tok], weights.w1(l), weights.w2(l), act, I,
                         fc2_input_scale, None if gate_alpha is None else gate_alpha[l])
        for key in ("preact", "act_bf16", "icodes", "isf", "rows", "y2"):
            res[key][prow] = r[key]
    res["out"] = finalize(np.nan_to_num(res["rows"]), topk_weights, plan["token_to_row"],
                          routed_scaling_factor)
    if out_prev is not None:
        res["out_acc"] = combine_accumulate(out_prev, np.nan_to_num(res["y2"]), topk_weights,
                                            plan["token_to_row"], routed_scaling_factor)
    res["plan"] = plan
    return res


def forward_tokens(tokens: Sequence[int], xq: np.ndarray, xsf: np.ndarray, xs: np.ndarray,
                   topk_ids: np.ndarray, topk_weights: np.ndarray, weights: ExpertWeights,
                   act: str, local_expert_offset: int = 0,
                   fc2_input_scale: float = 1.0, routed_scaling_factor: float = 1.0,
                   gate_alpha: Optional[np.ndarray] = None, out_prev: Optional[np.ndarray] = None) -> dict:
    """Output rows of selected tokens only, each computed on its own.

    Every step of the path is row-local (per-token scales, static FC2 input
    scale), so a token's output depends only on its own activations and the
    weights of its routed local experts. Returns ``out`` [len(tokens), H] and
    the expert rows ``rows[(t, j)]``; with ``out_prev`` [len(tokens), H] also ``out_acc``,
    the accumulated output of those tokens.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    M, k = ids.shape
    I = weights.inter
    rows, y2 = {}, {}
    for t in tokens:
        A = dequantize_rows(xq[t:t + 1], xsf[t:t + 1])
        for j in range(k):
            l = int(ids[t, j]) - local_expert_offset
            if 0 <= l < weights.num_local:
                r = expert_chain(A, xs[t:t + 1], weights.w1(l), weights.w2(l), act, I,
                                 fc2_input_scale, None if gate_alpha is None else gate_alpha[l])
                rows[(t, j)] = r["rows"][0]
                y2[(t, j)] = r["y2"][0]
    sub_rows, sub_y2 = [], []
    t2r = np.full((len(tokens), k), -1, dtype=np.int64)
    for i, t in enumerate(tokens):
        for j in range(k):
            if (t, j) in rows:
                t2r[i, j] = len(sub_rows)
                sub_rows.append(rows[(t, j)])
                sub_y2.append(y2[(t, j)])
    R = np.array(sub_rows) if sub_rows else np.zeros((1, weights.hidden))
    w = np.asarray(topk_weights)[list(tokens)]
    res = {"out": finalize(R, w, t2r, routed_scaling_factor), "rows": rows}
    if out_prev is not None:
        Y = np.array(sub_y2) if sub_y2 else np.zeros((1, weights.hidden))
        res["out_acc"] = combine_accumulate(out_prev, Y, w, t2r, routed_scaling_factor)
    return res
