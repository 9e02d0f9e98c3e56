"""User-facing wrapper: owns the capacity-sized buffers and makes the C-ABI calls.

``NVFP4RoutedMoE.forward`` is one moe_routed_forward call (the whole layer from BF16
hidden states); ``forward_steps`` makes the separate calls moe_quantize_input ->
moe_plan -> moe_grouped_fp4_forward and keeps every intermediate buffer. Both run on
torch's current stream and every step runs in the library's kernels; torch only
allocates device memory (once per batch shape) and supplies the stream.
"""
from __future__ import annotations

import torch

from . import _lib as L


def quantize_weights(w_bf16: torch.Tensor):
    """BF16 expert stack [E, rows, cols] -> (data [E, rows, cols/2] u8, sf [E, rows, cols/16] u8,
    alpha [E] f32) with one FP32 global scale per expert (moe_quantize_weights)."""
    E, R, C = w_bf16.shape
    dev = w_bf16.device
    data = torch.empty(E, R, C // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(E, R, C // 16, dtype=torch.uint8, device=dev)
    alpha = torch.empty(E, dtype=torch.float32, device=dev)
    scratch = torch.empty(E, dtype=torch.float32, device=dev)
    L.moe_quantize_weights(w_bf16.contiguous().view(torch.int16), data, sf, alpha, scratch)
    return data, sf, alpha


class NVFP4RoutedMoE:
    """Routed-MoE expert layer on NVFP4 weights (linear boundary layout, on the GPU)."""

    def __init__(self, w1, w1_sf, w1_alpha, w2, w2_sf, w2_alpha, activation: str = "swiglu",
                 num_experts: int | None = None, local_expert_offset: int = 0,
                 fc2_input_scale: float = 1.0, scale_mode: str = "per_token",
                 routed_scaling_factor: float = 1.0, w1_gate_alpha=None):
        """w1_gate_alpha [E_local] f32 (optional): separate dequant scalars of the gate rows of a
        gated W1; w1_alpha then scales the up rows only."""
        El, N1, Hh = w1.shape
        self.El = El
        self.H = Hh * 2
        self.I = w2.shape[2] * 2
        if activation not in L.ACTIVATIONS:
            raise ValueError(f"activation must be one of {sorted(L.ACTIVATIONS)}")
        self.act = L.ACTIVATIONS[activation]
        self.num_experts = num_experts if num_experts is not None else El + local_expert_offset
        self.local_expert_offset = local_expert_offset
        self.fc2_input_scale = float(fc2_input_scale)
        self.routed_scaling_factor = float(routed_scaling_factor)
        self.scale_mode = L.MOE_SCALE_PER_TOKEN if scale_mode == "per_token" else L.MOE_SCALE_GLOBAL_ONE
        self.device = w1.device
        self.linear = (w1, w1_sf, w1_alpha, w2, w2_sf, w2_alpha, w1_gate_alpha)
        self.w = L.make_weights(El, self.H, self.I, self.act, w1, w1_sf, w1_alpha, w2, w2_sf, w2_alpha,
                                w1_gate_alpha)
        nbytes = L.moe_prepared_weights_bytes(self.w)
        self.prepared = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        L.moe_prepare_weights(self.w, self.prepared)
        self._bufs = {}

    def refresh(self):
        """Re-prepare from the (updated) linear weights into the same buffer."""
        L.moe_prepare_weights(self.w, self.prepared)

    def routed_buffers(self, M: int, top_k: int, do_finalize) -> dict:
        """Buffers of the one-call path for one batch shape (workspace, token_to_row, outputs)."""
        mode = int(do_finalize)
        key = ("routed", M, top_k, mode)
        if key in self._bufs:
            return self._bufs[key]
        dev = self.device
        cap = L.moe_plan_capacity(M, top_k, self.El)
        b = {
            "ws": torch.empty(max(L.moe_routed_forward_workspace_bytes(M, top_k, self.w, mode), 16),
                              dtype=torch.uint8, device=dev),
            "token_to_row": torch.empty(M, top_k, dtype=torch.int32, device=dev),
            "dev_status": torch.zeros(4, dtype=torch.int32, device=dev),
            "out": torch.empty(M, self.H, dtype=torch.bfloat16, device=dev)
            if mode == L.MOE_OUTPUT_FINALIZED else None,
            "gemm2_out": torch.empty(max(cap, 1), self.H, dtype=torch.bfloat16, device=dev)
            if mode == L.MOE_OUTPUT_UNFINALIZED else None,
            "capacity": cap,
        }
        self._bufs[key] = b
        return b

    def buffers(self, M: int, top_k: int, do_finalize) -> dict:
        """Buffers of the separate-call path for one batch shape. do_finalize: False/0
        unfinalized rows, True/1 finalized output, 2 accumulated output (the caller's out)."""
        mode = int(do_finalize)
        key = (M, top_k, mode)
        if key in self._bufs:
            return self._bufs[key]
        dev = self.device
        cap = L.moe_plan_capacity(M, top_k, self.El)
        b = {
            "xq": torch.empty(M, self.H // 2, dtype=torch.uint8, device=dev),
            "xsf": torch.empty(M, self.H // 16, dtype=torch.uint8, device=dev),
            "xs": torch.empty(M, dtype=torch.float32, device=dev),
            "counts": torch.empty(self.El, dtype=torch.int32, device=dev),
            "padded_offsets": torch.empty(self.El + 1, dtype=torch.int32, device=dev),
            "row_to_slot": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
            "token_to_row": torch.empty(M, top_k, dtype=torch.int32, device=dev),
            "plan_ws": torch.empty(max(L.moe_plan_workspace_bytes(M, top_k, self.El), 16),
                                   dtype=torch.uint8, device=dev),
            "ws": torch.empty(max(L.moe_forward_workspace_bytes(M, top_k, self.w, mode), 16),
                              dtype=torch.uint8, device=dev),
            "dev_status": torch.zeros(4, dtype=torch.int32, device=dev),
            "out": torch.empty(M, self.H, dtype=torch.bfloat16, device=dev)
            if mode == L.MOE_OUTPUT_FINALIZED else None,
            "gemm2_out": torch.empty(max(cap, 1), self.H, dtype=torch.bfloat16, device=dev)
            if mode == L.MOE_OUTPUT_UNFINALIZED else None,
            "capacity": cap,
        }
        self._bufs[key] = b
        return b

    def quantize(self, x: torch.Tensor, b: dict):
        L.moe_quantize_input(x.view(torch.int16), self.scale_mode, b["xq"], b["xsf"], b["xs"])

    def plan(self, topk_ids: torch.Tensor, b: dict, packed: bool = False):
        L.moe_plan(topk_ids, self.num_experts, self.local_expert_offset, self.El, b["counts"],
                   b["padded_offsets"], b["row_to_slot"], b["token_to_row"], b["plan_ws"], b["dev_status"],
                   packed=packed)

    def experts(self, topk_weights: torch.Tensor, b: dict, do_finalize, step_events=None, out=None):
        L.moe_grouped_fp4_forward(b["padded_offsets"], b["row_to_slot"], b["token_to_row"], b["xq"], b["xsf"],
                                  b["xs"], self.w, self.prepared, topk_weights, self.fc2_input_scale,
                                  int(do_finalize), out if out is not None else b["out"], b["gemm2_out"],
                                  b["ws"], b["dev_status"], step_events=step_events,
                                  routed_scaling_factor=self.routed_scaling_factor)

    def routed(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor, b: dict, do_finalize,
               packed: bool = False, step_events=None, out=None, test_options=None):
        """One moe_routed_forward call into the buffers ``b`` of routed_buffers() (with
        ``test_options``, the test build's moe_test_routed_forward)."""
        L.moe_routed_forward(x.view(torch.int16), self.scale_mode, topk_ids, self.num_experts,
                             self.local_expert_offset, topk_weights, self.w, self.prepared, self.fc2_input_scale,
                             int(do_finalize), out if out is not None else b["out"], b["gemm2_out"],
                             b["token_to_row"], b["ws"], b["dev_status"], step_events=step_events,
                             routed_scaling_factor=self.routed_scaling_factor, packed=packed,
                             test_options=test_options)

    @staticmethod
    def _prefix(x, topk_ids, topk_weights, out, token_capacity):
        if token_capacity is None:
            return x, topk_ids, topk_weights, out
        T = int(token_capacity)
        if not 0 <= T <= x.shape[0]:
            raise ValueError("token_capacity must lie in [0, M]")
        return x[:T], topk_ids[:T], topk_weights[:T], (out[:T] if out is not None else None)

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor | None,
                do_finalize=True, step_events=None, out: torch.Tensor | None = None,
                token_capacity: int | None = None):
        """x [M, H] bf16, topk_ids [M, k] int32, topk_weights [M, k] f32 or bf16 (all on the GPU).

        One moe_routed_forward call (the small-batch prologue fuses quantiser, plan and
        permutation). Arguments and results as forward_steps; ``step_events`` (5 recorded
        events) mark the prologue, GEMM1, GEMM2, the combine and the end.
        """
        packed = topk_weights is None
        if packed:
            topk_weights = topk_ids
        mode = int(do_finalize)
        if mode == L.MOE_OUTPUT_ACCUMULATE and out is None:
            raise ValueError("do_finalize=2 (accumulate) needs the caller's out tensor")
        x, topk_ids, topk_weights, out = self._prefix(x, topk_ids, topk_weights, out, token_capacity)
        M, k = topk_ids.shape
        b = self.routed_buffers(M, k, mode)
        self.routed(x, topk_ids, topk_weights, b, mode, packed, step_events, out)
        if mode == L.MOE_OUTPUT_UNFINALIZED:
            return b["gemm2_out"], topk_weights, b["token_to_row"]
        return out if out is not None else b["out"]

    def forward_steps(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor | None,
                      do_finalize=True, step_events=None, out: torch.Tensor | None = None,
                      token_capacity: int | None = None):
        """The separate calls: moe_quantize_input, moe_plan, moe_grouped_fp4_forward.

        x [M, H] bf16, topk_ids [M, k] int32, topk_weights [M, k] f32 or bf16 (all on the GPU).

        topk_weights None: topk_ids holds packed routing slots (int32: BF16 score in bits
        31..16, expert id in bits 15..0) and supplies both the ids and the scores.
        do_finalize: True/1 returns out [M, H] bf16 (ordered combine); False/0 returns
        (gemm2_out [capacity, H], topk_weights, token_to_row); 2 adds the routed
        contributions in FP32 to the caller's ``out`` [M, H] bf16 (required) and returns it.
        out (finalized mode, optional): write into this [M, H] tensor instead of the layer's.
        token_capacity: process only the first token_capacity rows of x and the routing
        (a fixed prefix of a graph-stable dispatcher buffer); rows of ``out`` past it are left
        untouched. Returned tensors other than a caller's out are the layer's reusable buffers.
        """
        packed = topk_weights is None
        if packed:
            topk_weights = topk_ids
        mode = int(do_finalize)
        if mode == L.MOE_OUTPUT_ACCUMULATE and out is None:
            raise ValueError("do_finalize=2 (accumulate) needs the caller's out tensor")
        x, topk_ids, topk_weights, out = self._prefix(x, topk_ids, topk_weights, out, token_capacity)
        M, k = topk_ids.shape
        b = self.buffers(M, k, mode)
        self.quantize(x, b)
        self.plan(topk_ids, b, packed)
        self.experts(topk_weights, b, mode, step_events, out)
        if mode == L.MOE_OUTPUT_UNFINALIZED:
            return b["gemm2_out"], topk_weights, b["token_to_row"]
        return out if out is not None else b["out"]

    def capture(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor | None,
                do_finalize=True, step_events=None, out: torch.Tensor | None = None) -> torch.cuda.CUDAGraph:
        """Capture one forward (the one-call path) in a CUDA graph.

        The graph reads x, topk_ids and topk_weights at their current addresses and writes the
        layer's buffers; refill the inputs in place and call ``replay()``. Any routing of the
        same (M, top_k) replays correctly: the kernels size their work from the device-side
        plan. ``step_events`` (5 recorded torch events, optional) mark the step boundaries
        inside the graph: before the prologue, GEMM1, GEMM2, the combine, and the end.
        """
        M, k = topk_ids.shape
        mode = int(do_finalize)
        packed = topk_weights is None
        if packed:
            topk_weights = topk_ids
        b = self.routed_buffers(M, k, mode)
        if mode == L.MOE_OUTPUT_ACCUMULATE and out is None:
            raise ValueError("do_finalize=2 (accumulate) needs the caller's out tensor")
        # warm-up outside the capture (an accumulating warm-up writes a copy of out)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            warm_out = out.clone() if mode == L.MOE_OUTPUT_ACCUMULATE else out
            self.forward(x, topk_ids, None if packed else topk_weights, mode, out=warm_out)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.routed(x, topk_ids, topk_weights, b, mode, packed, step_events, out)
        return g

    # Host traffic (inputs + output) up to which capture_host lets the kernels read and write
    # the pinned buffers in place. Measured on GB300 (NVLink-C2C): in place saves the copy
    # nodes' fixed latency (decode T=8: 55 -> 43 us per step) but moves data more slowly than
    # the copy engine (prefill 4k, 118 MB: 1.88 -> 2.04 ms); the two cross near 8 MB.
    DIRECT_HOST_BYTES = 8 << 20

    def capture_host(self, staging: "HostStaging", host_out: torch.Tensor,
                     direct: bool | None = None) -> torch.cuda.CUDAGraph:
        """Capture one forward from host buffers to a host buffer in a CUDA graph (the one-call
        path, finalized output [M, H] bf16 into the pinned ``host_out``). Refill
        ``staging.x`` / ``.ids`` / ``.weights`` in place and call ``replay()``; the output is
        in ``host_out`` once the stream reaches the end of the replay.

        direct=False: the graph copies the staging buffer to the device (one transfer), runs
        the forward and copies the output back. direct=True: the kernels read the pinned
        inputs and write the pinned output in place (over the CPU-GPU link; no copy nodes).
        None picks direct when the host traffic is at most DIRECT_HOST_BYTES. The choice is
        recorded in ``staging.direct``.
        """
        if not host_out.is_pinned() or host_out.dtype != torch.bfloat16 or tuple(host_out.shape) != (staging.M, staging.H):
            raise ValueError("host_out must be a pinned bf16 tensor of shape [M, H]")
        if direct is None:
            direct = staging.nbytes + host_out.numel() * 2 <= self.DIRECT_HOST_BYTES
        mode = L.MOE_OUTPUT_FINALIZED
        b = self.routed_buffers(staging.M, staging.top_k, mode)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            staging.device.copy_(staging.host, non_blocking=True)
            self.forward(staging.dev_x, staging.dev_ids, staging.dev_weights, mode)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if direct:
                self.routed(staging.x, staging.ids, staging.weights, b, mode, out=host_out)
            else:
                staging.device.copy_(staging.host, non_blocking=True)
                self.routed(staging.dev_x, staging.dev_ids, staging.dev_weights, b, mode)
                host_out.copy_(b["out"], non_blocking=True)
        staging.direct = direct
        return g

    def device_status(self, M: int, top_k: int, do_finalize, routed: bool = True) -> int:
        b = self.routed_buffers(M, top_k, do_finalize) if routed else self.buffers(M, top_k, do_finalize)
        return int(b["dev_status"][0].item())


class HostStaging:
    """One step's inputs in a single pinned host buffer (hidden states [M, H] bf16, routing ids
    [M, k] int32, routing weights [M, k] f32, at 256-byte aligned offsets) and its device
    mirror, so that NVFP4RoutedMoE.capture_host copies them to the device in one transfer."""

    def __init__(self, M: int, H: int, top_k: int, device):
        self.M, self.H, self.top_k = M, H, top_k
        nb_x, nb_ids = M * H * 2, M * top_k * 4
        off_ids = (nb_x + 255) // 256 * 256
        off_w = off_ids + (nb_ids + 255) // 256 * 256
        total = off_w + nb_ids
        self.host = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.device = torch.empty(total, dtype=torch.uint8, device=device)

        def views(buf):
            return (buf[:nb_x].view(torch.bfloat16).view(M, H),
                    buf[off_ids:off_ids + nb_ids].view(torch.int32).view(M, top_k),
                    buf[off_w:off_w + nb_ids].view(torch.float32).view(M, top_k))

        self.x, self.ids, self.weights = views(self.host)
        self.dev_x, self.dev_ids, self.dev_weights = views(self.device)
        self.nbytes = total
        self.direct = None  # set by NVFP4RoutedMoE.capture_host: in place (True) or copies (False)
