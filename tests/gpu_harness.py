"""Shared set-up of the GPU parity tests: seeded inputs on both sides, the CUDA path
through the C ABI, and the oracle on the same inputs.

The GPU side quantises the seeded BF16 weights with moe_quantize_weights; the oracle
quantises the same BF16 values with its own quantiser. Tests assert the two weight
encodings are identical before they compare anything downstream.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

import moe_inputs as mi
import nvfp4_routed_moe_sort_gb300 as pkg
from oracle import formats as F
from oracle import moe as O
from oracle import quantize as Q

DEV = torch.device("cuda:0")

# final BF16 output tolerance of the path (relative Frobenius, max-abs relative to max|ref|)
REL_FRO_TOL = 1e-2
MAX_ABS_TOL = 2e-2


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def bf16_np(t: torch.Tensor) -> np.ndarray:
    # capacity-sized buffers keep whatever their untouched padding rows held (NaN patterns
    # included); the tests compare real rows only
    with np.errstate(invalid="ignore"):
        return t.detach().float().cpu().numpy().astype(np.float64)


@functools.lru_cache(maxsize=256)
def oracle_expert(cfg_key: tuple, l: int):
    """Oracle-quantised (W1, W2) packs of one expert; BF16 drawn on the GPU, copied back."""
    cfg = mi.MoEConfig(*cfg_key)
    w1 = mi.expert_w1_bf16(cfg, l, DEV).float().cpu().numpy()
    w2 = mi.expert_w2_bf16(cfg, l, DEV).float().cpu().numpy()
    return Q.quantize_weight(w1), Q.quantize_weight(w2)


def cfg_key(cfg: mi.MoEConfig) -> tuple:
    # only what the weights depend on (name and routing fields do not matter)
    return ("w", 0, cfg.H, cfg.I, cfg.E, 1, cfg.act, "per_token", 0, cfg.weight_seed, 0.0,
            cfg.local_offset, cfg.num_local, 1.0, 1.0)


def oracle_weights(cfg: mi.MoEConfig) -> O.ExpertWeights:
    key = cfg_key(cfg)
    return O.ExpertWeights(cfg.El, cfg.H, cfg.I, cfg.gated, lambda l: oracle_expert(key, l))


class Problem:
    """One seeded problem on the GPU (inputs, quantised weights, prepared layer)."""

    def __init__(self, cfg: mi.MoEConfig, ids: np.ndarray | None = None, tw: np.ndarray | None = None,
                 gate_factor: np.ndarray | None = None):
        """gate_factor [E_local] (optional): the layer gets separate gate-row scalars
        fp32(alpha1 * factor), with alpha1 taken from the oracle's own quantisation."""
        self.cfg = cfg
        self.x = mi.hidden_bf16(cfg, DEV)
        if ids is None:
            ids, tw = mi.routing(cfg)
        self.ids, self.tw = ids, tw
        self.ids_t = torch.from_numpy(np.ascontiguousarray(ids)).to(DEV)
        self.tw_t = torch.from_numpy(np.ascontiguousarray(tw)).to(DEV)
        El = cfg.El
        self.w1_bf16 = torch.stack([mi.expert_w1_bf16(cfg, l, DEV) for l in range(El)])
        self.w2_bf16 = torch.stack([mi.expert_w2_bf16(cfg, l, DEV) for l in range(El)])
        self.q1 = pkg.quantize_weights(self.w1_bf16)
        self.q2 = pkg.quantize_weights(self.w2_bf16)
        self.gate_alpha = None
        if gate_factor is not None:
            W = oracle_weights(cfg)
            self.gate_alpha = np.array([np.float32(W.w1(l)[2]) * np.float32(gate_factor[l]) for l in range(El)],
                                       dtype=np.float32)
            self.gate_alpha_t = torch.from_numpy(self.gate_alpha).to(DEV)
        self.layer = pkg.NVFP4RoutedMoE(*self.q1, *self.q2, activation=cfg.act, num_experts=cfg.E,
                                        local_expert_offset=cfg.local_offset,
                                        fc2_input_scale=cfg.fc2_input_scale, scale_mode=cfg.scale_mode,
                                        routed_scaling_factor=cfg.routed_scaling_factor,
                                        w1_gate_alpha=None if gate_factor is None else self.gate_alpha_t)

    def run(self, do_finalize=True):
        """The separate calls (quantize, plan, forward): every intermediate stays in bufs()."""
        res = self.layer.forward_steps(self.x, self.ids_t, self.tw_t, do_finalize=do_finalize)
        torch.cuda.synchronize()
        return res

    def run_routed(self, do_finalize=True):
        """The one-call path (moe_routed_forward), as the benchmark times it."""
        res = self.layer.forward(self.x, self.ids_t, self.tw_t, do_finalize=do_finalize)
        torch.cuda.synchronize()
        return res

    def bufs(self, do_finalize=True):
        return self.layer.buffers(self.cfg.M, self.cfg.top_k, do_finalize)

    def oracle_inputs(self):
        xf = self.x.float().cpu().numpy()
        return Q.quantize_activations(xf, self.cfg.scale_mode)

    def oracle_forward(self, **kw):
        xq, xsf, xs = self.oracle_inputs()
        return O.forward(xq, xsf, xs, self.ids, self.tw, oracle_weights(self.cfg), self.cfg.act,
                         local_expert_offset=self.cfg.local_offset,
                         fc2_input_scale=self.cfg.fc2_input_scale,
                         routed_scaling_factor=self.cfg.routed_scaling_factor, gate_alpha=self.gate_alpha,
                         **kw)


def assert_close_output(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = got - ref
    ref_n = np.linalg.norm(ref)
    rel = np.linalg.norm(err) / ref_n if ref_n > 0 else np.linalg.norm(err)
    mx = np.abs(err).max() if err.size else 0.0
    bound = MAX_ABS_TOL * (np.abs(ref).max() if ref.size else 0.0)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert rel <= REL_FRO_TOL, f"{what}: relative Frobenius error {rel:.3e} > {REL_FRO_TOL}"
    assert mx <= bound + 1e-30, f"{what}: max |err| {mx:.3e} > {bound:.3e}"
    return rel, mx


def sf_tiles_to_linear(tiles: np.ndarray, rows: int, kcols: int) -> np.ndarray:
    """Undo the 128-row x 4-scale tile layout: byte (r, c) of a [rows, kcols] scale matrix
    sits at tile (r // 128, c // 4) (tiles row-major with ceil-to-256-of-K columns), inside
    the tile at (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4."""
    kcols_p = (kcols + 15) // 16 * 16
    r = np.arange(rows)[:, None]
    c = np.arange(kcols)[None, :]
    off = ((r // 128) * (kcols_p // 4) + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
    return tiles[off]


def e2m1_bytes_equal(a: np.ndarray, b: np.ndarray) -> bool:
    return np.array_equal(np.asarray(a, np.uint8), np.asarray(b, np.uint8))


__all__ = ["DEV", "Problem", "assert_close_output", "oracle_weights", "oracle_expert", "to_np", "bf16_np",
           "sf_tiles_to_linear", "F", "O", "Q", "mi", "pkg"]
