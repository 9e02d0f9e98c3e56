"""Seeded synthetic inputs for the NVFP4 routed-MoE expert path.

This module is shared by the CPU oracle and the GPU path. It holds no step of
the method: it only draws the BF16 hidden states, the router logits (and the
routing taken from them), and the BF16 expert weights that both sides then
quantise and run on their own.

Every value is a pure function of (seed, tensor id, element index), built from
a published 32-bit integer hash ("lowbias32", C. Wellons, *Prospecting for hash
functions*, 2018) and the Irwin-Hall sum of twelve uniforms for N(0, 1). All of
it is integer arithmetic plus one power-of-two division, so a tensor drawn with
torch on the CPU and one drawn on a GPU are identical bit for bit; weights for
the large workloads are drawn on the GPU, one expert at a time.

The routing (softmax of the logits, top-k by value, renormalised weights) is
computed once on the host in float32 numpy and handed to both sides unchanged.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

M32 = 0xFFFFFFFF

# Tensor ids of the counter-based generator.
TID_HIDDEN = 1
TID_LOGITS = 2
TID_ZIPF_PERM = 5
TID_W1_BASE = 1000  # W1 of global expert e: TID_W1_BASE + 2 * e
TID_W2_BASE = 1001  # W2 of global expert e: TID_W2_BASE + 2 * e

WEIGHT_STD = 0.02


# --------------------------------------------------------------------------
# counter-based generator
# --------------------------------------------------------------------------
def _hash32_int(x: int) -> int:
    """lowbias32 on a Python int (used for key derivation)."""
    x &= M32
    x ^= x >> 16
    x = (x * 0x7FEB352D) & M32
    x ^= x >> 15
    x = (x * 0x846CA68B) & M32
    x ^= x >> 16
    return x


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for 0 <= x < 2**32 without any int64 overflow."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def _hash32(x: torch.Tensor) -> torch.Tensor:
    """lowbias32 on an int64 tensor holding values in [0, 2**32)."""
    x = x ^ (x >> 16)
    x = _mul32(x, 0x7FEB352D)
    x = x ^ (x >> 15)
    x = _mul32(x, 0x846CA68B)
    x = x ^ (x >> 16)
    return x


def stream_key(seed: int, tensor_id: int) -> int:
    return _hash32_int(_hash32_int(seed ^ 0x5EED1234) ^ _hash32_int(tensor_id + 0x632BE5AB))


def normal_f32(seed: int, tensor_id: int, start: int, n: int,
               device: torch.device | str = "cpu") -> torch.Tensor:
    """n float32 draws of N(0,1) (Irwin-Hall of 12 uniforms), elements start..start+n-1.

    Each element sums the two 16-bit halves of six hashed counters; the sum
    minus its mean, divided by 2**16, is exact in float32 and lies in [-6, 6].
    """
    key = stream_key(seed, tensor_id)
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    acc = torch.zeros(n, dtype=torch.int64, device=device)
    for d in range(6):
        c = idx * 8 + d
        h = _hash32(_hash32((c & M32) ^ key) ^ (c >> 32))
        acc += (h & 0xFFFF) + (h >> 16)
    return (acc - 393210).to(torch.float32) / 65536.0


def uniform_u32(seed: int, tensor_id: int, n: int, device="cpu") -> torch.Tensor:
    key = stream_key(seed, tensor_id)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    return _hash32(_hash32((idx & M32) ^ key) ^ (idx >> 32))


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    M: int                 # tokens
    H: int                 # hidden size
    I: int                 # intermediate size
    E: int                 # global experts
    top_k: int
    act: str = "swiglu"    # gated: "swiglu", "geglu"; non-gated: "relu2", "gelu", "relu", "silu", "identity"
    scale_mode: str = "per_token"   # "global_one" | "per_token"
    seed: int = 0          # hidden + routing
    weight_seed: int = 0   # expert weights
    skew: float = 0.0      # Zipf exponent of the per-expert logit bias (0 = uniform)
    local_offset: int = 0
    num_local: Optional[int] = None
    fc2_input_scale: float = 1.0
    routed_scaling_factor: float = 1.0

    @property
    def El(self) -> int:
        return self.E if self.num_local is None else self.num_local

    @property
    def gated(self) -> bool:
        return self.act in ("swiglu", "geglu")

    @property
    def N1(self) -> int:
        return 2 * self.I if self.gated else self.I

    def with_(self, **kw) -> "MoEConfig":
        return dataclasses.replace(self, **kw)


CONFIGS = {
    "tiny": MoEConfig("tiny", M=4, H=128, I=128, E=4, top_k=2, scale_mode="global_one",
                      seed=0, weight_seed=0),
    "decode_t4": MoEConfig("decode_t4", M=4, H=2048, I=512, E=128, top_k=10,
                           seed=1, weight_seed=1),
    "decode_t8": MoEConfig("decode_t8", M=8, H=2048, I=512, E=128, top_k=10,
                           seed=2, weight_seed=1),
    "wide_decode": MoEConfig("wide_decode", M=8, H=7168, I=2048, E=256, top_k=8,
                             seed=3, weight_seed=4),
    "prefill_uniform": MoEConfig("prefill_uniform", M=4096, H=7168, I=2048, E=256, top_k=8,
                                 seed=4, weight_seed=4),
    "prefill_skewed": MoEConfig("prefill_skewed", M=4096, H=7168, I=2048, E=256, top_k=8,
                                seed=5, weight_seed=4, skew=1.2),
    "relu2_ep": MoEConfig("relu2_ep", M=16384, H=4096, I=1536, E=128, top_k=6, act="relu2",
                          seed=6, weight_seed=6, local_offset=0, num_local=64),
}


def hidden_bf16(cfg: MoEConfig, device="cpu") -> torch.Tensor:
    """BF16 hidden states [M, H], N(0,1) rounded to nearest-even BF16."""
    z = normal_f32(cfg.seed, TID_HIDDEN, 0, cfg.M * cfg.H, device)
    return z.to(torch.bfloat16).reshape(cfg.M, cfg.H)


def router_logits(cfg: MoEConfig) -> np.ndarray:
    """float32 router logits [M, E] (N(0,1), plus the Zipf bias when skewed)."""
    z = normal_f32(cfg.seed, TID_LOGITS, 0, cfg.M * cfg.E, "cpu").numpy().reshape(cfg.M, cfg.E)
    if cfg.skew:
        # a seeded permutation gives each expert a popularity rank 1..E; the
        # bias is the log of a Zipf(s) probability, up to a constant
        u = uniform_u32(cfg.seed, TID_ZIPF_PERM, cfg.E).numpy()
        rank = np.empty(cfg.E, dtype=np.int64)
        rank[np.argsort(u, kind="stable")] = np.arange(1, cfg.E + 1)
        bias = (-np.float32(cfg.skew) * np.log(rank.astype(np.float32))).astype(np.float32)
        z = (z + bias[None, :]).astype(np.float32)
    return z


def routing(cfg: MoEConfig) -> tuple[np.ndarray, np.ndarray]:
    """(topk_ids int32 [M,k], topk_weights float32 [M,k]).

    float32 softmax over all E experts, the k largest probabilities (ties to
    the lower expert id), renormalised to sum to one in ascending-slot order.
    """
    logits = router_logits(cfg)
    m = logits.max(axis=1, keepdims=True)
    e = np.exp((logits - m).astype(np.float32)).astype(np.float32)
    p = (e / e.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
    order = np.argsort(-p, axis=1, kind="stable")[:, : cfg.top_k]
    ids = order.astype(np.int32)
    pk = np.take_along_axis(p, order, axis=1).astype(np.float32)
    s = np.zeros(cfg.M, dtype=np.float32)
    for j in range(cfg.top_k):
        s = (s + pk[:, j]).astype(np.float32)
    w = (pk / s[:, None]).astype(np.float32)
    return ids, w


def expert_w1_bf16(cfg: MoEConfig, local_expert: int, device="cpu") -> torch.Tensor:
    """BF16 W1 of one local expert, [N1, H]; SwiGLU rows are [gate; up]."""
    e = cfg.local_offset + local_expert
    z = normal_f32(cfg.weight_seed, TID_W1_BASE + 2 * e, 0, cfg.N1 * cfg.H, device)
    return (z * torch.tensor(WEIGHT_STD, dtype=torch.float32, device=device)).to(
        torch.bfloat16).reshape(cfg.N1, cfg.H)


def expert_w2_bf16(cfg: MoEConfig, local_expert: int, device="cpu") -> torch.Tensor:
    """BF16 W2 of one local expert, [H, I]."""
    e = cfg.local_offset + local_expert
    z = normal_f32(cfg.weight_seed, TID_W2_BASE + 2 * e, 0, cfg.H * cfg.I, device)
    return (z * torch.tensor(WEIGHT_STD, dtype=torch.float32, device=device)).to(
        torch.bfloat16).reshape(cfg.H, cfg.I)


def with_unrouted(ids: np.ndarray, frac: float, seed: int, num_experts: int) -> np.ndarray:
    """Copy of ids with a seeded fraction of slots set to -1 or to ids >= E.

    Unrouted and out-of-range slots are part of the routing contract: they
    must contribute nothing.
    """
    ids = ids.copy()
    u = uniform_u32(seed, 77, ids.size).numpy().reshape(ids.shape)
    thresh = int(frac * 2**32)
    sel = u < thresh
    alt = (u & 1) == 1
    ids[sel & alt] = -1
    ids[sel & ~alt] = num_experts + (u[sel & ~alt] % 7).astype(np.int32)
    return ids


def expected_rows(ids: np.ndarray, off: int, El: int) -> int:
    """Number of routed local (token, slot) pairs: the algorithmic row count R."""
    l = ids.astype(np.int64) - off
    return int(((l >= 0) & (l < El)).sum())


def algorithmic_work(cfg: MoEConfig, ids: np.ndarray, finalize: bool = True) -> dict:
    """FLOPs and HBM bytes the method must move for one forward (no padding rows)."""
    l = ids.astype(np.int64).ravel() - cfg.local_offset
    l = l[(l >= 0) & (l < cfg.El)]
    R = int(l.size)
    active = int(np.unique(l).size)
    flops = 2.0 * R * cfg.H * cfg.N1 + 2.0 * R * cfg.I * cfg.H
    nv = 0.5 + 1.0 / 16.0
    wbytes = active * (cfg.N1 * cfg.H + cfg.H * cfg.I) * nv + 8.0 * cfg.El
    io = cfg.M * cfg.H * 2.0 + (cfg.M * cfg.H * 2.0 if finalize else R * cfg.H * 2.0) \
        + cfg.M * cfg.top_k * 8.0
    return {"R": R, "active_experts": active, "flops": flops, "bytes": wbytes + io,
            "weight_bytes": wbytes}
