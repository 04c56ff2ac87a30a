"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random numbers and lays out tensors; it holds none of the
layer's arithmetic.  Both the CUDA library's tests/bench and the CPU oracle take
their inputs from here, so the two sides always see the same values.

Distributions (as the workloads state them): x ~ N(0, 1); router weights
W_r ~ N(0, variance 1/H); expert and shared-expert weights ~ N(0, sd 0.02).  bf16
workloads round every value to bf16 (round-to-nearest-even), the toy workload stays
in float32.  Uneven expert load comes from a per-expert router bias b[E] (float32):
  * "normal": b_e ~ N(0, 1);
  * "zipf":   a seeded random permutation gives each expert a popularity rank
              rho_e in 1..E and b_e = -s * ln(rho_e)  (log of a Zipf(s) law up to a
              constant), s = 1.1.
Each tensor is drawn from its own seeded torch.Generator stream, so changing one
shape does not shift the values of another tensor.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """One workload: tokens T, hidden H, experts E, top-K, expert intermediate I."""

    name: str
    T: int
    H: int
    E: int
    K: int
    I: int
    I_shared: int = 0          # 0 = no shared expert
    theta: float = 0.0         # gate-drop threshold, 0 = off
    dtype: str = "bf16"        # "bf16" or "f32" (activations and weights)
    bias: str = "none"         # "none" | "normal" | "zipf"
    zipf_s: float = 1.1
    seed: int = 0

    def with_(self, **kw) -> "MoEShape":
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32


WORKLOADS = {
    # small fp32 layer: T=256, H=512, E=8, top-2, I=1024
    "toy": MoEShape("toy", T=256, H=512, E=8, K=2, I=1024, dtype="f32"),
    # Mixtral-8x7B-shaped prefill: near-uniform load
    "mixtral": MoEShape("mixtral", T=4096, H=4096, E=8, K=2, I=14336),
    # Qwen3-30B-A3B-shaped prefill: per-expert N(0,1) logit bias, uneven groups
    "qwen_prefill": MoEShape("qwen_prefill", T=8192, H=2048, E=128, K=8, I=768, bias="normal"),
    # Qwen3-30B-A3B-shaped decode step (T in {1, 8, 32, 64}); same generators
    "qwen_decode": MoEShape("qwen_decode", T=64, H=2048, E=128, K=8, I=768, bias="normal"),
    # DeepSeek-style: 256 routed experts top-8 + one shared expert, Zipf popularity,
    # gates below 0.05 dropped
    "deepseek": MoEShape("deepseek", T=16384, H=7168, E=256, K=8, I=2048, I_shared=2048,
                         theta=0.05, bias="zipf"),
}

DECODE_TOKENS = (1, 8, 32, 64)


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + stream)
    return g


def _normal(shape, sd, dtype, device, g, chunk_dim0: Optional[int] = None):
    """N(0, sd^2) drawn in float32 and rounded once to ``dtype``.

    Large tensors are drawn slice by slice along dim 0 to bound the float32
    temporary; the slices come from the same generator in order.
    """
    out = torch.empty(shape, dtype=dtype, device=device)
    if chunk_dim0 is None or shape[0] <= chunk_dim0:
        out.copy_(torch.randn(shape, generator=g, device=device, dtype=torch.float32) * sd)
        return out
    for i in range(0, shape[0], chunk_dim0):
        j = min(shape[0], i + chunk_dim0)
        out[i:j].copy_(torch.randn((j - i,) + tuple(shape[1:]), generator=g, device=device,
                                   dtype=torch.float32) * sd)
    return out


def router_bias(shape: MoEShape, device="cpu") -> Optional[torch.Tensor]:
    """Per-expert float32 router bias that makes the expert load uneven (or None)."""
    if shape.bias == "none":
        return None
    g = _gen(device, shape.seed, 5)
    if shape.bias == "normal":
        return torch.randn((shape.E,), generator=g, device=device, dtype=torch.float32)
    if shape.bias == "zipf":
        rank = torch.randperm(shape.E, generator=g, device=device).to(torch.float64) + 1.0
        return (-shape.zipf_s * torch.log(rank)).to(torch.float32)
    raise ValueError(shape.bias)


def make_inputs(shape: MoEShape, device="cpu", T: Optional[int] = None, weights: bool = True):
    """All inputs of one workload as torch tensors on ``device``.

    Returns a dict: x [T,H], w_router [E,H], w_gate_up [E,2I,H] (rows 0..I-1 gate,
    I..2I-1 up), w_down [E,H,I], router_bias [E] float32 or None, and, when
    I_shared > 0, w_shared_gate_up [2I_s,H] and w_shared_down [H,I_s].
    ``T`` overrides the token count: the first T rows of the workload's token
    stream (the stream is drawn for max(T, shape.T) rows).
    """
    dt = shape.torch_dtype
    Tn = shape.T if T is None else T
    Tdraw = max(Tn, shape.T)
    H, E, I = shape.H, shape.E, shape.I
    out = {}
    out["x"] = _normal((Tdraw, H), 1.0, dt, device, _gen(device, shape.seed, 1), 4096)[:Tn].contiguous()
    out["w_router"] = _normal((E, H), 1.0 / math.sqrt(H), dt, device, _gen(device, shape.seed, 2))
    out["router_bias"] = router_bias(shape, device)
    if weights:
        out["w_gate_up"] = _normal((E, 2 * I, H), 0.02, dt, device, _gen(device, shape.seed, 3), 1)
        out["w_down"] = _normal((E, H, I), 0.02, dt, device, _gen(device, shape.seed, 4), 1)
        if shape.I_shared > 0:
            Is = shape.I_shared
            out["w_shared_gate_up"] = _normal((2 * Is, H), 0.02, dt, device, _gen(device, shape.seed, 6))
            out["w_shared_down"] = _normal((H, Is), 0.02, dt, device, _gen(device, shape.seed, 7))
    return out


def random_logits(T: int, E: int, seed: int = 0, device="cpu", scale: float = 1.0,
                  bias: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Float32 router logits drawn directly (for routing-stage tests): N(0, scale^2) + bias."""
    g = _gen(device, seed, 11)
    L = torch.randn((T, E), generator=g, device=device, dtype=torch.float32) * scale
    if bias is not None:
        L = L + bias.to(device)[None, :]
    return L


def to_numpy_f64(t: torch.Tensor):
    """Exact widening of a (bf16 or fp32) tensor to a float64 NumPy array on the host."""
    return t.detach().to("cpu", torch.float64).numpy()
