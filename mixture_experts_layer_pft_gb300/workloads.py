"""Seeded synthetic workloads for the padding-free MoE layer.

This module only draws inputs; it holds none of the layer's arithmetic, so both the CUDA
path and the CPU oracle may consume what it makes.  Shapes follow the model table of the
X-MoE review (§5 "Benchmarks": Small h=2048 f=1408 E=64 k=6 s=2048; Medium h=5120 f=1536
E=128 k=6 s=4096; Large h=7168 f=2048 E=256 k=8 s=4096; Super h=7168 f=2560 E=256 k=8
s=4096) and the FlashDMoE blog §6
(synthetic inputs, up to 16k tokens, k=2, up to 128 experts, FP32).

Recipe (every workload): one ``torch.Generator`` on the target device seeded with the
workload's seed; draw order x, W_g, W1, W3, W2, dy; x ~ N(0,1), W_g ~ N(0,1/h),
W1, W3 ~ N(0,1/h), W2 ~ N(0,1/f), dy ~ N(0,1); values are drawn in fp32 and cast to the
activation type.  The router weight and bias stay fp32.  Skewed workloads add a fixed
per-expert logit bias b_e = 2·log((e+1)^-0.8) (Zipf-like load, many experts near empty).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    h: int
    E: int
    k: int
    f: int
    dtype: str  # "f32" or "bf16": activations and expert weights
    skew: bool  # add the Zipf-like router bias
    backward: bool  # the timed step includes the backward pass
    seed: int

    @property
    def Tk(self) -> int:
        return self.T * self.k

    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_tokens(self, T: int) -> "Workload":
        return Workload(self.name, T, self.h, self.E, self.k, self.f, self.dtype, self.skew,
                        self.backward, self.seed)


WORKLOADS = [
    Workload("tiny-fp32", 256, 128, 8, 2, 64, "f32", False, True, 0),
    Workload("xmoe-small-bf16", 2048, 2048, 64, 6, 1408, "bf16", False, True, 1),
    Workload("xmoe-medium-bf16-zipf", 4096, 5120, 128, 6, 1536, "bf16", True, True, 2),
    Workload("xmoe-large-bf16", 4096, 7168, 256, 8, 2048, "bf16", False, True, 3),
    Workload("longseq-fp32-fwd-zipf", 16384, 2048, 128, 2, 2048, "f32", True, False, 4),
    # the X-MoE Super layer (same table): the Large layer with a wider expert FFN
    Workload("xmoe-super-bf16", 4096, 7168, 256, 8, 2560, "bf16", False, True, 5),
]


def skew_bias(E: int, device="cpu") -> torch.Tensor:
    """b_e = 2·log(1/(e+1)^0.8) = -1.6·ln(e+1), fp32 [E]."""
    e = torch.arange(E, dtype=torch.float64)
    return (-1.6 * torch.log(e + 1.0)).to(torch.float32).to(device)


def _normal(gen, shape, std, device, out_dtype):
    return (torch.randn(*shape, generator=gen, device=device, dtype=torch.float32) * std).to(out_dtype)


def make_inputs(w: Workload, device="cpu", T: int | None = None, seed: int | None = None,
                token_seed: int | None = None):
    """Draw x, W_g, bias, W1, W3, W2, dy for workload ``w`` on ``device``.

    ``T`` overrides the token count; ``seed`` overrides the workload's seed.  With
    ``token_seed`` the tokens x and dy come from a second generator seeded with it (x, then
    dy) while the weights keep the workload's draws: the data-parallel replicas of one
    layer see different tokens and identical weights.
    """
    T = w.T if T is None else T
    seed = w.seed if seed is None else seed
    dt = w.torch_dtype()
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tgen = gen
    if token_seed is not None:
        tgen = torch.Generator(device=device)
        tgen.manual_seed(token_seed)
    x = _normal(tgen, (T, w.h), 1.0, device, dt)
    Wg = _normal(gen, (w.h, w.E), 1.0 / math.sqrt(w.h), device, torch.float32)
    W1 = torch.empty(w.E, w.h, w.f, dtype=dt, device=device)
    W3 = torch.empty(w.E, w.h, w.f, dtype=dt, device=device)
    W2 = torch.empty(w.E, w.f, w.h, dtype=dt, device=device)
    # one expert at a time keeps the fp32 staging tensor small at the large shapes
    for e in range(w.E):
        W1[e] = _normal(gen, (w.h, w.f), 1.0 / math.sqrt(w.h), device, dt)
    for e in range(w.E):
        W3[e] = _normal(gen, (w.h, w.f), 1.0 / math.sqrt(w.h), device, dt)
    for e in range(w.E):
        W2[e] = _normal(gen, (w.f, w.h), 1.0 / math.sqrt(w.f), device, dt)
    dy = _normal(tgen, (T, w.h), 1.0, device, dt)
    bias = skew_bias(w.E, device) if w.skew else None
    return {"x": x, "Wg": Wg, "bias": bias, "W1": W1, "W3": W3, "W2": W2, "dy": dy}


def random_logits(T: int, E: int, seed: int, device="cpu", scale: float = 1.0):
    """Router logits drawn directly (fp32 N(0, scale^2)), for gating tests that must feed
    identical logits to both sides."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randn(T, E, generator=gen, device=device, dtype=torch.float32) * scale


def random_tensor(shape, seed: int, dtype=torch.float32, device="cpu", std: float = 1.0):
    """A seeded N(0, std^2) tensor of ``shape`` in ``dtype``."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return _normal(gen, shape, std, device, dtype)


def make_token_sample(w: Workload, T: int, device="cpu"):
    """x, W_g, bias and dy for T tokens of workload ``w`` with no expert weights: the seeded
    recipe's router weight and token draws (x, then W_g, from the workload's seed; dy from a
    second generator seeded with seed + 1), for the oracle's timing samples, which fetch expert
    weights only for the experts their tokens reach (``make_expert_sample``)."""
    dt = w.torch_dtype()
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    x = _normal(gen, (T, w.h), 1.0, device, dt)
    Wg = _normal(gen, (w.h, w.E), 1.0 / math.sqrt(w.h), device, torch.float32)
    dgen = torch.Generator(device=device)
    dgen.manual_seed(w.seed + 1)
    dy = _normal(dgen, (T, w.h), 1.0, device, dt)
    bias = skew_bias(w.E, device) if w.skew else None
    return {"x": x, "Wg": Wg, "bias": bias, "dy": dy}


def make_expert_sample(w: Workload, experts, device="cpu"):
    """{e: (W1[e], W3[e], W2[e])} for the listed experts, each drawn from its own generator
    (seeded from the workload's seed and e) with the recipe's distributions: timing samples for
    the oracle, not the values make_inputs draws."""
    dt = w.torch_dtype()
    out = {}
    for e in experts:
        gen = torch.Generator(device=device)
        gen.manual_seed(1_000_003 * (w.seed + 1) + int(e))
        out[int(e)] = (_normal(gen, (w.h, w.f), 1.0 / math.sqrt(w.h), device, dt),
                       _normal(gen, (w.h, w.f), 1.0 / math.sqrt(w.h), device, dt),
                       _normal(gen, (w.f, w.h), 1.0 / math.sqrt(w.f), device, dt))
    return out
