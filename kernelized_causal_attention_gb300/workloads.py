"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and describes shapes; it holds none of
the attention arithmetic, so the CUDA path and the CPU oracle can both be fed
from it without sharing any of the method.

Recipe (the same for every workload): a ``torch.Generator('cpu')`` seeded with
the workload's seed draws, in this order, the valid lengths (non-causal only,
uniform integers in [lo, hi]), then Q, K, V and the upstream gradient G, each
i.i.d. N(0, 1) in fp32, and only then casts to the workload's dtype.  Decode
draws q_t, k_t, v_t (in that order) once per step from one generator.  The
projected decode step draws x ~ N(0, 1) [B, d_model], then W ~ N(0, 1/d_model)
[d_model, H(2D+M)] (so that the projections come out near unit variance), then
a state standing in for t earlier tokens: S_0 entries N(0, t) and Z_0 entries
uniform in [t/2, 3t/2] (positive, like a sum of t positive features).

The shapes follow the pages' workloads: 784-token (28x28) and 3072-token
(32x32x3) autoregressive image sequences with 8 heads of 64 dims, long
speech-like non-causal sequences with 6 heads and lengths between 800 and 2048,
and 256 independent decode streams; for the projected step, 256 streams with
d_model = 512 and, as in the MNIST generation test of §4.2.1 (10,000 images
decoded at once), 10,000 streams with d_model = 256 and 8 heads of 32.  The pages' datasets (MNIST, CIFAR-10, WSJ)
are not used: these normal draws stand in for their activations.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "causal" | "noncausal" | "decode" | "decode_proj"
    B: int
    H: int
    N: int  # sequence length; decode: number of steps T
    D: int
    M: int
    dtype: str  # "f32" | "bf16"
    seed: int
    len_range: tuple = field(default=None)  # non-causal: (lo, hi) inclusive
    d_model: int = 0  # projected decode: width of the layer input x

    @property
    def torch_dtype(self):
        return DTYPES[self.dtype]


WORKLOADS = {
    "causal_tiny_f32": Workload("causal_tiny_f32", "causal", 1, 1, 64, 16, 16, "f32", 1),
    "causal_mnist_bf16": Workload("causal_mnist_bf16", "causal", 8, 8, 784, 64, 64, "bf16", 2),
    "causal_cifar_bf16": Workload("causal_cifar_bf16", "causal", 4, 8, 3072, 64, 64, "bf16", 3),
    # the pages' models' head size: 256 / 8 = 32
    "causal_cifar_d32_bf16": Workload("causal_cifar_d32_bf16", "causal", 4, 8, 3072, 32, 32, "bf16", 8),
    # the 3072-token images with fp32 inputs (the fp32-accurate path)
    "causal_cifar_f32": Workload("causal_cifar_f32", "causal", 4, 8, 3072, 64, 64, "f32", 9),
    "noncausal_speech_f32": Workload("noncausal_speech_f32", "noncausal", 16, 6, 2048, 64, 64,
                                     "f32", 4, (800, 2048)),
    "decode_f32": Workload("decode_f32", "decode", 256, 8, 3072, 64, 64, "f32", 5),
    # N is the number of earlier tokens the stand-in state represents
    "decode_proj_bf16": Workload("decode_proj_bf16", "decode_proj", 256, 8, 392, 64, 64, "bf16", 6,
                                 d_model=512),
    "decode_proj_mnist_bf16": Workload("decode_proj_mnist_bf16", "decode_proj", 10000, 8, 392, 32,
                                       32, "bf16", 7, d_model=256),
}


def causal_inputs(B, H, N, D, M, dtype="f32", seed=0):
    """q, k [B,H,N,D]; v, g [B,H,N,M] on the CPU in the requested dtype."""
    gen = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn(B, H, N, D, generator=gen)
    k = torch.randn(B, H, N, D, generator=gen)
    v = torch.randn(B, H, N, M, generator=gen)
    g = torch.randn(B, H, N, M, generator=gen)
    dt = DTYPES[dtype]
    return q.to(dt), k.to(dt), v.to(dt), g.to(dt)


def noncausal_inputs(B, H, N, D, M, dtype="f32", seed=0, len_range=None):
    """(lengths int32 [B], q, k, v, g); lengths drawn first, uniform in
    [lo, hi] (all N when len_range is None)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    if len_range is None:
        lengths = torch.full((B,), N, dtype=torch.int32)
    else:
        lo, hi = len_range
        lengths = torch.randint(lo, hi + 1, (B,), generator=gen).to(torch.int32)
    q = torch.randn(B, H, N, D, generator=gen)
    k = torch.randn(B, H, N, D, generator=gen)
    v = torch.randn(B, H, N, M, generator=gen)
    g = torch.randn(B, H, N, M, generator=gen)
    dt = DTYPES[dtype]
    return lengths, q.to(dt), k.to(dt), v.to(dt), g.to(dt)


class DecodeStream:
    """Per-step decode inputs: each call to ``step()`` draws q_t, k_t [B,H,D]
    and v_t [B,H,M] from one seeded generator."""

    def __init__(self, B, H, D, M, dtype="f32", seed=0):
        self.B, self.H, self.D, self.M = B, H, D, M
        self.dt = DTYPES[dtype]
        self.gen = torch.Generator("cpu").manual_seed(seed)

    def step(self):
        q = torch.randn(self.B, self.H, self.D, generator=self.gen)
        k = torch.randn(self.B, self.H, self.D, generator=self.gen)
        v = torch.randn(self.B, self.H, self.M, generator=self.gen)
        return q.to(self.dt), k.to(self.dt), v.to(self.dt)

    def steps(self, T):
        """T steps stacked: q, k [T,B,H,D]; v [T,B,H,M]."""
        qs, ks, vs = zip(*(self.step() for _ in range(T)))
        return torch.stack(qs), torch.stack(ks), torch.stack(vs)


def proj_inputs(B, d_model, H, D, M, t=100, seed=0):
    """x bf16 [B, d_model], W bf16 [d_model, H(2D+M)], S_0 float32 [B,H,D,M],
    Z_0 float32 [B,H,D], all on the CPU (recipe in the module docstring)."""
    gen = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(B, d_model, generator=gen)
    W = torch.randn(d_model, H * (2 * D + M), generator=gen) / d_model ** 0.5
    S = torch.randn(B, H, D, M, generator=gen) * t ** 0.5
    Z = (torch.rand(B, H, D, generator=gen) + 0.5) * t
    return x.to(torch.bfloat16), W.to(torch.bfloat16), S, Z


def workload_inputs(w: Workload):
    """Inputs of a named workload (causal: q,k,v,g; non-causal: lengths,q,k,v,g)."""
    if w.kind == "causal":
        return causal_inputs(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed)
    if w.kind == "noncausal":
        return noncausal_inputs(w.B, w.H, w.N, w.D, w.M, w.dtype, w.seed, w.len_range)
    raise ValueError("decode workloads are drawn step by step with DecodeStream")
