"""Seeded synthetic workloads for the ZeRO optimizer step.

This module holds only sizes and random numbers: the five parameter-set shapes, per-tensor
gradient scales, and the seeded generators of gradients and initial master weights. It
holds none of the step's arithmetic (no layout, reduction, norm or optimizer), so that the
GPU path and the CPU oracle can both be fed from it without sharing code.

Gradients are produced in each rank's *unpadded* tensor order; placing them into a padded
flat buffer is the caller's job (the library's planner for the GPU path, the oracle's
planner for the oracle).

Shapes follow the dense-transformer parameter count of "并行策略总览：六个维度各切什么、
怎么通信" (blog.javazero.top), section 先把要切的东西摆出来: a layer holds about 12 d^2
weights (attention 4 d^2, MLP 8 d^2), plus a 50257 x d embedding.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

BASE_SEED = 20261202
VOCAB = 50257
MIB = 1024 * 1024


@dataclass(frozen=True)
class Workload:
    name: str
    numel: tuple          # tensor sizes in declared order
    M: int                # emulated data-parallel ranks
    stage: int            # ZeRO stage 1/2/3
    bucket_bytes: int     # bf16 gradient bytes per bucket (0 = one bucket)
    clip: float | None    # global-norm clip threshold (None = no clipping)
    steps: int
    sigma_mode: str       # "const" or "loguniform"
    sigma_const: float = 1e-3
    zero_frac: float = 0.0  # probability that a (rank, element) gradient is exactly +0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    master_std: float = 0.02
    seed: int = BASE_SEED

    @property
    def N(self) -> int:
        return int(sum(self.numel))


def _transformer_numel(d: int, layers: int, layernorm: bool) -> tuple:
    sizes = [VOCAB * d]
    for _ in range(layers):
        if layernorm:
            sizes += [d, d]                      # ln1.weight, ln1.bias
        sizes += [d * 3 * d, d * d]              # qkv, attention projection (4 d^2)
        if layernorm:
            sizes += [d, d]                      # ln2.weight, ln2.bias
        sizes += [d * 4 * d, 4 * d * d]          # MLP fc, fc projection (8 d^2)
    if layernorm:
        sizes += [d, d]                          # final LayerNorm
    return tuple(sizes)


def _is_prime(n: int) -> bool:
    if n < 2:
        return False
    if n % 2 == 0:
        return n == 2
    f = 3
    while f * f <= n:
        if n % f == 0:
            return False
        f += 2
    return True


def _next_prime(n: int) -> int:
    while not _is_prime(n):
        n += 1
    return n


def ragged_numel(count: int = 2000, lo: int = 2 ** 10, hi: int = 2 ** 22, seed: int = BASE_SEED) -> tuple:
    """Sizes log-uniform in [lo, hi]; every 10th replaced by the next prime >= it; every
    4th (offset 1) forced odd, so at least a quarter of the sizes are odd and thus not
    divisible by any even rank count."""
    g = torch.Generator(device="cpu").manual_seed(seed + 3)
    u = torch.rand(count, generator=g, dtype=torch.float64).numpy()
    sizes = []
    for i in range(count):
        n = int(math.floor(math.exp(math.log(lo) + u[i] * (math.log(hi) - math.log(lo)))))
        n = min(max(n, lo), hi)
        if i % 10 == 0:
            n = _next_prime(n)
        elif i % 4 == 1:
            n |= 1
        sizes.append(n)
    return tuple(sizes)


KEYS = ("tiny", "gpt2s", "1p3b", "ragged", "4b")


def workload(key: str) -> Workload:
    """The five standard workloads, by short name: "tiny" (4096 params, M=2), "gpt2s"
    (GPT-2-small shaped, M=8), "1p3b" (1.3B dense, M=8), "ragged" (2000 tensors, M=16),
    "4b" (4B dense, M=4)."""
    if key == "tiny":
        return Workload("tiny: one 4096-element tensor, M=2, ZeRO-1, no clip, 3 steps",
                        (4096,), M=2, stage=1, bucket_bytes=0, clip=None, steps=3, sigma_mode="const")
    if key == "gpt2s":
        return Workload("GPT-2-small shaped (123,570,432 params, d=768, 12 layers), M=8, ZeRO-2, 25 MiB buckets, "
                        "no clip, 10 steps",
                        _transformer_numel(768, 12, True), M=8, stage=2, bucket_bytes=25 * MIB, clip=None,
                        steps=10, sigma_mode="loguniform")
    if key == "1p3b":
        return Workload("1.3B dense transformer shaped (1,310,885,888 params, d=2048, 24 layers), M=8, ZeRO-1, "
                        "clip 1.0, 5 steps",
                        _transformer_numel(2048, 24, False), M=8, stage=1, bucket_bytes=0, clip=1.0, steps=5,
                        sigma_mode="loguniform")
    if key == "ragged":
        return Workload("ragged: 2000 tensors log-uniform in 1K..4M with primes, M=16, ZeRO-3, clip 1.0, "
                        "1% exact zeros, 5 steps",
                        ragged_numel(), M=16, stage=3, bucket_bytes=0, clip=1.0, steps=5, sigma_mode="const",
                        zero_frac=0.01)
    if key == "4b":
        return Workload("4B dense transformer shaped (4,092,982,400 params, d=3200, 32 layers), M=4, ZeRO-3, "
                        "clip 1.0, 3 steps",
                        _transformer_numel(3200, 32, False), M=4, stage=3, bucket_bytes=0, clip=1.0, steps=3,
                        sigma_mode="loguniform")
    raise ValueError(f"no workload {key!r} (known: {', '.join(KEYS)})")


def small_variant(w: Workload, numel: tuple, name: str | None = None, **kw) -> Workload:
    """The same recipe on smaller tensors (for element-by-element parity)."""
    from dataclasses import replace
    return replace(w, numel=tuple(int(x) for x in numel), name=name or (w.name + " (reduced)"), **kw)


def sigmas(w: Workload) -> np.ndarray:
    """Per-tensor gradient standard deviation (float64)."""
    T = len(w.numel)
    if w.sigma_mode == "const":
        return np.full(T, w.sigma_const, dtype=np.float64)
    out = np.empty(T, dtype=np.float64)
    lo, hi = math.log(1e-5), math.log(1e-2)
    for t in range(T):
        g = torch.Generator(device="cpu").manual_seed(w.seed ^ t)
        u = float(torch.rand(1, generator=g, dtype=torch.float64))
        out[t] = math.exp(lo + u * (hi - lo))
    return out


def _grad_seed(w: Workload, rank: int, step: int) -> int:
    return (w.seed * 1_000_003 + rank * 10_007 + step * 101 + 17) % (2 ** 62)


def fill_grads(w: Workload, rank: int, step: int, out: torch.Tensor, tensor_offsets, sig=None) -> None:
    """Write rank `rank`'s bf16 gradient of step `step` into the flat bf16 buffer `out`,
    tensor t at element offset tensor_offsets[t]. Lanes outside the tensors are untouched
    (callers zero them). Values: bf16(sigma_t * z), z ~ N(0, 1); with zero_frac > 0 a
    Bernoulli(zero_frac) mask sets elements to +0."""
    assert out.dtype == torch.bfloat16
    dev = out.device
    sig = sigmas(w) if sig is None else sig
    g = torch.Generator(device=dev).manual_seed(_grad_seed(w, rank, step))
    for t, n in enumerate(w.numel):
        if n == 0:
            continue
        off = int(tensor_offsets[t])
        z = torch.randn(n, generator=g, device=dev, dtype=torch.float32)
        z.mul_(float(sig[t]))
        if w.zero_frac > 0:
            masked = torch.rand(n, generator=g, device=dev) < w.zero_frac
            z.masked_fill_(masked, 0.0)   # exactly +0
        out[off:off + n].copy_(z)
        del z


def master_init(w: Workload, device="cpu") -> torch.Tensor:
    """Initial fp32 master weights ~ N(0, master_std), unpadded tensor order."""
    g = torch.Generator(device=device).manual_seed(w.seed + 1)
    x = torch.randn(w.N, generator=g, device=device, dtype=torch.float32)
    return x.mul_(w.master_std)
