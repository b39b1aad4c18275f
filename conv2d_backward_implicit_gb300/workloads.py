"""Seeded synthetic inputs for conv2d dgrad: the configurations and their generators.

This module holds no arithmetic of the method.  It only names the workloads
(shapes, dtypes, value distributions; every size is written out literally)
and draws their random inputs.  Both the CUDA-path tests and the oracle take
their inputs from here; nothing here imports either of them.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` (0 by default) draws
grad_out first, then weight, in float32; the tensors are then rounded once
(round-to-nearest-even) to the workload's input dtype.  The GPU and the
oracle consume the identical rounded values (the oracle widens them exactly
to float64).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int
    Ci: int
    H: int
    W: int
    Co: int
    kH: int
    kW: int
    stride: int
    padding_h: int
    padding_w: int
    OH: int
    OW: int
    dtype: str            # "f32" (TF32 tensor cores), "bf16" or "f16"
    dist: str             # "uniform" (both U[-1,1]) or "normal" (g ~ N(0,1), w ~ N(0, w_std))
    w_std: float = 1.0

    @property
    def grad_out_shape(self):
        return (self.N, self.Co, self.OH, self.OW)

    @property
    def weight_shape(self):
        return (self.Co, self.Ci, self.kH, self.kW)

    @property
    def grad_in_shape(self):
        return (self.N, self.Ci, self.H, self.W)

    def with_batch(self, n: int) -> "Workload":
        return dataclasses.replace(self, N=n, name=f"{self.name}[N={n}]")


TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}

# The five workloads: a tiny fp32 case, ResNet 3x3, a strided downsample, a
# pointwise (pure GEMM) layer and a Ci=3 stem.  Output sizes are written out.
TINY = Workload("tiny fp32 3x3 s1 p1", 1, 8, 8, 8, 16, 3, 3, 1, 1, 1, 8, 8, "f32", "uniform")
RESNET = Workload("resnet 3x3 s1 p1", 32, 64, 56, 56, 64, 3, 3, 1, 1, 1, 56, 56, "bf16", "normal",
                  math.sqrt(2.0 / (64 * 9)))
STRIDED = Workload("strided 3x3 s2 p1", 32, 128, 56, 56, 256, 3, 3, 2, 1, 1, 28, 28, "bf16",
                   "normal", math.sqrt(2.0 / (128 * 9)))
POINTWISE = Workload("pointwise 1x1", 64, 256, 14, 14, 1024, 1, 1, 1, 0, 0, 14, 14, "f16",
                     "normal", math.sqrt(2.0 / 256))
STEM = Workload("stem 7x7 s2 p3", 16, 3, 224, 224, 64, 7, 7, 2, 3, 3, 112, 112, "f32", "normal",
                math.sqrt(2.0 / (3 * 49)))

ALL = (TINY, RESNET, STRIDED, POINTWISE, STEM)
BY_KEY = {"tiny": TINY, "resnet": RESNET, "strided": STRIDED, "pointwise": POINTWISE, "stem": STEM}


def make_inputs(wl: Workload, seed: int = 0):
    """(grad_out, weight) as CPU tensors in the workload's input dtype."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    if wl.dist == "uniform":
        g = torch.rand(wl.grad_out_shape, generator=gen, dtype=torch.float32) * 2 - 1
        w = torch.rand(wl.weight_shape, generator=gen, dtype=torch.float32) * 2 - 1
    elif wl.dist == "normal":
        g = torch.randn(wl.grad_out_shape, generator=gen, dtype=torch.float32)
        w = torch.randn(wl.weight_shape, generator=gen, dtype=torch.float32) * wl.w_std
    else:
        raise ValueError(wl.dist)
    dt = TORCH_DTYPE[wl.dtype]
    return g.to(dt), w.to(dt)


def make_tensor(shape, seed: int, dtype: str = "f32", dist: str = "uniform") -> torch.Tensor:
    """One seeded tensor (used for the forward input x in adjoint checks and for sweeps)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    if dist == "uniform":
        t = torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
    else:
        t = torch.randn(shape, generator=gen, dtype=torch.float32)
    return t.to(TORCH_DTYPE[dtype])


def random_small_shapes(count: int, seed: int = 1234, max_hw: int = 9, max_c: int = 5,
                        max_k: int = 5, strides=(1, 2, 3)):
    """Random tiny problem shapes (N, Ci, H, W, Co, kH, kW, s, ph, pw), output size left to the caller.

    Rectangular kernels, padding_h != padding_w, strides 1-3, padding up to
    the kernel size and stride above the kernel size all occur.
    """
    gen = torch.Generator(device="cpu").manual_seed(seed)

    def ri(lo, hi):
        return int(torch.randint(lo, hi + 1, (1,), generator=gen).item())

    out = []
    while len(out) < count:
        kH, kW = ri(1, max_k), ri(1, max_k)
        s = strides[ri(0, len(strides) - 1)]
        ph, pw = ri(0, kH), ri(0, kW)
        H, W = ri(1, max_hw), ri(1, max_hw)
        if H + 2 * ph < kH or W + 2 * pw < kW:
            continue
        out.append((ri(1, 2), ri(1, max_c), H, W, ri(1, max_c), kH, kW, s, ph, pw))
    return out
