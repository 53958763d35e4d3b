"""Seeded synthetic workloads for the MLP training step.

This module is the only code that the CUDA path and the CPU oracle share: it
draws inputs (batches, labels, initial parameters) and holds the workload
table.  It contains none of the step's arithmetic.  Every array it returns is a
CPU torch tensor; callers copy it to the device or hand it to the oracle.

Workloads (shapes, distributions, optimiser settings) follow the five MLP
training configurations this library is measured on: a 784-256-128-10 ReLU
net (the MNIST-shaped network of noeira.ai "Neural networks", section "A
complete example") in fp32 at batch 64 and 4096; a CIFAR-shaped
3072-1024-1024-1024-10 ReLU net in bf16; a token-level 1024-4096(GELU)-1024
block with a 32000-way head in bf16; and a deep narrow 512x8 ReLU net with 100
classes in bf16.  The synthetic data stands in for MNIST / CIFAR-10 / a token
stream, none of which is needed or present.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

ACT_NONE, ACT_RELU, ACT_GELU_TANH = 0, 1, 2
F32, BF16 = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Tuple[int, ...]          # [in, h1, ..., C]
    acts: Tuple[int, ...]          # one per hidden layer (len(dims) - 2)
    dtype: int                     # F32 or BF16 (bf16 compute, fp32 master)
    batch: int
    steps: int
    lr: float
    beta1: float
    beta2: float
    eps: float
    wd: float
    x_dist: str                    # "uniform01" or "normal"
    seed: int
    graph_steps: int = 1           # steps captured per CUDA-graph launch

    @property
    def n_layers(self) -> int:
        return len(self.dims) - 1

    @property
    def n_classes(self) -> int:
        return self.dims[-1]

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def param_shapes(self) -> List[Tuple[Tuple[int, int], Tuple[int]]]:
        return [((self.dims[l + 1], self.dims[l]), (self.dims[l + 1],))
                for l in range(self.n_layers)]

    def n_params(self) -> int:
        return sum(a * b + a for (a, b), _ in self.param_shapes())

    def gemm_flops(self) -> int:
        """Algorithmic GEMM FLOPs of one training step: forward, wgrad for
        every layer, dgrad for every layer but the first."""
        B = self.batch
        f = 0
        for l in range(self.n_layers):
            k, n = self.dims[l], self.dims[l + 1]
            f += 2 * B * k * n * (3 if l > 0 else 2)
        return f


_R, _G = ACT_RELU, ACT_GELU_TANH

WORKLOADS = {
    "mnist_mlp_b64": Workload(
        "mnist_mlp_b64", (784, 256, 128, 10), (_R, _R), F32, 64, 1,
        1e-3, 0.9, 0.999, 1e-8, 0.01, "uniform01", 1001),
    "mnist_mlp_b4096": Workload(
        "mnist_mlp_b4096", (784, 256, 128, 10), (_R, _R), F32, 4096, 100,
        1e-3, 0.9, 0.999, 1e-8, 0.01, "uniform01", 1002),
    "cifar_mlp_b8192": Workload(
        "cifar_mlp_b8192", (3072, 1024, 1024, 1024, 10), (_R, _R, _R), BF16,
        8192, 20, 3e-4, 0.9, 0.999, 1e-8, 0.05, "normal", 1003),
    "lm_block_t16384": Workload(
        "lm_block_t16384", (1024, 4096, 1024, 32000), (_G, ACT_NONE), BF16,
        16384, 10, 1e-4, 0.9, 0.999, 1e-8, 0.1, "normal", 1004),
    "deep_narrow_b65536": Workload(
        "deep_narrow_b65536", (512,) + (512,) * 8 + (100,), (_R,) * 8, BF16,
        65536, 50, 1e-3, 0.9, 0.999, 1e-8, 0.01, "normal", 1005,
        graph_steps=50),
}
# The order the configurations are listed in (small fp32 case first).
WORKLOAD_ORDER = ["mnist_mlp_b64", "mnist_mlp_b4096", "cifar_mlp_b8192",
                  "lm_block_t16384", "deep_narrow_b65536"]


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def make_batch(w: Workload, step: int, batch: Optional[int] = None
               ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Batch `step` of workload `w`: (x, labels).

    x is [B, dims[0]] float32 (F32 workloads) or bfloat16 (BF16 workloads,
    drawn in fp32 and converted by torch's round-to-nearest-even cast);
    labels are int32 uniform in [0, C).
    """
    B = w.batch if batch is None else batch
    rng = _rng(w.seed, 1, step)
    if w.x_dist == "uniform01":
        x = rng.random((B, w.dims[0]), dtype=np.float32)
    else:
        x = rng.standard_normal((B, w.dims[0]), dtype=np.float32)
    labels = rng.integers(0, w.n_classes, size=(B,), dtype=np.int32)
    xt = torch.from_numpy(x)
    if w.dtype == BF16:
        xt = xt.to(torch.bfloat16)
    return xt, torch.from_numpy(labels)


def make_params(w: Workload, seed: Optional[int] = None) -> List[torch.Tensor]:
    """Initial parameters [W1, b1, ..., WL, bL] as fp32 CPU tensors.

    Weights are Kaiming-normal in fan-in mode with the ReLU gain,
    std = sqrt(2 / fan_in), for every layer; biases are zero.  (The MNIST MLP
    of noeira.ai "Neural networks", "A complete example", is built with the
    Kaiming initializer.)
    """
    rng = _rng(w.seed if seed is None else seed, 2)
    out = []
    for (n, k), _ in w.param_shapes():
        W = rng.standard_normal((n, k), dtype=np.float32) * np.float32(math.sqrt(2.0 / k))
        out += [torch.from_numpy(W.astype(np.float32)), torch.zeros(n, dtype=torch.float32)]
    return out


def make_uniform(shape: Sequence[int], lo: float, hi: float, *key: int,
                 dtype=torch.float32) -> torch.Tensor:
    """Generic seeded uniform tensor for op-level tests."""
    a = _rng(*key).uniform(lo, hi, size=tuple(shape)).astype(np.float32)
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def make_normal(shape: Sequence[int], std: float, *key: int,
                dtype=torch.float32) -> torch.Tensor:
    """Generic seeded normal tensor for op-level tests."""
    a = (_rng(*key).standard_normal(tuple(shape), dtype=np.float32) * np.float32(std))
    t = torch.from_numpy(a)
    return t.to(dtype) if dtype != torch.float32 else t


def make_labels(n: int, C: int, *key: int) -> torch.Tensor:
    return torch.from_numpy(_rng(*key).integers(0, C, size=(n,), dtype=np.int32))


def make_targets(w: Workload, step: int, batch: Optional[int] = None) -> torch.Tensor:
    """Regression targets of batch `step` for an MSE step: float32 [B, C],
    standard normal (the real-valued outputs MuNet's "Python training"
    example fits with mse_loss; the pages fix no distribution)."""
    B = w.batch if batch is None else batch
    return torch.from_numpy(_rng(w.seed, 3, step).standard_normal((B, w.n_classes), dtype=np.float32))
