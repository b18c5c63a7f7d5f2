"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws numbers (and rounds activations to bf16, the storage
type of the workloads); it holds none of the method's arithmetic.  The tests
feed the same arrays to the CUDA library and to the CPU oracle.

Two generators with the same distributions:
  * numpy PCG64 on the host (``*_np``) for parity tests and oracle samples;
  * torch Philox on the device (``*_torch``) for the large benchmark stacks,
    where drawing gigabytes on the host would dominate the run.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# ------------------------------------------------------------------ host --


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 (finite inputs); returns uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def weights_np(N: int, K: int, dist: str = "normal", scale: float = 0.02, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    if dist == "normal":
        return (rng.standard_normal((N, K)) * scale).astype(np.float32)
    if dist == "laplace":
        return rng.laplace(0.0, scale, (N, K)).astype(np.float32)
    raise ValueError(dist)


def acts_np(M: int, K: int, dist: str = "normal", seed: int = 0, outlier_p: float = 0.0,
            outlier_mult: float = 20.0, bf16: bool = True):
    """Returns (bits uint16 or None, fp32 values).  fp32 values are the exact
    bf16 values when bf16=True."""
    rng = np.random.default_rng(seed)
    if dist == "normal":
        x = rng.standard_normal((M, K))
    elif dist == "student_t4":
        x = rng.standard_t(4, size=(M, K))
    else:
        raise ValueError(dist)
    if outlier_p > 0:
        mask = rng.random((M, K)) < outlier_p
        x = np.where(mask, x * outlier_mult, x)
    x = x.astype(np.float32)
    if not bf16:
        return None, x
    bits = f32_to_bf16_bits(x)
    return bits, bf16_bits_to_f32(bits)


# ---------------------------------------------------------------- device --


def _gen(seed: int, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def weights_torch(N: int, K: int, dist: str, scale: float, seed: int, device):
    import torch

    g = _gen(seed, device)
    if dist == "normal":
        return torch.randn((N, K), generator=g, device=device, dtype=torch.float32) * scale
    if dist == "laplace":
        # difference of two Exp(1) draws; 1 - U lies in (0, 1], so the logs are finite
        e1 = -torch.log1p(-torch.rand((N, K), generator=g, device=device, dtype=torch.float32))
        e2 = -torch.log1p(-torch.rand((N, K), generator=g, device=device, dtype=torch.float32))
        return scale * (e1 - e2)
    raise ValueError(dist)


def acts_torch(M: int, K: int, dist: str, seed: int, device, outlier_p: float = 0.0, outlier_mult: float = 20.0):
    import torch

    g = _gen(seed, device)
    if dist == "normal":
        x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    elif dist == "student_t4":
        z = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
        c = torch.randn((4, M, K), generator=g, device=device, dtype=torch.float32).pow(2).sum(0) / 4.0
        x = z / c.sqrt()
    else:
        raise ValueError(dist)
    if outlier_p > 0:
        mask = torch.rand((M, K), generator=g, device=device) < outlier_p
        x = torch.where(mask, x * outlier_mult, x)
    return x.to(torch.bfloat16)


# ----------------------------------------------------------- workloads --


@dataclass
class Layer:
    name: str
    N: int
    K: int
    w_dist: str
    w_scale: float
    w_seed: int
    x_dist: str
    x_seed: int
    outlier_p: float = 0.0
    x_bf16: bool = True


@dataclass
class Workload:
    name: str
    description: str
    M: list
    layers: list = field(default_factory=list)


def workload(name: str) -> Workload:
    """The workloads (sizes, distributions and seeds): the five matmul
    workloads and the feed-forward decode built on them."""
    if name == "bitlinear-1024":
        return Workload(name, "single BitLinear decode: W N(0,0.02) [1024,1024], x fp32 N(0,1) [1,1024]", [1],
                        [Layer("linear", 1024, 1024, "normal", 0.02, 0, "normal", 0, x_bf16=False)])
    if name == "2b-decode":
        shapes = [("q_proj", 2560, 2560), ("o_proj", 2560, 2560), ("gate_proj", 6912, 2560),
                  ("up_proj", 6912, 2560), ("down_proj", 2560, 6912)]
        return Workload(name, "2B-shaped decode GEMVs, M=1, bf16 N(0,1) activations with 0.1% x20 outliers",
                        [1], [Layer(n, N, K, "normal", 0.02, 10 + i, "normal", 20 + i, outlier_p=0.001)
                              for i, (n, N, K) in enumerate(shapes)])
    if name == "gateup-sweep":
        return Workload(name, "batched decode sweep on the fused gate+up layer N=13824, K=2560",
                        [1, 2, 4, 8, 16, 32, 64], [Layer("gate_up", 13824, 2560, "normal", 0.02, 30, "normal", 31)])
    if name == "prefill-2048":
        return Workload(name, "prefill GEMM M=2048, Student-t(4) bf16 activations",
                        [2048], [Layer("k2560_n6912", 6912, 2560, "normal", 0.02, 40, "student_t4", 42),
                                 Layer("k6912_n2560", 2560, 6912, "normal", 0.02, 41, "student_t4", 43)])
    if name == "ffn-2b-decode":
        return Workload(name, "2B-shaped feed-forward decode: silu(gate(h)) * up(h) from the fused gate+up matrix "
                              "[13824, 2560], then down [2560, 6912]; h bf16 N(0,1) with 0.1% x20 outliers",
                        [1], [Layer("gate_up", 13824, 2560, "normal", 0.02, 50, "normal", 51, outlier_p=0.001),
                              Layer("down", 2560, 6912, "normal", 0.02, 52, "normal", 53)])
    if name == "100b-stream":
        return Workload(name, "100B-class layer stream: 30 GEMVs N=28672, K=8192, Laplace(0,0.01) weights",
                        [1, 16], [Layer(f"layer{i}", 28672, 8192, "laplace", 0.01, 100 + i, "normal", 99)
                                  for i in range(30)])
    raise KeyError(name)


WORKLOADS = ["bitlinear-1024", "2b-decode", "gateup-sweep", "prefill-2048", "100b-stream", "ffn-2b-decode"]
