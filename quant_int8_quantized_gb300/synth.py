"""Seeded synthetic inputs for the block-quantized matmul path.

This module is shared by the CUDA-path tests, the bench and the CPU oracle's
callers. It holds none of the method's arithmetic: it only draws seeded random
numbers and places them into the input layouts (f32 activations, raw q4_K /
q6_K / q5_K super-block bytes, raw q4_0 / q4_1 block bytes).

Every tensor is drawn from its own stream, seeded by (seed, name), so a tensor
does not depend on which other tensors were drawn before it.

Workload recipe (the pages measure real 7B/14B GGUF models; these synthetic
tensors of the same shapes stand in for them):
  * activations: f32 N(0, 1);
  * RMSNorm weight: f32 N(1, 0.1);
  * q4_K super-block (144 B): every byte uniform, so the 4-bit quants are
    uniform in 0..15 and each packed 6-bit scale and min is uniform in 0..63;
    then bytes 0..1 (d) and 2..3 (dmin) are overwritten with f16 |N(0, 0.01)|;
  * q6_K super-block (210 B): every byte uniform, so the 6-bit quants are
    uniform in 0..63 and the int8 sub-block scales uniform in -128..127; then
    bytes 208..209 (d) are overwritten with f16 |N(0, 0.01)|;
  * q5_K super-block (176 B): every byte uniform (nibbles and fifth bits, so q
    is uniform in 0..31; scales and mins as in q4_K); bytes 0..1 (d) and 2..3
    (dmin) overwritten with f16 |N(0, 0.01)|;
  * q4_0 block (18 B per 32): nibbles uniform; d (bytes 0..1) f16 N(0, 0.01)
    (signed, as a q4_0 quantizer emits);
  * q4_1 block (20 B per 32): nibbles uniform; d f16 |N(0, 0.01)|, m f16
    N(0, 0.08);
  * "outlier" activations: each entry independently multiplied by 50 with
    probability 0.01.
"""
from __future__ import annotations

import zlib

import torch

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
Q5K_BLOCK_BYTES = 176
Q4_0_BLOCK_BYTES = 18
Q4_1_BLOCK_BYTES = 20
QK_K = 256


def _generator(seed: int, name: str, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed((int(seed) * 1_000_003 + zlib.crc32(name.encode())) & 0x7FFF_FFFF_FFFF)
    return g


def normal(shape, seed: int, name: str, mean: float = 0.0, std: float = 1.0,
           device="cpu") -> torch.Tensor:
    """f32 tensor of N(mean, std) draws."""
    g = _generator(seed, name, device)
    x = torch.randn(tuple(shape), generator=g, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def with_outliers(x: torch.Tensor, seed: int, name: str, p: float = 0.01,
                  factor: float = 50.0) -> torch.Tensor:
    """Return x with each entry independently scaled by `factor` with probability p."""
    g = _generator(seed, name + "#outliers", x.device)
    u = torch.rand(x.shape, generator=g, dtype=torch.float32, device=x.device)
    return torch.where(u < p, x * factor, x)


def _f16_abs_normal(n: int, std: float, g: torch.Generator, device) -> torch.Tensor:
    v = torch.randn((n,), generator=g, dtype=torch.float32, device=device).abs_().mul_(std)
    return v.to(torch.float16).view(torch.uint8).view(n, 2)


def _f16_normal(n: int, std: float, g: torch.Generator, device) -> torch.Tensor:
    v = torch.randn((n,), generator=g, dtype=torch.float32, device=device).mul_(std)
    return v.to(torch.float16).view(torch.uint8).view(n, 2)


def _random_bytes(n: int, g: torch.Generator, device) -> torch.Tensor:
    return torch.randint(0, 256, (n,), generator=g, dtype=torch.uint8, device=device)


def q4k_weights(N: int, K: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    """Raw q4_K bytes for an N x K weight, shape [N, K/256*144], uint8."""
    assert K % QK_K == 0
    S = K // QK_K
    g = _generator(seed, name, device)
    w = _random_bytes(N * S * Q4K_BLOCK_BYTES, g, device).view(N * S, Q4K_BLOCK_BYTES)
    w[:, 0:2] = _f16_abs_normal(N * S, 0.01, g, device)
    w[:, 2:4] = _f16_abs_normal(N * S, 0.01, g, device)
    return w.view(N, S * Q4K_BLOCK_BYTES)


def q6k_weights(N: int, K: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    """Raw q6_K bytes for an N x K weight, shape [N, K/256*210], uint8."""
    assert K % QK_K == 0
    S = K // QK_K
    g = _generator(seed, name, device)
    w = _random_bytes(N * S * Q6K_BLOCK_BYTES, g, device).view(N * S, Q6K_BLOCK_BYTES)
    w[:, 208:210] = _f16_abs_normal(N * S, 0.01, g, device)
    return w.view(N, S * Q6K_BLOCK_BYTES)


def q5k_weights(N: int, K: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    """Raw q5_K bytes for an N x K weight, shape [N, K/256*176], uint8."""
    assert K % QK_K == 0
    S = K // QK_K
    g = _generator(seed, name, device)
    w = _random_bytes(N * S * Q5K_BLOCK_BYTES, g, device).view(N * S, Q5K_BLOCK_BYTES)
    w[:, 0:2] = _f16_abs_normal(N * S, 0.01, g, device)
    w[:, 2:4] = _f16_abs_normal(N * S, 0.01, g, device)
    return w.view(N, S * Q5K_BLOCK_BYTES)


def q4_0_weights(N: int, K: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    """Raw q4_0 bytes for an N x K weight, shape [N, K/32*18], uint8."""
    assert K % 32 == 0
    B = K // 32
    g = _generator(seed, name, device)
    w = _random_bytes(N * B * Q4_0_BLOCK_BYTES, g, device).view(N * B, Q4_0_BLOCK_BYTES)
    w[:, 0:2] = _f16_normal(N * B, 0.01, g, device)
    return w.view(N, B * Q4_0_BLOCK_BYTES)


def q4_1_weights(N: int, K: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    """Raw q4_1 bytes for an N x K weight, shape [N, K/32*20], uint8."""
    assert K % 32 == 0
    B = K // 32
    g = _generator(seed, name, device)
    w = _random_bytes(N * B * Q4_1_BLOCK_BYTES, g, device).view(N * B, Q4_1_BLOCK_BYTES)
    w[:, 0:2] = _f16_abs_normal(N * B, 0.01, g, device)
    w[:, 2:4] = _f16_normal(N * B, 0.08, g, device)
    return w.view(N, B * Q4_1_BLOCK_BYTES)


def weights(kind: str, N: int, K: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    gen = {"q4k": q4k_weights, "q6k": q6k_weights, "q5k": q5k_weights, "q4_0": q4_0_weights,
           "q4_1": q4_1_weights}
    if kind not in gen:
        raise ValueError(kind)
    return gen[kind](N, K, seed, name, device)
