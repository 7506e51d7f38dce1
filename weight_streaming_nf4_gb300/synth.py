"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the method itself: it only draws random
tensors (numpy's PCG64 generator, one independent stream per named tensor)
and stores them in the dtypes the hot path consumes (bf16 bit patterns as
uint16, fp32).  Both the CUDA path and the CPU oracle receive the very same
arrays from here.

Distributions follow the workloads the method is measured on: activations
x ~ N(0, 1) in bf16, frozen base weights W ~ N(0, 0.02) in bf16 before NF4
quantisation, LoRA A ~ U(-1/sqrt(K), 1/sqrt(K)) (the Kaiming-uniform bound
PEFT uses for A), LoRA B ~ N(0, 0.01) (non-zero so the up projection and dB
are exercised), upstream gradient dY ~ N(0, 1) in bf16.
"""
from __future__ import annotations

import hashlib

import numpy as np


def _rng(seed: int, name: str) -> np.random.Generator:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return np.random.default_rng(int.from_bytes(h[:8], "little"))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Store float values as bf16 (round to nearest even), returned as uint16."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    return to_bf16_bits(_rng(seed, name).normal(0.0, std, size=shape))


def normal_f32(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    return _rng(seed, name).normal(0.0, std, size=shape).astype(np.float32)


def uniform_f32(seed: int, name: str, shape, bound: float) -> np.ndarray:
    return _rng(seed, name).uniform(-bound, bound, size=shape).astype(np.float32)


def linear_inputs(seed: int, M: int, N: int, K: int, r: int = 16, tag: str = "lin"):
    """One NF4-LoRA linear: x [M,K] bf16, W [N,K] bf16, A [r,K], B [N,r], dY [M,N] bf16."""
    return dict(
        x=normal_bf16(seed, f"{tag}.x", (M, K), 1.0),
        W=normal_bf16(seed, f"{tag}.W", (N, K), 0.02),
        A=uniform_f32(seed, f"{tag}.A", (r, K), 1.0 / np.sqrt(K)),
        B=normal_f32(seed, f"{tag}.B", (N, r), 0.01),
        dY=normal_bf16(seed, f"{tag}.dY", (M, N), 1.0),
    )


def stack_h0(seed: int, step: int, M: int, H: int) -> np.ndarray:
    """Residual-stream input of one step (fp32, N(0,1)); regenerated per step."""
    return normal_f32(seed, f"h0.step{step}", (M, H), 1.0)


def stack_weights(seed: int, layer: int, lin: str, N: int, K: int, r: int = 16):
    """Base weight (bf16 bits) and LoRA A, B of one linear of the stack."""
    t = f"L{layer}.{lin}"
    return (normal_bf16(seed, t + ".W", (N, K), 0.02),
            uniform_f32(seed, t + ".A", (r, K), 1.0 / np.sqrt(K)),
            normal_f32(seed, t + ".B", (N, r), 0.01))
