"""Helpers shared by the GPU tests: numpy <-> torch transfers and error norms."""
import numpy as np
import torch


def dev():
    return torch.device("cuda:0")


def bf16_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())


def f32_to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel(a, b) -> float:
    """Normwise relative error ||a - b||_F / ||b||_F."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


# Tolerance of the floating-point outputs against the fp64 oracle: bf16
# inputs, fp32 accumulation, normwise relative error (bf16 output rounding
# alone accounts for about 1.5e-3 of it).
TOL = 2e-3
