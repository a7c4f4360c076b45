"""fp64 oracle of the strict RMSNorm that produces the head's hidden states.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"vLLM RL-Kernel v0.1.0: ROCm 上でのビット単位のトレーニング-ロールアウト一貫性",
strict-path boundary table, row "RMSNorm": its reduction domain, epsilon,
residual add and output boundary are fixed.  The definition, per row t:

    x'[t]   = x[t] + residual[t]                (if a residual is given)
    y[t, i] = x'[t, i] / sqrt(mean_i(x'[t, i]^2) + eps) * gamma[i]

The residual sum is an output boundary of its own (the next layer's
residual stream, bf16): it is the fp32 sum of the two bf16 inputs rounded
to bf16, which this oracle forms exactly that way so the boundary can be
compared bit for bit.  Everything after it is fp64.
"""
from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def encode_bf16(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bits, round to nearest even (finite values)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def residual_add(x_bits: np.ndarray, r_bits: np.ndarray) -> np.ndarray:
    """bf16 bits of bf16_RN(fp32_RN(x + r))."""
    xs = (np.ascontiguousarray(x_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
    rs = (np.ascontiguousarray(r_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
    return encode_bf16((xs + rs).astype(np.float32))


def rmsnorm(x_bits: np.ndarray, gamma_bits: np.ndarray, eps: float,
            residual_bits: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """(y fp64 [T, H], x' bf16 bits [T, H])."""
    xr = x_bits if residual_bits is None else residual_add(x_bits, residual_bits)
    x = decode_bf16(xr)
    g = decode_bf16(gamma_bits)
    ms = (x * x).mean(axis=1)
    y = x / np.sqrt(ms + eps)[:, None] * g[None, :]
    return y, np.ascontiguousarray(xr, dtype=np.uint16)
