"""Normalised Sylvester-Hadamard rotation — oracle (test infrastructure).

Restates [vLLM-TQ] section "为什么先旋转" / subsection "为什么 vLLM 选了 Hadamard
而不是随机正交矩阵": H_1 = [1], H_{2n} = [[H_n, H_n], [H_n, -H_n]]; the rotation
is H / sqrt(d), which is orthonormal and symmetric, so it is its own inverse;
no random sign flips are applied. [TQ-intro] section "1. Walsh-Hadamard 旋转"
states H H^T = d I for the unnormalised matrix.

The oracle applies the rotation as the plain dense product (the definition),
not as a butterfly.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = ["sylvester_hadamard", "rotate"]


def sylvester_hadamard(d: int) -> np.ndarray:
    """Unnormalised d x d Sylvester-Hadamard matrix (entries +-1), float64."""
    if d < 1 or (d & (d - 1)) != 0:
        raise ValueError("d must be a power of two")
    h = np.array([[1.0]])
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(x: np.ndarray) -> np.ndarray:
    """y = (H / sqrt(d)) x along the last axis, float64."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = sylvester_hadamard(d) / math.sqrt(d)
    return x @ h.T
