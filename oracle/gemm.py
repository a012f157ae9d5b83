"""Oracle: the GEMM producer's product and the error metric.  TEST INFRASTRUCTURE ONLY.

The Iris "Triggered Plans" page (section Model) names a GEMM as the typical tiled producer whose
tiles ``tile_chunks()`` groups.  Each virtual rank r computes C_r = A_r @ B from bf16 operands;
the reference result here is the exact-as-fp64 product of the same bf16 values (numpy matmul is
the library primitive), and the check is the relative Frobenius error
||C_gpu - C_ref||_F / ||C_ref||_F.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def product(A: np.ndarray, Bt: np.ndarray) -> np.ndarray:
    """C = A @ B with A [M, K] and Bt = B^T [N, K], both float64 values of bf16 numbers."""
    return np.asarray(A, dtype=np.float64) @ np.asarray(Bt, dtype=np.float64).T


def rel_frobenius(C: np.ndarray, C_ref: np.ndarray) -> float:
    C = np.asarray(C, dtype=np.float64)
    C_ref = np.asarray(C_ref, dtype=np.float64)
    den = np.linalg.norm(C_ref)
    return float(np.linalg.norm(C - C_ref) / den) if den else float(np.linalg.norm(C))
