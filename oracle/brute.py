"""Pure-Python brute force of Y = SiLU(A x W1) (.) (A x W2), for tiny shapes.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

A second implementation, independent of numpy and BLAS, used to pin
``oracle.swiglu_ref``. Source: "Tile-Level Activation Overlap for Efficient LLM
Inference" (gist.science technical summary), section "Problem Statement".

Each Gate / Up entry is the exactly rounded float64 value of the exact sum: the
products of two bf16 values are exact in float64 (8 + 8 significant bits) and
``math.fsum`` rounds their exact sum once. SiLU uses ``math.exp``.
"""
from __future__ import annotations

import math


def _sigmoid(x: float) -> float:
    # exp(-x) overflows a float for x < about -709.78; sigmoid is then 0.
    if -x > 709.0:
        return 0.0
    return 1.0 / (1.0 + math.exp(-x))


def silu_scalar(x: float) -> float:
    """SiLU(x) = x * sigmoid(x) for one float."""
    return x * _sigmoid(x)


def gate_up_brute(a, w1, w2):
    """Gate[m][n] = sum_k a[m][k] * w1[k][n], Up likewise with w2 (lists)."""
    m_rows, k_dim = len(a), len(a[0])
    n_cols = len(w1[0])
    gate = [[math.fsum(a[m][k] * w1[k][n] for k in range(k_dim)) for n in range(n_cols)]
            for m in range(m_rows)]
    up = [[math.fsum(a[m][k] * w2[k][n] for k in range(k_dim)) for n in range(n_cols)]
          for m in range(m_rows)]
    return gate, up


def swiglu_brute(a, w1, w2):
    """Y[m][n] = SiLU(Gate[m][n]) * Up[m][n] as nested lists of floats."""
    gate, up = gate_up_brute(a, w1, w2)
    return [[silu_scalar(g) * u for g, u in zip(grow, urow)] for grow, urow in zip(gate, up)]
