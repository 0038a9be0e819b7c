"""float64 reference of Y = SiLU(A x W1) (.) (A x W2).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): never imported by the
product path.

Source: "Tile-Level Activation Overlap for Efficient LLM Inference" (gist.science
technical summary), section "Problem Statement": the gated MLP computes
Y = SiLU(A x W1) (.) (A x W2), two independent GEMMs followed by an elementwise
gated activation. Section "Methodology / Kernel-1" names the activation on the
Gate accumulator "Swish (SiLU(Gate))"; it is read here as SiLU(x) = x * sigmoid(x)
(Swish with beta = 1). Shapes: A [M, K], W1 and W2 [K, N], Y [M, N].

Precision: inputs are bf16 and are converted exactly to float64. Gate and Up are
never rounded (the fused method keeps them in the accumulator, section "Key
Contributions", tile-level fusion). The float64 result may then be rounded once,
to nearest-even, to bf16.

The contraction uses numpy's float64 matmul as a library step; the sum over k
is the definition's sum, in whatever order the BLAS takes, which is exact up to
float64 rounding (about K * 2**-53 relative, far below bf16 resolution).
"""
from __future__ import annotations

import numpy as np

BF16_MAX = float.fromhex("0x1.fep127")  # largest finite bf16: (2 - 2**-7) * 2**127


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact float64 values of bf16 bit patterns (uint16 array)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 values to bf16 (round to nearest, ties to even), once.

    bf16 keeps 8 significant bits and float32's exponent range: normal numbers
    down to 2**-126, then subnormals with a fixed spacing of 2**-133. A value
    a = m * 2**e (m in [0.5, 1)) has spacing 2**(max(e, -125) - 8) on the bf16
    grid; it is scaled to that grid, rounded half-to-even to an integer and
    scaled back (all exact in float64). Magnitudes that round above the largest
    finite bf16 become infinity; NaN becomes the canonical quiet NaN 0x7FC0.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(invalid="ignore", over="ignore"):
        _, e = np.frexp(a)
        e_eff = np.maximum(e, -125).astype(np.int64)
        q = np.rint(np.ldexp(a, -(e_eff - 8)))
        r = np.ldexp(q, e_eff - 8)
    over = ~(r <= BF16_MAX)  # also true for inf and nan
    r_safe = np.where(over, 0.0, r)
    bits = (r_safe.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(over, np.uint16(0x7F80), bits)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    bits = np.where(np.signbit(x) & ~np.isnan(x), bits | np.uint16(0x8000), bits)
    return bits.astype(np.uint16)


def silu(x) -> np.ndarray:
    """SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x)), in float64.

    For very negative x, exp(-x) overflows to +inf and the quotient is -0.0,
    which is the correctly signed limit; no NaN arises for finite x.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def gate_up_f64(a: np.ndarray, w1: np.ndarray, w2: np.ndarray):
    """Gate = A x W1 and Up = A x W2 in float64 (no rounding to bf16)."""
    a = np.asarray(a, dtype=np.float64)
    gate = a @ np.asarray(w1, dtype=np.float64)
    up = a @ np.asarray(w2, dtype=np.float64)
    return gate, up


def swiglu_f64_values(a: np.ndarray, w1: np.ndarray, w2: np.ndarray) -> np.ndarray:
    """Y = SiLU(A x W1) (.) (A x W2) on float64 value arrays."""
    gate, up = gate_up_f64(a, w1, w2)
    return silu(gate) * up


def swiglu_f64(a_bits, w1_bits, w2_bits, rows=None) -> np.ndarray:
    """Reference Y (float64) for bf16 inputs given as uint16 bit arrays.

    a_bits [M, K], w1_bits / w2_bits [K, N]. ``rows`` (optional integer array)
    selects which rows of A, hence of Y, are computed; the result then has
    len(rows) rows in that order. Rows are independent in the definition, so a
    row subset is the same computation restricted, not an approximation.
    """
    a_bits = np.asarray(a_bits, dtype=np.uint16)
    if rows is not None:
        a_bits = a_bits[np.asarray(rows, dtype=np.int64)]
    a = bf16_bits_to_f64(a_bits)
    w1 = bf16_bits_to_f64(w1_bits)
    w2 = bf16_bits_to_f64(w2_bits)
    return swiglu_f64_values(a, w1, w2)
