"""FP8 (E4M3) variant of the reference: decoding and Y from scaled FP8 inputs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages note that quantisation to FP8 raises tensor-core density and so
makes the memory-bound SwiGLU steps relatively costlier ("Tile-Level
Activation Overlap for Efficient LLM Inference", gist.science, section
"Problem Statement"); they give no scaling convention. The reading taken here
is the plainest one: each input tensor is E4M3 values times one fp32 scale,
  A = s_a * A8,   W1 = s_1 * W1_8,   W2 = s_2 * W2_8,
and Y = SiLU(A x W1) (.) (A x W2) as in ``swiglu_ref``, in float64 on the exact
decoded values, rounded once to bf16.

E4M3 (OCP FP8, "fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
bits; exponent 0 encodes subnormals m/8 * 2^-6; S.1111.111 is NaN; there are
no infinities; the largest finite magnitude is 448.
"""
from __future__ import annotations

import numpy as np

from .swiglu_ref import swiglu_f64_values


def e4m3_bits_to_f64(bits) -> np.ndarray:
    """Exact float64 values of E4M3 bit patterns (uint8 array)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    subnormal = np.ldexp(m / 8.0, -6)
    v = sign * np.where(e == 0, subnormal, normal)
    return np.where((e == 15) & ((b & 0x7) == 7), np.nan, v)


def swiglu_f64_fp8(a_bits, w1_bits, w2_bits, scale_a: float, scale_w1: float, scale_w2: float,
                   rows=None) -> np.ndarray:
    """Reference Y (float64) for E4M3 inputs (uint8 bit arrays) and per-tensor scales.

    a_bits [M, K], w1_bits / w2_bits [K, N]; ``rows`` selects rows of A and Y.
    """
    a_bits = np.asarray(a_bits, dtype=np.uint8)
    if rows is not None:
        a_bits = a_bits[np.asarray(rows, dtype=np.int64)]
    a = np.float64(np.float32(scale_a)) * e4m3_bits_to_f64(a_bits)
    w1 = np.float64(np.float32(scale_w1)) * e4m3_bits_to_f64(w1_bits)
    w2 = np.float64(np.float32(scale_w2)) * e4m3_bits_to_f64(w2_bits)
    return swiglu_f64_values(a, w1, w2)
