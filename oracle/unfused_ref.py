"""Rounding model of the unfused gated MLP: Gate and Up stored as bf16.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): never imported by the
product path.

Source: "Tile-Level Activation Overlap for Efficient LLM Inference" (gist.science
technical summary), section "Key Contributions", item "Numerical Superiority":
the fused kernels have no outputs more than 1% away from an FP32 reference,
while the cuBLAS baseline has a few percent, which the pages put down to bf16
partial accumulation across tiles. cuBLAS accumulates bf16 GEMMs in fp32, so
the reading taken here is another one: the unfused path rounds to bf16 three
times before the output's own rounding, once per tensor it writes to memory.

    g16 = bf16(A x W1)            first GEMM's output
    u16 = bf16(A x W2)            second GEMM's output
    s16 = bf16(SiLU(g16))         the activation kernel's output
    y16 = bf16(s16 * u16)         the multiply kernel's output

Each rounding is to nearest, ties to even. Gate and Up are taken as the exact
sums (float64, as in ``swiglu_ref``); the fp32 accumulation of a real GEMM
changes a bf16 rounding only where the exact sum lies within a few fp32 ulps of
a bf16 rounding boundary. The product of two bf16 values is exact in float64,
so ``y16`` is that product rounded once.
"""
from __future__ import annotations

import numpy as np

from oracle.swiglu_ref import bf16_bits_to_f64, f64_to_bf16_bits, gate_up_f64, silu


def unfused_bf16_stages(a_bits, w1_bits, w2_bits, rows=None):
    """(g16, u16, s16, y16) bf16 bit arrays of the unfused path (see the module text).

    a_bits [M, K], w1_bits / w2_bits [K, N] as uint16 bf16 bit patterns; ``rows``
    optionally selects rows of A (and of every result), as in ``swiglu_f64``.
    """
    a_bits = np.asarray(a_bits, dtype=np.uint16)
    if rows is not None:
        a_bits = a_bits[np.asarray(rows, dtype=np.int64)]
    gate, up = gate_up_f64(bf16_bits_to_f64(a_bits), bf16_bits_to_f64(w1_bits),
                           bf16_bits_to_f64(w2_bits))
    g16 = f64_to_bf16_bits(gate)
    u16 = f64_to_bf16_bits(up)
    s16 = f64_to_bf16_bits(silu(bf16_bits_to_f64(g16)))
    y16 = f64_to_bf16_bits(bf16_bits_to_f64(s16) * bf16_bits_to_f64(u16))
    return g16, u16, s16, y16


def unfused_bf16(a_bits, w1_bits, w2_bits, rows=None) -> np.ndarray:
    """Y of the unfused path as bf16 bits (the last element of ``unfused_bf16_stages``)."""
    return unfused_bf16_stages(a_bits, w1_bits, w2_bits, rows=rows)[3]
