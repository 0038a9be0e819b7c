"""float64 reference of the gated MLP's down-projection: Out = Y x W3 + R.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages' gated MLP ("Tile-Level Activation Overlap for Efficient LLM
Inference", gist.science, section "Problem Statement") produces
Y = SiLU(A x W1) (.) (A x W2); in the models it names (Qwen-2.5 and others)
the MLP's next step projects Y back to the hidden size with a third weight
and adds the block's residual input. The pages say nothing more about it; the
reading taken is the plain one: Out [M, H] = Y [M, N] x W3 [N, H] + R [M, H],
all bf16 in and out, computed here in float64 on the exact inputs (R may be
absent: zero).
"""
from __future__ import annotations

import numpy as np

from .swiglu_ref import bf16_bits_to_f64


def down_f64_values(y: np.ndarray, w3: np.ndarray, r: np.ndarray | None) -> np.ndarray:
    out = np.asarray(y, dtype=np.float64) @ np.asarray(w3, dtype=np.float64)
    if r is not None:
        out = out + np.asarray(r, dtype=np.float64)
    return out


def down_f64(y_bits, w3_bits, r_bits=None, rows=None) -> np.ndarray:
    """Out (float64) for bf16 bit arrays Y [M, N], W3 [N, H], R [M, H] (or None)."""
    y_bits = np.asarray(y_bits, dtype=np.uint16)
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        y_bits = y_bits[rows]
        if r_bits is not None:
            r_bits = np.asarray(r_bits, dtype=np.uint16)[rows]
    r = bf16_bits_to_f64(r_bits) if r_bits is not None else None
    return down_f64_values(bf16_bits_to_f64(y_bits), bf16_bits_to_f64(w3_bits), r)


def pack_down_reference(w3_bits: np.ndarray) -> np.ndarray:
    """Packed W3 [Hp/256, Np/64, 256, 64] from W3 [N, H] (bf16 bits).

    Tile (j, b) row i is output column 256 j + i over the 64 K values
    (rows of W3) 64 b .. 64 b + 63; zero past H and past N.
    """
    w3_bits = np.asarray(w3_bits, dtype=np.uint16)
    n_dim, h_dim = w3_bits.shape
    blocks = -(-h_dim // 256)
    slices = -(-n_dim // 64)
    out = np.zeros((blocks, slices, 256, 64), dtype=np.uint16)
    for j in range(blocks):
        h0 = j * 256
        cols = min(256, h_dim - h0)
        for b in range(slices):
            k0 = b * 64
            depth = min(64, n_dim - k0)
            out[j, b, :cols, :depth] = w3_bits[k0:k0 + depth, h0:h0 + cols].T
    return out
