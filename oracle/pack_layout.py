"""The packed gate/up weight layout, stated plainly, on the CPU.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages fuse W1 and W2 into one K x 2N weight so that one GEMM produces
matching Gate and Up columns side by side ("Tile-Level Activation Overlap for
Efficient LLM Inference", gist.science technical summary, section
"Methodology / Kernel-2": W_fused with interleaved columns, even = Gate,
odd = Up). This library interleaves by blocks instead of single columns and
stores each (column block, 64-deep K slice) tile contiguously:

* NB = 128 columns per block; N is zero-padded to Np = ceil(N / 128) * 128.
* KB = 64 K-values per slice; K is zero-padded to Kp = ceil(K / 64) * 64.
* Packed array P has shape [Np / 128, Kp / 64, 256, 64] (bf16):
  P[j, b, i, t]       = W1[64 b + t, 128 j + i]   for i in [0, 128)   (gate)
  P[j, b, 128 + i, t] = W2[64 b + t, 128 j + i]   for i in [0, 128)   (up)
  and 0 where 128 j + i >= N or 64 b + t >= K.

The layout only moves bits; results do not depend on it. This module is the
byte-level specification the CUDA pack kernel is checked against.
"""
from __future__ import annotations

import numpy as np

PACK_BLOCK_N = 128
PACK_BLOCK_K = 64


def padded_n(n: int) -> int:
    """N rounded up to a whole number of 128-column blocks."""
    return -(-n // PACK_BLOCK_N) * PACK_BLOCK_N


def padded_k(k: int) -> int:
    """K rounded up to a whole number of 64-deep slices."""
    return -(-k // PACK_BLOCK_K) * PACK_BLOCK_K


def pack_reference(w1_bits: np.ndarray, w2_bits: np.ndarray, slice_k: int = PACK_BLOCK_K):
    """Packed array [Np/128, Kp/slice_k, 256, slice_k] from W1, W2 [K, N] (bit arrays).

    slice_k = 64 for bf16 (uint16 bits, 128-byte rows); the FP8 layout uses
    slice_k = 128 (uint8 bits, also 128-byte rows).
    """
    w1_bits = np.asarray(w1_bits)
    w2_bits = np.asarray(w2_bits)
    k_dim, n_dim = w1_bits.shape
    n_blocks = padded_n(n_dim) // PACK_BLOCK_N
    k_slices = -(-k_dim // slice_k)
    out = np.zeros((n_blocks, k_slices, 2 * PACK_BLOCK_N, slice_k), dtype=w1_bits.dtype)
    for j in range(n_blocks):
        n0 = j * PACK_BLOCK_N
        cols = min(PACK_BLOCK_N, n_dim - n0)          # real columns in this block
        for b in range(k_slices):
            k0 = b * slice_k
            depth = min(slice_k, k_dim - k0)          # real K values in this slice
            # row i of the tile is weight column n0 + i, over k0 .. k0 + depth
            out[j, b, :cols, :depth] = w1_bits[k0:k0 + depth, n0:n0 + cols].T
            out[j, b, PACK_BLOCK_N:PACK_BLOCK_N + cols, :depth] = \
                w2_bits[k0:k0 + depth, n0:n0 + cols].T
    return out


def unpack_reference(packed: np.ndarray, k_dim: int, n_dim: int, slice_k: int = PACK_BLOCK_K):
    """Inverse of ``pack_reference`` with the same ``slice_k``: (W1, W2) as [K, N] arrays.

    The element type is kept (uint16 bf16 bits for slice_k = 64, uint8 E4M3
    bits for slice_k = 128).
    """
    p = np.asarray(packed)
    n_blocks = padded_n(n_dim) // PACK_BLOCK_N
    k_slices = -(-k_dim // slice_k)
    p = p.reshape(n_blocks, k_slices, 2 * PACK_BLOCK_N, slice_k)
    # [j, b, i, t] -> column 128 j + i, row slice_k * b + t
    gate = p[:, :, :PACK_BLOCK_N, :].transpose(1, 3, 0, 2).reshape(k_slices * slice_k, -1)
    up = p[:, :, PACK_BLOCK_N:, :].transpose(1, 3, 0, 2).reshape(k_slices * slice_k, -1)
    return (np.ascontiguousarray(gate[:k_dim, :n_dim]), np.ascontiguousarray(up[:k_dim, :n_dim]))
