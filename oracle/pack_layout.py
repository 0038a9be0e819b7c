"""The packed gate/up weight layout, stated plainly, on the CPU.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages fuse W1 and W2 into one K x 2N weight so that one GEMM produces
matching Gate and Up columns side by side ("Tile-Level Activation Overlap for
Efficient LLM Inference", gist.science technical summary, section
"Methodology / Kernel-2": W_fused with interleaved columns, even = Gate,
odd = Up). This library interleaves by blocks instead of single columns, and
stores the result K-contiguous (each packed row is one weight column):

* NB = 128 columns per block; N is zero-padded to Np = ceil(N / 128) * 128.
* Packed array P has shape [Np / 128, 256, K] (bf16), i.e. [2 * Np, K]:
  P[j, i, k]       = W1[k, j * 128 + i]   for i in [0, 128)   (gate rows)
  P[j, 128 + i, k] = W2[k, j * 128 + i]   for i in [0, 128)   (up rows)
  and 0 where j * 128 + i >= N.

The layout only moves bits; results do not depend on it. This module is the
byte-level specification the CUDA pack kernel is checked against.
"""
from __future__ import annotations

import numpy as np

PACK_BLOCK_N = 128


def padded_n(n: int) -> int:
    """N rounded up to a whole number of 128-column blocks."""
    return -(-n // PACK_BLOCK_N) * PACK_BLOCK_N


def pack_reference(w1_bits: np.ndarray, w2_bits: np.ndarray) -> np.ndarray:
    """Packed array [2 * Np, K] (uint16 bf16 bits) from W1, W2 [K, N] (uint16)."""
    w1_bits = np.asarray(w1_bits, dtype=np.uint16)
    w2_bits = np.asarray(w2_bits, dtype=np.uint16)
    k_dim, n_dim = w1_bits.shape
    n_pad = padded_n(n_dim)
    out = np.zeros((n_pad // PACK_BLOCK_N, 2 * PACK_BLOCK_N, k_dim), dtype=np.uint16)
    for j in range(n_pad // PACK_BLOCK_N):
        for i in range(PACK_BLOCK_N):
            n = j * PACK_BLOCK_N + i
            if n < n_dim:
                out[j, i, :] = w1_bits[:, n]
                out[j, PACK_BLOCK_N + i, :] = w2_bits[:, n]
    return out.reshape(2 * n_pad, k_dim)


def unpack_reference(packed: np.ndarray, n_dim: int):
    """Inverse of ``pack_reference``: (W1, W2) as [K, N] uint16 arrays."""
    packed = np.asarray(packed, dtype=np.uint16)
    two_np, k_dim = packed.shape
    blocks = packed.reshape(two_np // (2 * PACK_BLOCK_N), 2 * PACK_BLOCK_N, k_dim)
    gate = blocks[:, :PACK_BLOCK_N, :].reshape(-1, k_dim)[:n_dim]  # [N, K]
    up = blocks[:, PACK_BLOCK_N:, :].reshape(-1, k_dim)[:n_dim]
    return np.ascontiguousarray(gate.T), np.ascontiguousarray(up.T)
