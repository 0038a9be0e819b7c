"""Block-scaled FP8 (MX) variant of the reference, and its scale-factor layouts.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The pages name FP8 quantisation only as the reason the SwiGLU steps weigh more
once the GEMMs run faster ("Tile-Level Activation Overlap for Efficient LLM
Inference", gist.science, section "Problem Statement"); they give no scaling
convention. This module takes the block-scaled reading: every input is stored
as E4M3 values, and each run of 32 consecutive values along the contraction
dimension K shares one power-of-two scale, stored as an 8-bit exponent
(UE8M0):

  A[m, k]  = e4m3(A8[m, k])  * 2**(SA[m, k // 32] - 127)
  W1[k, n] = e4m3(W1_8[k, n]) * 2**(S1[k // 32, n] - 127)     (W2 likewise)

so A's scales run along its rows and W's along its columns, and one scale
group never straddles two K values of different groups. Y = SiLU(A x W1) (.)
(A x W2) in float64 on these exact values, rounded once to bf16, as in
``swiglu_ref``. UE8M0: value 2**(e - 127) for e in 0..254; e = 255 is NaN.

Layouts (byte specifications the CUDA pack kernels are checked against):

* ``scale_tile_offset``: a block of 128 rows x 4 scale groups occupies 512
  bytes; row r, group g sits at byte (r % 32) * 16 + (r // 32) * 4 + g.
* ``tile_act_scales``: A's scales [M, K/32] as such blocks, ordered
  [ceil(M/128)][ceil(K/128)]; positions past M or past K hold 127 (2**0).
* ``pack_weight_scales``: for each packed weight tile (128-column block j,
  128-deep K slice b, in the packed weight's tile order) 1024 bytes: the block
  of W1's scales for columns 128 j .. 128 j + 127 and groups 4 b .. 4 b + 3,
  then the same block of W2's scales; padding holds 127.
"""
from __future__ import annotations

import numpy as np

from .fp8 import e4m3_bits_to_f64
from .swiglu_ref import swiglu_f64_values

GROUP = 32          # K values per scale
PAD_SCALE = 127     # 2**0: the scale written where no value exists


def ue8m0_to_f64(bits) -> np.ndarray:
    """Exact float64 values 2**(e - 127) of UE8M0 scale bytes; 255 is NaN."""
    e = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    v = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, v)


def mx_values_rows(q_bits, s_bits) -> np.ndarray:
    """Values of a [R, K] E4M3 array whose scales [R, K/32] run along each row."""
    q = e4m3_bits_to_f64(q_bits)
    s = ue8m0_to_f64(s_bits)
    k = q.shape[1]
    return q * np.repeat(s, GROUP, axis=1)[:, :k]


def mx_values_cols(q_bits, s_bits) -> np.ndarray:
    """Values of a [K, N] E4M3 array whose scales [K/32, N] run down each column."""
    q = e4m3_bits_to_f64(q_bits)
    s = ue8m0_to_f64(s_bits)
    k = q.shape[0]
    return q * np.repeat(s, GROUP, axis=0)[:k, :]


def swiglu_f64_mxfp8(a_bits, sa_bits, w1_bits, s1_bits, w2_bits, s2_bits,
                     rows=None) -> np.ndarray:
    """Reference Y (float64) for block-scaled E4M3 inputs.

    a_bits [M, K] and sa_bits [M, K/32] (uint8); w1_bits / w2_bits [K, N] and
    s1_bits / s2_bits [K/32, N]. ``rows`` selects rows of A, hence of Y.
    """
    a_bits = np.asarray(a_bits, dtype=np.uint8)
    sa_bits = np.asarray(sa_bits, dtype=np.uint8)
    if rows is not None:
        idx = np.asarray(rows, dtype=np.int64)
        a_bits, sa_bits = a_bits[idx], sa_bits[idx]
    a = mx_values_rows(a_bits, sa_bits)
    w1 = mx_values_cols(w1_bits, s1_bits)
    w2 = mx_values_cols(w2_bits, s2_bits)
    return swiglu_f64_values(a, w1, w2)


def scale_tile_offset(r, g):
    """Byte offset of (row r in 0..127, group g in 0..3) inside a 512-byte block."""
    r = np.asarray(r)
    g = np.asarray(g)
    return (r % 32) * 16 + (r // 32) * 4 + g


def _block(src, r0: int, g0: int) -> np.ndarray:
    """One 512-byte block from src[rows r0.., groups g0..] (rows x groups array)."""
    out = np.full(512, PAD_SCALE, dtype=np.uint8)
    rows, groups = src.shape
    for r in range(128):
        for g in range(4):
            if r0 + r < rows and g0 + g < groups:
                out[scale_tile_offset(r, g)] = src[r0 + r, g0 + g]
    return out


def tile_act_scales(sa_bits, m_dim: int, k_dim: int) -> np.ndarray:
    """A's scales [M, K/32] in the tiled layout (flat uint8 array)."""
    sa = np.asarray(sa_bits, dtype=np.uint8).reshape(m_dim, -(-k_dim // GROUP))
    m_blocks = -(-m_dim // 128)
    k_slices = -(-k_dim // 128)
    blocks = [_block(sa, 128 * i, 4 * b) for i in range(m_blocks) for b in range(k_slices)]
    return np.concatenate(blocks) if blocks else np.zeros(0, dtype=np.uint8)


def pack_weight_scales(s1_bits, s2_bits, k_dim: int, n_dim: int) -> np.ndarray:
    """W1's and W2's scales [K/32, N] in the packed tile order (flat uint8 array)."""
    groups = -(-k_dim // GROUP)
    s1 = np.asarray(s1_bits, dtype=np.uint8).reshape(groups, n_dim).T   # [N, groups]
    s2 = np.asarray(s2_bits, dtype=np.uint8).reshape(groups, n_dim).T
    n_blocks = -(-n_dim // 128)
    k_slices = -(-k_dim // 128)
    out = []
    for j in range(n_blocks):
        for b in range(k_slices):
            out.append(_block(s1, 128 * j, 4 * b))
            out.append(_block(s2, 128 * j, 4 * b))
    return np.concatenate(out)
