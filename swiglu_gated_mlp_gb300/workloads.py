"""Seeded synthetic inputs for the fused SwiGLU projection, and the named workloads.

This module draws random numbers and rounds them to bf16; it holds none of the
method's arithmetic. Both the CUDA path's tests / benchmark and the CPU oracle
receive the arrays it returns.

Workloads are the gate/up projection shapes of the Qwen-2.5 MLPs the pages
evaluate on ("Tile-Level Activation Overlap for Efficient LLM Inference",
gist.science, section "Results": Qwen-2.5 0.5B to 72B on H100): M tokens,
K = hidden size, N = intermediate size. The pages do not print the shapes or
batch sizes; the ones below are the models' published MLP dimensions.

Recipe (one ``torch.Generator`` seeded with the workload's seed, CPU float32,
then rounded to bf16 with round-to-nearest-even):
  A  = randn(M, K)                 -> A  ~ N(0, 1)
  W1 = randn(K, N) * K**-0.5       -> W1 ~ N(0, 1/K)   (gate)
  W2 = randn(K, N) * K**-0.5       -> W2 ~ N(0, 1/K)   (up)
drawn in that order. Gate and Up entries are then roughly N(0, 1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    K: int
    N: int
    seed: int
    note: str

    @property
    def flops(self) -> int:
        """Contraction FLOPs counted as 4*M*K*N (two GEMMs, multiply + add)."""
        return 4 * self.M * self.K * self.N

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes the fused op must move: A once, W1 and W2 once, Y once (bf16)."""
        return 2 * self.M * self.K + 4 * self.K * self.N + 2 * self.M * self.N


WORKLOADS = {
    w.name: w
    for w in [
        Workload("qwen2.5-0.5b-mlp-m128", 128, 896, 4864, 0,
                 "Qwen-2.5-0.5B MLP gate/up, 128 tokens"),
        Workload("qwen2.5-7b-decode-m16", 16, 3584, 18944, 1,
                 "Qwen-2.5-7B MLP gate/up, decode batch of 16 tokens (weight-bandwidth bound)"),
        Workload("qwen2.5-7b-prefill-m4096", 4096, 3584, 18944, 2,
                 "Qwen-2.5-7B MLP gate/up, prefill of 4096 tokens"),
        Workload("qwen2.5-32b-prefill-m4096", 4096, 5120, 27648, 3,
                 "Qwen-2.5-32B MLP gate/up, prefill of 4096 tokens"),
        Workload("qwen2.5-72b-prefill-m8192", 8192, 8192, 29568, 4,
                 "Qwen-2.5-72B MLP gate/up, prefill of 8192 tokens"),
    ]
}

# Token-count sweep at the Qwen-2.5-32B shape (K=5120, N=27648), seed 3.
SWEEP_32B_M = (1, 64, 512, 2048)


def sweep_32b(m: int) -> Workload:
    return Workload(f"qwen2.5-32b-m{m}", m, 5120, 27648, 3,
                    f"Qwen-2.5-32B MLP gate/up, {m} tokens")


def make_inputs(M: int, K: int, N: int, seed: int):
    """(A [M,K], W1 [K,N], W2 [K,N]) as contiguous CPU bf16 tensors."""
    g = torch.Generator().manual_seed(int(seed))
    a = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(K)
    w1 = (torch.randn(K, N, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)
    w2 = (torch.randn(K, N, generator=g, dtype=torch.float32) * scale).to(torch.bfloat16)
    return a.contiguous(), w1.contiguous(), w2.contiguous()


def make_workload_inputs(w: Workload):
    return make_inputs(w.M, w.K, w.N, w.seed)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw bf16 bit patterns of a CPU tensor as a numpy uint16 array (a view)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(M: int, count: int, seed: int) -> np.ndarray:
    """Sorted seeded subset of row indices of size min(count, M), always with 0 and M-1."""
    if count >= M:
        return np.arange(M, dtype=np.int64)
    rng = np.random.default_rng(seed + 7919)
    inner = rng.choice(np.arange(1, M - 1), size=max(count - 2, 0), replace=False)
    return np.unique(np.concatenate([[0, M - 1], inner]).astype(np.int64))


def make_inputs_fp8(M: int, K: int, N: int, seed: int):
    """FP8 (E4M3) inputs with one fp32 scale per tensor, for the FP8 path.

    The same seeded draws as ``make_inputs`` (float32, before any rounding),
    each quantised as x ~= s * q with s = max|x| / 448 and q = RNE_E4M3(x / s).
    Returns (A8 [M,K], W1_8 [K,N], W2_8 [K,N]) as CPU float8_e4m3fn tensors and
    the scales (s_a, s_1, s_2) as Python floats (exact fp32 values).
    """
    g = torch.Generator().manual_seed(int(seed))
    a = torch.randn(M, K, generator=g, dtype=torch.float32)
    scale = 1.0 / math.sqrt(K)
    w1 = torch.randn(K, N, generator=g, dtype=torch.float32) * scale
    w2 = torch.randn(K, N, generator=g, dtype=torch.float32) * scale
    out, scales = [], []
    for x in (a, w1, w2):
        s = torch.clamp(x.abs().max() / 448.0, min=1e-30).to(torch.float32)
        out.append((x / s).to(torch.float8_e4m3fn).contiguous())
        scales.append(float(s))
    return out[0], out[1], out[2], tuple(scales)


def fp8_bits(t: torch.Tensor) -> np.ndarray:
    """The raw E4M3 bit patterns of a CPU float8 tensor as a numpy uint8 array."""
    assert t.dtype == torch.float8_e4m3fn
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


MX_GROUP = 32  # K values that share one scale in the block-scaled FP8 inputs


def _mx_quantise(x: torch.Tensor, dim: int):
    """E4M3 values and UE8M0 scale exponents of x, one scale per 32 values along `dim`.

    For each group, e = floor(log2(max|x|)) - 8 (E4M3's largest exponent is 8,
    its largest value 448 = 1.75 * 2^8), clamped to [-127, 127]; the values are
    x / 2^e rounded to nearest even in E4M3 after saturation to +-448, and the
    stored scale byte is e + 127. All-zero groups get e = -127 (byte 0).
    """
    xt = x.movedim(dim, -1)
    k = xt.shape[-1]
    groups = -(-k // MX_GROUP)
    pad = groups * MX_GROUP - k
    xp = torch.nn.functional.pad(xt, (0, pad)) if pad else xt
    xg = xp.reshape(*xp.shape[:-1], groups, MX_GROUP)
    amax = xg.abs().amax(dim=-1)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax)) - 8, torch.full_like(amax, -127.0))
    e = e.clamp(-127, 127)
    q = (xg / torch.exp2(e).unsqueeze(-1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    q = q.reshape(*xp.shape)[..., :k].movedim(-1, dim).contiguous()
    s = (e + 127).to(torch.uint8).movedim(-1, dim).contiguous()
    return q, s


def make_inputs_mxfp8(M: int, K: int, N: int, seed: int):
    """Block-scaled FP8 inputs for the MX path, from the same draws as ``make_inputs``.

    The float32 draws (before any rounding) are quantised in groups of 32
    consecutive K values: A's groups run along its rows, W1's and W2's down
    their columns. Returns CPU tensors (A8 [M,K], SA [M,K/32], W1_8 [K,N],
    S1 [K/32,N], W2_8 [K,N], S2 [K/32,N]); values float8_e4m3fn, scales uint8.
    """
    g = torch.Generator().manual_seed(int(seed))
    a = torch.randn(M, K, generator=g, dtype=torch.float32)
    scale = 1.0 / math.sqrt(K)
    w1 = torch.randn(K, N, generator=g, dtype=torch.float32) * scale
    w2 = torch.randn(K, N, generator=g, dtype=torch.float32) * scale
    a8, sa = _mx_quantise(a, 1)
    w18, s1 = _mx_quantise(w1, 0)
    w28, s2 = _mx_quantise(w2, 0)
    return a8, sa, w18, s1, w28, s2
