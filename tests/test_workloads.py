"""Seeded input generator: determinism, shapes and value distributions (no GPU)."""
import numpy as np
import torch

from swiglu_gated_mlp_gb300.workloads import (SWEEP_32B_M, WORKLOADS, bf16_bits, make_inputs,
                                              sample_rows, sweep_32b)


def test_same_seed_same_inputs_and_order():
    a1, w11, w21 = make_inputs(8, 64, 32, seed=5)
    a2, w12, w22 = make_inputs(8, 64, 32, seed=5)
    assert torch.equal(a1, a2) and torch.equal(w11, w12) and torch.equal(w21, w22)
    a3, _, _ = make_inputs(8, 64, 32, seed=6)
    assert not torch.equal(a1, a3)
    assert not torch.equal(w11, w21)


def test_shapes_dtypes_and_moments():
    a, w1, w2 = make_inputs(256, 1024, 512, seed=2)
    assert a.shape == (256, 1024) and w1.shape == (1024, 512) and w2.shape == (1024, 512)
    assert a.dtype == w1.dtype == w2.dtype == torch.bfloat16
    assert abs(a.float().mean()) < 0.01 and abs(a.float().std() - 1) < 0.01
    assert abs(w1.float().std() * 32 - 1) < 0.01  # N(0, 1/K), K = 1024


def test_bf16_bits_is_a_view_of_the_bits():
    t = torch.tensor([1.0, -2.0, 0.0], dtype=torch.bfloat16)
    assert bf16_bits(t).tolist() == [0x3F80, 0xC000, 0x0000]


def test_sample_rows_keeps_ends_and_is_seeded():
    r = sample_rows(4096, 512, seed=3)
    assert r[0] == 0 and r[-1] == 4095 and len(r) == 512 and np.all(np.diff(r) > 0)
    assert np.array_equal(r, sample_rows(4096, 512, seed=3))
    assert np.array_equal(sample_rows(10, 64, seed=1), np.arange(10))


def test_named_workloads():
    w = WORKLOADS["qwen2.5-7b-decode-m16"]
    assert (w.M, w.K, w.N, w.seed) == (16, 3584, 18944, 1)
    assert w.flops == 4 * 16 * 3584 * 18944
    assert w.algorithmic_bytes == 2 * 16 * 3584 + 4 * 3584 * 18944 + 2 * 16 * 18944
    assert [sweep_32b(m).M for m in SWEEP_32B_M] == [1, 64, 512, 2048]
