"""Parity of the FP8 (E4M3) path with the FP8 oracle (needs a GB300).

Inputs are E4M3 values with one fp32 scale per tensor (the reading taken for
the pages' remark on FP8 quantisation, "Problem Statement"); the oracle
computes Y in float64 from the exact decoded values. Same pass rule as the
bf16 path: |y - ref| <= 1e-2 |ref| + 1e-3 for every compared element.
"""
import numpy as np
import pytest
import torch

from oracle import compare, pack_layout
from oracle.fp8 import swiglu_f64_fp8
from swiglu_gated_mlp_gb300.workloads import (WORKLOADS, bf16_bits, fp8_bits, make_inputs_fp8,
                                              sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


def run_fp8(native, M, K, N, seed, rows=None):
    a8, w18, w28, (sa, s1, s2) = make_inputs_fp8(M, K, N, seed)
    wp = native.swiglu_pack_weights_fp8(w18.cuda(), w28.cuda())
    y = native.swiglu_forward_fp8(a8.cuda(), wp, N, sa, s1, s2)
    native.swiglu_check_device_status()
    yb = bf16_bits(y.cpu())
    if rows is not None:
        yb = yb[rows]
    ref = swiglu_f64_fp8(fp8_bits(a8), fp8_bits(w18), fp8_bits(w28), sa, s1, s2, rows=rows)
    rep = compare.report(yb, ref)
    assert rep["nonfinite"] == 0, rep
    assert rep["tolerance_pass"], rep
    return rep


@pytest.mark.parametrize("K,N", [(128, 128), (144, 136), (400, 264), (896, 4864)])
def test_fp8_pack_is_bit_exact(native, K, N):
    _, w18, w28, _ = make_inputs_fp8(1, K, N, seed=K + N)
    wp = native.swiglu_pack_weights_fp8(w18.cuda(), w28.cuda())
    torch.cuda.synchronize()
    want = pack_layout.pack_reference(fp8_bits(w18), fp8_bits(w28), slice_k=128)
    got = wp.cpu().numpy().reshape(-1)
    assert got.size == native.swiglu_packed_weight_bytes_fp8(K, N)
    assert np.array_equal(got, want.reshape(-1))


# decode kernel (M <= 64), with and without K split over clusters, and the
# CTA-pair kernel (M > 64); K multiples of 16 with ragged 128-value slices
CASES = [
    (1, 128, 128), (16, 3584, 1280), (16, 144, 136), (33, 400, 264), (64, 896, 4864),
    (16, 896, 4864), (65, 256, 512), (100, 400, 264), (256, 1024, 1024), (300, 512, 1000),
    (1000, 2048, 768), (48, 512, 20480),
]


@pytest.mark.parametrize("M,K,N", CASES)
def test_fp8_forward_matches_oracle(native, M, K, N):
    run_fp8(native, M, K, N, seed=M + 3 * K + N)


@pytest.mark.parametrize("M", [1, 2, 3, 7, 15, 16, 17, 127, 128, 129])
def test_fp8_small_token_counts_match_oracle(native, M):
    run_fp8(native, M, 400, 264, seed=3000 + M)


def _repeat_rows(t, M):
    """The rows of a CPU block repeated down to M rows, on the device (bytes as uint8)."""
    reps = (M + t.shape[0] - 1) // t.shape[0]
    return t.cuda().view(torch.uint8).repeat(reps, 1)[:M].view(t.dtype)


def test_fp8_largest_m_matches_oracle(native):
    # 2^31 - 1 tokens (the largest M the ABI accepts) on the CTA-pair kernel:
    # A is a seeded 4096-row block repeated down the rows, so each sampled
    # row's oracle is its row in the block (about 69 GB on the device)
    M, K, N, blk = (1 << 31) - 1, 16, 8, 4096
    a8, w18, w28, (sa, s1, s2) = make_inputs_fp8(blk, K, N, seed=67)
    ad = y = None
    try:
        ad = _repeat_rows(a8, M)
        wp = native.swiglu_pack_weights_fp8(w18.cuda(), w28.cuda())
        y = native.swiglu_forward_fp8(ad, wp, N, sa, s1, s2)
        native.swiglu_check_device_status()
        rows = np.array([0, 1, blk - 1, blk, 1 << 30, M - 257, M - 256, M - 129, M - 2, M - 1],
                        dtype=np.int64)
        got = bf16_bits(y[torch.from_numpy(rows).cuda()].cpu())
        ref = swiglu_f64_fp8(fp8_bits(a8), fp8_bits(w18), fp8_bits(w28), sa, s1, s2,
                             rows=rows % blk)
        rep = compare.report(got, ref)
        assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep
    finally:
        ad = y = None
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["qwen2.5-7b-decode-m16", "qwen2.5-7b-prefill-m4096",
                                  "qwen2.5-72b-prefill-m8192"])
def test_fp8_full_size_workloads(native, name):
    # 512 sampled rows (0 and M-1 included) x every column, as for bf16
    w = WORKLOADS[name]
    rows = sample_rows(w.M, 512, seed=w.seed)
    rep = run_fp8(native, w.M, w.K, w.N, seed=w.seed, rows=rows)
    assert rep["mismatch_rate"] == 0.0


def test_fp8_zero_activations_give_zero(native):
    _, w18, w28, (_, s1, s2) = make_inputs_fp8(1, 256, 384, seed=9)
    wp = native.swiglu_pack_weights_fp8(w18.cuda(), w28.cuda())
    for M in (16, 200):
        a8 = torch.zeros(M, 256, dtype=torch.float8_e4m3fn, device="cuda")
        y = native.swiglu_forward_fp8(a8, wp, 384, 1.0, s1, s2)
        torch.cuda.synchronize()
        assert torch.count_nonzero(y.float()) == 0


def test_fp8_rejects_bad_arguments(native):
    lib = native.lib
    fake = 0x10000
    assert lib.swiglu_forward_fp8(fake, fake * 64, fake * 256, 4, 72, 64, 1.0, 1.0, 1.0,
                                  None) == native.SWIGLU_ERR_UNSUPPORTED  # K % 16
    assert lib.swiglu_forward_fp8(fake, fake * 64, fake * 256, 4, 64, 64, float("nan"), 1.0,
                                  1.0, None) == native.SWIGLU_ERR_INVALID_ARG


def test_fp8_plan_string_names_the_kernel(native):
    # decode kernel up to 80 tokens when the 7B shape's 148 column blocks fill the SMs;
    # CTA pairs for the 32B shape's 216 blocks above 32 tokens
    assert native.swiglu_plan_string_fp8(16, 3584, 18944).startswith("fp8 small_m")
    assert native.swiglu_plan_string_fp8(64, 3584, 18944).startswith("fp8 small_m")
    assert native.swiglu_plan_string_fp8(48, 5120, 27648).startswith("fp8 large_m_pair")
    assert native.swiglu_plan_string_fp8(4096, 3584, 18944).startswith("fp8 large_m_pair")
