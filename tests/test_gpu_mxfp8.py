"""Parity of the block-scaled FP8 (MX) path with the MX oracle (needs a GB300).

Inputs are E4M3 values with one UE8M0 power-of-two scale per 32 consecutive K
values (A's along its rows, W1's and W2's down their columns): the
block-scaled reading of the pages' remark on FP8 quantisation ("Problem
Statement"). The oracle decodes values and scales exactly and computes Y in
float64. Same pass rule as the other paths: |y - ref| <= 1e-2 |ref| + 1e-3
for every compared element.

The seeded generator's scales vary little from group to group (mostly by
one step), so the forward is also checked with every scale byte moved at
random by up to +-2 steps, independently per group, per row and per column:
a scale applied to the wrong group, row or column is then off by up to 2^4.
The moves stay small and centred on each group's own scale on purpose: the
pass rule's absolute floor (1e-3) assumes outputs of order one, and bytes
drawn around 2^0 instead scale the outputs to 1e10 and beyond, where an fp32
accumulation of random-signed terms that cancel is no longer within 1 %
(an error model with fp32 rounding alone puts elements outside the rule).
"""
import numpy as np
import pytest
import torch

from oracle import compare, pack_layout
from oracle.mxfp8 import pack_weight_scales, swiglu_f64_mxfp8, tile_act_scales
from swiglu_gated_mlp_gb300.workloads import (WORKLOADS, bf16_bits, fp8_bits, make_inputs_mxfp8,
                                              sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


def _random_scales(inputs, seed, spread=2):
    """The same E4M3 values with each scale byte moved by a random step in [-spread, spread]."""
    a8, sa, w18, s1, w28, s2 = inputs
    g = torch.Generator().manual_seed(seed)

    def rnd(t):
        step = torch.randint(-spread, spread + 1, t.shape, generator=g, dtype=torch.int32)
        return (t.to(torch.int32) + step).clamp(1, 254).to(torch.uint8)
    return a8, rnd(sa), w18, rnd(s1), w28, rnd(s2)


def _uniform_bytes(t, seed, lo, hi):
    """Scale bytes drawn uniformly in [lo, hi) (for layout tests only)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi, t.shape, generator=g, dtype=torch.int32).to(torch.uint8)


def run_mx(native, M, K, N, seed, rows=None, random_scales=False):
    inputs = make_inputs_mxfp8(M, K, N, seed)
    if random_scales:
        inputs = _random_scales(inputs, seed)
    a8, sa, w18, s1, w28, s2 = inputs
    wp = native.swiglu_pack_weights_mxfp8(w18.cuda(), s1.cuda(), w28.cuda(), s2.cuda())
    sat = native.swiglu_pack_act_scales_mxfp8(sa.cuda())
    y = native.swiglu_forward_mxfp8(a8.cuda(), sat, wp, N)
    native.swiglu_check_device_status()
    yb = bf16_bits(y.cpu())
    if rows is not None:
        yb = yb[rows]
    ref = swiglu_f64_mxfp8(fp8_bits(a8), sa.numpy(), fp8_bits(w18), s1.numpy(), fp8_bits(w28),
                           s2.numpy(), rows=rows)
    rep = compare.report(yb, ref)
    assert rep["nonfinite"] == 0, rep
    assert rep["tolerance_pass"], rep
    return rep


@pytest.mark.parametrize("K,N", [(128, 128), (160, 136), (384, 264), (896, 4864)])
def test_mx_weight_pack_is_bit_exact(native, K, N):
    _, _, w18, s1, w28, s2 = make_inputs_mxfp8(1, K, N, seed=K + N)
    s1, s2 = _uniform_bytes(s1, K, 0, 255), _uniform_bytes(s2, K + 1, 0, 255)
    wp = native.swiglu_pack_weights_mxfp8(w18.cuda(), s1.cuda(), w28.cuda(), s2.cuda())
    torch.cuda.synchronize()
    got = wp.cpu().numpy()
    assert got.size == native.swiglu_packed_weight_bytes_mxfp8(K, N)
    values = pack_layout.pack_reference(fp8_bits(w18), fp8_bits(w28), slice_k=128).reshape(-1)
    assert np.array_equal(got[:values.size], values)
    assert np.array_equal(got[values.size:], pack_weight_scales(s1.numpy(), s2.numpy(), K, N))


@pytest.mark.parametrize("M,K", [(1, 32), (130, 160), (256, 1024), (300, 96)])
def test_mx_act_scale_tiles_are_bit_exact(native, M, K):
    sa = _uniform_bytes(make_inputs_mxfp8(M, K, 8, seed=M + K)[1], M, 0, 255)
    sat = native.swiglu_pack_act_scales_mxfp8(sa.cuda())
    torch.cuda.synchronize()
    n = native.swiglu_act_scale_bytes_mxfp8(M, K)
    assert np.array_equal(sat.cpu().numpy()[:n], tile_act_scales(sa.numpy(), M, K))


# decode kernel (few tokens; narrow N splits K over clusters) and the CTA-pair
# kernel; K multiples of 32 with ragged 128-value slices, ragged N
CASES = [
    (1, 128, 128), (16, 3584, 1280), (16, 160, 136), (33, 416, 264), (64, 896, 4864),
    (16, 896, 4864), (48, 512, 20480), (1, 512, 27648), (100, 416, 264), (128, 1024, 1024),
    (200, 512, 1000),
    (300, 512, 1000), (1000, 2048, 768), (257, 160, 136), (300, 416, 264), (513, 96, 4864),
]


@pytest.mark.parametrize("M,K,N", CASES)
def test_mx_forward_matches_oracle(native, M, K, N):
    run_mx(native, M, K, N, seed=M + 5 * K + N)


@pytest.mark.parametrize("M", [1, 2, 3, 7, 15, 16, 17, 127, 128, 129])
def test_mx_small_token_counts_match_oracle(native, M):
    run_mx(native, M, 416, 264, seed=2000 + M)


def test_mx_largest_m_matches_oracle(native):
    # 2^31 - 1 tokens (the largest M the ABI accepts) on the CTA-pair kernel,
    # with the activation-scale tiling at that size: A and its scales are a
    # seeded 4096-row block repeated down the rows, so each sampled row's
    # oracle is its row in the block (about 115 GB on the device)
    M, K, N, blk = (1 << 31) - 1, 32, 8, 4096
    a8, sa, w18, s1, w28, s2 = make_inputs_mxfp8(blk, K, N, seed=71)
    reps = (M + blk - 1) // blk
    ad = sad = sat = y = None
    try:
        ad = a8.cuda().view(torch.uint8).repeat(reps, 1)[:M].view(a8.dtype)
        sad = sa.cuda().repeat(reps, 1)[:M]
        wp = native.swiglu_pack_weights_mxfp8(w18.cuda(), s1.cuda(), w28.cuda(), s2.cuda())
        sat = native.swiglu_pack_act_scales_mxfp8(sad)
        sad = None
        y = native.swiglu_forward_mxfp8(ad, sat, wp, N)
        native.swiglu_check_device_status()
        rows = np.array([0, 1, blk - 1, blk, 1 << 30, M - 257, M - 256, M - 129, M - 2, M - 1],
                        dtype=np.int64)
        got = bf16_bits(y[torch.from_numpy(rows).cuda()].cpu())
        ref = swiglu_f64_mxfp8(fp8_bits(a8), sa.numpy(), fp8_bits(w18), s1.numpy(), fp8_bits(w28),
                               s2.numpy(), rows=rows % blk)
        rep = compare.report(got, ref)
        assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep
    finally:
        ad = sad = sat = y = None
        torch.cuda.empty_cache()


@pytest.mark.parametrize("M,K,N", [(16, 1024, 1280), (33, 416, 264), (64, 896, 4864),
                                   (16, 896, 4864), (300, 512, 1000), (512, 1024, 2048),
                                   (1000, 2048, 768)])
def test_mx_forward_with_scales_random_per_group(native, M, K, N):
    run_mx(native, M, K, N, seed=7 * M + K + N, random_scales=True)


def test_mx_plan_string_names_the_kernel(native):
    assert native.swiglu_plan_string_mxfp8(16, 3584, 18944).startswith("mxfp8 small_m")
    # 216 column blocks for 152 SMs: two decode CTAs per SM (3 stages each)
    assert "stages=3 " in native.swiglu_plan_string_mxfp8(1, 5120, 27648)
    assert native.swiglu_plan_string_mxfp8(4096, 3584, 18944).startswith("mxfp8 large_m_pair")
    assert "splits=1 " not in native.swiglu_plan_string_mxfp8(16, 896, 4864)


@pytest.mark.parametrize("name", ["qwen2.5-7b-decode-m16", "qwen2.5-7b-prefill-m4096",
                                  "qwen2.5-72b-prefill-m8192"])
def test_mx_full_size_workloads(native, name):
    w = WORKLOADS[name]
    rows = sample_rows(w.M, 512, seed=w.seed)
    rep = run_mx(native, w.M, w.K, w.N, seed=w.seed, rows=rows)
    assert rep["mismatch_rate"] == 0.0


def test_mx_zero_activations_give_zero(native):
    _, _, w18, s1, w28, s2 = make_inputs_mxfp8(1, 256, 384, seed=9)
    wp = native.swiglu_pack_weights_mxfp8(w18.cuda(), s1.cuda(), w28.cuda(), s2.cuda())
    for M in (16, 200):
        a8 = torch.zeros(M, 256, dtype=torch.float8_e4m3fn, device="cuda")
        sa = torch.full((M, 8), 127, dtype=torch.uint8, device="cuda")
        y = native.swiglu_forward_mxfp8(a8, native.swiglu_pack_act_scales_mxfp8(sa), wp, 384)
        torch.cuda.synchronize()
        assert torch.count_nonzero(y.float()) == 0


def test_mx_rejects_bad_arguments(native):
    lib = native.lib
    fake = 0x10000
    # K not a multiple of 32
    assert lib.swiglu_forward_mxfp8(fake, fake * 2, fake * 64, fake * 256, 4, 48, 64,
                                    None) == native.SWIGLU_ERR_UNSUPPORTED
    assert lib.swiglu_pack_weights_mxfp8(fake, fake, fake, fake, fake * 64, 48, 64,
                                         None) == native.SWIGLU_ERR_UNSUPPORTED
    # misaligned block-scale pointer
    assert lib.swiglu_forward_mxfp8(fake, fake * 2 + 8, fake * 64, fake * 256, 4, 64, 64,
                                    None) == native.SWIGLU_ERR_INVALID_ARG
    assert native.swiglu_packed_weight_bytes_mxfp8(64, 128) == 2 * 128 * 128 + 1024
    assert native.swiglu_act_scale_bytes_mxfp8(129, 64) == 2 * 512
