"""Parity of the CUDA path with the CPU oracle (needs a GB300).

Element-by-element comparison on seeded inputs at sizes the oracle finishes in
seconds, spanning several tiles and ragged tails in M, K and N, for both
kernels and the automatic choice. Pass rule: |y - ref| <= 1e-2 |ref| + 1e-3
for every element; no non-finite outputs.
"""
import numpy as np
import pytest
import torch

from oracle import pack_layout
from oracle.swiglu_ref import swiglu_f64_values, f64_to_bf16_bits, swiglu_f64
from swiglu_gated_mlp_gb300.workloads import bf16_bits, make_inputs

from gpu_helpers import (check_against_oracle, run_forward, sentinel_buffer, sentinel_intact,
                         to_dev)

pytestmark = pytest.mark.gpu

AUTO, LARGE, SMALL, PAIR, SEQ, SPLIT, RESIDENT = 0, 1, 2, 3, 4, 5, 6


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


# ------------------------------------------------------------------ pack ----

@pytest.mark.parametrize("K,N", [(64, 128), (72, 136), (200, 264), (896, 4864), (8, 8)])
def test_pack_is_bit_exact(native, K, N):
    _, w1, w2 = make_inputs(1, K, N, seed=K + N)
    w1d, w2d = to_dev(w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    torch.cuda.synchronize()
    want = pack_layout.pack_reference(bf16_bits(w1), bf16_bits(w2))
    got = bf16_bits(wp.cpu()).reshape(-1)
    assert got.size * 2 == native.swiglu_packed_weight_bytes(K, N)
    assert np.array_equal(got, want.reshape(-1))


# --------------------------------------------------------------- forward ----

SMALL_CASES = [
    (1, 64, 128), (2, 72, 136), (7, 200, 264), (16, 256, 1024), (17, 128, 384),
    (33, 520, 256), (64, 1024, 512), (100, 136, 392), (256, 192, 256), (16, 3584, 640),
]

LARGE_CASES = [
    (1, 64, 128), (100, 200, 264), (128, 64, 128), (129, 136, 256), (300, 512, 1000),
    (1000, 256, 512), (513, 896, 4864), (256, 3584, 1024), (384, 72, 8), (2048, 128, 2048),
]

AUTO_CASES = [(16, 3584, 1280), (64, 512, 768), (65, 512, 768), (128, 896, 4864), (1024, 1024, 1024),
              (48, 256, 18944), (100, 256, 27648)]


# Few column blocks: the decode kernel splits K over clusters of 2, 4 or 8 CTAs
# and reduces the partial accumulators through distributed shared memory.
SPLIT_CASES = [
    (1, 896, 4864), (64, 896, 4864), (48, 896, 4864), (16, 128, 1024), (64, 136, 392),
    (33, 520, 8), (7, 4096, 640), (60, 200, 264),
]


@pytest.mark.parametrize("M,K,N", SPLIT_CASES)
def test_small_m_split_k_matches_oracle(native, M, K, N):
    plan = native.swiglu_plan_string(M, K, N, SMALL)
    assert "splits=1 " not in plan, plan
    check_against_oracle(native, M, K, N, seed=M * 11 + K + N, variant=SMALL)


# More than 64 tokens on few column blocks: 64-token groups, each group's K
# range split over a cluster.
GROUP_CASES = [(128, 896, 4864), (65, 256, 256), (100, 1000, 1032), (200, 512, 1000),
               (256, 384, 264)]


@pytest.mark.parametrize("M,K,N", GROUP_CASES)
def test_small_m_token_groups_match_oracle(native, M, K, N):
    plan = native.swiglu_plan_string(M, K, N, SMALL)
    assert "groups=1 " not in plan, plan
    check_against_oracle(native, M, K, N, seed=M * 17 + K + N, variant=SMALL)


@pytest.mark.parametrize("M,K,N", SMALL_CASES)
def test_small_m_kernel_matches_oracle(native, M, K, N):
    check_against_oracle(native, M, K, N, seed=M * 7 + K + N, variant=SMALL)


@pytest.mark.parametrize("M,K,N", LARGE_CASES)
def test_large_m_kernel_matches_oracle(native, M, K, N):
    check_against_oracle(native, M, K, N, seed=M * 5 + K + N, variant=LARGE)


PAIR_CASES = [
    (1, 64, 128), (100, 200, 264), (256, 64, 128), (257, 136, 256), (300, 512, 1000),
    (1000, 256, 512), (513, 896, 4864), (512, 3584, 1024), (384, 72, 8), (2048, 128, 2048),
]


@pytest.mark.parametrize("M,K,N", PAIR_CASES)
def test_pair_kernel_matches_oracle(native, M, K, N):
    check_against_oracle(native, M, K, N, seed=M * 3 + K + N, variant=PAIR)


# K split over the two CTAs of a cluster, one 128 x 64 tile per cluster: the
# 0.5B shape, ragged K (a CTA with no K slice when K is one slice), ragged N,
# two row tiles, and a long K loop that wraps the 7-stage ring.
SPLITK_CASES = [(128, 896, 4864), (100, 200, 264), (1, 64, 128), (129, 136, 256),
                (300, 512, 1000), (256, 3584, 1024), (90, 8, 8)]


@pytest.mark.parametrize("M,K,N", SPLITK_CASES)
def test_split_k_kernel_matches_oracle(native, M, K, N):
    assert native.swiglu_plan_string(M, K, N, SPLIT).startswith("split_k"), (M, K, N)
    check_against_oracle(native, M, K, N, seed=M * 19 + K + N, variant=SPLIT)


# Every K slice resident in shared memory (K <= 896): 128 x 64 tiles on CTA
# pairs with M = 128 MMAs; the 0.5B shape, ragged M, K and N, more tiles than
# SMs, a single K slice.
RESIDENT_CASES = [(128, 896, 4864), (100, 200, 264), (1, 64, 128), (129, 136, 256),
                  (300, 512, 1000), (65, 896, 520), (257, 832, 4864), (90, 8, 8), (64, 72, 64)]


@pytest.mark.parametrize("M,K,N", RESIDENT_CASES)
def test_resident_pair_kernel_matches_oracle(native, M, K, N):
    assert native.swiglu_plan_string(M, K, N, RESIDENT).startswith("resident_pair"), (M, K, N)
    check_against_oracle(native, M, K, N, seed=M * 23 + K + N, variant=RESIDENT)


def test_resident_pair_rejects_long_k(native):
    # K = 960 needs 15 slices: more than shared memory holds at once
    a, w1, w2 = make_inputs(16, 960, 128, seed=3)
    with pytest.raises(native.SwigluError) as err:
        run_forward(native, a, w1, w2, RESIDENT)
    assert err.value.code == native.SWIGLU_ERR_UNSUPPORTED


# The pages' Kernel-1 schedule (gate K loop, then up K loop), kept for comparison.
SEQ_CASES = [(1, 64, 128), (100, 200, 264), (129, 136, 256), (300, 512, 1000), (513, 896, 4864),
             (2048, 128, 2048)]


@pytest.mark.parametrize("M,K,N", SEQ_CASES)
def test_sequential_kernel_matches_oracle(native, M, K, N):
    check_against_oracle(native, M, K, N, seed=M * 13 + K + N, variant=SEQ)


@pytest.mark.parametrize("M,K,N", AUTO_CASES)
def test_auto_choice_matches_oracle(native, M, K, N):
    check_against_oracle(native, M, K, N, seed=M + K + N, variant=AUTO)


@pytest.mark.parametrize("variant", [LARGE, SMALL, PAIR, SEQ, SPLIT, RESIDENT])
def test_variants_agree(native, variant):
    # both kernels accumulate in fp32; their bf16 outputs agree within 1 ulp-ish
    a, w1, w2 = make_inputs(48, 640, 512, seed=77)
    y_auto, _ = run_forward(native, a, w1, w2, AUTO)
    y_var, _ = run_forward(native, a, w1, w2, variant)
    assert torch.allclose(y_auto.float(), y_var.float(), rtol=1e-2, atol=1e-3)


# Every token count from 1 to 17 and around one 128-row tile, on every kernel
# (ragged K slice and ragged column block): the decode kernel's token padding
# to 16, the row tails of the 128- and 256-row tiles.
TOKEN_COUNTS = list(range(1, 18)) + [127, 128, 129]


@pytest.mark.parametrize("variant", [AUTO, SMALL, LARGE, PAIR, SPLIT, RESIDENT])
@pytest.mark.parametrize("M", TOKEN_COUNTS)
def test_every_small_token_count_matches_oracle(native, M, variant):
    check_against_oracle(native, M, 200, 264, seed=1000 + M, variant=variant)


# ------------------------------------------------------------ extremes ----

# Long K (hundreds of pipeline phases per tile), wide N with short K (many
# column blocks, persistent tile loops), and a tall M (many tiles per CTA).
EXTREME_CASES = [
    (16, 32768, 384, SMALL), (300, 32768, 256, LARGE), (512, 16384, 256, PAIR),
    (16, 64, 131072, SMALL), (200, 64, 65536, AUTO), (20000, 128, 256, AUTO),
]


@pytest.mark.parametrize("M,K,N,variant", EXTREME_CASES)
def test_extreme_shapes_match_oracle(native, M, K, N, variant):
    from swiglu_gated_mlp_gb300.workloads import sample_rows
    rows = sample_rows(M, 128, seed=M + K + N)
    check_against_oracle(native, M, K, N, seed=M + 2 * K + N, variant=variant, rows=rows)


# The limits of the boundary: K or N at 2^21 (the largest the ABI accepts),
# and the smallest K and N (8, one 16-byte row) on every kernel.
MAX_CASES = [(1, 1 << 21, 128), (3, 64, 1 << 21)]


@pytest.mark.parametrize("M,K,N", MAX_CASES)
def test_largest_k_and_n_match_oracle(native, M, K, N):
    check_against_oracle(native, M, K, N, seed=M + 5, variant=AUTO)
    torch.cuda.empty_cache()


# The largest M the ABI accepts (2^31 - 1 tokens, a ragged last row tile) on
# the row-tiled kernels: row coordinates near 2^31 in the loads, stores and
# tile loops. A is a seeded 4096-row block repeated down the rows, so each
# sampled row's oracle is that of its row in the block (about 69 GB on the
# device: A and Y, 34 GB each).
@pytest.mark.parametrize("variant", [AUTO, LARGE, PAIR])
def test_largest_m_matches_oracle(native, variant):
    from oracle import compare
    M, K, N, blk = (1 << 31) - 1, 8, 8, 4096
    a, w1, w2 = make_inputs(blk, K, N, seed=61)
    ad = y = None
    try:
        ad = a.cuda().repeat((M + blk - 1) // blk, 1)[:M]
        wp = native.swiglu_pack_weights(w1.cuda(), w2.cuda())
        y = native.swiglu_forward_variant(ad, wp, N, variant)
        native.swiglu_check_device_status()
        rows = np.array([0, 1, blk - 1, blk, 1 << 30, M - 257, M - 256, M - 129, M - 2, M - 1],
                        dtype=np.int64)
        got = bf16_bits(y[torch.from_numpy(rows).cuda()].cpu())
        ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2), rows=rows % blk)
        rep = compare.report(got, ref)
        assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep
    finally:
        ad = y = None
        torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", [AUTO, LARGE, SMALL, PAIR, SEQ, SPLIT, RESIDENT])
@pytest.mark.parametrize("M", [1, 9, 130])
def test_smallest_k_and_n_match_oracle(native, variant, M):
    check_against_oracle(native, M, 8, 8, seed=M + variant, variant=variant)


# ------------------------------------------------------- special values ----

def test_empty_batch_on_every_entry_point(native):
    # M = 0 tokens: every forward entry point (each bf16 variant, host buffers,
    # per-tensor and block-scaled FP8, the down-projection with and without a
    # workspace) returns an empty output and leaves the device status clean
    from swiglu_gated_mlp_gb300.workloads import make_inputs_fp8, make_inputs_mxfp8
    K, N, H = 256, 264, 264
    _, w1, w2 = make_inputs(1, K, N, seed=5)
    wp = native.swiglu_pack_weights(w1.cuda(), w2.cuda())
    a0 = torch.empty(0, K, dtype=torch.bfloat16, device="cuda")
    for variant in (AUTO, LARGE, SMALL, PAIR, SEQ, SPLIT, RESIDENT):
        assert tuple(native.swiglu_forward_variant(a0, wp, N, variant).shape) == (0, N)
    y_host = torch.empty(0, N, dtype=torch.bfloat16)
    native.swiglu_forward_from_host(torch.empty(0, K, dtype=torch.bfloat16), wp, N, y_host, a0,
                                    torch.empty(0, N, dtype=torch.bfloat16, device="cuda"))
    a8, w18, w28, scales = make_inputs_fp8(1, K, N, seed=6)
    wp8 = native.swiglu_pack_weights_fp8(w18.cuda(), w28.cuda())
    assert tuple(native.swiglu_forward_fp8(a8.cuda()[:0], wp8, N, *scales).shape) == (0, N)
    a8, sa, w18, s1, w28, s2 = make_inputs_mxfp8(1, K, N, seed=7)
    wpm = native.swiglu_pack_weights_mxfp8(w18.cuda(), s1.cuda(), w28.cuda(), s2.cuda())
    sat = native.swiglu_pack_act_scales_mxfp8(sa.cuda()[:0])
    assert tuple(native.swiglu_forward_mxfp8(a8.cuda()[:0], sat, wpm, N).shape) == (0, N)
    _, w3, _ = make_inputs(1, N, H, seed=8)
    w3p = native.swiglu_pack_down_weights(w3.cuda())
    y0 = torch.empty(0, N, dtype=torch.bfloat16, device="cuda")
    assert tuple(native.swiglu_down_forward(y0, w3p, H).shape) == (0, H)
    ws = native.swiglu_down_workspace(16, N, H)
    assert tuple(native.swiglu_down_forward(y0, w3p, H, workspace=ws).shape) == (0, H)
    torch.cuda.synchronize()
    native.swiglu_check_device_status()


@pytest.mark.parametrize("variant", [LARGE, SMALL])
def test_zero_activations_give_exact_zero(native, variant):
    _, w1, w2 = make_inputs(1, 256, 384, seed=4)
    a = torch.zeros(40, 256, dtype=torch.bfloat16)
    y, _ = run_forward(native, a, w1, w2, variant)
    assert torch.count_nonzero(y.float()) == 0


@pytest.mark.parametrize("variant", [LARGE, SMALL])
def test_large_gate_magnitudes_stay_finite(native, variant):
    # Gate values spread over [-240, 240]: SiLU's exp overflows for the most
    # negative ones; the result must be the signed-zero limit, never NaN.
    K, N, M = 64, 256, 32
    a = torch.zeros(M, K, dtype=torch.bfloat16)
    a[:, 0] = torch.linspace(-15, 15, M).to(torch.bfloat16)
    w1 = torch.zeros(K, N, dtype=torch.bfloat16)
    w1[0, :] = torch.linspace(-16, 16, N).to(torch.bfloat16)
    w2 = torch.ones(K, N, dtype=torch.bfloat16)
    y, _ = run_forward(native, a, w1, w2, variant)
    assert torch.isfinite(y.float()).all()
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2))
    from oracle import compare
    assert compare.report(bf16_bits(y), ref)["tolerance_pass"]


@pytest.mark.parametrize("variant", [LARGE, SMALL])
def test_identity_slice(native, variant):
    # K = N, W1 = W2 = I  =>  Y = SiLU(A) (.) A
    K = N = 128
    a, _, _ = make_inputs(64, K, N, seed=31)
    eye = torch.eye(K, dtype=torch.bfloat16)
    y, _ = run_forward(native, a, eye, eye, variant)
    av = a.double().numpy()
    want = swiglu_f64_values(av, np.eye(K), np.eye(K))
    from oracle import compare
    assert compare.report(bf16_bits(y), want)["tolerance_pass"]


# ------------------------------------------------- memory and streams ----

@pytest.mark.parametrize("variant,M", [(LARGE, 200), (SMALL, 9), (LARGE, 5), (PAIR, 300), (SEQ, 150)])
def test_writes_stay_inside_y(native, variant, M):
    K, N, pad = 128, 392, 4096
    a, w1, w2 = make_inputs(M, K, N, seed=8)
    ad, w1d, w2d = to_dev(a, w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    buf = sentinel_buffer(M * N, pad)
    y = buf[pad:pad + M * N].view(M, N)
    native.swiglu_forward_variant(ad, wp, N, variant, Y=y)
    native.swiglu_check_device_status()
    assert sentinel_intact(buf, pad)
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2))
    from oracle import compare
    assert compare.report(bf16_bits(y.cpu()), ref)["tolerance_pass"]


def test_runs_on_a_side_stream(native):
    a, w1, w2 = make_inputs(96, 256, 512, seed=10)
    ad, w1d, w2d = to_dev(a, w1, w2)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        wp = native.swiglu_pack_weights(w1d, w2d)
        y = native.swiglu_forward(ad, wp, 512)
    s.synchronize()
    native.swiglu_check_device_status(stream=s)
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2))
    from oracle import compare
    assert compare.report(bf16_bits(y.cpu()), ref)["tolerance_pass"]


def test_repeated_calls_are_identical(native):
    a, w1, w2 = make_inputs(300, 512, 640, seed=12)
    ad, w1d, w2d = to_dev(a, w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    y1 = native.swiglu_forward(ad, wp, 640).clone()
    for _ in range(5):
        y2 = native.swiglu_forward(ad, wp, 640)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("M,K,N", [(16, 1024, 2048), (40, 896, 4864)])
def test_forward_sees_weights_repacked_in_place(native, M, K, N):
    # One packed buffer, two weight sets, alternately packed into it and used by
    # a forward call on one stream with no synchronisation in between. The decode
    # kernel stages weight tiles in L2 before it waits for the kernel ahead of it;
    # every call must still compute with the weights packed just before it.
    from oracle import compare
    a, w1, w2 = make_inputs(M, K, N, seed=91)
    _, v1, v2 = make_inputs(M, K, N, seed=92)
    ad, w1d, w2d, v1d, v2d = to_dev(a, w1, w2, v1, v2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    ys = []
    for i in range(6):
        if i:
            native.swiglu_pack_weights(*((v1d, v2d) if i % 2 else (w1d, w2d)), Wpacked=wp)
        ys.append(native.swiglu_forward(ad, wp, N))
    native.swiglu_check_device_status()
    ab = bf16_bits(a)
    refs = [swiglu_f64(ab, bf16_bits(w1), bf16_bits(w2)), swiglu_f64(ab, bf16_bits(v1), bf16_bits(v2))]
    for i, y in enumerate(ys):
        rep = compare.report(bf16_bits(y.cpu()), refs[i % 2])
        assert rep["tolerance_pass"] and rep["nonfinite"] == 0, (i, rep)


def test_forward_from_host_buffers(native):
    M, K, N = 16, 512, 640
    a, w1, w2 = make_inputs(M, K, N, seed=14)
    w1d, w2d = to_dev(w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    a_host = a.pin_memory()
    y_host = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    a_dev = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    y_dev = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    native.swiglu_forward_from_host(a_host, wp, N, y_host, a_dev, y_dev)
    torch.cuda.synchronize()
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2))
    from oracle import compare
    assert compare.report(bf16_bits(y_host), ref)["tolerance_pass"]


def test_auto_choice_follows_the_token_sweep(native):
    # the automatic choice on a 152-SM GB300 (from timing every kernel at M = 1..128)
    assert native.swiglu_plan_string(48, 3584, 18944).startswith("small_m")     # 148 blocks
    assert native.swiglu_plan_string(96, 3584, 18944).startswith("large_m bn")
    assert native.swiglu_plan_string(64, 5120, 27648).startswith("large_m bn")  # 216 blocks
    assert native.swiglu_plan_string(256, 5120, 27648).startswith("large_m_pair")
    assert native.swiglu_plan_string(72, 896, 4864).startswith("large_m bn")    # 38 blocks


def test_plan_string_names_a_kernel(native):
    assert native.swiglu_plan_string(16, 3584, 18944).startswith("small_m")
    assert native.swiglu_plan_string(4096, 3584, 18944).startswith("large_m_pair bn=128")
    assert native.swiglu_plan_string(4096, 3584, 18944, 1).startswith("large_m bn=128")


@pytest.mark.parametrize("n_streams", [2, 3])
def test_pair_kernel_launches_on_several_streams_at_once(native, n_streams):
    # The pair kernel keeps its tile rounds loosely in step through per-round
    # counters in global memory, tagged per launch (bf16, K >= 8192). Launches
    # in flight at once (separate streams) share those counters; with three
    # streams the CTAs of two launches can also start interleaved and draw
    # from each other's launch numbers. Each launch must still give the
    # oracle's result (a pacing wait that finds a later launch's counter, or
    # runs out, only stops pacing). 1024 x 8192 outputs: 256 tiles, about 3.4
    # tile rounds a pair, so the waits before the third and fourth rounds are
    # exercised.
    from oracle import compare
    from swiglu_gated_mlp_gb300.workloads import sample_rows
    M, K, N = 1024, 8192, 8192
    inputs = [make_inputs(M, K, N, seed=31 + i) for i in range(n_streams)]
    dev = [tuple(t.cuda() for t in x) for x in inputs]
    wps = [native.swiglu_pack_weights(w1, w2) for _, w1, w2 in dev]
    streams = [torch.cuda.Stream() for _ in range(n_streams)]
    ys = [torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(n_streams)]
    torch.cuda.synchronize()
    for _ in range(4):
        for i in range(n_streams):
            native.swiglu_forward_variant(dev[i][0], wps[i], N, PAIR, Y=ys[i], stream=streams[i])
    torch.cuda.synchronize()
    native.swiglu_check_device_status()
    rows = sample_rows(M, 64, seed=5)
    for i in range(n_streams):
        a, w1, w2 = inputs[i]
        ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2), rows=rows)
        rep = compare.report(bf16_bits(ys[i].cpu())[rows], ref)
        assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep


def test_round_pacing_stays_aligned_after_a_small_grid(native):
    # Launch numbers of the pair kernel's round pacing are drawn on the device
    # from a global ticket, one fixed-size block per launch whatever its number
    # of pairs. A launch with 16 pairs between paced launches (bf16, K = 8192,
    # 512 tiles on 76 pairs: several rounds) must leave every paced launch
    # with one launch number: none of their waits may run out (a misaligned
    # number splits a launch in two, and then its waits run out every time).
    from oracle import compare
    from swiglu_gated_mlp_gb300.workloads import sample_rows
    sm, sk, sn = 256, 1024, 2048
    small = tuple(t.cuda() for t in make_inputs(sm, sk, sn, seed=41))
    swp = native.swiglu_pack_weights(small[1], small[2])
    ys = torch.empty(sm, sn, dtype=torch.bfloat16, device="cuda")
    assert "grid=32 " in native.swiglu_plan_string(sm, sk, sn, PAIR) + " "
    M, K, N = 2048, 8192, 8192
    a, w1, w2 = make_inputs(M, K, N, seed=43)
    ad = a.cuda()
    wp = native.swiglu_pack_weights(w1.cuda(), w2.cuda())
    assert native.swiglu_plan_string(M, K, N).startswith("large_m_pair")
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    before = native.swiglu_testing_pace_run_out()
    for _ in range(3):
        native.swiglu_forward_variant(small[0], swp, sn, PAIR, Y=ys)
        native.swiglu_forward(ad, wp, N, Y=y)
    torch.cuda.synchronize()
    native.swiglu_check_device_status()
    assert native.swiglu_testing_pace_run_out() == before
    rows = sample_rows(M, 16, seed=7)
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2), rows=rows)
    rep = compare.report(bf16_bits(y.cpu())[rows], ref)
    assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep
