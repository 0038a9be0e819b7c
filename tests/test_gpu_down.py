"""Parity of the down-projection Out = Y x W3 + R with the oracle (needs a GB300).

Inputs: Y [M, N] ~ N(0, 1), W3 [N, H] ~ N(0, 1/N), R [M, H] ~ N(0, 1), all
bf16 from the seeded generator. Pass rule as for the fused forward:
|out - ref| <= 1e-2 |ref| + 1e-3 for every compared element.
"""
import numpy as np
import pytest
import torch

from oracle import compare
from oracle.down_ref import down_f64, pack_down_reference
from swiglu_gated_mlp_gb300.workloads import bf16_bits, make_inputs, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


def down_inputs(M, N, H, seed):
    y, w3, _ = make_inputs(M, N, H, seed)
    r = make_inputs(M, H, 8, seed + 1)[0]
    return y, w3, r


def run_down(native, M, N, H, seed, residual=True, in_place=False, rows=None):
    y, w3, r = down_inputs(M, N, H, seed)
    wp = native.swiglu_pack_down_weights(w3.cuda())
    rd = r.cuda() if residual else None
    out = native.swiglu_down_forward(y.cuda(), wp, H, R=rd, Out=rd if in_place else None)
    native.swiglu_check_device_status()
    ob = bf16_bits(out.cpu())
    if rows is not None:
        ob = ob[rows]
    ref = down_f64(bf16_bits(y), bf16_bits(w3), bf16_bits(r) if residual else None, rows=rows)
    rep = compare.report(ob, ref)
    assert rep["nonfinite"] == 0, rep
    assert rep["tolerance_pass"], rep
    return rep


@pytest.mark.parametrize("N,H", [(64, 256), (200, 264), (4864, 896)])
def test_down_pack_is_bit_exact(native, N, H):
    _, w3, _ = make_inputs(1, N, H, seed=N + H)
    wp = native.swiglu_pack_down_weights(w3.cuda())
    torch.cuda.synchronize()
    got = bf16_bits(wp.cpu()).reshape(-1)
    assert got.size * 2 == native.swiglu_down_packed_bytes(N, H)
    assert np.array_equal(got, pack_down_reference(bf16_bits(w3)).reshape(-1))


# decode kernel (M <= 64; narrow H splits K over clusters) and CTA pairs (M > 64)
CASES = [
    (1, 512, 256), (16, 1000, 264), (33, 4864, 896), (64, 2048, 3584), (16, 18944, 512),
    (65, 512, 256), (300, 1000, 1032), (1000, 256, 3584), (257, 4864, 896),
    (128, 4864, 896), (100, 2048, 264),
]


@pytest.mark.parametrize("M,N,H", CASES)
def test_down_matches_oracle(native, M, N, H):
    run_down(native, M, N, H, seed=M + N + H)


def test_down_largest_m_matches_oracle(native):
    # 2^31 - 1 tokens (the largest M the ABI accepts) on the CTA-pair kernel,
    # with the residual read at row offsets near 2^31: Y and R are seeded
    # 4096-row blocks repeated down the rows, so each sampled row's oracle is
    # its row in the block (about 103 GB on the device)
    M, N, H, blk = (1 << 31) - 1, 8, 8, 4096
    y, w3, r = down_inputs(blk, N, H, seed=73)
    reps = (M + blk - 1) // blk
    yd = rd = out = None
    try:
        yd = y.cuda().repeat(reps, 1)[:M]
        rd = r.cuda().repeat(reps, 1)[:M]
        wp = native.swiglu_pack_down_weights(w3.cuda())
        out = native.swiglu_down_forward(yd, wp, H, R=rd)
        native.swiglu_check_device_status()
        rows = np.array([0, 1, blk - 1, blk, 1 << 30, M - 257, M - 256, M - 129, M - 2, M - 1],
                        dtype=np.int64)
        got = bf16_bits(out[torch.from_numpy(rows).cuda()].cpu())
        ref = down_f64(bf16_bits(y), bf16_bits(w3), bf16_bits(r), rows=rows % blk)
        rep = compare.report(got, ref)
        assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep
    finally:
        yd = rd = out = None
        torch.cuda.empty_cache()


@pytest.mark.parametrize("M", [16, 300])
def test_down_without_residual(native, M):
    run_down(native, M, 1024, 520, seed=M + 1, residual=False)


@pytest.mark.parametrize("M", [16, 300])
def test_down_in_place_residual(native, M):
    run_down(native, M, 1024, 520, seed=M + 2, in_place=True)


@pytest.mark.parametrize("M", [16, 4096])
def test_down_qwen7b_shape(native, M):
    # Qwen-2.5-7B MLP down-projection: N = 18944 intermediate, H = 3584 hidden
    rows = sample_rows(M, 64, seed=M)
    rep = run_down(native, M, 18944, 3584, seed=7 + M, rows=rows)
    assert rep["mismatch_rate"] == 0.0


def test_down_plan_string_names_the_kernel(native):
    assert native.swiglu_down_plan_string(16, 18944, 3584).startswith("down small_m")
    assert native.swiglu_down_plan_string(4096, 18944, 3584).startswith("down large_m_pair")


# K split across clusters with a caller workspace (decode kernel, few output
# blocks): on GB300 the 32B decode shape (20 blocks: 2 x 3 clusters), 10, 5,
# 6 (ragged H) and 2 blocks (4 x 3, 8 x 3, 8 x 2, 8 x 2), 32 tokens; and
# shapes whose plan keeps one cluster per block (7B decode, 64-token tiles,
# the 0.5B shape, a single block with 8 K slices)
WS_CASES = [
    (1, 27648, 5120), (16, 4096, 5120), (32, 2048, 5120), (8, 2048, 2560), (16, 4096, 1280),
    (5, 3000, 1288), (7, 27648, 5120),
    (16, 18944, 3584), (64, 27648, 5120), (128, 4864, 896), (16, 1000, 264), (1, 512, 256),
]
WS_SPLIT = {(1, 27648, 5120), (16, 4096, 5120), (32, 2048, 5120), (8, 2048, 2560),
            (16, 4096, 1280), (5, 3000, 1288), (7, 27648, 5120), (16, 1000, 264)}


def _plan_fields(plan):
    return {k: int(v) for k, _, v in (f.partition("=") for f in plan.split()) if v.isdigit()}


def _counters_are_zero(native, ws, M, N, H):
    f = _plan_fields(native.swiglu_down_plan_string_ws(M, N, H))
    n = f["blocks"] * f["groups"] * f["splits"] * 4
    torch.cuda.synchronize()
    return int(torch.count_nonzero(ws[:n])) == 0


def run_down_ws(native, M, N, H, seed, ws=None, rows=None):
    y, w3, r = down_inputs(M, N, H, seed)
    wp = native.swiglu_pack_down_weights(w3.cuda())
    if ws is None:
        ws = native.swiglu_down_workspace(M, N, H)
    out = native.swiglu_down_forward(y.cuda(), wp, H, R=r.cuda(), workspace=ws)
    native.swiglu_check_device_status()
    ob = bf16_bits(out.cpu())
    if rows is not None:
        ob = ob[rows]
    ref = down_f64(bf16_bits(y), bf16_bits(w3), bf16_bits(r), rows=rows)
    rep = compare.report(ob, ref)
    assert rep["nonfinite"] == 0, rep
    assert rep["tolerance_pass"], rep
    return out, ws


@pytest.mark.parametrize("M,N,H", WS_CASES)
def test_down_with_workspace_matches_oracle(native, M, N, H):
    plan = native.swiglu_down_plan_string_ws(M, N, H)
    nbytes = native.swiglu_down_workspace_bytes(M, N, H)
    assert (nbytes > 0) == (_plan_fields(plan)["clusters"] > 1), plan
    assert ((M, N, H) in WS_SPLIT) == (nbytes > 0), plan
    out, ws = run_down_ws(native, M, N, H, seed=3 * M + N + H)
    if ws is not None:
        assert _counters_are_zero(native, ws, M, N, H)


@pytest.mark.parametrize("M", [1, 16, 32])
def test_down_32b_decode_splits_across_clusters(native, M):
    # the 32B decode down-projection: 120 CTAs (2 x 3 clusters per block) instead of 80
    f = _plan_fields(native.swiglu_down_plan_string_ws(M, 27648, 5120))
    g = _plan_fields(native.swiglu_down_plan_string(M, 27648, 5120))
    assert f["clusters"] > 1 and g["clusters"] == 1
    assert f["grid"] * 10 >= g["grid"] * 14


@pytest.mark.parametrize("M,N,H", [(16, 18944, 3584), (64, 27648, 5120), (16, 29568, 8192)])
def test_down_other_shapes_keep_one_cluster_per_block(native, M, N, H):
    # measured slower across clusters: 7B decode, 64-token tiles, 72B decode
    assert native.swiglu_down_plan_string_ws(M, N, H) == native.swiglu_down_plan_string(M, N, H)
    assert native.swiglu_down_workspace_bytes(M, N, H) == 0


def test_down_workspace_reused_and_deterministic(native):
    M, N, H = 16, 27648, 5120
    out1, ws = run_down_ws(native, M, N, H, seed=41)
    outs = [run_down_ws(native, M, N, H, seed=41, ws=ws)[0] for _ in range(3)]
    for o in outs:  # same inputs, same cluster order: bit-identical outputs
        assert torch.equal(o, out1)
    assert _counters_are_zero(native, ws, M, N, H)


def test_down_workspace_too_small_is_rejected(native):
    M, N, H = 16, 27648, 5120
    n = native.swiglu_down_workspace_bytes(M, N, H)
    assert n > 0
    y, w3, r = down_inputs(M, N, H, seed=5)
    wp = native.swiglu_pack_down_weights(w3.cuda())
    small = torch.zeros(n - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(native.SwigluError) as err:
        native.swiglu_down_forward(y.cuda(), wp, H, workspace=small)
    assert err.value.code == native.SWIGLU_ERR_INVALID_ARG


def test_down_workspace_after_a_timeout(native):
    # every cluster counts itself in even when its waits gave up, so the
    # counters are zero again and the next call with the same workspace is right
    M, N, H = 16, 27648, 5120
    y, w3, r = down_inputs(M, N, H, seed=9)
    wp = native.swiglu_pack_down_weights(w3.cuda())
    ws = native.swiglu_down_workspace(M, N, H)
    native.swiglu_check_device_status()
    native.swiglu_testing_inject_stall(True, timeout_ms=200)
    try:
        native.swiglu_down_forward(y.cuda(), wp, H, R=r.cuda(), workspace=ws)
        with pytest.raises(native.SwigluError) as err:
            native.swiglu_check_device_status()
        assert err.value.code == native.SWIGLU_ERR_TIMEOUT
    finally:
        native.swiglu_testing_inject_stall(False, timeout_ms=1000)
    assert _counters_are_zero(native, ws, M, N, H)
    run_down_ws(native, M, N, H, seed=9, ws=ws)
