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
