"""Failure detection without a GPU fault (needs a GB300).

The kernels bound every pipeline wait. A testing hook makes the next launches
leave one pipeline stage unfilled, so the MMA issuer's wait on it runs out
after a short limit; the kernel then stops cleanly (in-flight copies and MMAs
drained, tensor memory released) and the host reads SWIGLU_ERR_TIMEOUT from
the status word. The context must stay usable: the next normal call is
checked against the oracle.
"""
import pytest
import torch

from gpu_helpers import check_against_oracle, to_dev
from oracle import compare
from oracle.fp8 import swiglu_f64_fp8
from oracle.mxfp8 import swiglu_f64_mxfp8
from swiglu_gated_mlp_gb300.workloads import (bf16_bits, fp8_bits, make_inputs, make_inputs_fp8,
                                              make_inputs_mxfp8)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


@pytest.mark.parametrize("variant,M", [(1, 64), (2, 16), (1, 300), (3, 300), (4, 200), (5, 128),
                                       (6, 128)])
def test_stalled_pipeline_reports_timeout_and_context_survives(native, variant, M):
    K, N = 256, 384
    a, w1, w2 = make_inputs(M, K, N, seed=5)
    ad, w1d, w2d = to_dev(a, w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    native.swiglu_check_device_status()
    native.swiglu_testing_inject_stall(True, timeout_ms=200)
    try:
        native.swiglu_forward_variant(ad, wp, N, variant)
        with pytest.raises(native.SwigluError) as err:
            native.swiglu_check_device_status()
        assert err.value.code == native.SWIGLU_ERR_TIMEOUT
    finally:
        native.swiglu_testing_inject_stall(False, timeout_ms=1000)
    native.swiglu_check_device_status()  # cleared by the previous read
    check_against_oracle(native, M, K, N, seed=5, variant=variant)


def _fp8_call(native, M, K, N, seed):
    a8, w18, w28, (sa, s1, s2) = make_inputs_fp8(M, K, N, seed)
    wp = native.swiglu_pack_weights_fp8(w18.cuda(), w28.cuda())
    a8d = a8.cuda()
    plan = native.swiglu_plan_string_fp8(M, K, N)

    def run():
        return native.swiglu_forward_fp8(a8d, wp, N, sa, s1, s2)

    def ref():
        return swiglu_f64_fp8(fp8_bits(a8), fp8_bits(w18), fp8_bits(w28), sa, s1, s2)
    return plan, run, ref


def _mx_call(native, M, K, N, seed):
    a8, sa, w18, s1, w28, s2 = make_inputs_mxfp8(M, K, N, seed)
    wp = native.swiglu_pack_weights_mxfp8(w18.cuda(), s1.cuda(), w28.cuda(), s2.cuda())
    sat = native.swiglu_pack_act_scales_mxfp8(sa.cuda())
    a8d = a8.cuda()
    plan = native.swiglu_plan_string_mxfp8(M, K, N)

    def run():
        return native.swiglu_forward_mxfp8(a8d, sat, wp, N)

    def ref():
        return swiglu_f64_mxfp8(fp8_bits(a8), sa.numpy(), fp8_bits(w18), s1.numpy(),
                                fp8_bits(w28), s2.numpy())
    return plan, run, ref


# the FP8 forms: decode kernel (16 tokens) and CTA pairs (300 tokens); the
# block-scaled pair kernel's scale-copy warp waits on the unfilled stage too
@pytest.mark.parametrize("form,M,kernel", [("fp8", 16, "small_m"), ("fp8", 300, "large_m_pair"),
                                           ("mxfp8", 16, "small_m"),
                                           ("mxfp8", 300, "large_m_pair")])
def test_fp8_forms_report_timeout_and_context_survives(native, form, M, kernel):
    K, N = 256, 384
    plan, run, ref = (_fp8_call if form == "fp8" else _mx_call)(native, M, K, N, seed=11)
    assert kernel in plan, plan
    native.swiglu_check_device_status()
    native.swiglu_testing_inject_stall(True, timeout_ms=200)
    try:
        run()
        with pytest.raises(native.SwigluError) as err:
            native.swiglu_check_device_status()
        assert err.value.code == native.SWIGLU_ERR_TIMEOUT
    finally:
        native.swiglu_testing_inject_stall(False, timeout_ms=1000)
    native.swiglu_check_device_status()
    y = run()
    native.swiglu_check_device_status()
    rep = compare.report(bf16_bits(y.cpu()), ref())
    assert rep["nonfinite"] == 0 and rep["tolerance_pass"], rep
