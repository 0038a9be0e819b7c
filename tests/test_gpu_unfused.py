"""Accuracy of the fused path beside the unfused one (needs a GB300).

The pages report zero mismatches (outputs with more than 1% relative error
against a higher-precision reference) for the fused kernels and 4.5-11% for
the cuBLAS-based PyTorch path ("Tile-Level Activation Overlap for Efficient
LLM Inference", gist.science, section "Key Contributions"). Here both run on
the same seeded inputs: the fused kernel, and PyTorch eager with bf16 Gate
and Up written out, SiLU and the product as separate bf16 kernels. Both are
compared with the float64 oracle under the rule |y - ref| <= 1e-2 |ref| + 1e-3.
The fused path must have no mismatch; the unfused rate is reported (it comes
from rounding Gate, Up and SiLU(Gate) to bf16 between the steps).
"""
import pytest
import torch

from oracle import compare
from oracle.swiglu_ref import swiglu_f64
from swiglu_gated_mlp_gb300.workloads import (WORKLOADS, bf16_bits, make_workload_inputs,
                                              sample_rows)

pytestmark = pytest.mark.gpu

CASES = ["qwen2.5-0.5b-mlp-m128", "qwen2.5-7b-decode-m16", "qwen2.5-7b-prefill-m4096"]


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


@pytest.mark.parametrize("name", CASES)
def test_fused_has_no_mismatch_and_unfused_rate_is_reported(native, name, record_property):
    w = WORKLOADS[name]
    a, w1, w2 = make_workload_inputs(w)
    ad, w1d, w2d = a.cuda(), w1.cuda(), w2.cuda()
    wp = native.swiglu_pack_weights(w1d, w2d)
    y_fused = native.swiglu_forward(ad, wp, w.N)
    y_unfused = torch.nn.functional.silu(ad @ w1d) * (ad @ w2d)
    native.swiglu_check_device_status()
    rows = sample_rows(w.M, 64, seed=w.seed)
    idx = torch.from_numpy(rows).cuda()
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2), rows=rows)
    fused = compare.report(bf16_bits(y_fused[idx].cpu()), ref)
    unfused = compare.report(bf16_bits(y_unfused[idx].cpu()), ref)
    record_property("fused_mismatch_rate", fused["mismatch_rate"])
    record_property("unfused_mismatch_rate", unfused["mismatch_rate"])
    print(f"{name}: fused mismatch {fused['mismatch_rate']:.6f} "
          f"(ulp>1 {fused['bf16_ulp_gt1_rate']:.6f}); unfused mismatch "
          f"{unfused['mismatch_rate']:.6f} (ulp>1 {unfused['bf16_ulp_gt1_rate']:.6f}, "
          f"relative>1% {unfused['relative_mismatch_rate']:.6f})")
    assert fused["mismatch_rate"] == 0.0 and fused["tolerance_pass"], fused
    assert unfused["nonfinite"] == 0


@pytest.mark.parametrize("name", CASES)
def test_unfused_error_is_the_bf16_rounding_of_the_intermediates(native, name):
    # torch eager against the model that rounds Gate, Up, SiLU(Gate) and the
    # product to bf16 once each: the same mismatch rates and nearly all bits,
    # with cuBLAS's reduced-precision reductions allowed or not.
    from oracle.unfused_ref import unfused_bf16
    w = WORKLOADS[name]
    a, w1, w2 = make_workload_inputs(w)
    ad, w1d, w2d = a.cuda(), w1.cuda(), w2.cuda()
    rows = sample_rows(w.M, 64, seed=w.seed)
    idx = torch.from_numpy(rows).cuda()
    ab, w1b, w2b = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    ref = swiglu_f64(ab, w1b, w2b, rows=rows)
    model = unfused_bf16(ab, w1b, w2b, rows=rows)
    rep_model = compare.report(model, ref)
    flag = torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction
    try:
        outs = []
        for allow in (True, False):
            torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction = allow
            outs.append(bf16_bits((torch.nn.functional.silu(ad @ w1d) * (ad @ w2d))[idx].cpu()))
    finally:
        torch.backends.cuda.matmul.allow_bf16_reduced_precision_reduction = flag
    for eager in outs:
        rep = compare.report(eager, ref)
        assert float((eager == model).mean()) >= 0.99
        assert abs(rep["mismatch_rate"] - rep_model["mismatch_rate"]) <= 5e-5
        assert abs(rep["relative_mismatch_rate"] - rep_model["relative_mismatch_rate"]) <= 2e-4
