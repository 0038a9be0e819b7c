"""Parity at the full workload sizes, in the launch configuration bench.py times
(automatic kernel choice), on seeded rows the oracle computes one by one.

Workloads: the Qwen-2.5 MLP gate/up shapes (0.5B M=128; 7B decode M=16; 7B
prefill M=4096; 32B prefill M=4096 and its M sweep 1/64/512/2048; 72B prefill
M=8192). Up to 512 seeded rows per workload, always with the first and the
last, are checked on every column (all rows when M <= 512); every output of
the whole Y is also checked to be finite.
"""
import numpy as np
import pytest
import torch

from oracle import compare
from oracle.swiglu_ref import swiglu_f64
from swiglu_gated_mlp_gb300.workloads import (SWEEP_32B_M, WORKLOADS, bf16_bits,
                                              make_workload_inputs, sample_rows, sweep_32b)

pytestmark = pytest.mark.gpu

CASES = list(WORKLOADS.values()) + [sweep_32b(m) for m in SWEEP_32B_M]


@pytest.fixture(scope="module")
def native(native_lib):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return native_lib


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_full_size_workload_matches_oracle_on_sampled_rows(native, w):
    a, w1, w2 = make_workload_inputs(w)
    wp = native.swiglu_pack_weights(w1.cuda(), w2.cuda())
    y = native.swiglu_forward(a.cuda(), wp, w.N)
    native.swiglu_check_device_status()
    assert torch.isfinite(y).all().item()
    rows = sample_rows(w.M, 512, seed=w.seed)
    y_rows = bf16_bits(y[torch.from_numpy(rows).cuda()].cpu())
    del y, wp
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2), rows=rows)
    rep = compare.report(y_rows, ref)
    assert rep["tolerance_pass"] and rep["nonfinite"] == 0, rep
    assert rep["mismatch_rate"] == 0.0
    torch.cuda.empty_cache()
