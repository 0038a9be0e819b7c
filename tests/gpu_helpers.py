"""Shared helpers of the GPU tests: run the CUDA path through the binding and
compare with the oracle on the same seeded inputs."""
import numpy as np
import torch

from oracle import compare
from oracle.swiglu_ref import swiglu_f64
from swiglu_gated_mlp_gb300.workloads import bf16_bits, make_inputs


def to_dev(*ts):
    return [t.cuda() for t in ts]


def run_forward(native, a, w1, w2, variant=0):
    """Pack on the GPU, run the fused forward, return (Y on the CPU, packed weight)."""
    ad, w1d, w2d = to_dev(a, w1, w2)
    wp = native.swiglu_pack_weights(w1d, w2d)
    y = native.swiglu_forward_variant(ad, wp, w1.shape[1], variant)
    native.swiglu_check_device_status()
    return y.cpu(), wp


def check_against_oracle(native, M, K, N, seed, variant=0, rows=None):
    a, w1, w2 = make_inputs(M, K, N, seed)
    y, _ = run_forward(native, a, w1, w2, variant)
    yb = bf16_bits(y)
    if rows is not None:
        yb = yb[rows]
    ref = swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2), rows=rows)
    rep = compare.report(yb, ref)
    assert rep["nonfinite"] == 0, rep
    assert rep["tolerance_pass"], rep
    return rep


def sentinel_buffer(n_elems, pad, device="cuda"):
    """A bf16 buffer of n_elems + 2*pad elements filled with a NaN sentinel."""
    buf = torch.empty(n_elems + 2 * pad, dtype=torch.bfloat16, device=device)
    buf.view(torch.int16).fill_(0x7FBF)
    return buf


def sentinel_intact(buf, pad):
    head = buf[:pad].view(torch.int16).cpu().numpy()
    tail = buf[-pad:].view(torch.int16).cpu().numpy()
    return bool(np.all(head == 0x7FBF) and np.all(tail == 0x7FBF))
