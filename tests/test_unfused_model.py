"""Pins of the unfused rounding model (``oracle.unfused_ref``), no GPU.

The model rounds Gate, Up, SiLU(Gate) and the product to bf16, once each. The
pins are hand-derived values for one element, a property that holds whenever
Gate and Up are already bf16 values, and the zero case.
"""
import numpy as np

from oracle import brute, compare
from oracle.swiglu_ref import bf16_bits_to_f64, f64_to_bf16_bits, swiglu_f64
from oracle.unfused_ref import unfused_bf16, unfused_bf16_stages
from swiglu_gated_mlp_gb300.workloads import bf16_bits, make_inputs


def test_single_element_by_hand():
    # K = 1, a = 1.5, w1 = w2 = 1 + 2**-7 (both bf16): Gate = Up = 1.51171875,
    # which is 193.5 steps of 2**-7 above 0; ties go to the even step, 194, so
    # g16 = u16 = 1.515625 = 0x3FC2.
    a = np.array([[0x3FC0]], dtype=np.uint16)   # 1.5
    w = np.array([[0x3F81]], dtype=np.uint16)   # 1.0078125
    g16, u16, s16, y16 = unfused_bf16_stages(a, w, w)
    assert int(g16[0, 0]) == 0x3FC2 and int(u16[0, 0]) == 0x3FC2
    # SiLU(1.515625) = 1.24265...; the nearest bf16 is 1.2421875 = 1 + 31/128 = 0x3F9F
    assert abs(brute.silu_scalar(1.515625) - 1.2426508) < 1e-6
    assert int(s16[0, 0]) == 0x3F9F
    # 1.2421875 * 1.515625 = 1.88269..., 240.98 steps of 2**-7: 241 -> 1.8828125 = 0x3FF1
    assert int(y16[0, 0]) == 0x3FF1
    # the single rounding of the exact result: SiLU(1.51171875) * 1.51171875 =
    # 1.87236..., 239.66 steps: 240 -> 1.875 = 0x3FF0, one bf16 step away
    ref = swiglu_f64(a, w, w)
    assert int(f64_to_bf16_bits(ref)[0, 0]) == 0x3FF0
    assert abs(float(ref[0, 0]) - 1.87236) < 1e-4


def test_exact_gate_and_up_give_at_most_one_step_from_the_rounded_result():
    # One-hot rows of A pick rows of W1 and W2, so Gate and Up are bf16 values and
    # only SiLU and the product are rounded: at most one bf16 step from the
    # correctly rounded result, and never a transposed or swapped operand.
    _, w1, w2 = make_inputs(1, 40, 96, seed=31)
    w1b, w2b = bf16_bits(w1), bf16_bits(w2)
    a = np.zeros((40, 40))
    a[np.arange(40), np.arange(40)[::-1]] = 1.0
    ab = f64_to_bf16_bits(a)
    g16, u16, _, y16 = unfused_bf16_stages(ab, w1b, w2b)
    assert np.array_equal(g16, w1b[::-1]) and np.array_equal(u16, w2b[::-1])
    ref = swiglu_f64(ab, w1b, w2b)
    assert compare.bf16_ulp_distance(y16, ref).max() <= 1


def test_zero_activations_give_zero():
    _, w1, w2 = make_inputs(1, 64, 32, seed=3)
    y = unfused_bf16(np.zeros((4, 64), dtype=np.uint16), bf16_bits(w1), bf16_bits(w2))
    assert np.all(bf16_bits_to_f64(y) == 0.0)


def test_model_shows_the_unfused_error_the_single_rounding_does_not():
    a, w1, w2 = make_inputs(64, 512, 256, seed=5)
    ab, w1b, w2b = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    ref = swiglu_f64(ab, w1b, w2b)
    model = compare.report(unfused_bf16(ab, w1b, w2b), ref)
    once = compare.report(f64_to_bf16_bits(ref), ref)
    assert once["bf16_ulp_gt1_rate"] == 0.0 and once["mismatch_rate"] == 0.0
    assert model["bf16_ulp_gt1_rate"] > 0.005 and model["max_bf16_ulp"] >= 2
    assert model["nonfinite"] == 0
