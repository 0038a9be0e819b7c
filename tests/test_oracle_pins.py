"""Pins of the CPU oracle against things other than itself (no GPU).

Each pin is chosen so that a plausible slip in the oracle fails it: a wrong sign
in SiLU, sigmoid(-x) for sigmoid(x), a transposed operand, W1 and W2 swapped, a
dropped term of the sum, rounding through float32 before bf16, or a wrong
index in the packed layout.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import brute, compare, pack_layout
from oracle.swiglu_ref import (bf16_bits_to_f64, f64_to_bf16_bits, gate_up_f64, silu,
                               swiglu_f64, swiglu_f64_values)
from swiglu_gated_mlp_gb300.workloads import bf16_bits, make_inputs

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))


def _frac(s):
    from fractions import Fraction
    return float(Fraction(s))


def _example():
    ex = GOLDEN["worked_example"]
    a = np.array([[_frac(v) for v in r] for r in ex["A"]])
    w1 = np.array([[_frac(v) for v in r] for r in ex["W1"]])
    w2 = np.array([[_frac(v) for v in r] for r in ex["W2"]])
    y = np.array([[float(v) for v in r] for r in ex["Y"]])
    gate = np.array([[_frac(v) for v in r] for r in ex["gate_exact"]])
    up = np.array([[_frac(v) for v in r] for r in ex["up_exact"]])
    return a, w1, w2, gate, up, y


# ---------------------------------------------------------------- SiLU ----

@pytest.mark.parametrize("row", GOLDEN["silu"], ids=lambda r: r["x_name"])
def test_silu_matches_symbolic_values(row):
    x = float(row["x"])
    want = float(row["silu"])
    got = float(silu(np.float64(x)))
    assert got == pytest.approx(want, rel=4e-16, abs=1e-300)


@pytest.mark.parametrize("row", GOLDEN["silu_closed_forms"], ids=["ln3", "-ln3"])
def test_silu_closed_forms(row):
    assert float(silu(float(row["x"]))) == pytest.approx(float(row["silu"]), rel=4e-16)


def test_silu_odd_part_is_identity():
    # SiLU(x) - SiLU(-x) = x (sigmoid(x) + sigmoid(-x) = 1)
    x = np.random.default_rng(0).normal(size=1000) * 8
    assert np.allclose(silu(x) - silu(-x), x, rtol=1e-14, atol=1e-14)


def test_silu_extremes_are_finite_and_signed():
    assert silu(0.0) == 0.0
    neg = silu(np.array([-1e4, -1e308, -800.0]))
    assert np.all(neg == 0.0) and np.all(np.signbit(neg))
    pos = silu(np.array([1e4, 800.0]))
    assert np.array_equal(pos, [1e4, 800.0])
    # -100 * e^-100 / (1 + e^-100), well inside float64 range
    assert float(silu(-100.0)) == pytest.approx(-100.0 * math.exp(-100.0), rel=1e-15)


# ------------------------------------------------------- worked example ----

def test_worked_example_gate_up_exact():
    a, w1, w2, gate, up, _ = _example()
    g, u = gate_up_f64(a, w1, w2)
    assert np.array_equal(g, gate) and np.array_equal(u, up)


def test_worked_example_y():
    a, w1, w2, _, _, y = _example()
    assert np.allclose(swiglu_f64_values(a, w1, w2), y, rtol=1e-15, atol=0)


def test_worked_example_through_bf16_bits():
    a, w1, w2, _, _, y = _example()
    got = swiglu_f64(f64_to_bf16_bits(a), f64_to_bf16_bits(w1), f64_to_bf16_bits(w2))
    assert np.allclose(got, y, rtol=1e-15, atol=0)


def test_brute_matches_worked_example():
    a, w1, w2, _, _, y = _example()
    got = np.array(brute.swiglu_brute(a.tolist(), w1.tolist(), w2.tolist()))
    assert np.allclose(got, y, rtol=1e-15, atol=0)


def test_swapping_w1_w2_changes_result():
    a, w1, w2, _, _, y = _example()
    assert not np.allclose(swiglu_f64_values(a, w2, w1), y, rtol=1e-3)


def test_transposed_operand_is_caught():
    # A (2x3) @ W (3x4): using W^T would need a 4x3 weight; a square case with a
    # non-symmetric W shows the orientation instead.
    a = np.array([[1.0, 2.0]])
    w1 = np.array([[1.0, 0.0], [1.0, 1.0]])   # A @ W1 = [3, 2];  A @ W1^T = [1, 3]
    w2 = np.eye(2)
    y = swiglu_f64_values(a, w1, w2)
    s = {r["x_name"]: float(r["silu"]) for r in GOLDEN["silu"]}
    # Y = [SiLU(3) * 1, SiLU(2) * 2];  SiLU(3) = 3 sigmoid(3)
    assert y[0, 1] == pytest.approx(s["2"] * 2, rel=1e-15)
    assert y[0, 0] == pytest.approx(3.0 / (1.0 + math.exp(-3.0)), rel=1e-15)


# ------------------------------------------------- brute force, tiny ----

@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (8, 16, 8), (9, 17, 33), (5, 64, 3)])
def test_oracle_matches_brute_force(shape):
    m, k, n = shape
    a, w1, w2 = make_inputs(m, k, n, seed=m * 100 + k + n)
    ab, w1b, w2b = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    av, w1v, w2v = (bf16_bits_to_f64(x) for x in (ab, w1b, w2b))
    g_ref, u_ref = brute.gate_up_brute(av.tolist(), w1v.tolist(), w2v.tolist())
    g, u = gate_up_f64(av, w1v, w2v)
    # brute force is the exactly rounded sum; BLAS float64 is within K ulps
    assert np.allclose(g, g_ref, rtol=k * 2.3e-16, atol=1e-300)
    assert np.allclose(u, u_ref, rtol=k * 2.3e-16, atol=1e-300)
    y_ref = np.array(brute.swiglu_brute(av.tolist(), w1v.tolist(), w2v.tolist()))
    assert np.allclose(swiglu_f64(ab, w1b, w2b), y_ref, rtol=1e-13, atol=1e-15)


def test_dropped_term_would_be_seen():
    # every k contributes: zeroing one column of A changes Y on random data
    a, w1, w2 = make_inputs(4, 32, 8, seed=11)
    ab, w1b, w2b = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    y = swiglu_f64(ab, w1b, w2b)
    for k in (0, 31):
        ab2 = ab.copy()
        ab2[:, k] = 0
        assert not np.allclose(swiglu_f64(ab2, w1b, w2b), y, rtol=1e-6)


# --------------------------------------------------------- identities ----

def test_zero_activations_give_zero():
    _, w1, w2 = make_inputs(1, 64, 40, seed=3)
    a0 = np.zeros((7, 64), dtype=np.uint16)
    y = swiglu_f64(a0, bf16_bits(w1), bf16_bits(w2))
    assert np.array_equal(y, np.zeros((7, 40)))


def test_linearity_in_w2():
    a, w1, w2 = make_inputs(6, 48, 24, seed=5)
    _, _, w2b = make_inputs(6, 48, 24, seed=6)
    av, w1v, w2v, w2bv = (bf16_bits_to_f64(bf16_bits(x)) for x in (a, w1, w2, w2b))
    y = swiglu_f64_values(av, w1v, w2v)
    # scaling by 2 is exact in float64
    assert np.array_equal(swiglu_f64_values(av, w1v, 2.0 * w2v), 2.0 * y)
    y_sum = swiglu_f64_values(av, w1v, w2v + w2bv)
    assert np.allclose(y_sum, y + swiglu_f64_values(av, w1v, w2bv), rtol=1e-12, atol=1e-13)


def test_identity_slice_gives_silu_times_a():
    # K = N, W1 = W2 = I:  Y = SiLU(A) (.) A; checked against the symbolic table
    table = GOLDEN["silu"]
    xs = np.array([float(r["x"]) for r in table])
    want = np.array([float(r["silu"]) for r in table]) * xs
    eye = np.eye(len(xs))
    y = swiglu_f64_values(xs[None, :], eye, eye)[0]
    assert np.allclose(y, want, rtol=1e-15, atol=1e-300)


def test_one_hot_rows_select_weight_rows():
    _, w1, w2 = make_inputs(1, 16, 12, seed=9)
    w1v, w2v = bf16_bits_to_f64(bf16_bits(w1)), bf16_bits_to_f64(bf16_bits(w2))
    a = np.zeros((3, 16))
    picks = [0, 7, 15]
    for m, k in enumerate(picks):
        a[m, k] = 1.0
    y = swiglu_f64_values(a, w1v, w2v)
    want = np.array([[brute.silu_scalar(w1v[k, n]) * w2v[k, n] for n in range(12)] for k in picks])
    assert np.allclose(y, want, rtol=1e-15, atol=0)


def test_row_and_column_permutation_equivariance():
    a, w1, w2 = make_inputs(10, 40, 20, seed=12)
    ab, w1b, w2b = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    y = swiglu_f64(ab, w1b, w2b)
    rp = np.random.default_rng(1).permutation(10)
    cp = np.random.default_rng(2).permutation(20)
    assert np.allclose(swiglu_f64(ab[rp], w1b, w2b), y[rp], rtol=1e-14, atol=1e-15)
    assert np.allclose(swiglu_f64(ab, w1b[:, cp], w2b[:, cp]), y[:, cp], rtol=1e-14, atol=1e-15)


def test_row_subset_equals_full_rows():
    a, w1, w2 = make_inputs(33, 24, 16, seed=13)
    ab, w1b, w2b = bf16_bits(a), bf16_bits(w1), bf16_bits(w2)
    rows = np.array([0, 5, 32])
    assert np.array_equal(swiglu_f64(ab, w1b, w2b, rows=rows), swiglu_f64(ab, w1b, w2b)[rows])


# ------------------------------------------------------ bf16 rounding ----

def test_bf16_bits_decode_known_patterns():
    bits = np.array([0x3F80, 0xBF80, 0x0000, 0x8000, 0x7F80, 0x0001, 0x7F7F], dtype=np.uint16)
    v = bf16_bits_to_f64(bits)
    assert v[0] == 1.0 and v[1] == -1.0 and v[2] == 0.0 and np.signbit(v[3])
    assert v[4] == np.inf and v[5] == 2.0 ** -133
    assert v[6] == (2 - 2 ** -7) * 2.0 ** 127


def test_bf16_rounding_ties_to_even_and_single_rounding():
    one = 1.0
    cases = {
        one + 2 ** -8: 0x3F80,                 # halfway, round to even (down)
        one + 3 * 2 ** -8: 0x3F82,             # halfway, round to even (up)
        one + 2 ** -8 + 2 ** -30: 0x3F81,      # just above half: up; via float32 it would tie down
        one + 2 ** -8 - 2 ** -30: 0x3F80,
        -(one + 2 ** -8 + 2 ** -30): 0xBF81,
        2.0 ** -130: 0x0008,                   # subnormal, exact
        2.0 ** -134: 0x0000,                   # half the smallest subnormal: ties to even (0)
        3 * 2.0 ** -134: 0x0002,               # 1.5 smallest subnormals: ties to even (2)
        float.fromhex("0x1.ffp127"): 0x7F80,  # rounds past the largest finite: inf
        float.fromhex("0x1.fe8p127") - 2.0 ** 100: 0x7F7F,  # just below the overflow threshold
        -0.0: 0x8000,
    }
    xs = np.array(list(cases.keys()))
    want = np.array(list(cases.values()), dtype=np.uint16)
    assert np.array_equal(f64_to_bf16_bits(xs), want)
    assert f64_to_bf16_bits(np.array([np.nan]))[0] == 0x7FC0


def test_bf16_rounding_agrees_with_torch_on_float32_values():
    # for values that are exactly float32, one rounding from float64 equals
    # torch's float32 -> bf16 round-to-nearest-even
    rng = np.random.default_rng(4)
    x32 = np.concatenate([
        rng.normal(size=20000).astype(np.float32) * np.float32(3),
        (rng.normal(size=2000) * 1e-39).astype(np.float32),      # subnormals
        rng.integers(0, 2 ** 32, size=20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x32 = x32[np.isfinite(x32)]
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = f64_to_bf16_bits(x32.astype(np.float64))
    assert np.array_equal(got, want)


# ------------------------------------------------------- comparison ----

def test_ulp_distance_counts_bf16_steps():
    ref = bf16_bits_to_f64(np.array([0x3F80, 0x3F80, 0x0000, 0x8001], dtype=np.uint16))
    y = np.array([0x3F81, 0x3F7F, 0x8000, 0x0001], dtype=np.uint16)
    assert compare.bf16_ulp_distance(y, ref).tolist() == [1, 1, 0, 2]


def test_tolerance_rule_boundaries():
    ref = np.array([1.0, 0.0, -2.0])
    # bounds: 0.011 at ref=1, 0.001 at ref=0, 0.021 at ref=-2
    y_ok = f64_to_bf16_bits(np.array([1.0078125, 0.0009765625, -2.015625]))
    assert compare.within_tolerance(y_ok, ref).all()
    y_bad = f64_to_bf16_bits(np.array([1.015625, 0.001953125, -2.0625]))
    assert not compare.within_tolerance(y_bad, ref).any()
    assert compare.mismatch_rate(y_bad, ref) == 1.0


def test_relative_mismatch_rate_hand_values():
    # the pages' accuracy figure: share of outputs more than 1 % from the
    # reference, read over |ref| >= 1e-3 (the floor is included, ref = 0 is not)
    bf = lambda v: f64_to_bf16_bits(np.array(v, dtype=np.float64))
    # |ref| = 1e-3 exactly is compared (y = 0 is 100 % off); 0.99e-3 and 0 are not
    ref = np.array([1e-3, 0.99e-3, 0.0, 0.5])
    assert compare.relative_mismatch_rate(bf([0.0, 0.0, 0.25, 0.5]), ref) == 0.5
    # the denominator is |ref|, not |y|: d = 0.00995 is 1.005 % of 0.99005 but
    # 0.995 % of y = 1; the sign does not matter
    assert compare.relative_mismatch_rate(bf([1.0]), np.array([0.99005])) == 1.0
    assert compare.relative_mismatch_rate(bf([-1.0]), np.array([-0.99005])) == 1.0
    # just under and just over 1 % (y exact in bf16): 2^-7 / (1 - 2^-7) = 0.787 %,
    # 3 * 2^-8 / (1 - 3 * 2^-8) = 1.186 %
    assert compare.relative_mismatch_rate(bf([1.0]), np.array([1.0 - 2.0 ** -7])) == 0.0
    assert compare.relative_mismatch_rate(bf([1.0]), np.array([1.0 - 3 * 2.0 ** -8])) == 1.0
    # the rate is over the compared elements only: 1 of 4 compared, 4 ignored
    ref = np.array([1.0, 1.0, 1.0, 1.0, 1e-4, -1e-4, 0.0, 5e-4])
    y = bf([1.0, 1.0, 1.0, 2.0, 1.0, 1.0, 1.0, 1.0])
    assert compare.relative_mismatch_rate(y, ref) == 0.25
    # nothing compared: 0, not NaN
    assert compare.relative_mismatch_rate(bf([1.0, -1.0]), np.array([0.0, 1e-5])) == 0.0
    assert compare.relative_mismatch_rate(bf([]), np.array([])) == 0.0


def test_report_fields_on_hand_values():
    # y as raw bf16 bits against a float64 reference, every field worked by hand
    y = np.array([0x3F80,   # 1.0 against 1.0: exact
                  0x3F81,   # 1.0078125 against 1.0: one bf16 step, within tolerance
                  0x8001,   # -2^-133 against +0: one step across the signed zeros
                  0x0002,   # 2 * 2^-133 against -2^-133 (bf16 0x8001)
                  0x4000],  # 2.0 against 1.0: outside tolerance, 128 steps
                 dtype=np.uint16)
    tiny = 2.0 ** -133
    ref = np.array([1.0, 1.0, 0.0, -tiny, 1.0])
    rep = compare.report(y, ref)
    assert rep["n"] == 5
    assert rep["max_abs_err"] == 1.0
    assert rep["max_excess"] == 1.0 - (1e-2 * 1.0 + 1e-3)
    assert rep["tolerance_pass"] is False
    assert rep["tolerance_pass"] == bool(compare.within_tolerance(y, ref).all())
    assert rep["mismatch_rate"] == pytest.approx(0.2, abs=1e-15)
    assert rep["relative_mismatch_rate"] == 1.0 / 3.0       # |ref| >= 1e-3: three, one off
    # steps: 0, 1, 1 (0x8001 vs +0), 3 (0x0002 vs 0x8001 = -1 on the ordered line), 128
    assert compare.bf16_ulp_distance(y, ref).tolist() == [0, 1, 1, 3, 128]
    assert rep["max_bf16_ulp"] == 128
    assert rep["bf16_ulp_gt1_rate"] == pytest.approx(0.4, abs=1e-15)
    assert rep["nonfinite"] == 0
    # dropping the failing element passes
    assert compare.report(y[:4], ref[:4])["tolerance_pass"] is True


def test_report_counts_non_finite_outputs_and_fails_them():
    y = np.array([0x7FC0, 0x7F80, 0xFF80, 0x3F80, 0xFFC1], dtype=np.uint16)  # NaN, +inf, -inf, 1, NaN
    ref = np.ones(5)
    rep = compare.report(y, ref)
    assert rep["nonfinite"] == 4
    assert rep["tolerance_pass"] is False
    assert compare.within_tolerance(y, ref).tolist() == [False, False, False, True, False]
    assert rep["mismatch_rate"] == pytest.approx(0.8, abs=1e-15)
    # an empty comparison passes vacuously and reports zeros
    empty = compare.report(np.zeros(0, dtype=np.uint16), np.zeros(0))
    assert empty["n"] == 0 and empty["tolerance_pass"] and empty["max_bf16_ulp"] == 0


# ------------------------------------------------------ packed layout ----

def test_pack_layout_indices_and_padding():
    _, w1, w2 = make_inputs(1, 100, 200, seed=21)
    w1b, w2b = bf16_bits(w1), bf16_bits(w2)
    p = pack_layout.pack_reference(w1b, w2b)
    assert p.shape == (2, 2, 256, 64)      # Np = 256, Kp = 128
    for n in (0, 1, 127, 128, 150, 199):
        j, i = divmod(n, 128)
        for k in (0, 5, 63, 64, 99):
            b, t = divmod(k, 64)
            assert p[j, b, i, t] == w1b[k, n]
            assert p[j, b, 128 + i, t] == w2b[k, n]
    assert not p[1, :, 72:128].any() and not p[1, :, 128 + 72:].any()   # columns >= N
    assert not p[:, 1, :, 36:].any()                                    # K values >= K


def test_pack_layout_round_trip():
    _, w1, w2 = make_inputs(1, 40, 264, seed=22)
    w1b, w2b = bf16_bits(w1), bf16_bits(w2)
    u1, u2 = pack_layout.unpack_reference(pack_layout.pack_reference(w1b, w2b), 40, 264)
    assert np.array_equal(u1, w1b) and np.array_equal(u2, w2b)


def test_pack_layout_matches_elementwise_definition():
    # the slicing in pack_reference against the definition, element by element
    _, w1, w2 = make_inputs(1, 72, 136, seed=23)
    w1b, w2b = bf16_bits(w1), bf16_bits(w2)
    p = pack_layout.pack_reference(w1b, w2b)
    for j in range(p.shape[0]):
        for b in range(p.shape[1]):
            for i in range(256):
                n = 128 * j + (i % 128)
                for t in range(64):
                    k = 64 * b + t
                    src = w1b if i < 128 else w2b
                    want = src[k, n] if (k < 72 and n < 136) else 0
                    assert p[j, b, i, t] == want


# ------------------------------------------------------------- FP8 path ----

def test_e4m3_decode_known_patterns():
    from oracle.fp8 import e4m3_bits_to_f64
    bits = np.array([0x00, 0x38, 0xB8, 0x7E, 0x08, 0x01, 0x07, 0x80, 0x40], dtype=np.uint8)
    v = e4m3_bits_to_f64(bits)
    assert v.tolist()[:7] == [0.0, 1.0, -1.0, 448.0, 2.0 ** -6, 2.0 ** -9, 7 * 2.0 ** -9]
    assert v[7] == 0.0 and np.signbit(v[7]) and v[8] == 2.0
    assert np.isnan(e4m3_bits_to_f64(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_decode_agrees_with_torch_on_all_patterns():
    from oracle.fp8 import e4m3_bits_to_f64
    bits = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    got = e4m3_bits_to_f64(bits)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok].astype(np.float64))


def test_fp8_reference_reduces_to_the_bf16_reference():
    # with unit scales, E4M3 values are exact in bf16: both references agree exactly
    from oracle.fp8 import e4m3_bits_to_f64, swiglu_f64_fp8
    rng = np.random.default_rng(3)
    a8 = rng.integers(0, 256, size=(5, 48), dtype=np.uint8)
    w18 = rng.integers(0, 256, size=(48, 24), dtype=np.uint8)
    w28 = rng.integers(0, 256, size=(48, 24), dtype=np.uint8)
    for arr in (a8, w18, w28):                     # no NaN patterns
        arr[(arr & 0x7F) == 0x7F] = 0x38
    got = swiglu_f64_fp8(a8, w18, w28, 1.0, 1.0, 1.0)
    to_bf16 = lambda b: f64_to_bf16_bits(e4m3_bits_to_f64(b))
    want = swiglu_f64(to_bf16(a8), to_bf16(w18), to_bf16(w28))
    assert np.array_equal(got, want)


def test_fp8_reference_scales():
    from oracle.fp8 import swiglu_f64_fp8
    rng = np.random.default_rng(4)
    a8 = rng.integers(0, 0x70, size=(3, 32), dtype=np.uint8)
    w18 = rng.integers(0, 0x70, size=(32, 16), dtype=np.uint8)
    w28 = rng.integers(0x80, 0xF0, size=(32, 16), dtype=np.uint8)
    y = swiglu_f64_fp8(a8, w18, w28, 0.5, 0.25, 0.125)
    # Y is linear in the up scale (exact for a power of two)
    assert np.array_equal(swiglu_f64_fp8(a8, w18, w28, 0.5, 0.25, 0.25), 2.0 * y)
    # rows subset
    assert np.array_equal(swiglu_f64_fp8(a8, w18, w28, 0.5, 0.25, 0.125, rows=[2, 0]), y[[2, 0]])


def test_fp8_pack_layout_uses_128_value_slices():
    rng = np.random.default_rng(5)
    w1 = rng.integers(0, 256, size=(200, 136), dtype=np.uint8)
    w2 = rng.integers(0, 256, size=(200, 136), dtype=np.uint8)
    p = pack_layout.pack_reference(w1, w2, slice_k=128)
    assert p.shape == (2, 2, 256, 128) and p.dtype == np.uint8
    for n in (0, 127, 128, 135):
        j, i = divmod(n, 128)
        for k in (0, 127, 128, 199):
            b, t = divmod(k, 128)
            assert p[j, b, i, t] == w1[k, n] and p[j, b, 128 + i, t] == w2[k, n]
    assert not p[1, :, 8:128].any() and not p[:, 1, :, 72:].any()


def test_fp8_pack_layout_round_trip():
    rng = np.random.default_rng(6)
    w1 = rng.integers(0, 256, size=(144, 264), dtype=np.uint8)
    w2 = rng.integers(0, 256, size=(144, 264), dtype=np.uint8)
    p = pack_layout.pack_reference(w1, w2, slice_k=128)
    u1, u2 = pack_layout.unpack_reference(p, 144, 264, slice_k=128)
    assert u1.dtype == np.uint8 and np.array_equal(u1, w1) and np.array_equal(u2, w2)
    # the bf16 slicing does not invert the FP8 layout
    with pytest.raises(ValueError):
        pack_layout.unpack_reference(p, 144, 264)


# ----------------------------------------------------- down-projection ----

def test_down_reference_matches_brute_force():
    from oracle.down_ref import down_f64
    import math as _m
    y, w3, _ = make_inputs(5, 24, 9, seed=31)          # Y [5, 24], W3 [24, 9]
    r, _, _ = make_inputs(5, 9, 1, seed=32)            # R [5, 9]
    yb, w3b, rb = bf16_bits(y), bf16_bits(w3), bf16_bits(r)
    yv, w3v, rv = (bf16_bits_to_f64(x) for x in (yb, w3b, rb))
    want = np.array([[_m.fsum([*(yv[m, k] * w3v[k, h] for k in range(24)), rv[m, h]])
                      for h in range(9)] for m in range(5)])
    assert np.allclose(down_f64(yb, w3b, rb), want, rtol=1e-14, atol=1e-15)
    assert np.allclose(down_f64(yb, w3b, None), want - rv, rtol=1e-13, atol=1e-14)


def test_down_reference_identity_and_rows():
    from oracle.down_ref import down_f64_values, down_f64
    y = np.array([[1.0, -2.0, 0.5]])
    assert np.array_equal(down_f64_values(y, np.eye(3), np.array([[1.0, 1.0, 1.0]])),
                          [[2.0, -1.0, 1.5]])
    yv, w3, _ = make_inputs(7, 16, 5, seed=33)
    full = down_f64(bf16_bits(yv), bf16_bits(w3))
    assert np.array_equal(down_f64(bf16_bits(yv), bf16_bits(w3), rows=[6, 1]), full[[6, 1]])


def test_down_pack_layout():
    from oracle.down_ref import pack_down_reference
    rng = np.random.default_rng(8)
    w3 = rng.integers(0, 2 ** 16, size=(100, 300), dtype=np.uint16)   # N=100, H=300
    p = pack_down_reference(w3)
    assert p.shape == (2, 2, 256, 64)
    for h in (0, 255, 256, 299):
        j, i = divmod(h, 256)
        for k in (0, 63, 64, 99):
            b, t = divmod(k, 64)
            assert p[j, b, i, t] == w3[k, h]
    assert not p[1, :, 44:].any() and not p[:, 1, :, 36:].any()


# ------------------------------------------------- block-scaled FP8 (MX) ----

def test_ue8m0_decode_known_patterns():
    from oracle.mxfp8 import ue8m0_to_f64
    v = ue8m0_to_f64(np.array([0, 1, 126, 127, 128, 134, 254, 255], dtype=np.uint8))
    assert v.tolist()[:7] == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 128.0, 2.0 ** 127]
    assert np.isnan(v[7])


def test_mx_reference_with_unit_scales_is_the_per_tensor_reference():
    from oracle.fp8 import swiglu_f64_fp8
    from oracle.mxfp8 import swiglu_f64_mxfp8
    rng = np.random.default_rng(11)
    a8 = rng.integers(0, 256, size=(4, 96), dtype=np.uint8)
    w18 = rng.integers(0, 256, size=(96, 40), dtype=np.uint8)
    w28 = rng.integers(0, 256, size=(96, 40), dtype=np.uint8)
    for arr in (a8, w18, w28):
        arr[(arr & 0x7F) == 0x7F] = 0x30                    # no NaN patterns
    ones_a = np.full((4, 3), 127, dtype=np.uint8)
    ones_w = np.full((3, 40), 127, dtype=np.uint8)
    got = swiglu_f64_mxfp8(a8, ones_a, w18, ones_w, w28, ones_w)
    assert np.array_equal(got, swiglu_f64_fp8(a8, w18, w28, 1.0, 1.0, 1.0))


def _mx_brute(a8, sa, w18, s1, w28, s2):
    """Pure-Python triple loop: every product scaled by its own two group exponents."""
    import math as _m
    from oracle.fp8 import e4m3_bits_to_f64
    from oracle.brute import silu_scalar
    av, w1v, w2v = (e4m3_bits_to_f64(x) for x in (a8, w18, w28))
    M, K = a8.shape
    N = w18.shape[1]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            g = _m.fsum(_m.ldexp(float(av[m, k]) * float(w1v[k, n]),
                                int(sa[m, k // 32]) + int(s1[k // 32, n]) - 254) for k in range(K))
            u = _m.fsum(_m.ldexp(float(av[m, k]) * float(w2v[k, n]),
                                int(sa[m, k // 32]) + int(s2[k // 32, n]) - 254) for k in range(K))
            y[m, n] = silu_scalar(g) * u
    return y


@pytest.mark.parametrize("M,K,N", [(3, 64, 5), (2, 96, 7), (1, 32, 3)])
def test_mx_reference_matches_brute_force(M, K, N):
    from oracle.mxfp8 import swiglu_f64_mxfp8
    rng = np.random.default_rng(M * 100 + K + N)
    a8 = rng.integers(0, 0x78, size=(M, K), dtype=np.uint8) | (rng.integers(0, 2, size=(M, K)) << 7).astype(np.uint8)
    w18 = rng.integers(0, 0x78, size=(K, N), dtype=np.uint8)
    w28 = rng.integers(0x80, 0xF8, size=(K, N), dtype=np.uint8)
    # scales that differ per group, per row of A and per column of W, so a
    # scale applied along the wrong axis or to the wrong group is seen
    sa = rng.integers(118, 136, size=(M, K // 32), dtype=np.uint8)
    s1 = rng.integers(118, 136, size=(K // 32, N), dtype=np.uint8)
    s2 = rng.integers(118, 136, size=(K // 32, N), dtype=np.uint8)
    got = swiglu_f64_mxfp8(a8, sa, w18, s1, w28, s2)
    want = _mx_brute(a8, sa, w18, s1, w28, s2)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-300)
    # transposed scale arrays give a different result (the axis matters)
    if K // 32 > 1:
        wrong = swiglu_f64_mxfp8(a8, sa, w18, s1[::-1], w28, s2)
        assert not np.allclose(wrong, want, rtol=1e-6)


def test_mx_scale_is_an_exact_power_of_two_per_group():
    # raising one group's exponent by 3 equals multiplying that group's values by 8
    from oracle.mxfp8 import mx_values_rows, mx_values_cols
    q = np.array([[0x38, 0x40, 0xB8] * 22], dtype=np.uint8)[:, :64]   # 1, 2, -1, ...
    s = np.array([[127, 127]], dtype=np.uint8)
    base = mx_values_rows(q, s)
    s2 = s.copy()
    s2[0, 1] += 3
    got = mx_values_rows(q, s2)
    assert np.array_equal(got[:, :32], base[:, :32])
    assert np.array_equal(got[:, 32:], 8.0 * base[:, 32:])
    # columns: the same along K for a [K, N] array
    assert np.array_equal(mx_values_cols(q.T, s2.T), got.T)


def test_scale_tile_layout_is_a_bijection_with_the_stated_offsets():
    from oracle.mxfp8 import scale_tile_offset
    r, g = np.meshgrid(np.arange(128), np.arange(4), indexing="ij")
    off = scale_tile_offset(r, g)
    assert sorted(off.ravel().tolist()) == list(range(512))
    assert scale_tile_offset(0, 0) == 0 and scale_tile_offset(0, 3) == 3
    assert scale_tile_offset(32, 0) == 4 and scale_tile_offset(1, 0) == 16
    assert scale_tile_offset(127, 3) == 31 * 16 + 3 * 4 + 3


def test_act_scale_tiles_element_by_element():
    from oracle.mxfp8 import tile_act_scales, scale_tile_offset
    rng = np.random.default_rng(12)
    M, K = 130, 160                       # 2 row blocks, 2 K slices (the second ragged)
    sa = rng.integers(0, 255, size=(M, K // 32), dtype=np.uint8)
    t = tile_act_scales(sa, M, K)
    assert t.size == 2 * 2 * 512
    for m in range(256):
        for grp in range(8):
            blk = (m // 128) * 2 + grp // 4
            got = t[blk * 512 + scale_tile_offset(m % 128, grp % 4)]
            want = sa[m, grp] if (m < M and grp < K // 32) else 127
            assert got == want


def test_weight_scale_pack_element_by_element():
    from oracle.mxfp8 import pack_weight_scales, scale_tile_offset
    rng = np.random.default_rng(13)
    K, N = 192, 136                       # 2 K slices (ragged), 2 column blocks (ragged)
    s1 = rng.integers(0, 255, size=(K // 32, N), dtype=np.uint8)
    s2 = rng.integers(0, 255, size=(K // 32, N), dtype=np.uint8)
    p = pack_weight_scales(s1, s2, K, N)
    assert p.size == 2 * 2 * 1024
    for j in range(2):
        for b in range(2):
            tile = p[(j * 2 + b) * 1024:(j * 2 + b + 1) * 1024]
            for half, src in ((0, s1), (1, s2)):
                for i in range(128):
                    for grp in range(4):
                        n, kg = 128 * j + i, 4 * b + grp
                        want = src[kg, n] if (n < N and kg < K // 32) else 127
                        assert tile[half * 512 + scale_tile_offset(i, grp)] == want
