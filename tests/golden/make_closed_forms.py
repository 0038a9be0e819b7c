"""Writes closed_forms.json: SiLU constants and one hand-sized worked example.

Run from the repository root:  python tests/golden/make_closed_forms.py

The values come from exact symbolic arithmetic (sympy), never from the oracle
or the CUDA path, so they pin both independently.

* SiLU(x) = x * sigmoid(x) = x / (1 + e^-x) ("Tile-Level Activation Overlap for
  Efficient LLM Inference", gist.science, section "Methodology / Kernel-1":
  Swish on the Gate accumulator, beta = 1). Includes the two values with a
  finite closed form, SiLU(ln 3) = (3/4) ln 3 and SiLU(-ln 3) = -(1/4) ln 3.
* A 2 x 3 by 3 x 4 example of Y = SiLU(A x W1) (.) (A x W2) (same page, section
  "Problem Statement"), with small dyadic inputs that bf16 holds exactly; W1 is
  not symmetric and the shapes are not square, so a transposed operand, a
  swapped W1 / W2 or a dropped term gives different numbers.
"""
import json
import os

import sympy as sp

DIGITS = 30


def silu(x):
    return x / (1 + sp.exp(-x))


def main():
    xs = {
        "0": sp.Integer(0), "1": sp.Integer(1), "-1": sp.Integer(-1),
        "2": sp.Integer(2), "-2": sp.Integer(-2), "0.5": sp.Rational(1, 2),
        "-0.5": sp.Rational(-1, 2), "10": sp.Integer(10), "-10": sp.Integer(-10),
        "30": sp.Integer(30), "-30": sp.Integer(-30), "ln3": sp.log(3), "-ln3": -sp.log(3),
    }
    silu_table = []
    for name, x in xs.items():
        silu_table.append({"x_name": name, "x": str(sp.N(x, DIGITS)),
                           "silu": str(sp.N(silu(x), DIGITS))})
    closed = [
        {"x": str(sp.N(sp.log(3), DIGITS)), "silu": str(sp.N(sp.Rational(3, 4) * sp.log(3), DIGITS)),
         "why": "sigmoid(ln 3) = 1 / (1 + 1/3) = 3/4"},
        {"x": str(sp.N(-sp.log(3), DIGITS)), "silu": str(sp.N(-sp.Rational(1, 4) * sp.log(3), DIGITS)),
         "why": "sigmoid(-ln 3) = 1 / (1 + 3) = 1/4"},
    ]

    R = sp.Rational
    a = sp.Matrix([[1, R(-1, 2), 2], [R(1, 4), R(3, 2), -1]])
    w1 = sp.Matrix([[R(1, 2), -1, 0, R(5, 4)], [1, R(3, 4), R(-1, 2), 0], [R(-1, 4), R(1, 2), 1, -1]])
    w2 = sp.Matrix([[1, 0, -2, R(1, 2)], [R(1, 2), -1, R(1, 4), 1], [0, 2, 1, R(-3, 4)]])
    gate = a * w1
    up = a * w2
    y = sp.Matrix(gate.rows, gate.cols, lambda i, j: silu(gate[i, j]) * up[i, j])
    example = {
        "A": [[str(v) for v in row] for row in a.tolist()],
        "W1": [[str(v) for v in row] for row in w1.tolist()],
        "W2": [[str(v) for v in row] for row in w2.tolist()],
        "gate_exact": [[str(v) for v in row] for row in gate.tolist()],
        "up_exact": [[str(v) for v in row] for row in up.tolist()],
        "Y": [[str(sp.N(v, DIGITS)) for v in row] for row in y.tolist()],
    }
    out = {
        "source": "sympy exact arithmetic; definition from 'Tile-Level Activation Overlap for "
                  "Efficient LLM Inference' (gist.science), sections 'Problem Statement' and "
                  "'Methodology / Kernel-1'",
        "silu": silu_table,
        "silu_closed_forms": closed,
        "worked_example": example,
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
