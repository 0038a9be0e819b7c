"""Plain, slow, obviously correct CPU oracle for the fused SwiGLU gated-MLP projection.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or link
anything under ``oracle/``: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` use it. It shares no code with the
CUDA path (``swiglu_gated_mlp_gb300``) and imports nothing from it.

What it computes, and where that comes from ("Tile-Level Activation Overlap for
Efficient LLM Inference", gist.science technical summary):

* ``swiglu_ref.swiglu_f64``: Y = SiLU(A x W1) (.) (A x W2) (section "Problem
  Statement"), in float64 on the bf16-rounded inputs, with no intermediate
  rounding of Gate or Up (section "Key Contributions", tile-level fusion keeps
  Gate and Up out of HBM and out of bf16).
* ``swiglu_ref.silu``: SiLU(x) = x * sigmoid(x), the "Swish" of section
  "Methodology / Kernel-1" read with beta = 1.
* ``swiglu_ref.f64_to_bf16_bits``: one round-to-nearest-even from float64 to
  bf16, the single rounding of the bf16 output Y.
* ``brute.swiglu_brute``: a second, pure-Python implementation with exactly
  rounded sums (``math.fsum``) used to pin the first one on tiny shapes.
* ``pack_layout``: the packed gate/up weight layout, stated plainly; the pages
  concatenate W1 and W2 into one fused K x 2N matrix (section "Methodology /
  Kernel-2"); this library's layout is a block interleave of the same columns.
* ``mxfp8``: the block-scaled FP8 reading (E4M3 values, one power-of-two
  UE8M0 scale per 32 consecutive K values of A's rows and of W's columns) and
  the byte layouts of its scale factors; the pages name FP8 only as a reason
  the SwiGLU steps weigh more (section "Problem Statement").
* ``compare``: the pass rule |y - ref| <= 1e-2 |ref| + 1e-3 and the mismatch
  rates (section "Key Contributions", numerical superiority: share of outputs
  with more than 1% relative error against a higher-precision reference).

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, exact brute force and textbook identities; no function is "parity
unpinned".
"""
