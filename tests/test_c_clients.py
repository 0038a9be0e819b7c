"""The boundary from plain C: include/swiglu.h compiles as C99 and libswiglu.so
links and runs without Python or PyTorch (tests/c/*.c)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(src, out, extra):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    from swiglu_gated_mlp_gb300 import build as _build
    lib_dir = os.path.dirname(_build.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", src), "-o", str(out), "-L", lib_dir, "-lswiglu",
           f"-Wl,-rpath,{lib_dir}"] + extra
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr


def test_header_compiles_as_c99_and_the_library_links(native_lib, tmp_path):
    exe = tmp_path / "abi_no_device"
    _compile("abi_no_device.c", exe, ["-pedantic"])
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    assert "c abi ok" in res.stdout


@pytest.mark.gpu
def test_forward_from_plain_c_matches_oracle(native_lib, tmp_path):
    from oracle import compare
    from oracle.swiglu_ref import swiglu_f64
    from swiglu_gated_mlp_gb300.workloads import bf16_bits, make_inputs
    exe = tmp_path / "forward_from_c"
    _compile("forward_from_c.c", exe, ["-I", os.path.join(CUDA_HOME, "include"),
                                        "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart"])
    M, K, N = 33, 520, 1000
    a, w1, w2 = make_inputs(M, K, N, seed=123)
    paths = [tmp_path / n for n in ("a.bin", "w1.bin", "w2.bin", "y.bin")]
    for t, pth in zip((a, w1, w2), paths):
        bf16_bits(t).tofile(pth)
    res = subprocess.run([str(exe), str(M), str(K), str(N)] + [str(p) for p in paths],
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    y = np.fromfile(paths[3], dtype=np.uint16).reshape(M, N)
    rep = compare.report(y, swiglu_f64(bf16_bits(a), bf16_bits(w1), bf16_bits(w2)))
    assert rep["tolerance_pass"] and rep["nonfinite"] == 0, rep
