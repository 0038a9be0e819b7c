"""The C-ABI library: it builds, loads and exports every declared symbol; host-side
argument checks; the Python binding's checks. No kernel is launched here."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swiglu.h")

NO_GPU = not torch.cuda.is_available()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SWIGLU_API\s+[\w\s\*]+?\b(swiglu_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("swiglu_packed_weight_bytes", "swiglu_pack_weights", "swiglu_forward",
                     "swiglu_check_device_status", "swiglu_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(native_lib):
    lib = ctypes.CDLL(native_lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_only_swiglu_symbols_are_exported(native_lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", native_lib.LIB_PATH],
                         capture_output=True, text=True).stdout
    syms = [line.split()[-1] for line in out.splitlines() if " T " in line]
    assert syms and all(s.startswith("swiglu_") for s in syms), syms


def test_packed_weight_bytes(native_lib):
    f = native_lib.swiglu_packed_weight_bytes
    assert f(896, 4864) == 2 * 4864 * 896 * 2
    assert f(64, 130) == 2 * 256 * 64 * 2      # N padded to a multiple of 128
    assert f(0, 128) == 0 and f(64, 0) == 0 and f(-1, 8) == 0


def test_status_strings(native_lib):
    for code in range(6):
        assert native_lib.swiglu_status_string(code).startswith("SWIGLU_")
    assert "UNKNOWN" in native_lib.swiglu_status_string(99)


FAKE = 0x10000  # never dereferenced: every call below fails its argument checks first


@pytest.mark.parametrize("M,K,N,want", [
    (-1, 64, 64, 1),   # negative M
    (4, 0, 64, 1),     # K = 0
    (4, 64, 0, 1),     # N = 0
    (4, 60, 64, 2),    # K not a multiple of 8
    (4, 64, 12, 2),    # N not a multiple of 8
    (4, 1 << 22, 64, 2),
])
def test_forward_rejects_bad_shapes(native_lib, M, K, N, want):
    lib = native_lib.lib
    assert lib.swiglu_forward(FAKE, FAKE * 4, FAKE * 16, M, K, N, None) == want


def test_forward_rejects_null_misaligned_and_aliased(native_lib):
    lib = native_lib.lib
    assert lib.swiglu_forward(None, FAKE, FAKE * 64, 4, 64, 64, None) == 1
    assert lib.swiglu_forward(FAKE + 2, FAKE * 16, FAKE * 64, 4, 64, 64, None) == 1
    # Y overlapping A
    assert lib.swiglu_forward(FAKE, FAKE * 64, FAKE + 64, 4, 64, 64, None) == 1
    # Y overlapping the packed weight
    assert lib.swiglu_forward(FAKE, FAKE * 64, FAKE * 64 + 256, 4, 64, 64, None) == 1
    assert lib.swiglu_forward_variant(FAKE, FAKE * 64, FAKE * 128, 4, 64, 64, 7, None) == 1


def test_forward_variant_rejects_unknown_variant(native_lib):
    lib = native_lib.lib
    for bad in (-1, 7, 99):
        assert lib.swiglu_forward_variant(FAKE, FAKE * 64, FAKE * 256, 4, 64, 64, bad, None) == 1


def test_forward_m_zero_is_a_no_op(native_lib):
    assert native_lib.lib.swiglu_forward(None, None, None, 0, 64, 64, None) == 0


def test_pack_rejects_bad_arguments(native_lib):
    lib = native_lib.lib
    assert lib.swiglu_pack_weights(None, FAKE, FAKE * 64, 64, 64, None) == 1
    assert lib.swiglu_pack_weights(FAKE, FAKE * 2, FAKE * 64, 64, 60, None) == 2
    assert lib.swiglu_pack_weights(FAKE, FAKE * 4, FAKE, 64, 64, None) == 1  # overlap


def test_plan_string_rejects_bad_buffer(native_lib):
    assert native_lib.lib.swiglu_plan_string(16, 64, 64, 0, None, 0) == 1


@pytest.mark.skipif(not NO_GPU, reason="checks the no-device path; a GPU is present")
def test_valid_call_without_a_device_fails_loudly(native_lib):
    lib = native_lib.lib
    rc = lib.swiglu_forward(FAKE, FAKE * 64, FAKE * 256, 4, 64, 64, None)
    assert rc == native_lib.SWIGLU_ERR_NO_DEVICE
    buf = ctypes.create_string_buffer(64)
    assert lib.swiglu_plan_string(16, 64, 64, 0, buf, 64) == native_lib.SWIGLU_ERR_NO_DEVICE
    assert lib.swiglu_down_plan_string(512, 4096, 1024, buf, 64) == native_lib.SWIGLU_ERR_NO_DEVICE
    assert lib.swiglu_plan_string_fp8(16, 4096, 1024, buf, 64) == native_lib.SWIGLU_ERR_NO_DEVICE
    assert lib.swiglu_down_plan_string_ws(16, 4096, 1024, buf, 64) == native_lib.SWIGLU_ERR_NO_DEVICE
    # no device, no plan: no workspace is asked for; a call with one fails like the plain call
    assert native_lib.swiglu_down_workspace_bytes(16, 4096, 1024) == 0
    assert lib.swiglu_down_forward_ws(FAKE, FAKE * 64, None, FAKE * 256, 16, 4096, 1024,
                                      FAKE * 1024, 1 << 20, None) == native_lib.SWIGLU_ERR_NO_DEVICE


def test_down_plan_string_checks_arguments_first(native_lib):
    lib = native_lib.lib
    buf = ctypes.create_string_buffer(64)
    assert lib.swiglu_down_plan_string(512, 4096, 1024, None, 0) == native_lib.SWIGLU_ERR_INVALID_ARG
    assert lib.swiglu_down_plan_string(512, 4100, 1024, buf, 64) == native_lib.SWIGLU_ERR_UNSUPPORTED
    assert lib.swiglu_down_plan_string_ws(16, 4096, 1024, None, 0) == native_lib.SWIGLU_ERR_INVALID_ARG
    assert lib.swiglu_down_plan_string_ws(16, 4100, 1024, buf, 64) == native_lib.SWIGLU_ERR_UNSUPPORTED
    # shape errors come before any device or workspace check
    assert native_lib.swiglu_down_workspace_bytes(16, 4100, 1024) == 0
    assert lib.swiglu_down_forward_ws(FAKE, FAKE * 64, None, FAKE * 256, 16, 4100, 1024,
                                      FAKE * 1024, 1 << 20, None) == native_lib.SWIGLU_ERR_UNSUPPORTED
    assert lib.swiglu_down_forward_ws(FAKE, FAKE * 64, None, FAKE * 256, 0, 4096, 1024,
                                      None, 0, None) == native_lib.SWIGLU_OK
    assert lib.swiglu_plan_string_fp8(16, 4104, 1024, buf, 64) == native_lib.SWIGLU_ERR_UNSUPPORTED
    assert lib.swiglu_plan_string_fp8(16, 4096, 1024, None, 0) == native_lib.SWIGLU_ERR_INVALID_ARG


def test_binding_rejects_cpu_tensors(native_lib):
    a = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        native_lib.swiglu_forward(a, a, 64)
    with pytest.raises(ValueError):
        native_lib.swiglu_pack_weights(a, a)


def test_block_scaled_sizes(native_lib):
    f = native_lib.swiglu_packed_weight_bytes_mxfp8
    # values as the per-tensor FP8 layout, then 1 KB of scales per 32 KB tile
    assert f(128, 128) == 2 * 128 * 128 + 1024
    assert f(160, 136) == 2 * 256 * 256 + 4 * 1024     # Np = 256, Kp = 256: 4 tiles
    assert f(0, 128) == 0
    g = native_lib.swiglu_act_scale_bytes_mxfp8
    assert g(128, 128) == 512 and g(129, 128) == 1024 and g(1, 160) == 1024
    assert g(0, 128) == 0 and g(5, 0) == 0


def test_block_scaled_argument_checks(native_lib):
    lib = native_lib.lib
    # K not a multiple of 32 (the scale group): UNSUPPORTED before any device work
    assert lib.swiglu_forward_mxfp8(FAKE, FAKE, FAKE, FAKE * 64, 4, 48, 64, None) == 2
    assert lib.swiglu_pack_weights_mxfp8(FAKE, FAKE, FAKE, FAKE, FAKE * 64, 48, 64, None) == 2
    assert lib.swiglu_pack_act_scales_mxfp8(FAKE, FAKE * 4, 4, 48, None) == 2
    # null scale pointer, misaligned block scales: INVALID_ARG
    assert lib.swiglu_forward_mxfp8(FAKE, None, FAKE, FAKE * 64, 4, 64, 64, None) == 1
    assert lib.swiglu_forward_mxfp8(FAKE, FAKE + 8, FAKE * 16, FAKE * 64, 4, 64, 64, None) == 1
    # M = 0 is a no-op
    assert lib.swiglu_forward_mxfp8(FAKE, FAKE, FAKE, FAKE, 0, 64, 64, None) == 0
