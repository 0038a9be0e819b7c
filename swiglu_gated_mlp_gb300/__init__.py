"""Fused SwiGLU gated-MLP projection for NVIDIA GB300 (sm_103a).

    Y = SiLU(A W1) * (A W2),   A [M, K], W1 / W2 [K, N], Y [M, N], all bf16.

The public functions mirror the C ABI in include/swiglu.h (same names):
``swiglu_pack_weights``, ``swiglu_forward``, ``swiglu_forward_variant``,
``swiglu_forward_from_host``, ``swiglu_packed_weight_bytes``,
``swiglu_check_device_status``, ``swiglu_status_string``, ``swiglu_plan_string``
and the FP8, down-projection and allocation-free forms; ``pack(W1, W2)`` and
``forward(A, Wp, N)`` are short names of the first two.
They load the compiled library on first use and raise if it is missing; there
is no CPU or PyTorch fallback.
"""
_EXPORTS = {
    "pack", "forward",
    "swiglu_packed_weight_bytes_mxfp8", "swiglu_pack_weights_mxfp8", "swiglu_act_scale_bytes_mxfp8",
    "swiglu_pack_act_scales_mxfp8", "swiglu_forward_mxfp8", "swiglu_plan_string_mxfp8",
    "swiglu_pack_weights", "swiglu_forward", "swiglu_forward_variant", "swiglu_forward_from_host",
    "swiglu_forward_noalloc", "swiglu_pack_weights_fp8", "swiglu_forward_fp8",
    "swiglu_packed_weight_bytes_fp8", "swiglu_down_packed_bytes", "swiglu_pack_down_weights",
    "swiglu_down_forward", "swiglu_down_plan_string", "swiglu_plan_string_fp8",
    "swiglu_down_workspace_bytes", "swiglu_down_workspace", "swiglu_down_plan_string_ws",
    "swiglu_packed_weight_bytes", "swiglu_check_device_status", "swiglu_status_string",
    "swiglu_plan_string", "swiglu_testing_inject_stall", "swiglu_testing_pace_run_out",
    "SwigluError",
    "SWIGLU_VARIANT_AUTO", "SWIGLU_VARIANT_LARGE_M", "SWIGLU_VARIANT_SMALL_M",
    "SWIGLU_VARIANT_LARGE_M_PAIR", "SWIGLU_VARIANT_SEQUENTIAL", "SWIGLU_VARIANT_SPLIT_K",
    "SWIGLU_VARIANT_RESIDENT_PAIR",
}


def __getattr__(name):
    if name in _EXPORTS:
        from . import _native
        return getattr(_native, name)
    raise AttributeError(name)
