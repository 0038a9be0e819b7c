"""Thin ctypes binding of libswiglu (include/swiglu.h), with the same names.

Argument marshalling only: every step of the computation runs in the library's
CUDA kernels. PyTorch supplies device memory and the current stream. There is
no fallback: if the library is not built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

SWIGLU_OK = 0
SWIGLU_ERR_INVALID_ARG = 1
SWIGLU_ERR_UNSUPPORTED = 2
SWIGLU_ERR_CUDA = 3
SWIGLU_ERR_TIMEOUT = 4
SWIGLU_ERR_NO_DEVICE = 5

SWIGLU_VARIANT_AUTO = 0
SWIGLU_VARIANT_LARGE_M = 1
SWIGLU_VARIANT_SMALL_M = 2
SWIGLU_VARIANT_LARGE_M_PAIR = 3
SWIGLU_VARIANT_SEQUENTIAL = 4
SWIGLU_VARIANT_SPLIT_K = 5
SWIGLU_VARIANT_RESIDENT_PAIR = 6

PACK_BLOCK_N = 128

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is not built; run `python -m swiglu_gated_mlp_gb300.build` "
        "(or __graft_entry__.build()) first")

lib = ctypes.CDLL(LIB_PATH)

_i64, _vp, _sz, _int, _u32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
lib.swiglu_packed_weight_bytes.argtypes = [_i64, _i64]
lib.swiglu_packed_weight_bytes.restype = _sz
lib.swiglu_pack_weights.argtypes = [_vp, _vp, _vp, _i64, _i64, _vp]
lib.swiglu_pack_weights.restype = _int
lib.swiglu_forward.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _vp]
lib.swiglu_forward.restype = _int
lib.swiglu_forward_variant.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]
lib.swiglu_forward_variant.restype = _int
lib.swiglu_forward_from_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]
lib.swiglu_forward_from_host.restype = _int
lib.swiglu_check_device_status.argtypes = [_vp]
lib.swiglu_check_device_status.restype = _int
lib.swiglu_status_string.argtypes = [_int]
lib.swiglu_status_string.restype = ctypes.c_char_p
lib.swiglu_plan_string.argtypes = [_i64, _i64, _i64, _int, ctypes.c_char_p, _sz]
lib.swiglu_plan_string.restype = _int
lib.swiglu_packed_weight_bytes_fp8.argtypes = [_i64, _i64]
lib.swiglu_packed_weight_bytes_fp8.restype = _sz
lib.swiglu_pack_weights_fp8.argtypes = [_vp, _vp, _vp, _i64, _i64, _vp]
lib.swiglu_pack_weights_fp8.restype = _int
lib.swiglu_forward_fp8.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_float, ctypes.c_float,
                                   ctypes.c_float, _vp]
lib.swiglu_forward_fp8.restype = _int
lib.swiglu_down_packed_bytes.argtypes = [_i64, _i64]
lib.swiglu_down_packed_bytes.restype = _sz
lib.swiglu_pack_down_weights.argtypes = [_vp, _vp, _i64, _i64, _vp]
lib.swiglu_pack_down_weights.restype = _int
lib.swiglu_down_forward.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]
lib.swiglu_down_forward.restype = _int
lib.swiglu_down_plan_string.argtypes = [_i64, _i64, _i64, ctypes.c_char_p, _sz]
lib.swiglu_down_plan_string.restype = _int
lib.swiglu_down_workspace_bytes.argtypes = [_i64, _i64, _i64]
lib.swiglu_down_workspace_bytes.restype = _sz
lib.swiglu_down_forward_ws.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz, _vp]
lib.swiglu_down_forward_ws.restype = _int
lib.swiglu_down_plan_string_ws.argtypes = [_i64, _i64, _i64, ctypes.c_char_p, _sz]
lib.swiglu_down_plan_string_ws.restype = _int
lib.swiglu_plan_string_fp8.argtypes = [_i64, _i64, _i64, ctypes.c_char_p, _sz]
lib.swiglu_plan_string_fp8.restype = _int
lib.swiglu_packed_weight_bytes_mxfp8.argtypes = [_i64, _i64]
lib.swiglu_packed_weight_bytes_mxfp8.restype = _sz
lib.swiglu_pack_weights_mxfp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp]
lib.swiglu_pack_weights_mxfp8.restype = _int
lib.swiglu_act_scale_bytes_mxfp8.argtypes = [_i64, _i64]
lib.swiglu_act_scale_bytes_mxfp8.restype = _sz
lib.swiglu_pack_act_scales_mxfp8.argtypes = [_vp, _vp, _i64, _i64, _vp]
lib.swiglu_pack_act_scales_mxfp8.restype = _int
lib.swiglu_forward_mxfp8.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp]
lib.swiglu_forward_mxfp8.restype = _int
lib.swiglu_plan_string_mxfp8.argtypes = [_i64, _i64, _i64, ctypes.c_char_p, _sz]
lib.swiglu_plan_string_mxfp8.restype = _int
lib.swiglu_forward_noalloc.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]
lib.swiglu_forward_noalloc.restype = _int
lib.swiglu_testing_inject_stall.argtypes = [_int, _u32]
lib.swiglu_testing_inject_stall.restype = None
lib.swiglu_testing_pace_run_out.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
lib.swiglu_testing_pace_run_out.restype = _int


class SwigluError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {swiglu_status_string(code)}")


def _check(code: int, where: str) -> None:
    if code != SWIGLU_OK:
        raise SwigluError(code, where)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device) -> int:
    if stream is None:
        if _raw_stream is not None:  # the current stream's handle without a Stream object
            return _raw_stream(device.index if device.index is not None
                               else torch.cuda.current_device())
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if isinstance(stream, torch.cuda.Stream) else int(stream)


class _on_device:
    """Makes `device` current for the library call (a no-op when it already is)."""
    __slots__ = ("idx", "prev")

    def __init__(self, device):
        self.idx = device.index if device.index is not None else torch.cuda.current_device()

    def __enter__(self):
        self.prev = torch.cuda.current_device()
        if self.prev != self.idx:
            torch.cuda.set_device(self.idx)

    def __exit__(self, *exc):
        if self.prev != self.idx:
            torch.cuda.set_device(self.prev)
        return False


def _dev_bf16(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def padded_n(n: int) -> int:
    return -(-int(n) // PACK_BLOCK_N) * PACK_BLOCK_N


def swiglu_status_string(code: int) -> str:
    return lib.swiglu_status_string(int(code)).decode()


def swiglu_packed_weight_bytes(K: int, N: int) -> int:
    return int(lib.swiglu_packed_weight_bytes(int(K), int(N)))


def swiglu_pack_weights(W1: torch.Tensor, W2: torch.Tensor, Wpacked: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Packed gate/up weight (flat bf16 buffer) from W1, W2 [K, N] (bf16, CUDA)."""
    _dev_bf16(W1, "W1")
    _dev_bf16(W2, "W2")
    if W1.dim() != 2 or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must both be [K, N]")
    K, N = W1.shape
    if Wpacked is None:  # opaque buffer of swiglu_packed_weight_bytes(K, N) bytes
        Wpacked = torch.empty(swiglu_packed_weight_bytes(K, N) // 2, dtype=torch.bfloat16,
                              device=W1.device)
    _dev_bf16(Wpacked, "Wpacked")
    if Wpacked.numel() * 2 < swiglu_packed_weight_bytes(K, N):
        raise ValueError("Wpacked is too small")
    with _on_device(W1.device):
        _check(lib.swiglu_pack_weights(W1.data_ptr(), W2.data_ptr(), Wpacked.data_ptr(), K, N,
                                       _stream_handle(stream, W1.device)), "swiglu_pack_weights")
    return Wpacked


def swiglu_forward_variant(A: torch.Tensor, Wpacked: torch.Tensor, N: int, variant: int,
                           Y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _dev_bf16(A, "A")
    _dev_bf16(Wpacked, "Wpacked")
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    if Wpacked.numel() * 2 < swiglu_packed_weight_bytes(K, N):
        raise ValueError("Wpacked does not hold a packed weight for this K and N")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _dev_bf16(Y, "Y")
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [M, N]")
    with _on_device(A.device):
        _check(lib.swiglu_forward_variant(A.data_ptr(), Wpacked.data_ptr(), Y.data_ptr(), M, K, N,
                                          int(variant), _stream_handle(stream, A.device)),
               "swiglu_forward")
    return Y


def swiglu_forward(A: torch.Tensor, Wpacked: torch.Tensor, N: int, Y: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Y [M, N] = SiLU(A W1) * (A W2) from A [M, K] and the packed weight."""
    return swiglu_forward_variant(A, Wpacked, N, SWIGLU_VARIANT_AUTO, Y=Y, stream=stream)


def pack(W1: torch.Tensor, W2: torch.Tensor) -> torch.Tensor:
    """Short name of swiglu_pack_weights: the packed gate/up weight Wp from W1, W2 [K, N]."""
    return swiglu_pack_weights(W1, W2)


def forward(A: torch.Tensor, Wp: torch.Tensor, N: int) -> torch.Tensor:
    """Short name of swiglu_forward: Y [M, N] = SiLU(A W1) * (A W2) on the current stream."""
    return swiglu_forward(A, Wp, N)


def _dev_fp8(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float8_e4m3fn:
        raise ValueError(f"{name} must be float8_e4m3fn, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def swiglu_packed_weight_bytes_fp8(K: int, N: int) -> int:
    return int(lib.swiglu_packed_weight_bytes_fp8(int(K), int(N)))


def swiglu_pack_weights_fp8(W1: torch.Tensor, W2: torch.Tensor, Wpacked: torch.Tensor | None = None,
                            stream=None) -> torch.Tensor:
    """Packed FP8 gate/up weight (flat uint8 buffer) from E4M3 W1, W2 [K, N] (CUDA)."""
    _dev_fp8(W1, "W1")
    _dev_fp8(W2, "W2")
    if W1.dim() != 2 or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must both be [K, N]")
    K, N = W1.shape
    if Wpacked is None:
        Wpacked = torch.empty(swiglu_packed_weight_bytes_fp8(K, N), dtype=torch.uint8,
                              device=W1.device)
    if Wpacked.numel() * Wpacked.element_size() < swiglu_packed_weight_bytes_fp8(K, N):
        raise ValueError("Wpacked is too small")
    with _on_device(W1.device):
        _check(lib.swiglu_pack_weights_fp8(W1.data_ptr(), W2.data_ptr(), Wpacked.data_ptr(), K, N,
                                           _stream_handle(stream, W1.device)),
               "swiglu_pack_weights_fp8")
    return Wpacked


def swiglu_forward_fp8(A: torch.Tensor, Wpacked: torch.Tensor, N: int, scale_a: float,
                       scale_w1: float, scale_w2: float, Y: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Y [M, N] bf16 = SiLU(sa*A x s1*W1) * (sa*A x s2*W2) from E4M3 A [M, K] and the packed weight."""
    _dev_fp8(A, "A")
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    if Wpacked.numel() * Wpacked.element_size() < swiglu_packed_weight_bytes_fp8(K, N):
        raise ValueError("Wpacked does not hold a packed FP8 weight for this K and N")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _dev_bf16(Y, "Y")
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [M, N]")
    with _on_device(A.device):
        _check(lib.swiglu_forward_fp8(A.data_ptr(), Wpacked.data_ptr(), Y.data_ptr(), M, K, N,
                                      float(scale_a), float(scale_w1), float(scale_w2),
                                      _stream_handle(stream, A.device)),
               "swiglu_forward_fp8")
    return Y


def _dev_u8(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.uint8:
        raise ValueError(f"{name} must be uint8 (UE8M0 scale bytes), got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def swiglu_packed_weight_bytes_mxfp8(K: int, N: int) -> int:
    return int(lib.swiglu_packed_weight_bytes_mxfp8(int(K), int(N)))


def swiglu_act_scale_bytes_mxfp8(M: int, K: int) -> int:
    return int(lib.swiglu_act_scale_bytes_mxfp8(int(M), int(K)))


def swiglu_pack_weights_mxfp8(W1: torch.Tensor, S1: torch.Tensor, W2: torch.Tensor,
                              S2: torch.Tensor, Wpacked: torch.Tensor | None = None,
                              stream=None) -> torch.Tensor:
    """Packed block-scaled weight (flat uint8) from E4M3 W1, W2 [K, N] and UE8M0 S1, S2 [K/32, N]."""
    _dev_fp8(W1, "W1")
    _dev_fp8(W2, "W2")
    _dev_u8(S1, "S1")
    _dev_u8(S2, "S2")
    if W1.dim() != 2 or W1.shape != W2.shape:
        raise ValueError("W1 and W2 must both be [K, N]")
    K, N = W1.shape
    if tuple(S1.shape) != (K // 32, N) or tuple(S2.shape) != (K // 32, N):
        raise ValueError("S1 and S2 must be [K/32, N]")
    if Wpacked is None:
        Wpacked = torch.empty(swiglu_packed_weight_bytes_mxfp8(K, N), dtype=torch.uint8,
                              device=W1.device)
    if Wpacked.numel() * Wpacked.element_size() < swiglu_packed_weight_bytes_mxfp8(K, N):
        raise ValueError("Wpacked is too small")
    with _on_device(W1.device):
        _check(lib.swiglu_pack_weights_mxfp8(W1.data_ptr(), S1.data_ptr(), W2.data_ptr(),
                                             S2.data_ptr(), Wpacked.data_ptr(), K, N,
                                             _stream_handle(stream, W1.device)),
               "swiglu_pack_weights_mxfp8")
    return Wpacked


def swiglu_pack_act_scales_mxfp8(SA: torch.Tensor, SAtiled: torch.Tensor | None = None,
                                 stream=None) -> torch.Tensor:
    """A's UE8M0 scales [M, K/32] in the 512-byte block layout the forward reads."""
    _dev_u8(SA, "SA")
    if SA.dim() != 2:
        raise ValueError("SA must be [M, K/32]")
    M, K = SA.shape[0], 32 * SA.shape[1]
    if SAtiled is None:
        SAtiled = torch.empty(max(swiglu_act_scale_bytes_mxfp8(M, K), 16), dtype=torch.uint8,
                              device=SA.device)
    if SAtiled.numel() * SAtiled.element_size() < swiglu_act_scale_bytes_mxfp8(M, K):
        raise ValueError("SAtiled is too small")
    with _on_device(SA.device):
        _check(lib.swiglu_pack_act_scales_mxfp8(SA.data_ptr(), SAtiled.data_ptr(), M, K,
                                                _stream_handle(stream, SA.device)),
               "swiglu_pack_act_scales_mxfp8")
    return SAtiled


def swiglu_forward_mxfp8(A: torch.Tensor, SAtiled: torch.Tensor, Wpacked: torch.Tensor, N: int,
                         Y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y [M, N] bf16 = SiLU(A x W1) * (A x W2) from block-scaled E4M3 A [M, K] and the packed weight."""
    _dev_fp8(A, "A")
    if A.dim() != 2:
        raise ValueError("A must be [M, K]")
    M, K = A.shape
    if Wpacked.numel() * Wpacked.element_size() < swiglu_packed_weight_bytes_mxfp8(K, N):
        raise ValueError("Wpacked does not hold a packed block-scaled weight for this K and N")
    if SAtiled.numel() * SAtiled.element_size() < swiglu_act_scale_bytes_mxfp8(M, K):
        raise ValueError("SAtiled does not hold A's scales for this M and K")
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _dev_bf16(Y, "Y")
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [M, N]")
    with _on_device(A.device):
        _check(lib.swiglu_forward_mxfp8(A.data_ptr(), SAtiled.data_ptr(), Wpacked.data_ptr(),
                                        Y.data_ptr(), M, K, N, _stream_handle(stream, A.device)),
               "swiglu_forward_mxfp8")
    return Y


def swiglu_plan_string_mxfp8(M: int, K: int, N: int) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(lib.swiglu_plan_string_mxfp8(int(M), int(K), int(N), buf, 256),
           "swiglu_plan_string_mxfp8")
    return buf.value.decode()


def swiglu_down_packed_bytes(N: int, H: int) -> int:
    return int(lib.swiglu_down_packed_bytes(int(N), int(H)))


def swiglu_pack_down_weights(W3: torch.Tensor, W3packed: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """Packed down-projection weight (flat bf16 buffer) from W3 [N, H] (bf16, CUDA)."""
    _dev_bf16(W3, "W3")
    if W3.dim() != 2:
        raise ValueError("W3 must be [N, H]")
    N, H = W3.shape
    if W3packed is None:
        W3packed = torch.empty(swiglu_down_packed_bytes(N, H) // 2, dtype=torch.bfloat16,
                               device=W3.device)
    _dev_bf16(W3packed, "W3packed")
    if W3packed.numel() * 2 < swiglu_down_packed_bytes(N, H):
        raise ValueError("W3packed is too small")
    with _on_device(W3.device):
        _check(lib.swiglu_pack_down_weights(W3.data_ptr(), W3packed.data_ptr(), N, H,
                                            _stream_handle(stream, W3.device)),
               "swiglu_pack_down_weights")
    return W3packed


def swiglu_plan_string_fp8(M: int, K: int, N: int) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(lib.swiglu_plan_string_fp8(int(M), int(K), int(N), buf, 256), "swiglu_plan_string_fp8")
    return buf.value.decode()


def swiglu_down_plan_string(M: int, N: int, H: int) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(lib.swiglu_down_plan_string(int(M), int(N), int(H), buf, 256),
           "swiglu_down_plan_string")
    return buf.value.decode()


def swiglu_down_plan_string_ws(M: int, N: int, H: int) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(lib.swiglu_down_plan_string_ws(int(M), int(N), int(H), buf, 256),
           "swiglu_down_plan_string_ws")
    return buf.value.decode()


def swiglu_down_workspace_bytes(M: int, N: int, H: int) -> int:
    return int(lib.swiglu_down_workspace_bytes(int(M), int(N), int(H)))


def swiglu_down_workspace(M: int, N: int, H: int, device=None) -> torch.Tensor | None:
    """A zero-filled workspace for swiglu_down_forward(..., workspace=) at (M, N, H), or None.

    One workspace serves any number of calls in stream order (each call leaves
    its counters at zero); calls that may overlap in time need one each.
    """
    if device is None:
        device = torch.device("cuda", torch.cuda.current_device())
    device = torch.device(device)
    with _on_device(device):
        n = swiglu_down_workspace_bytes(M, N, H)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def swiglu_down_forward(Y: torch.Tensor, W3packed: torch.Tensor, H: int,
                        R: torch.Tensor | None = None, Out: torch.Tensor | None = None,
                        stream=None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Out [M, H] = Y [M, N] x W3 + R (R optional; Out may be R for an in-place add).

    With `workspace` (from swiglu_down_workspace, on Y's device) the decode
    kernel may also split K across clusters (swiglu_down_forward_ws).
    """
    _dev_bf16(Y, "Y")
    _dev_bf16(W3packed, "W3packed")
    if Y.dim() != 2:
        raise ValueError("Y must be [M, N]")
    M, N = Y.shape
    if W3packed.numel() * 2 < swiglu_down_packed_bytes(N, H):
        raise ValueError("W3packed does not hold a packed W3 for this N and H")
    if R is not None:
        _dev_bf16(R, "R")
        if tuple(R.shape) != (M, H):
            raise ValueError("R must be [M, H]")
    if Out is None:
        Out = torch.empty((M, H), dtype=torch.bfloat16, device=Y.device)
    _dev_bf16(Out, "Out")
    if tuple(Out.shape) != (M, H):
        raise ValueError("Out must be [M, H]")
    if workspace is not None:
        if not workspace.is_cuda or workspace.device != Y.device or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor on Y's device")
        with _on_device(Y.device):
            _check(lib.swiglu_down_forward_ws(
                Y.data_ptr(), W3packed.data_ptr(), R.data_ptr() if R is not None else None,
                Out.data_ptr(), M, N, H, workspace.data_ptr(),
                workspace.numel() * workspace.element_size(), _stream_handle(stream, Y.device)),
                "swiglu_down_forward_ws")
        return Out
    with _on_device(Y.device):
        _check(lib.swiglu_down_forward(Y.data_ptr(), W3packed.data_ptr(),
                                       R.data_ptr() if R is not None else None, Out.data_ptr(),
                                       M, N, H, _stream_handle(stream, Y.device)),
               "swiglu_down_forward")
    return Out


def swiglu_forward_from_host(A_host: torch.Tensor, Wpacked: torch.Tensor, N: int,
                             Y_host: torch.Tensor, A_dev: torch.Tensor, Y_dev: torch.Tensor,
                             stream=None) -> torch.Tensor:
    """Host A -> device, fused forward, device Y -> host, all enqueued on `stream`."""
    for t, name in ((A_host, "A_host"), (Y_host, "Y_host")):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 host tensor")
    _dev_bf16(Wpacked, "Wpacked")
    _dev_bf16(A_dev, "A_dev")
    _dev_bf16(Y_dev, "Y_dev")
    M, K = A_host.shape
    if tuple(A_dev.shape) != (M, K) or tuple(Y_host.shape) != (M, N) or tuple(Y_dev.shape) != (M, N):
        raise ValueError("shape mismatch between host and device buffers")
    with _on_device(A_dev.device):
        _check(lib.swiglu_forward_from_host(A_host.data_ptr(), Wpacked.data_ptr(), Y_host.data_ptr(),
                                            A_dev.data_ptr(), Y_dev.data_ptr(), M, K, N,
                                            _stream_handle(stream, A_dev.device)),
               "swiglu_forward_from_host")
    return Y_host


def swiglu_forward_noalloc(A: torch.Tensor, Wpacked: torch.Tensor, N: int, Y: torch.Tensor,
                           status_out=None, stream=None) -> torch.Tensor:
    """Allocation-free decode forward (M <= 256) into a caller-provided Y.

    `status_out`: optional host buffer of 4 x 32-bit words that receives the
    kernel's status record once the stream synchronises: a ctypes uint32
    array, or a CPU int32 tensor (page-locked keeps the copy asynchronous).
    """
    _dev_bf16(A, "A")
    _dev_bf16(Wpacked, "Wpacked")
    _dev_bf16(Y, "Y")
    M, K = A.shape
    if tuple(Y.shape) != (M, N):
        raise ValueError("Y must be [M, N]")
    if status_out is None:
        ptr = None
    elif isinstance(status_out, torch.Tensor):
        if (status_out.is_cuda or status_out.dtype != torch.int32 or status_out.numel() < 4
                or not status_out.is_contiguous()):
            raise ValueError("status_out must be a contiguous host int32 tensor of 4 words")
        ptr = status_out.data_ptr()
    else:
        if ctypes.sizeof(status_out) < 16:
            raise ValueError("status_out must hold 4 x uint32")
        ptr = ctypes.addressof(status_out)
    with _on_device(A.device):
        _check(lib.swiglu_forward_noalloc(A.data_ptr(), Wpacked.data_ptr(), Y.data_ptr(), M, K, N,
                                          ptr, _stream_handle(stream, A.device)),
               "swiglu_forward_noalloc")
    return Y


def swiglu_check_device_status(stream=None, device=None) -> None:
    """Synchronises the stream; raises SwigluError if a kernel reported a timeout."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        _check(lib.swiglu_check_device_status(_stream_handle(stream, device)),
               "swiglu_check_device_status")


def swiglu_plan_string(M: int, K: int, N: int, variant: int = SWIGLU_VARIANT_AUTO) -> str:
    buf = ctypes.create_string_buffer(256)
    _check(lib.swiglu_plan_string(int(M), int(K), int(N), int(variant), buf, 256),
           "swiglu_plan_string")
    return buf.value.decode()


def swiglu_testing_inject_stall(enable: bool, timeout_ms: int = 0) -> None:
    lib.swiglu_testing_inject_stall(1 if enable else 0, int(timeout_ms))


def swiglu_testing_pace_run_out() -> int:
    """Pacing waits of the CTA-pair kernel that ran out on the current device."""
    v = ctypes.c_uint64(0)
    _check(lib.swiglu_testing_pace_run_out(ctypes.byref(v)), "swiglu_testing_pace_run_out")
    return v.value
