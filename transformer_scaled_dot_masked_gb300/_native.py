"""ctypes binding of libattn_gb300.so (argument marshalling only).

Every step of the computation runs in the library's CUDA kernels; this module
turns torch tensors into pointers and shapes, passes the current CUDA stream,
and turns status codes into exceptions.  It raises at import time when the
library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(_PKG, "libattn_gb300.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "attn.h")

if not os.path.exists(LIBRARY):
    raise ImportError(
        f"{LIBRARY} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")

# Keep these in step with include/attn.h (tests/test_abi.py checks them against the header).
ATTN_OK = 0
ATTN_ERR_DEVICE_TIMEOUT = 8
MASK_NONE, MASK_KEY_PADDING, MASK_CAUSAL, MASK_WINDOW = 0, 1, 2, 4
DTYPE_BF16, DTYPE_FP32 = 0, 1
# ATTN_SCALE_DEFAULT: the library substitutes the formula's scale, 1/sqrt(d_k)
SCALE_DEFAULT = -1.0
KERNEL_AUTO, KERNEL_FLASH, KERNEL_SHORT, KERNEL_SIMT, KERNEL_WIDE, KERNEL_RESIDENT = 0, 1, 2, 3, 4, 5
KERNEL_NAMES = {KERNEL_AUTO: "auto", KERNEL_FLASH: "flash", KERNEL_SHORT: "short", KERNEL_SIMT: "simt",
                KERNEL_WIDE: "wide", KERNEL_RESIDENT: "resident"}


class MhaDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("h", ctypes.c_int32), ("m", ctypes.c_int32),
                ("n", ctypes.c_int32), ("d_model", ctypes.c_int32), ("d_k", ctypes.c_int32)]


class AttnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("h", ctypes.c_int32), ("m", ctypes.c_int32),
                ("n", ctypes.c_int32), ("d_k", ctypes.c_int32), ("dtype", ctypes.c_int32)]


lib = ctypes.CDLL(LIBRARY)
_vp = ctypes.c_void_p
lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_float, _vp,
                         ctypes.POINTER(AttnDims), _vp]
lib.attn_fwd.restype = ctypes.c_int
lib.attn_fwd_kernel.argtypes = lib.attn_fwd.argtypes + [ctypes.c_int]
lib.attn_fwd_kernel.restype = ctypes.c_int
lib.attn_workspace_size.argtypes = []
lib.attn_workspace_size.restype = ctypes.c_size_t
lib.attn_fwd_ws.argtypes = lib.attn_fwd.argtypes + [_vp, ctypes.c_size_t]
lib.attn_fwd_ws.restype = ctypes.c_int
lib.attn_fwd_noalloc.argtypes = lib.attn_fwd.argtypes
lib.attn_fwd_host_workspace_size.argtypes = [ctypes.POINTER(AttnDims)]
lib.attn_fwd_host_workspace_size.restype = ctypes.c_size_t
lib.attn_fwd_host.argtypes = lib.attn_fwd.argtypes[:-1] + [_vp, ctypes.c_size_t, _vp]
lib.attn_fwd_host.restype = ctypes.c_int
lib.attn_fwd_noalloc.restype = ctypes.c_int
lib.attn_test_withheld_arrival.argtypes = lib.attn_fwd.argtypes[:-1] + [ctypes.c_uint64, _vp]
lib.attn_test_withheld_arrival.restype = ctypes.c_int
lib.attn_fwd_lse.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_float, _vp, _vp,
                             ctypes.POINTER(AttnDims), _vp]
lib.attn_fwd_lse.restype = ctypes.c_int
lib.attn_bwd_workspace_size.argtypes = [ctypes.POINTER(AttnDims)]
lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
lib.attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_float, _vp, _vp, _vp,
                         _vp, ctypes.c_size_t, ctypes.POINTER(AttnDims), _vp]
lib.attn_bwd.restype = ctypes.c_int
lib.attn_fwd_window.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_float, _vp,
                                ctypes.POINTER(AttnDims), _vp]
lib.attn_fwd_window.restype = ctypes.c_int
lib.attn_mha_workspace_size.argtypes = [ctypes.POINTER(MhaDims)]
lib.attn_mha_workspace_size.restype = ctypes.c_size_t
lib.attn_mha_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_float, _vp,
                             ctypes.POINTER(MhaDims), _vp, ctypes.c_size_t, _vp]
lib.attn_mha_fwd.restype = ctypes.c_int
lib.attn_decode_workspace_size.argtypes = [ctypes.POINTER(AttnDims)]
lib.attn_decode_workspace_size.restype = ctypes.c_size_t
lib.attn_decode.argtypes = [_vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, ctypes.POINTER(AttnDims), _vp,
                            ctypes.c_size_t, _vp]
lib.attn_decode.restype = ctypes.c_int
lib.attn_select_kernel.argtypes = [ctypes.POINTER(AttnDims), ctypes.c_int]
lib.attn_select_kernel.restype = ctypes.c_int
lib.attn_device_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int32)]
lib.attn_device_status.restype = ctypes.c_int
lib.attn_status_string.argtypes = [ctypes.c_int]
lib.attn_status_string.restype = ctypes.c_char_p
lib.attn_version.argtypes = []
lib.attn_version.restype = ctypes.c_int32


class AttnError(RuntimeError):
    def __init__(self, status: int):
        self.status = status
        super().__init__(f"attn status {status}: {status_string(status)}")


def status_string(status: int) -> str:
    return lib.attn_status_string(int(status)).decode()


def header_exports(path: str = HEADER):
    """Function names declared in include/attn.h."""
    text = open(path).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, re.M)))


def make_dims(B, h, m, n, d, dtype: int) -> AttnDims:
    return AttnDims(int(B), int(h), int(m), int(n), int(d), int(dtype))


def select_kernel(B, h, m, n, d, dtype: int, mask_kind: int) -> int:
    dims = make_dims(B, h, m, n, d, dtype)
    return lib.attn_select_kernel(ctypes.byref(dims), int(mask_kind))


def fwd_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, scale, out_ptr, dims: AttnDims, stream_ptr,
            kernel: int = KERNEL_AUTO) -> int:
    """Direct call with integer device pointers; returns the status code."""
    return lib.attn_fwd_kernel(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), float(scale), out_ptr,
                               ctypes.byref(dims), stream_ptr, int(kernel))


def workspace_size() -> int:
    return int(lib.attn_workspace_size())


def fwd_ws_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, scale, out_ptr, dims: AttnDims, stream_ptr,
               ws_ptr, ws_bytes) -> int:
    """attn_fwd_ws with integer device pointers; returns the status code."""
    return lib.attn_fwd_ws(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), float(scale), out_ptr,
                           ctypes.byref(dims), stream_ptr, ws_ptr, int(ws_bytes))


def host_workspace_size(dims: AttnDims) -> int:
    return int(lib.attn_fwd_host_workspace_size(ctypes.byref(dims)))


def fwd_host_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, scale, out_ptr, dims: AttnDims, ws_ptr, ws_bytes,
                 stream_ptr) -> int:
    """attn_fwd_host with integer host pointers (device workspace); returns the status code."""
    return lib.attn_fwd_host(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), float(scale), out_ptr,
                             ctypes.byref(dims), ws_ptr, int(ws_bytes), stream_ptr)


def test_withheld_arrival_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, scale, out_ptr, dims: AttnDims,
                              wait_ns: int, stream_ptr) -> int:
    """attn_test_withheld_arrival (failure-detection test hook); returns the status code."""
    return lib.attn_test_withheld_arrival(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), float(scale), out_ptr,
                                          ctypes.byref(dims), int(wait_ns), stream_ptr)


def fwd_noalloc_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, scale, out_ptr, dims: AttnDims,
                    stream_ptr) -> int:
    """attn_fwd_noalloc with integer device pointers; returns the status code."""
    return lib.attn_fwd_noalloc(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), float(scale), out_ptr,
                                ctypes.byref(dims), stream_ptr)


def fwd_lse_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, scale, out_ptr, lse_ptr, dims: AttnDims,
                stream_ptr) -> int:
    """attn_fwd_lse with integer device pointers; returns the status code."""
    return lib.attn_fwd_lse(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), float(scale), out_ptr, lse_ptr,
                            ctypes.byref(dims), stream_ptr)


def bwd_workspace_size(dims: AttnDims) -> int:
    return int(lib.attn_bwd_workspace_size(ctypes.byref(dims)))


def bwd_raw(q_ptr, k_ptr, v_ptr, out_ptr, dout_ptr, lse_ptr, lens_ptr, mask_kind, scale, dq_ptr, dk_ptr,
            dv_ptr, ws_ptr, ws_bytes, dims: AttnDims, stream_ptr) -> int:
    """attn_bwd with integer device pointers; returns the status code."""
    return lib.attn_bwd(q_ptr, k_ptr, v_ptr, out_ptr, dout_ptr, lse_ptr, lens_ptr, int(mask_kind),
                        float(scale), dq_ptr, dk_ptr, dv_ptr, ws_ptr, int(ws_bytes), ctypes.byref(dims),
                        stream_ptr)


def fwd_window_raw(q_ptr, k_ptr, v_ptr, lens_ptr, mask_kind, window, scale, out_ptr, dims: AttnDims,
                   stream_ptr) -> int:
    """attn_fwd_window with integer device pointers; returns the status code."""
    return lib.attn_fwd_window(q_ptr, k_ptr, v_ptr, lens_ptr, int(mask_kind), int(window), float(scale), out_ptr,
                               ctypes.byref(dims), stream_ptr)


def decode_workspace_size(dims: AttnDims) -> int:
    return int(lib.attn_decode_workspace_size(ctypes.byref(dims)))


def decode_raw(q_ptr, k_ptr, v_ptr, lens_ptr, scale, out_ptr, lse_ptr, dims: AttnDims, ws_ptr, ws_bytes,
               stream_ptr) -> int:
    """attn_decode with integer device pointers; returns the status code."""
    return lib.attn_decode(q_ptr, k_ptr, v_ptr, lens_ptr, float(scale), out_ptr, lse_ptr, ctypes.byref(dims),
                           ws_ptr, int(ws_bytes), stream_ptr)


def mha_workspace_size(B, h, m, n, d_model, d_k=64) -> int:
    d = MhaDims(int(B), int(h), int(m), int(n), int(d_model), int(d_k))
    return int(lib.attn_mha_workspace_size(ctypes.byref(d)))


def mha_raw(xq, xkv, wq, wk, wv, wo, lens_ptr, mask_kind, scale, out_ptr, B, h, m, n, d_model, ws_ptr, ws_bytes,
            stream_ptr, d_k=64) -> int:
    """attn_mha_fwd with integer device pointers; returns the status code."""
    d = MhaDims(int(B), int(h), int(m), int(n), int(d_model), int(d_k))
    return lib.attn_mha_fwd(xq, xkv, wq, wk, wv, wo, lens_ptr, int(mask_kind), float(scale), out_ptr,
                            ctypes.byref(d), ws_ptr, int(ws_bytes), stream_ptr)


def device_status(stream_ptr=None):
    info = ctypes.c_int32(0)
    st = lib.attn_device_status(stream_ptr, ctypes.byref(info))
    return st, info.value
