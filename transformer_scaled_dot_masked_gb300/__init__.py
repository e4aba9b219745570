"""GB300 (sm_103a) masked scaled dot-product multi-head attention.

    out = attn_fwd(q, k, v, key_lengths, mask_kind, scale)
    out, lse = attn_fwd_lse(q, k, v, key_lengths, mask_kind, scale)
    dq, dk, dv = attn_bwd(q, k, v, out, dout, lse, key_lengths, mask_kind, scale)
    out = attn_decode(q_new, k_cache, v_cache, cache_lengths, scale)

computes softmax(scale * Q K^T + M) V for every (batch, head) on the GPU, and
its gradients (the chain rule of that equation),
through the C ABI in ``include/attn.h`` ("Paper Deep Reading: Attention Is All
You Need", §04 attention equation with the additive mask M).  Importing the
package fails when the CUDA library has not been built.
"""
from __future__ import annotations

from typing import Optional

from . import _native
from ._native import (AttnError, KERNEL_AUTO, KERNEL_FLASH, KERNEL_SHORT, KERNEL_SIMT, KERNEL_WIDE, KERNEL_RESIDENT, MASK_CAUSAL,
                      MASK_KEY_PADDING, MASK_NONE, MASK_WINDOW, DTYPE_BF16, DTYPE_FP32, SCALE_DEFAULT)

__all__ = ["attn_fwd", "attn_fwd_host", "host_workspace_size", "attn_mha_fwd", "mha_workspace_size", "attn_fwd_window", "attn_fwd_lse", "MASK_WINDOW", "attn_bwd", "bwd_workspace_size", "attn_decode", "decode_workspace_size", "AttnError", "select_kernel", "device_status", "make_workspace", "workspace_size", "MASK_NONE", "MASK_KEY_PADDING",
           "MASK_CAUSAL", "KERNEL_AUTO", "KERNEL_FLASH", "KERNEL_SHORT", "KERNEL_SIMT", "KERNEL_WIDE", "KERNEL_RESIDENT"]


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise TypeError(f"attn_fwd supports bfloat16 and float32 tensors, got {t.dtype}")


def workspace_size() -> int:
    """Bytes of device workspace ``attn_fwd(..., workspace=...)`` needs."""
    return _native.workspace_size()


def make_workspace(device=None):
    """A zero-filled workspace for ``attn_fwd(..., workspace=...)`` (torch allocation)."""
    import torch
    return torch.zeros(workspace_size(), dtype=torch.uint8, device=device or "cuda")


def attn_fwd(q, k, v, key_lengths=None, mask_kind: int = MASK_NONE, scale: Optional[float] = None,
             out=None, kernel: int = KERNEL_AUTO, stream=None, workspace=None):
    """Masked scaled dot-product attention over [B, h, len, d_k] CUDA tensors.

    q: [B, h, m, d_k]; k, v: [B, h, n, d_k]; same dtype (bf16 or fp32), contiguous,
    on the current CUDA device.  key_lengths: int32 [B] CUDA tensor (needed for
    MASK_KEY_PADDING).  scale defaults to 1/sqrt(d_k), which the library computes (ATTN_SCALE_DEFAULT).  out: optional preallocated
    [B, h, m, d_k] tensor.  Enqueued on ``stream`` (default: torch's current stream).
    workspace: optional zero-filled CUDA buffer from ``make_workspace`` (selects the
    dynamic tile schedule, attn_fwd_ws; not combinable with an explicit kernel).
    Calls that may overlap on the GPU need different workspaces.
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, len, d_k]")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, h, m, d = q.shape
    n = k.shape[2]
    if k.shape != (B, h, n, d) or v.shape != k.shape or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError(f"shape/dtype mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = SCALE_DEFAULT
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or not out.is_cuda:
        raise ValueError("out must be a contiguous CUDA tensor shaped and typed like q")
    lens_ptr = None
    if mask_kind & MASK_KEY_PADDING:
        if key_lengths is None or key_lengths.dtype != torch.int32 or not key_lengths.is_cuda \
                or key_lengths.numel() != B:
            raise ValueError("key padding needs key_lengths: int32 CUDA tensor of B elements")
        lens_ptr = key_lengths.data_ptr()
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    dims = _native.make_dims(B, h, m, n, d, _dtype_code(q))
    if workspace is not None:
        if kernel != KERNEL_AUTO:
            raise ValueError("a workspace call always uses the automatic kernel choice")
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        st = _native.fwd_ws_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), lens_ptr, mask_kind, scale,
                                out.data_ptr(), dims, stream.cuda_stream, workspace.data_ptr(),
                                workspace.numel() * workspace.element_size())
    else:
        st = _native.fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), lens_ptr, mask_kind, scale,
                             out.data_ptr(), dims, stream.cuda_stream, kernel)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return out


def host_workspace_size(B, h, m, n, d, dtype: int = DTYPE_BF16) -> int:
    """Bytes of device workspace attn_fwd_host needs (0 for invalid sizes)."""
    return _native.host_workspace_size(_native.make_dims(B, h, m, n, d, dtype))


def attn_fwd_host(q, k, v, key_lengths=None, mask_kind: int = MASK_NONE, scale: Optional[float] = None,
                  out=None, workspace=None, stream=None, device=None):
    """attn_fwd on host (CPU) tensors: the C-ABI call copies the inputs in, runs the
    kernels and copies the output back, chunk by chunk so that the three overlap.

    q: [B, h, m, d_k]; k, v: [B, h, n, d_k] contiguous CPU tensors (bf16 or fp32; pinned
    memory for full-speed asynchronous copies).  key_lengths: int32 [B] CPU tensor
    (needed for MASK_KEY_PADDING).  out: optional preallocated CPU tensor.  workspace:
    optional CUDA uint8 buffer of at least host_workspace_size(...) bytes (allocated on
    ``device`` when omitted).  Enqueued on ``stream`` (default: torch's current stream on
    the device); ``out`` is valid after that stream is synchronised.
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, len, d_k]")
    for t in (q, k, v):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CPU tensors")
    B, h, m, d = q.shape
    n = k.shape[2]
    if k.shape != (B, h, n, d) or v.shape != k.shape or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError(f"shape/dtype mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    if scale is None:
        scale = SCALE_DEFAULT
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.is_cuda:
        raise ValueError("out must be a contiguous CPU tensor shaped and typed like q")
    lens_ptr = None
    if mask_kind & MASK_KEY_PADDING:
        if key_lengths is None or key_lengths.dtype != torch.int32 or key_lengths.is_cuda \
                or key_lengths.numel() != B or not key_lengths.is_contiguous():
            raise ValueError("key padding needs key_lengths: contiguous int32 CPU tensor of B elements")
        lens_ptr = key_lengths.data_ptr()
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    dims = _native.make_dims(B, h, m, n, d, _dtype_code(q))
    need = _native.host_workspace_size(dims)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    elif not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    with torch.cuda.device(workspace.device):
        st = _native.fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), lens_ptr, mask_kind, scale,
                                  out.data_ptr(), dims, workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), stream.cuda_stream)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return out


def select_kernel(B, h, m, n, d, dtype: int, mask_kind: int) -> int:
    return _native.select_kernel(B, h, m, n, d, dtype, mask_kind)


def device_status(stream=None):
    """(status, info) of the bounded-wait record; synchronises the stream."""
    return _native.device_status(None if stream is None else stream.cuda_stream)


def _check_qkv(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, h, len, d_k]")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, h, m, d = q.shape
    n = k.shape[2]
    if k.shape != (B, h, n, d) or v.shape != k.shape or q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError(f"shape/dtype mismatch: q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return B, h, m, n, d


def _lengths_ptr(key_lengths, mask_kind, B):
    import torch
    if not mask_kind & MASK_KEY_PADDING:
        return None
    if key_lengths is None or key_lengths.dtype != torch.int32 or not key_lengths.is_cuda \
            or key_lengths.numel() != B:
        raise ValueError("key padding needs key_lengths: int32 CUDA tensor of B elements")
    return key_lengths.data_ptr()


def _like(t, ref, name):
    if t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA tensor shaped and typed like {tuple(ref.shape)}")


def attn_fwd_lse(q, k, v, key_lengths=None, mask_kind: int = MASK_NONE, scale: Optional[float] = None,
                 out=None, lse=None, stream=None):
    """attn_fwd that also returns each query row's log-sum-exp (float32 [B, h, m], natural log),
    the statistic ``attn_bwd`` needs.  Returns (out, lse)."""
    import torch
    B, h, m, n, d = _check_qkv(q, k, v)
    scale = SCALE_DEFAULT if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    _like(out, q, "out")
    if lse is None:
        lse = torch.empty((B, h, m), dtype=torch.float32, device=q.device)
    elif lse.shape != (B, h, m) or lse.dtype != torch.float32 or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, h, m]")
    stream = torch.cuda.current_stream(q.device) if stream is None else stream
    dims = _native.make_dims(B, h, m, n, d, _dtype_code(q))
    st = _native.fwd_lse_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), _lengths_ptr(key_lengths, mask_kind, B),
                             mask_kind, scale, out.data_ptr(), lse.data_ptr(), dims, stream.cuda_stream)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return out, lse


def bwd_workspace_size(B, h, m, n, d, dtype: int = DTYPE_BF16) -> int:
    """Bytes of device workspace ``attn_bwd`` needs (0: those dims are not supported)."""
    return _native.bwd_workspace_size(_native.make_dims(B, h, m, n, d, dtype))


def attn_bwd(q, k, v, out, dout, lse, key_lengths=None, mask_kind: int = MASK_NONE,
             scale: Optional[float] = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out) for out = attention(q, k, v), bf16 with d_k a
    multiple of 8 up to 64.

    out and lse come from ``attn_fwd_lse`` on the same inputs, mask and scale.
    workspace: optional CUDA uint8 buffer of at least ``bwd_workspace_size(...)`` bytes
    (allocated per call otherwise); calls that may overlap on the GPU need different ones.
    """
    import torch
    B, h, m, n, d = _check_qkv(q, k, v)
    scale = SCALE_DEFAULT if scale is None else scale
    _like(out, q, "out")
    _like(dout, q, "dout")
    if lse.shape != (B, h, m) or lse.dtype != torch.float32 or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, h, m]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _like(dq, q, "dq")
    _like(dk, k, "dk")
    _like(dv, v, "dv")
    dims = _native.make_dims(B, h, m, n, d, _dtype_code(q))
    need = _native.bwd_workspace_size(dims)
    if need == 0:
        raise AttnError(3)  # ATTN_ERR_DTYPE: the backward runs bf16 with d_k a multiple of 8 up to 64
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    stream = torch.cuda.current_stream(q.device) if stream is None else stream
    st = _native.bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                         lse.data_ptr(), _lengths_ptr(key_lengths, mask_kind, B), mask_kind, scale,
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), dims, stream.cuda_stream)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return dq, dk, dv


def decode_workspace_size(B, h, m, n, d=64, dtype: int = DTYPE_BF16) -> int:
    """Bytes of device workspace ``attn_decode`` needs on the current device (0: none)."""
    return _native.decode_workspace_size(_native.make_dims(B, h, m, n, d, dtype))


def attn_decode(q, k_cache, v_cache, cache_lengths=None, scale: Optional[float] = None, out=None, lse=None,
                workspace=None, stream=None):
    """m (1..8) new query rows per (batch, head) against cached keys/values (bf16, d_k 16, 32,
    64 or 128).

    q: [B, h, m, d_k]; k_cache, v_cache: [B, h, n, d_k] (n = capacity); cache_lengths: int32 [B]
    CUDA tensor of valid cached rows per batch entry (None: all n).  Same result as
    ``attn_fwd`` with MASK_KEY_PADDING.  lse: optional float32 [B, h, m] output.
    """
    import torch
    B, h, m, n, d = _check_qkv(q, k_cache, v_cache)
    scale = SCALE_DEFAULT if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    _like(out, q, "out")
    lens_ptr = None
    if cache_lengths is not None:
        lens_ptr = _lengths_ptr(cache_lengths, MASK_KEY_PADDING, B)
    if lse is not None and (lse.shape != (B, h, m) or lse.dtype != torch.float32 or not lse.is_cuda
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, h, m]")
    dims = _native.make_dims(B, h, m, n, d, _dtype_code(q))
    need = _native.decode_workspace_size(dims)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    stream = torch.cuda.current_stream(q.device) if stream is None else stream
    st = _native.decode_raw(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), lens_ptr, scale, out.data_ptr(),
                            None if lse is None else lse.data_ptr(), dims,
                            None if workspace is None else workspace.data_ptr(),
                            0 if workspace is None else workspace.numel() * workspace.element_size(),
                            stream.cuda_stream)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return out


def attn_fwd_window(q, k, v, key_lengths=None, mask_kind: int = MASK_WINDOW, window: int = 0,
                    scale: Optional[float] = None, out=None, stream=None):
    """Restricted self-attention: attn_fwd where MASK_WINDOW in mask_kind keeps, for query i,
    the keys j with |i - j| <= window (combinable with MASK_CAUSAL and MASK_KEY_PADDING)."""
    import torch
    B, h, m, n, d = _check_qkv(q, k, v)
    scale = SCALE_DEFAULT if scale is None else scale
    if out is None:
        out = torch.empty_like(q)
    _like(out, q, "out")
    stream = torch.cuda.current_stream(q.device) if stream is None else stream
    dims = _native.make_dims(B, h, m, n, d, _dtype_code(q))
    st = _native.fwd_window_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), _lengths_ptr(key_lengths, mask_kind, B),
                                mask_kind, window, scale, out.data_ptr(), dims, stream.cuda_stream)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return out


def mha_workspace_size(B, h, m, n, d_model) -> int:
    """Bytes of device workspace ``attn_mha_fwd`` needs (0: shapes not supported)."""
    return _native.mha_workspace_size(B, h, m, n, d_model)


def attn_mha_fwd(xq, xkv, wq, wk, wv, wo, h: int, key_lengths=None, mask_kind: int = MASK_NONE,
                 scale: Optional[float] = None, out=None, workspace=None, stream=None):
    """Multi-head attention with its projections (bf16, d_k = 64 or 128, no biases).

    xq [B, m, d_model], xkv [B, n, d_model]; wq, wk, wv [d_model, h * d_k] (head i = columns
    i*d_k .. (i+1)*d_k - 1); wo [h * d_k, d_model]; d_k is read from the shape of wq.
    Returns out [B, m, d_model] = Concat(Attention(xq wq_i, xkv wk_i, xkv wv_i)) wo.
    """
    import torch
    for t in (xq, xkv, wq, wk, wv, wo):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError("inputs must be contiguous bf16 CUDA tensors")
    B, m, dm = xq.shape
    n = xkv.shape[1]
    if wq.dim() != 2 or wq.shape[1] % h:
        raise ValueError("wq must be [d_model, h * d_k]")
    dk = wq.shape[1] // h
    if xkv.shape != (B, n, dm) or wq.shape != (dm, h * dk) or wk.shape != wq.shape or wv.shape != wq.shape \
            or wo.shape != (h * dk, dm):
        raise ValueError("shape mismatch between inputs, projections and h")
    scale = SCALE_DEFAULT if scale is None else scale
    if out is None:
        out = torch.empty_like(xq)
    need = _native.mha_workspace_size(B, h, m, n, dm, dk)
    if need == 0:
        raise AttnError(2)  # ATTN_ERR_SHAPE (or a head width other than 64 and 128)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=xq.device)
    stream = torch.cuda.current_stream(xq.device) if stream is None else stream
    st = _native.mha_raw(xq.data_ptr(), xkv.data_ptr(), wq.data_ptr(), wk.data_ptr(), wv.data_ptr(), wo.data_ptr(),
                         _lengths_ptr(key_lengths, mask_kind, B), mask_kind, scale, out.data_ptr(), B, h, m, n, dm,
                         workspace.data_ptr(), workspace.numel() * workspace.element_size(), stream.cuda_stream,
                         dk)
    if st != _native.ATTN_OK:
        raise AttnError(st)
    return out

