"""The C-ABI library on the host: it loads, exports what include/attn.h declares,
and rejects bad arguments before touching the GPU (no compute calls here)."""
import ctypes
import re
import subprocess

import pytest

import transformer_scaled_dot_masked_gb300 as attn
from transformer_scaled_dot_masked_gb300 import _native as N

HEADER_TEXT = open(N.HEADER).read()


def _enum(name):
    return int(re.search(rf"\b{name}\s*=\s*(\d+)", HEADER_TEXT).group(1))


def test_library_exports_every_declared_function():
    declared = N.header_exports()
    assert set(declared) >= {"attn_fwd", "attn_fwd_kernel", "attn_select_kernel", "attn_device_status",
                             "attn_status_string", "attn_version"}
    out = subprocess.run(["nm", "-D", "--defined-only", N.LIBRARY], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(\w+)$", out, re.M))
    missing = [f for f in declared if f not in exported]
    assert not missing, f"declared in attn.h but not exported: {missing}"
    for f in declared:
        assert hasattr(N.lib, f)


def test_python_constants_match_header():
    assert N.ATTN_OK == _enum("ATTN_OK")
    assert N.ATTN_ERR_DEVICE_TIMEOUT == _enum("ATTN_ERR_DEVICE_TIMEOUT")
    assert (N.MASK_KEY_PADDING, N.MASK_CAUSAL) == (_enum("ATTN_MASK_KEY_PADDING"), _enum("ATTN_MASK_CAUSAL"))
    assert (N.DTYPE_BF16, N.DTYPE_FP32) == (_enum("ATTN_BF16"), _enum("ATTN_FP32"))
    assert (N.KERNEL_FLASH, N.KERNEL_SHORT, N.KERNEL_SIMT, N.KERNEL_WIDE, N.KERNEL_RESIDENT) == (
        _enum("ATTN_KERNEL_FLASH"), _enum("ATTN_KERNEL_SHORT"), _enum("ATTN_KERNEL_SIMT"),
        _enum("ATTN_KERNEL_WIDE"), _enum("ATTN_KERNEL_RESIDENT"))
    # the dims struct is six int32 fields in this order
    fields = re.search(r"typedef struct \{(.*?)\} attn_dims;", HEADER_TEXT, re.S).group(1)
    assert re.findall(r"int32_t (\w+);", fields) == [f for f, _ in N.AttnDims._fields_]


def test_status_strings_and_version():
    for code in range(0, 12):
        s = N.status_string(code)
        assert s and s != "unknown status"
    assert N.status_string(99) == "unknown status"
    assert N.lib.attn_version() >> 16 == 1


def test_kernel_selection():
    bf, f32 = N.DTYPE_BF16, N.DTYPE_FP32
    assert attn.select_kernel(64, 8, 100, 100, 64, bf, 1) == N.KERNEL_RESIDENT
    assert attn.select_kernel(32, 16, 128, 160, 64, bf, 1) == N.KERNEL_RESIDENT
    assert attn.select_kernel(32, 8, 128, 128, 64, bf, 2) == N.KERNEL_RESIDENT
    assert attn.select_kernel(2, 2, 128, 192, 64, bf, 0) == N.KERNEL_RESIDENT
    assert attn.select_kernel(2, 2, 128, 256, 64, bf, 0) == N.KERNEL_RESIDENT  # the most keys it holds
    assert attn.select_kernel(2, 2, 128, 257, 64, bf, 0) == N.KERNEL_SHORT
    assert attn.select_kernel(2, 2, 129, 100, 64, bf, 0) == N.KERNEL_RESIDENT  # one CTA per query tile
    assert attn.select_kernel(32, 16, 256, 256, 64, bf, 1) == N.KERNEL_RESIDENT
    assert attn.select_kernel(2, 2, 300, 257, 64, bf, 0) == N.KERNEL_FLASH
    assert attn.select_kernel(4, 16, 8192, 8192, 64, bf, 2) == N.KERNEL_FLASH
    assert attn.select_kernel(1, 1, 16, 16, 64, f32, 0) == N.KERNEL_SIMT
    # bf16 heads narrower than 64 (multiples of 8) run zero-padded on tensor cores
    assert attn.select_kernel(1, 1, 16, 16, 32, bf, 0) == N.KERNEL_RESIDENT
    assert attn.select_kernel(1, 1, 300, 300, 16, bf, 2) == N.KERNEL_FLASH
    assert attn.select_kernel(1, 1, 16, 16, 8, bf, 0) == N.KERNEL_RESIDENT
    assert attn.select_kernel(1, 1, 16, 16, 20, bf, 0) == N.KERNEL_SIMT    # not a multiple of 8
    assert attn.select_kernel(1, 1, 16, 16, 128, bf, 0) == N.KERNEL_WIDE   # 128 wide: its own kernel
    assert attn.select_kernel(1, 1, 16, 16, 96, bf, 0) == N.KERNEL_SIMT    # other widths above 64
    assert attn.select_kernel(1, 1, 16, 16, 128, f32, 0) == N.KERNEL_SIMT
    assert attn.select_kernel(1, 1, 16, 17, 64, bf, 2) == N.KERNEL_AUTO   # causal needs m == n
    assert attn.select_kernel(1, 1, 16, 16, 65, bf, 0) == N.KERNEL_SIMT   # d_k > 64: CUDA cores
    assert attn.select_kernel(1, 1, 16, 16, 129, bf, 0) == N.KERNEL_AUTO  # d_k > 128
    assert attn.select_kernel(1, 1, 16, 16, 64, bf, 4) == N.KERNEL_AUTO   # unknown mask bit
    assert attn.select_kernel(0, 1, 16, 16, 64, bf, 0) == N.KERNEL_AUTO


# Fake 16-byte-aligned "device" addresses: validation rejects these calls before
# any CUDA call is made, so nothing is ever dereferenced.
A, B_, C, O, L = 0x1000000, 0x2000000, 0x3000000, 0x4000000, 0x5000000


def _call(q=A, k=B_, v=C, lens=L, mask=0, scale=0.125, out=O, dims=(2, 2, 8, 8, 64, 0), kernel=0):
    d = N.make_dims(*dims)
    return N.fwd_raw(q, k, v, lens, mask, scale, out, d, None, kernel)


@pytest.mark.parametrize("kwargs,status", [
    (dict(q=None), 1), (dict(out=None), 1), (dict(lens=None, mask=1), 1),
    (dict(dims=(0, 2, 8, 8, 64, 0)), 2), (dict(dims=(2, 2, 8, 0, 64, 0)), 2),
    (dict(dims=(2, 2, 8, 9, 64, 0), mask=2), 2), (dict(dims=(70000, 1, 8, 8, 64, 0)), 2),
    (dict(dims=(2, 2, 8, 8, 129, 0)), 3), (dict(dims=(2, 2, 8, 8, 0, 0)), 3), (dict(dims=(2, 2, 8, 8, 64, 7)), 3),
    (dict(mask=4), 4), (dict(mask=-1), 4),
    (dict(q=A + 8), 5), (dict(out=O + 4), 5), (dict(lens=L + 2, mask=1), 5),
    (dict(scale=float("nan")), 9), (dict(scale=float("inf")), 9), (dict(scale=-0.5), 9),
    (dict(scale=-1.0001), 9), (dict(scale=N.SCALE_DEFAULT, q=A + 8), 5),  # the sentinel passes the scale check
    (dict(out=A), 10), (dict(out=B_ + 64), 10), (dict(out=L - 16, mask=1), 10),
])
def test_rejects_bad_arguments(kwargs, status):
    assert _call(**kwargs) == status


def test_rejects_unsupported_kernel_choice():
    # fp32 on a tensor-core kernel, SHORT with m > 128, head widths the tensor-core
    # kernels do not take, unknown kernel id
    assert _call(dims=(2, 2, 8, 8, 64, 1), kernel=N.KERNEL_FLASH) == 6
    assert _call(dims=(2, 2, 200, 200, 64, 0), kernel=N.KERNEL_SHORT) == 6
    assert _call(dims=(2, 2, 8, 8, 20, 0), kernel=N.KERNEL_SHORT) == 6   # d_k not a multiple of 8
    assert _call(dims=(2, 2, 8, 8, 128, 0), kernel=N.KERNEL_FLASH) == 6  # wider than 64
    assert _call(dims=(2, 2, 8, 8, 64, 0), kernel=N.KERNEL_WIDE) == 6    # the wide kernel: d_k 128 only
    assert _call(dims=(2, 2, 8, 8, 128, 1), kernel=N.KERNEL_WIDE) == 6   # and bf16 only
    assert _call(dims=(2, 2, 8, 257, 64, 0), kernel=N.KERNEL_RESIDENT) == 6  # more keys than it holds
    assert _call(dims=(2, 2, 8, 8, 64, 1), kernel=N.KERNEL_RESIDENT) == 6    # fp32
    assert _call(dims=(2, 2, 8, 8, 20, 0), kernel=N.KERNEL_RESIDENT) == 6    # d_k not a multiple of 8
    assert _call(kernel=17) == 6


def test_null_dims():
    assert N.lib.attn_fwd(A, B_, C, None, 0, ctypes.c_float(0.125), O, None, None) == 1


def _call_ws(ws=0x6000000, ws_bytes=None, **kw):
    d = N.make_dims(*(kw.pop("dims", (2, 2, 8, 8, 64, 0))))
    ws_bytes = N.workspace_size() if ws_bytes is None else ws_bytes
    return N.fwd_ws_raw(kw.get("q", A), B_, C, L, kw.get("mask", 0), 0.125, kw.get("out", O), d, None, ws,
                        ws_bytes)


def test_workspace_validation():
    assert N.workspace_size() >= 8
    assert _call_ws(ws=None) == 1
    assert _call_ws(ws_bytes=N.workspace_size() - 1) == 2
    assert _call_ws(ws=0x6000000 + 4) == 5
    assert _call_ws(ws=O + 64) == 10          # inside out
    assert _call_ws(ws=A) == 10               # inside Q
    assert _call_ws(q=A + 8) == 5             # tensor checks still apply
    assert _call_ws(ws=L, mask=1) == 10       # over the key lengths the kernel reads
    assert _call_ws(ws=L - 16, mask=1) == 10


# ---------------------------------------------------------------- host buffers
def _host_size(B, h, m, n, d, dtype):
    """The device workspace attn_fwd_host needs: Q, K, V, out (each rounded up to
    256 bytes), the int32 lengths (rounded up to 256) and two 256-byte tile counters."""
    r = lambda x: (x + 255) // 256 * 256
    esz = 2 if dtype == 0 else 4
    return 2 * r(B * h * m * d * esz) + 2 * r(B * h * n * d * esz) + r(4 * B) + 2 * 256


def test_host_workspace_size():
    for dims in [(2, 3, 300, 200, 64, 0), (1, 1, 1, 1, 1, 1), (9, 2, 100, 100, 64, 0), (3, 4, 37, 53, 3, 1)]:
        assert N.host_workspace_size(N.make_dims(*dims)) == _host_size(*dims)
    assert N.host_workspace_size(N.make_dims(0, 3, 300, 200, 64, 0)) == 0      # bad dims
    assert N.host_workspace_size(N.make_dims(2, 3, 300, 200, 200, 0)) == 0     # d_k too wide


def _call_host(ws=0x6000000, ws_bytes=None, mask=0, lens=None, **kw):
    dims = kw.pop("dims", (2, 2, 8, 8, 64, 0))
    d = N.make_dims(*dims)
    ws_bytes = _host_size(*dims) if ws_bytes is None else ws_bytes
    return N.fwd_host_raw(kw.get("q", A), B_, C, lens, mask, kw.get("scale", 0.125), kw.get("out", O), d, ws,
                          ws_bytes, None)


def test_host_validation():
    assert _call_host(ws=None) == 1                       # workspace NULL
    assert _call_host(q=None) == 1                        # tensor NULL
    assert _call_host(mask=1) == 1                        # padding without lengths
    assert _call_host(ws_bytes=_host_size(2, 2, 8, 8, 64, 0) - 1) == 2
    assert _call_host(ws=0x6000000 + 16) == 5             # workspace not 256-byte aligned
    assert _call_host(out=A + 64) == 10                   # out inside Q
    assert _call_host(out=L - 8, mask=1, lens=L) == 10    # out over the lengths
    assert _call_host(dims=(2, 2, 8, 9, 64, 0), mask=2) == 2   # causal with m != n
    assert _call_host(mask=8) == 4                        # unknown mask bit
    assert _call_host(scale=float("nan")) == 9
    assert _call_host(dims=(2, 2, 8, 8, 64, 7)) == 3      # unknown dtype


# ---------------------------------------------------------------- forward with lse, backward
LSE, DO, OUT2, DQ, DK, DV, WS = 0x7000000, 0x8000000, 0x9000000, 0xA000000, 0xB000000, 0xC000000, 0xD000000


def test_fwd_lse_validation():
    d = N.make_dims(2, 2, 8, 8, 64, 0)
    assert N.fwd_lse_raw(A, B_, C, None, 0, 0.125, O, None, d, None) == 1      # lse NULL
    assert N.fwd_lse_raw(A, B_, C, None, 0, 0.125, O, LSE + 2, d, None) == 5   # lse unaligned
    assert N.fwd_lse_raw(A, B_, C, None, 0, 0.125, O, O + 16, d, None) == 10   # lse inside out
    assert N.fwd_lse_raw(A, B_, C, None, 0, 0.125, O, A, d, None) == 10        # lse inside Q
    assert N.fwd_lse_raw(A + 8, B_, C, None, 0, 0.125, O, LSE, d, None) == 5   # forward checks apply


def test_bwd_workspace_size():
    assert N.bwd_workspace_size(N.make_dims(2, 3, 300, 200, 64, 0)) >= 2 * 3 * 300 * 64 * 4
    assert N.bwd_workspace_size(N.make_dims(2, 3, 300, 200, 32, 0)) >= 2 * 3 * 300 * 64 * 4  # zero-padded
    # CUDA-core backward (fp32, other bf16 widths up to 128): D, one float per query row
    assert N.bwd_workspace_size(N.make_dims(2, 3, 300, 200, 64, 1)) == 2 * 3 * 300 * 4
    assert N.bwd_workspace_size(N.make_dims(2, 3, 300, 200, 20, 0)) == 2 * 3 * 300 * 4
    assert N.bwd_workspace_size(N.make_dims(2, 3, 300, 200, 128, 0)) == 2 * 3 * 300 * 4
    assert N.bwd_workspace_size(N.make_dims(2, 3, 300, 200, 129, 0)) == 0  # wider than any kernel
    assert N.bwd_workspace_size(N.make_dims(0, 3, 300, 200, 64, 0)) == 0   # bad dims


def _call_bwd(dims=(2, 2, 8, 8, 64, 0), mask=0, lens=None, ws_bytes=None, **kw):
    d = N.make_dims(*dims)
    ws_bytes = N.bwd_workspace_size(N.make_dims(2, 2, 8, 8, 64, 0)) if ws_bytes is None else ws_bytes
    a = dict(q=A, k=B_, v=C, out=OUT2, dout=DO, lse=LSE, dq=DQ, dk=DK, dv=DV, ws=WS)
    a.update(kw)
    return N.bwd_raw(a["q"], a["k"], a["v"], a["out"], a["dout"], a["lse"], lens, mask, 0.125, a["dq"],
                     a["dk"], a["dv"], a["ws"], ws_bytes, d, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(out=None), 1), (dict(dout=None), 1), (dict(lse=None), 1), (dict(dq=None), 1), (dict(dk=None), 1),
    (dict(dv=None), 1), (dict(ws=None), 1), (dict(q=None), 1), (dict(mask=1), 1),
    (dict(dims=(2, 2, 8, 8, 129, 0)), 3), (dict(dims=(2, 2, 8, 8, 64, 7)), 3),
    (dict(dims=(2, 2, 8, 9, 64, 0), mask=2), 2), (dict(ws_bytes=64), 2),
    (dict(dout=DO + 8), 5), (dict(dk=DK + 2), 5), (dict(lse=LSE + 1), 5), (dict(ws=WS + 16), 5),
    (dict(dq=A), 10), (dict(dk=DQ + 32), 10), (dict(dv=DO), 10), (dict(ws=LSE), 10), (dict(dv=OUT2 + 16), 10),
])
def test_bwd_rejects_bad_arguments(kwargs, status):
    assert _call_bwd(**kwargs) == status


def _call_dec(dims=(2, 2, 1, 64, 64, 0), lens=L, lse=None, ws=None, ws_bytes=0, **kw):
    d = N.make_dims(*dims)
    return N.decode_raw(kw.get("q", A), kw.get("k", B_), kw.get("v", C), lens, kw.get("scale", 0.125),
                        kw.get("out", O), lse, d, ws, ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(q=None), 1), (dict(out=None), 1),
    (dict(dims=(2, 2, 1, 64, 64, 1)), 3), (dict(dims=(2, 2, 1, 64, 48, 0)), 3), (dict(dims=(2, 2, 1, 64, 8, 0)), 3),
    (dict(dims=(2, 2, 9, 64, 64, 0)), 2), (dict(dims=(2, 2, 0, 64, 64, 0)), 2),
    (dict(q=A + 8), 5), (dict(lens=L + 2), 5), (dict(lse=LSE + 2), 5),
    (dict(scale=float("nan")), 9), (dict(out=B_ + 64), 10), (dict(lse=O + 16), 10),
])
def test_decode_rejects_bad_arguments(kwargs, status):
    assert _call_dec(**kwargs) == status


def test_decode_workspace_size_rejects_bad_dims():
    assert N.decode_workspace_size(N.make_dims(2, 2, 9, 64, 64, 0)) == 0
    assert N.decode_workspace_size(N.make_dims(2, 2, 1, 64, 64, 1)) == 0


def test_window_mask_validation():
    assert N.MASK_WINDOW == _enum("ATTN_MASK_WINDOW")
    d = N.make_dims(2, 2, 8, 8, 64, 0)
    assert N.fwd_raw(A, B_, C, None, N.MASK_WINDOW, 0.125, O, d, None) == 4          # attn_fwd: no window bit
    assert N.fwd_window_raw(A, B_, C, None, N.MASK_WINDOW, -1, 0.125, O, d, None) == 9  # negative window
    assert N.fwd_window_raw(A, B_, C, None, 8, 3, 0.125, O, d, None) == 4              # unknown bit
    d2 = N.make_dims(2, 2, 8, 9, 64, 0)
    assert N.fwd_window_raw(A, B_, C, None, N.MASK_WINDOW, 3, 0.125, O, d2, None) == 2  # m != n
    assert N.fwd_window_raw(A + 8, B_, C, None, N.MASK_WINDOW, 3, 0.125, O, d, None) == 5


def _call_mha(dims=(2, 2, 8, 8, 128), mask=0, lens=None, ws=0xE000000, ws_bytes=None, **kw):
    ws_bytes = N.mha_workspace_size(*dims) if ws_bytes is None else ws_bytes
    a = dict(xq=A, xkv=B_, wq=C, wk=0x7000000, wv=0x8000000, wo=0x9000000, out=O)
    a.update(kw)
    return N.mha_raw(a["xq"], a["xkv"], a["wq"], a["wk"], a["wv"], a["wo"], lens, mask, 0.125, a["out"], *dims,
                     ws, ws_bytes, None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(xq=None), 1), (dict(wo=None), 1), (dict(ws=None), 1), (dict(mask=1), 1),
    (dict(dims=(2, 3, 8, 8, 128)), 2), (dict(dims=(2, 2, 8, 8, 96)), 2), (dict(dims=(2, 2, 8, 9, 128), mask=2), 2),
    (dict(ws_bytes=16), 2), (dict(mask=4), 4), (dict(wq=C + 8), 5), (dict(ws=0xE000000 + 16), 5),
    (dict(out=B_), 10), (dict(ws=0x9000000), 10),
])
def test_mha_rejects_bad_arguments(kwargs, status):
    assert _call_mha(**kwargs) == status


def test_mha_head_width():
    # the dims struct is six int32 fields in this order
    fields = re.search(r"typedef struct \{([^}]*)\} attn_mha_dims;", HEADER_TEXT).group(1)
    assert re.findall(r"int32_t (\w+);", fields) == [f for f, _ in N.MhaDims._fields_]
    assert N.mha_workspace_size(2, 2, 8, 8, 128, 128) == 2 * N.mha_workspace_size(2, 2, 8, 8, 128, 64)
    assert N.mha_workspace_size(2, 2, 8, 8, 128, 0) == N.mha_workspace_size(2, 2, 8, 8, 128, 64)  # 0 reads as 64
    # narrow heads: Q, K, V, O split plus the three concatenated products (O merges into Q's)
    assert N.mha_workspace_size(2, 4, 8, 8, 128, 32) == 7 * N.mha_workspace_size(2, 2, 8, 8, 128, 64) // 4
    assert N.mha_workspace_size(2, 2, 8, 8, 128, 32) == 0                                        # h * d_k = 64
    assert N.mha_workspace_size(2, 8, 8, 8, 128, 20) == 0                                        # not a multiple of 8
    assert N.mha_workspace_size(2, 1, 8, 8, 128, 128) > 0                                        # h * 128
    d = N.MhaDims(2, 2, 8, 8, 128, 96)
    assert N.lib.attn_mha_fwd(A, B_, C, 0x7000000, 0x8000000, 0x9000000, None, 0, ctypes.c_float(0.125), O,
                              ctypes.byref(d), 0xE000000, 1 << 20, None) == 3                   # ATTN_ERR_DTYPE
