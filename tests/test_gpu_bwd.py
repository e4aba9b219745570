"""Backward pass and the forward's log-sum-exp on the GPU against the fp64 oracle.

The oracle's gradients are the chain rule of the attention equation (pinned by
finite differences in the CPU tests).  Tolerance of the bf16 backward, from its
arithmetic: every gradient element is a sum of products in which the weights P
and the score gradients dS are rounded to bf16 (relative error up to 2^-8 each)
and the result is rounded to bf16 (2^-8 relative), with fp32 accumulation.  The
tests take a norm-wise bound of 2^-6 of the largest reference magnitude per
tensor for the worst element, and 2^-7 for the relative Frobenius error.  An
absolute floor of 1e-4 covers the fp32 rounding of the cancellation dP - D (a
sum of 64 products of magnitude ~10 each), which is all that remains when the
exact gradient is 0 (a single allowed key gives dS = 0).
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from workloads import WORKLOADS, MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE, Workload, draw, draw_dout

from gpu_helpers import as_f64, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def gpu_grads(inp, dout_bits):
    w = inp.workload
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    do = to_device(dout_bits, w.dtype)
    lens = torch.from_numpy(inp.key_lengths).cuda()
    out, lse = attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, out, do, lse, lens, w.mask, w.scale)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    return out, lse, dq, dk, dv


def check_grad(name, got, ref):
    got, ref = as_f64(got) if torch.is_tensor(got) else got, ref
    scale = max(np.abs(ref).max(), 1e-30)
    err = np.abs(got - ref)
    frob = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    assert err.max() <= 2.0 ** -6 * scale + 1e-4, f"{name}: max err {err.max():.3e} vs max |ref| {scale:.3e}"
    assert frob <= 2.0 ** -7 or np.linalg.norm(got - ref) <= 1e-4 * np.sqrt(ref.size), \
        f"{name}: relative Frobenius error {frob:.3e}"
    print(f"{name}: max err / max|ref| = {err.max() / scale:.2e}, relative Frobenius {frob:.2e}")
    return err.max() / scale, frob


BWD_CASES = [
    # name, B, h, m, n, mask, lengths
    ("self_causal_ragged", 2, 2, 300, 300, MASK_CAUSAL, None),
    ("self_none_exact_tiles", 1, 2, 256, 256, MASK_NONE, None),
    ("cross_padding_ragged", 3, 2, 200, 333, MASK_KEY_PADDING, (0, 333)),
    ("self_padding_causal", 2, 3, 130, 130, MASK_KEY_PADDING | MASK_CAUSAL, (1, 130)),
    ("single_query_tile", 4, 2, 77, 150, MASK_KEY_PADDING, (0, 150)),
    ("one_key", 2, 1, 40, 1, MASK_NONE, None),
]


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths", BWD_CASES, ids=[c[0] for c in BWD_CASES])
def test_bwd_matches_oracle(orc, name, B, h, m, n, mask, lengths):
    w = Workload(name, "bf16", B, h, m, n, 64, mask, 0.125, 77, lengths)
    inp = draw(w)
    dout = draw_dout(w)
    _, lse, dq, dk, dv = gpu_grads(inp, dout)
    rq, rk, rv = orc.attn_bwd(inp.q, inp.k, inp.v, dout, inp.key_lengths, w.mask, w.scale)
    check_grad("dV", dv, rv)
    check_grad("dK", dk, rk)
    check_grad("dQ", dq, rq)
    ref_lse = orc.attn_lse(inp.q, inp.k, inp.key_lengths, w.mask, w.scale)
    got_lse = lse.cpu().numpy().astype(np.float64)
    live = np.isfinite(ref_lse)
    assert (got_lse[~live] == -np.inf).all()
    assert np.abs(got_lse[live] - ref_lse[live]).max() <= 1e-3


NARROW_BWD = [
    # heads narrower than 64 (the model-variant table's d_k = 32 and 16, and other
    # multiples of 8): zero-padded to 64 inside the kernels, only d_k columns written
    ("d16_causal_ragged", 2, 2, 300, 300, 16, MASK_CAUSAL, None),
    ("d32_cross_padding", 3, 2, 200, 333, 32, MASK_KEY_PADDING, (0, 333)),
    ("d8_padding_causal", 2, 3, 130, 130, 8, MASK_KEY_PADDING | MASK_CAUSAL, (1, 130)),
    ("d48_short_heads", 4, 2, 100, 150, 48, MASK_KEY_PADDING, (0, 150)),
]


@pytest.mark.parametrize("name,B,h,m,n,d,mask,lengths", NARROW_BWD, ids=[c[0] for c in NARROW_BWD])
def test_bwd_narrow_heads(orc, name, B, h, m, n, d, mask, lengths):
    """Gradients of narrower heads against the oracle, written exactly into their
    [B, h, len, d_k] outputs (guard regions on both sides of each stay untouched)."""
    w = Workload(name, "bf16", B, h, m, n, d, mask, d ** -0.5, 78, lengths)
    inp = draw(w)
    dout = draw_dout(w)
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    do = to_device(dout, w.dtype)
    lens = torch.from_numpy(inp.key_lengths).cuda()
    out, lse = attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale)
    guard = 4096
    bufs, grads = [], []
    for like in (q, k, v):
        buf = torch.full((like.numel() + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
        bufs.append(buf)
        grads.append(buf[guard:guard + like.numel()].view(like.shape))
    attn.attn_bwd(q, k, v, out, do, lse, lens, w.mask, w.scale, dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    for buf in bufs:
        assert (buf[:guard] == -7.0).all() and (buf[-guard:] == -7.0).all()
    rq, rk, rv = orc.attn_bwd(inp.q, inp.k, inp.v, dout, inp.key_lengths, w.mask, w.scale)
    check_grad("dV", grads[2], rv)
    check_grad("dK", grads[1], rk)
    check_grad("dQ", grads[0], rq)


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_bwd_workloads(orc, cfg):
    w = WORKLOADS[cfg]
    inp = draw(w)
    dout = draw_dout(w)
    _, _, dq, dk, dv = gpu_grads(inp, dout)
    rq, rk, rv = orc.attn_bwd(inp.q, inp.k, inp.v, dout, inp.key_lengths, w.mask, w.scale)
    for name, g, r in (("dV", dv, rv), ("dK", dk, rk), ("dQ", dq, rq)):
        check_grad(name, g, r)


def test_bwd_long_causal_sampled_heads(orc):
    """B4 h16 n=m=8192 causal at full size; the oracle computes two whole heads."""
    w = WORKLOADS[5]
    inp = draw(w)
    dout = draw_dout(w)
    _, _, dq, dk, dv = gpu_grads(inp, dout)
    heads = np.array([0, w.B * w.h - 1])
    rq, rk, rv = orc.attn_bwd(inp.q, inp.k, inp.v, dout, inp.key_lengths, w.mask, w.scale, heads=heads)
    for name, g, r in (("dV", dv, rv), ("dK", dk, rk), ("dQ", dq, rq)):
        g = as_f64(g).reshape(w.B * w.h, -1, w.d)[heads]
        r = r.reshape(w.B * w.h, -1, w.d)[heads]
        check_grad(name, g, r)


def test_fwd_lse_on_every_kernel(orc):
    """lse from each forward kernel (and the output unchanged by asking for it)."""
    for w, kernels in ((Workload("lse_bf16", "bf16", 2, 3, 300, 300, 64, MASK_CAUSAL | MASK_KEY_PADDING,
                                 0.125, 5, (0, 300)), ["flash", "short", "simt"]),
                       (Workload("lse_fp32", "fp32", 2, 2, 50, 70, 33, MASK_KEY_PADDING, 0.2, 6, (0, 70)),
                        ["simt"])):
        inp = draw(w)
        q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
        lens = torch.from_numpy(inp.key_lengths).cuda()
        ref = orc.attn_lse(inp.q, inp.k, inp.key_lengths, w.mask, w.scale)
        out, lse = attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale)
        plain = attn.attn_fwd(q, k, v, lens, w.mask, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out, plain)
        got = lse.cpu().numpy().astype(np.float64)
        live = np.isfinite(ref)
        assert (got[~live] == -np.inf).all()
        assert np.abs(got[live] - ref[live]).max() <= 1e-3


def test_bwd_masked_keys_get_zero_and_dkdv_reproducible():
    """Keys no query may see get exactly zero gradients; dK and dV are bitwise
    reproducible (dQ sums tiles with atomics, so only its value is checked)."""
    w = Workload("zeros", "bf16", 3, 2, 200, 300, 64, MASK_KEY_PADDING, 0.125, 9, (0, 300))
    inp = draw(w)
    inp.key_lengths[:] = [0, 129, 300]
    dout = draw_dout(w)
    _, _, dq1, dk1, dv1 = gpu_grads(inp, dout)
    _, _, dq2, dk2, dv2 = gpu_grads(inp, dout)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dk1[0] == 0).all() and (dv1[0] == 0).all() and (dq1[0] == 0).all()
    assert (dk1[1, :, 129:] == 0).all() and (dv1[1, :, 129:] == 0).all()
    assert torch.allclose(dq1.float(), dq2.float(), atol=1e-2)


SIMT_BWD = [
    # the CUDA-core backward: heads of width 128 (the model-variant table's h = 4 row),
    # other bf16 widths, and fp32 (true fp32: its bound is far tighter than bf16's)
    ("d128_causal_ragged", "bf16", 2, 2, 300, 300, 128, MASK_CAUSAL, None),
    ("d128_cross_padding", "bf16", 3, 2, 100, 250, 128, MASK_KEY_PADDING, (0, 250)),
    ("d100_padding_causal", "bf16", 2, 2, 130, 130, 100, MASK_KEY_PADDING | MASK_CAUSAL, (1, 130)),
    ("fp32_d64_causal", "fp32", 2, 2, 200, 200, 64, MASK_CAUSAL, None),
    ("fp32_d33_cross_padding", "fp32", 2, 3, 50, 70, 33, MASK_KEY_PADDING, (0, 70)),
]


@pytest.mark.parametrize("name,dtype,B,h,m,n,d,mask,lengths", SIMT_BWD, ids=[c[0] for c in SIMT_BWD])
def test_bwd_cuda_cores(orc, name, dtype, B, h, m, n, d, mask, lengths):
    w = Workload(name, dtype, B, h, m, n, d, mask, d ** -0.5, 79, lengths)
    inp = draw(w)
    dout = draw_dout(w)
    _, lse, dq, dk, dv = gpu_grads(inp, dout)
    rq, rk, rv = orc.attn_bwd(inp.q, inp.k, inp.v, dout, inp.key_lengths, w.mask, w.scale)
    if dtype == "fp32":
        for name_, g, r in (("dV", dv, rv), ("dK", dk, rk), ("dQ", dq, rq)):
            err = np.abs(as_f64(g) - r).max()
            assert err <= 1e-4 * max(1.0, np.abs(r).max()), f"{name_}: max err {err:.3e}"
    else:
        check_grad("dV", dv, rv)
        check_grad("dK", dk, rk)
        check_grad("dQ", dq, rq)
