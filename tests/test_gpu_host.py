"""attn_fwd_host: the forward on host buffers, copied in and out chunk by chunk.

Against the fp64 oracle (tolerance 1e-2 bf16 / 1e-4 fp32, as for the forward), and
bitwise against attn_fwd on device copies of the same inputs: every (batch, head)
slice is computed by the same kernel either way, so cutting the problem into chunks
must not change a single bit.  The cases cover both ways of cutting (whole batches
when B >= 8, head ranges within a batch otherwise, with a ragged last range), the
single-chunk path (fp32 rows that are not whole 16-byte units), heads of width 128
(whose short-row launches pair heads, which a one-head chunk cannot), pageable
memory and the ordering on the caller's stream.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from workloads import MASK_CAUSAL, MASK_KEY_PADDING, Workload, draw

from gpu_helpers import as_f64, report, run, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def to_host(x: np.ndarray, dtype: str, pinned: bool):
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.pin_memory() if pinned else t.clone()


def run_host(inp, pinned=True, stream=None):
    w = inp.workload
    q, k, v = (to_host(x, w.dtype, pinned) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(np.ascontiguousarray(inp.key_lengths, dtype=np.int32))
    out = attn.attn_fwd_host(q, k, v, lens, w.mask, w.scale, stream=stream)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    return out


CASES = [
    # name, dtype, B, h, m, n, d, mask, lengths
    ("heads_split_ragged_causal", "bf16", 3, 5, 300, 300, 64, MASK_CAUSAL, None),
    ("heads_split_padding_cross", "bf16", 2, 7, 128, 160, 64, MASK_KEY_PADDING, (40, 160)),
    ("batches_whole_padding", "bf16", 9, 2, 100, 100, 64, MASK_KEY_PADDING, (10, 100)),
    ("batches_whole_causal_padding", "bf16", 17, 1, 257, 257, 64, MASK_CAUSAL | MASK_KEY_PADDING, (0, 257)),
    ("one_head", "bf16", 1, 1, 1000, 1000, 64, MASK_CAUSAL, None),
    ("fp32_odd_width_single_chunk", "fp32", 3, 4, 37, 53, 3, MASK_KEY_PADDING, (0, 53)),
    ("fp32_whole_rows", "fp32", 2, 5, 64, 64, 16, MASK_CAUSAL, None),
    ("narrow_heads_bf16", "bf16", 4, 3, 90, 90, 32, 0, None),
    # heads of width 128: long rows (query-tile pairs), and short rows, where the
    # whole problem runs as head pairs but a one-head chunk cannot
    ("wide_heads_causal", "bf16", 2, 3, 300, 300, 128, MASK_CAUSAL, None),
    ("wide_heads_short_padding", "bf16", 3, 3, 100, 100, 128, MASK_KEY_PADDING, (0, 100)),
]


@pytest.mark.parametrize("name,dtype,B,h,m,n,d,mask,lengths", CASES, ids=[c[0] for c in CASES])
def test_host_matches_oracle_and_device_path(orc, name, dtype, B, h, m, n, d, mask, lengths):
    w = Workload(name, dtype, B, h, m, n, d, mask, d ** -0.5, 61, lengths)
    inp = draw(w)
    got = as_f64(run_host(inp))
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, mask, w.scale)
    tol = tol_for(w)
    assert np.abs(got - ref).max() <= tol, report(got, ref, tol)
    dev = as_f64(run(inp))
    np.testing.assert_array_equal(got, dev)


def test_host_pageable_memory(orc):
    w = Workload("pageable", "bf16", 2, 4, 256, 256, 64, MASK_CAUSAL, 0.125, 62)
    inp = draw(w)
    got = as_f64(run_host(inp, pinned=False))
    np.testing.assert_array_equal(got, as_f64(run(inp)))


def test_host_result_ready_with_caller_stream():
    """The caller's stream waits for the last copy back: once an event recorded on it
    after the call has completed, the whole output is in host memory (checked before
    anything else synchronises), also when the stream was busy when the call was made."""
    w = Workload("ordered", "bf16", 4, 4, 512, 512, 64, MASK_CAUSAL, 0.125, 63)
    inp = draw(w)
    q, k, v = (to_host(x, w.dtype, True) for x in (inp.q, inp.k, inp.v))
    out = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    busy = torch.ones(64 << 20, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        busy.mul_(2.0)
        attn.attn_fwd_host(q, k, v, None, w.mask, w.scale, out=out, stream=s)
        ev = torch.cuda.Event()
        ev.record(s)
    ev.synchronize()
    got = as_f64(out)
    np.testing.assert_array_equal(got, as_f64(run(inp)))


def test_host_repeated_calls_reuse_workspace():
    w = Workload("repeat", "bf16", 2, 3, 384, 384, 64, MASK_CAUSAL, 0.125, 64)
    inp = draw(w)
    q, k, v = (to_host(x, w.dtype, True) for x in (inp.q, inp.k, inp.v))
    ws = torch.empty(attn.host_workspace_size(2, 3, 384, 384, 64), dtype=torch.uint8, device="cuda")
    outs = [attn.attn_fwd_host(q, k, v, None, w.mask, w.scale, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    ref = as_f64(run(inp))
    for o in outs:
        np.testing.assert_array_equal(as_f64(o), ref)


def test_host_full_size_long_causal_bitwise():
    """The long causal workload (B4 h16 n=8192, 268 MB of tensors, eight chunks) through
    the host-buffer path equals the device path bit for bit."""
    from workloads import WORKLOADS
    w = WORKLOADS[5]
    inp = draw(w)
    got = run_host(inp)
    dev = run(inp)
    assert torch.equal(got.view(torch.int16), dev.cpu().view(torch.int16))
