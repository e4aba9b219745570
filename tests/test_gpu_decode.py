"""attn_decode (m <= 8 new rows against a K/V cache) against the fp64 oracle.

Its definition is the attention equation with the key-padding mask, key_lengths
= the cache lengths, so the oracle is the same attn_fwd oracle; tolerance 1e-2
(bf16), as for the forward.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from workloads import DECODE, MASK_KEY_PADDING, MASK_NONE, Workload, draw, sample_rows

from gpu_helpers import as_f64, report, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def run_decode(inp, with_lengths=True, lse=False):
    w = inp.workload
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).cuda() if with_lengths else None
    lse_t = torch.empty((w.B, w.h, w.m), dtype=torch.float32, device="cuda") if lse else None
    out = attn.attn_decode(q, k, v, lens, w.scale, lse=lse_t)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    return out, lse_t


CASES = [
    # name, B, h, m, n, lengths
    ("one_query_short", 8, 4, 1, 100, (0, 100)),
    ("one_query_one_key", 3, 2, 1, 1, (0, 1)),
    ("two_queries", 4, 3, 2, 700, (1, 700)),
    ("three_queries_ragged", 5, 2, 3, 1000, (0, 1000)),
    ("five_queries", 2, 2, 5, 333, (300, 333)),
    ("eight_queries_long", 2, 2, 8, 5000, (4000, 5000)),
    ("few_heads_many_splits", 1, 1, 1, 20000, (19000, 20000)),
    ("many_heads_one_split", 64, 16, 1, 64, (1, 64)),
]


@pytest.mark.parametrize("name,B,h,m,n,lengths", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(orc, name, B, h, m, n, lengths):
    w = Workload(name, "bf16", B, h, m, n, 64, MASK_KEY_PADDING, 0.125, 31, lengths)
    inp = draw(w)
    inp.key_lengths[0] = lengths[0]
    out, lse = run_decode(inp, lse=True)
    got = as_f64(out)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, MASK_KEY_PADDING, w.scale)
    assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)
    ref_lse = orc.attn_lse(inp.q, inp.k, inp.key_lengths, MASK_KEY_PADDING, w.scale)
    g = lse.cpu().numpy().astype(np.float64)
    live = np.isfinite(ref_lse)
    assert (g[~live] == -np.inf).all()
    assert np.abs(g[live] - ref_lse[live]).max() <= 1e-3


def test_decode_without_lengths_sees_every_key(orc):
    w = Workload("no_lengths", "bf16", 3, 2, 1, 900, 64, MASK_NONE, 0.125, 32)
    inp = draw(w)
    out, _ = run_decode(inp, with_lengths=False)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, None, MASK_NONE, w.scale)
    assert np.abs(as_f64(out) - ref).max() <= 1e-2


def test_decode_step_workload_sampled(orc):
    """The benchmarked decode step at full size: B64 h16, caches of 4096."""
    w = DECODE
    inp = draw(w)
    out, _ = run_decode(inp)
    rows = sample_rows(w, 512)
    ref = orc.attn_rows(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale, rows)
    got = as_f64(out).reshape(-1, w.d)[rows]
    assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)


def test_decode_matches_forward_kernels():
    """Same inputs through attn_fwd (tensor-core split mode): agreement within bf16 rounding."""
    w = Workload("vs_fwd", "bf16", 6, 4, 4, 500, 64, MASK_KEY_PADDING, 0.125, 33, (0, 500))
    inp = draw(w)
    out, _ = run_decode(inp)
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    fwd = attn.attn_fwd(q, k, v, torch.from_numpy(inp.key_lengths).cuda(), MASK_KEY_PADDING, w.scale)
    torch.cuda.synchronize()
    assert (out.float() - fwd.float()).abs().max().item() <= 1.6e-2


WIDTH_CASES = [
    # the model-variant table's other head widths: d_k = 16 (h 32), 32 (h 16), 128 (h 4);
    # m from 1 to 8, ragged caches, one split and many
    ("d16_one_query", 16, 8, 4, 1, 700, (0, 700)),
    ("d16_eight_queries", 16, 2, 3, 8, 3000, (1, 3000)),
    ("d32_two_queries", 32, 4, 4, 2, 1500, (0, 1500)),
    ("d32_many_heads_one_split", 32, 64, 16, 1, 64, (1, 64)),
    ("d128_one_query_long", 128, 2, 2, 1, 9000, (8000, 9000)),
    ("d128_eight_queries", 128, 3, 2, 8, 600, (0, 600)),
    ("d128_five_queries", 128, 2, 2, 5, 333, (300, 333)),
]


@pytest.mark.parametrize("name,d,B,h,m,n,lengths", WIDTH_CASES, ids=[c[0] for c in WIDTH_CASES])
def test_decode_other_head_widths(orc, name, d, B, h, m, n, lengths):
    w = Workload(name, "bf16", B, h, m, n, d, MASK_KEY_PADDING, d ** -0.5, 34, lengths)
    inp = draw(w)
    inp.key_lengths[0] = lengths[0]
    out, lse = run_decode(inp, lse=True)
    got = as_f64(out)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, MASK_KEY_PADDING, w.scale)
    assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)
    ref_lse = orc.attn_lse(inp.q, inp.k, inp.key_lengths, MASK_KEY_PADDING, w.scale)
    g = lse.cpu().numpy().astype(np.float64)
    live = np.isfinite(ref_lse)
    assert (g[~live] == -np.inf).all()
    assert np.abs(g[live] - ref_lse[live]).max() <= 1e-3
