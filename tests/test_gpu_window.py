"""Restricted self-attention (ATTN_MASK_WINDOW) on every kernel against the fp64 oracle.

Keys with |i - j| <= window stay for query i; tolerance 1e-2 (bf16) / 1e-4 (fp32),
as for the forward.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from workloads import MASK_CAUSAL, MASK_KEY_PADDING, Workload, draw

from gpu_helpers import as_f64, report, to_device

pytestmark = pytest.mark.gpu

WIN = attn.MASK_WINDOW


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def run_window(inp, mask, window, kernel_m=None):
    w = inp.workload
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).cuda()
    out = attn.attn_fwd_window(q, k, v, lens, mask, window, w.scale)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    return as_f64(out)


CASES = [
    # name, dtype, B, h, n, extra mask, window, lengths
    ("pair_mode_w0", "bf16", 2, 2, 300, 0, 0, None),
    ("pair_mode_w1_causal", "bf16", 2, 2, 300, MASK_CAUSAL, 1, None),
    ("pair_mode_w127", "bf16", 1, 2, 700, 0, 127, None),
    ("pair_mode_w128_padding", "bf16", 3, 2, 700, MASK_KEY_PADDING, 128, (0, 700)),
    ("pair_mode_w200_causal_padding", "bf16", 2, 2, 1000, MASK_CAUSAL | MASK_KEY_PADDING, 200, (100, 1000)),
    ("pair_mode_long_w300", "bf16", 1, 4, 4096, 0, 300, None),
    ("pair_mode_covering_window", "bf16", 2, 2, 260, MASK_CAUSAL, 5000, None),
    ("resident_w10", "bf16", 3, 3, 100, MASK_KEY_PADDING, 10, (0, 100)),
    ("resident_w64_causal", "bf16", 4, 2, 128, MASK_CAUSAL, 64, None),
    ("resident_w0_causal_padding", "bf16", 3, 2, 128, MASK_CAUSAL | MASK_KEY_PADDING, 0, (0, 128)),
    ("resident_w40_m33", "bf16", 2, 3, 33, 0, 40, None),
    # the resident kernel's variant above 192 keys (O over the last S chunks, held
    # weights) with a window: two query tiles per head
    ("resident_long_w50_padding", "bf16", 2, 3, 256, MASK_KEY_PADDING, 50, (100, 256)),
    ("resident_long_w0_causal", "bf16", 2, 2, 224, MASK_CAUSAL, 0, None),
    ("resident_long_w130", "bf16", 2, 2, 250, 0, 130, None),
    ("fp32_w7", "fp32", 2, 2, 150, MASK_KEY_PADDING, 7, (1, 150)),
    ("narrow_heads_w3", "bf16_d32", 2, 2, 90, MASK_CAUSAL, 3, None),
    ("narrow_heads_pair_mode_w17", "bf16_d16", 2, 2, 300, MASK_KEY_PADDING, 17, (0, 300)),
    ("wide_heads_w0", "bf16_d128", 2, 2, 300, 0, 0, None),
    ("wide_heads_w127_causal", "bf16_d128", 2, 2, 700, MASK_CAUSAL, 127, None),
    ("wide_heads_w128_padding", "bf16_d128", 3, 2, 700, MASK_KEY_PADDING, 128, (0, 700)),
    ("wide_heads_w200_causal_padding", "bf16_d128", 2, 2, 1000, MASK_CAUSAL | MASK_KEY_PADDING, 200, (100, 1000)),
    ("wide_heads_covering_window", "bf16_d128", 2, 2, 260, 0, 5000, None),
    ("wide_heads_pairs_w5", "bf16_d128", 3, 1, 100, MASK_KEY_PADDING, 5, (0, 100)),
]


@pytest.mark.parametrize("name,dtype,B,h,n,mask,window,lengths", CASES, ids=[c[0] for c in CASES])
def test_window_matches_oracle(orc, name, dtype, B, h, n, mask, window, lengths):
    d = int(dtype.split("_d")[1]) if "_d" in dtype else 64
    w = Workload(name, dtype.split("_")[0], B, h, n, n, d, mask | WIN, d ** -0.5, 51, lengths)
    inp = draw(w)
    got = run_window(inp, mask | WIN, window)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, mask | WIN, w.scale, window=window)
    tol = 1e-4 if w.dtype == "fp32" else 1e-2
    assert np.abs(got - ref).max() <= tol, report(got, ref, tol)


@pytest.mark.parametrize("d", [64, 128])
def test_window_locality_bitwise(d):
    """Row i is bitwise unchanged when keys and values further than the window from it change."""
    w = Workload("loc", "bf16", 1, 2, 1024, 1024, d, WIN, d ** -0.5, 52)
    inp = draw(w)
    base = run_window(inp, WIN, 100)
    k2, v2 = inp.k.copy(), inp.v.copy()
    k2[:, :, 700:] ^= 0x0101
    v2[:, :, 700:] ^= 0x0101
    moved = run_window(type(inp)(w, inp.q, k2, v2, inp.key_lengths), WIN, 100)
    np.testing.assert_array_equal(moved[:, :, :600], base[:, :, :600])
    assert not np.array_equal(moved, base)


def test_window_benchmarked_size(orc):
    """The benchmarked call at full size: B4 h16 n=8192, window 256, the long workload's
    inputs; every row of two heads (first and last) and 2048 random rows elsewhere
    against the oracle."""
    from workloads import WORKLOADS
    w = WORKLOADS[5]
    inp = draw(w)
    got = run_window(inp, WIN, 256)
    rng = np.random.default_rng(53)
    m = w.m
    rows = np.concatenate([np.arange(0, m), np.arange((w.B * w.h - 1) * m, w.B * w.h * m),
                           rng.integers(0, w.B * w.h * m, size=2048)])
    ref = orc.attn_rows(inp.q, inp.k, inp.v, None, WIN, w.scale, rows, window=256)
    got_rows = got.reshape(-1, w.d)[rows]
    assert np.abs(got_rows - ref).max() <= 1e-2, report(got_rows, ref, 1e-2)
