"""GPU kernels against the fp64 oracle, element by element, on seeded inputs.

Tolerances: max abs error <= 1e-2 for bf16 inputs/outputs, <= 1e-4 for the
fp32 path.  Every kernel that can run a case is run on it.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from workloads import WORKLOADS, MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE, Workload, draw, round_to_bf16_bits, sample_rows

from gpu_helpers import as_f64, report, rounding_bound, run, to_device, tol_for

pytestmark = pytest.mark.gpu

K_FLASH, K_SHORT, K_SIMT, K_AUTO = attn.KERNEL_FLASH, attn.KERNEL_SHORT, attn.KERNEL_SIMT, attn.KERNEL_AUTO
K_WIDE, K_RESIDENT = attn.KERNEL_WIDE, attn.KERNEL_RESIDENT


def resident_fits(m, n, d=64, dtype="bf16"):
    return dtype == "bf16" and d % 8 == 0 and d <= 64 and n <= 256


def auto_for(m, n):
    """The tensor-core kernel the library picks for bf16 heads of width <= 64."""
    return K_RESIDENT if resident_fits(m, n) else (K_SHORT if m <= 128 else K_FLASH)


def kernels_for(w: Workload):
    ks = [K_SIMT]
    if w.dtype == "bf16" and w.d == 64:
        ks.append(K_FLASH)
        if w.m <= 128:
            ks.append(K_SHORT)
        if resident_fits(w.m, w.n):
            ks.append(K_RESIDENT)
    return ks


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def check_full(orc, w, kernel, inp=None, scale=None):
    inp = inp if inp is not None else draw(w)
    got = as_f64(run(inp, kernel, scale=scale))
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale if scale is None else scale)
    tol = tol_for(w)
    assert np.abs(got - ref).max() <= tol, report(got, ref, tol)
    return got, ref


# ---------------------------------------------------------------- the reference workloads
@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_workload_full(orc, cfg):
    w = WORKLOADS[cfg]
    inp = draw(w)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    for kern in [K_AUTO] + kernels_for(w):
        got = as_f64(run(inp, kern))
        assert np.abs(got - ref).max() <= tol_for(w), f"kernel {kern}: " + report(got, ref, tol_for(w))


def full_size_rows(w, m, extra):
    """Linear output-row ids ((b*h + head)*m + i) of a full-size check: every row of the
    first and the last head, the first and last row of every 128-row query tile of
    every head, and the rows in `extra`."""
    heads = np.concatenate([np.arange(m), (w.B * w.h - 1) * m + np.arange(m)])
    edges = (np.arange(w.B * w.h)[:, None] * m + np.array([0, 127])[None, :]
             + np.arange(0, m, 128)[:, None, None]).reshape(-1)
    rows = np.unique(np.concatenate([heads, edges, extra]))
    assert rows.size > 2 * m + w.B * w.h * (m // 128) and rows.max() < w.B * w.h * m
    return rows


def test_long_causal_sampled_rows(orc):
    """n = m = 8192 causal at full size, in the launch configuration the benchmark times;
    checked on every row of the first and the last head ((b, h) = (0, 0) and (3, 15)),
    the first and last row of every 128-row query tile of every head, and random rows."""
    w = WORKLOADS[5]
    inp = draw(w)
    assert attn.select_kernel(w.B, w.h, w.m, w.n, w.d, 0, w.mask) == K_FLASH
    got = as_f64(run(inp, K_AUTO)).reshape(-1, w.d)
    rows = full_size_rows(w, w.m, sample_rows(w, 1536))
    ref = orc.attn_rows(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale, rows)
    assert np.abs(got[rows] - ref).max() <= 1e-2, report(got[rows], ref, 1e-2)
    assert np.isfinite(got).all()
    # every row of a softmax-weighted mean lies inside the hull of the value rows it averages
    assert np.abs(got).max() <= 5.5


def test_wide_heads_benchmarked_sizes(orc):
    """The d_k = 128 calls the benchmark times, at full size on its inputs (the long
    workload with h = 8 and d_k = 128): causal n = 8192 through attn_fwd, no mask on the
    first 4096 positions, and windows of 256 and 1024 through attn_fwd_window; each
    checked on every row of the first and the last head, both edge rows of every
    query tile of every head, and random rows."""
    w = WORKLOADS[5].with_(h=8, d=128, scale=128 ** -0.5, name="long_causal_h8_d128")
    inp = draw(w)
    assert attn.select_kernel(w.B, w.h, w.m, w.n, w.d, 0, w.mask) == K_WIDE
    q, k, v = (to_device(x, "bf16") for x in (inp.q, inp.k, inp.v))
    half = w.n // 2
    qh, kh, vh = (x[:, :, :half].contiguous() for x in (q, k, v))
    host_half = tuple(np.ascontiguousarray(x[:, :, :half]) for x in (inp.q, inp.k, inp.v))
    full = (inp.q, inp.k, inp.v)
    cases = [
        ("causal", lambda: attn.attn_fwd(q, k, v, None, w.mask, w.scale), w.m, full, w.mask, None),
        ("no_mask_4096", lambda: attn.attn_fwd(qh, kh, vh, None, MASK_NONE, w.scale), half, host_half,
         MASK_NONE, None),
    ] + [(f"window_{win}", lambda win=win: attn.attn_fwd_window(q, k, v, None, attn.MASK_WINDOW, win, w.scale),
          w.m, full, attn.MASK_WINDOW, win) for win in (256, 1024)]
    rng = np.random.default_rng(61)
    for name, call, m, ins, mask, win in cases:
        got = as_f64(call()).reshape(-1, w.d)
        torch.cuda.synchronize()
        rows = full_size_rows(w, m, rng.integers(0, w.B * w.h * m, size=1024))
        ref = orc.attn_rows(*ins, None, mask, w.scale, rows, window=win)
        assert np.abs(got[rows] - ref).max() <= 1e-2, f"{name}: " + report(got[rows], ref, 1e-2)
        assert np.isfinite(got).all(), name
    assert attn.device_status() == (0, 0)


# ---------------------------------------------------------------- ragged and edge shapes
EDGE = [
    # name, B, h, m, n, mask, lengths
    ("causal_ragged_3tiles", 2, 3, 300, 300, MASK_CAUSAL, None),
    ("causal_one_tile_pair_tail", 1, 2, 129, 129, MASK_CAUSAL, None),
    ("cross_ragged", 2, 2, 200, 333, MASK_NONE, None),
    ("cross_padding_long", 3, 2, 190, 700, MASK_KEY_PADDING, (0, 700)),
    ("self_padding_causal", 3, 2, 260, 260, MASK_KEY_PADDING | MASK_CAUSAL, (1, 260)),
    ("short_padding_odd_heads", 3, 3, 77, 150, MASK_KEY_PADDING, (0, 150)),
    # h = 1: the two heads of a split-mode CTA tile belong to different sequences, so
    # their key tile counts differ (0 to 16) and their K/V rings run out of step
    ("short_single_head_ragged_keys", 9, 1, 128, 2000, MASK_KEY_PADDING, (0, 2000)),
    ("single_key", 2, 2, 50, 1, MASK_NONE, None),
    ("single_query", 2, 2, 1, 500, MASK_KEY_PADDING, (1, 500)),
    ("one_by_one_causal", 1, 1, 1, 1, MASK_CAUSAL, None),
    ("exact_tiles_no_mask", 1, 2, 256, 256, MASK_NONE, None),
    # the whole-head-resident kernel at the edges of its range: the most keys it holds,
    # one key box short of that, one query, lengths 0 .. n with causal, 17 keys
    ("resident_max_keys", 2, 3, 100, 192, MASK_KEY_PADDING, (0, 192)),
    ("resident_cross_191", 2, 2, 128, 191, MASK_NONE, None),
    ("resident_single_query", 3, 2, 1, 192, MASK_KEY_PADDING, (0, 192)),
    ("resident_causal_padding", 3, 2, 128, 128, MASK_CAUSAL | MASK_KEY_PADDING, (0, 128)),
    ("resident_17_keys", 2, 3, 33, 17, MASK_NONE, None),
    # above 192 keys (O over the last two chunks of S, their weights held first): the
    # most keys it holds, one chunk past 192 (one held chunk), a ragged box
    ("resident_256_keys", 2, 3, 100, 256, MASK_KEY_PADDING, (0, 256)),
    ("resident_208_keys", 2, 2, 128, 208, MASK_NONE, None),
    ("resident_250_keys_one_query", 3, 2, 1, 250, MASK_KEY_PADDING, (180, 250)),
    # several query tiles per head (one CTA each), causal and padded, ragged last tile
    ("resident_query_tiles_causal", 2, 3, 256, 256, MASK_CAUSAL, None),
    ("resident_query_tiles_ragged", 2, 2, 300, 230, MASK_KEY_PADDING, (0, 230)),
    ("resident_long_queries_short_keys", 1, 2, 1000, 60, MASK_KEY_PADDING, (1, 60)),
]


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths", EDGE, ids=[e[0] for e in EDGE])
def test_edge_shapes(orc, name, B, h, m, n, mask, lengths):
    w = Workload(name, "bf16", B, h, m, n, 64, mask, 0.125, 4242, lengths)
    inp = draw(w)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    for kern in kernels_for(w):
        got = as_f64(run(inp, kern))
        assert np.abs(got - ref).max() <= 1e-2, f"kernel {kern}: " + report(got, ref, 1e-2)


def test_zero_and_full_lengths(orc):
    """len_b = 0 (no allowed key: output 0), 1 (output = V[0]), n, and out-of-range lengths."""
    w = Workload("lengths", "bf16", 6, 2, 100, 140, 64, MASK_KEY_PADDING, 0.125, 77)
    inp = draw(w)
    inp.key_lengths[:] = [0, 1, 140, 129, -5, 1000]
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    for kern in kernels_for(w):
        got = as_f64(run(inp, kern))
        assert np.abs(got - ref).max() <= 1e-2, f"kernel {kern}: " + report(got, ref, 1e-2)
        assert (got[0] == 0).all() and (got[4] == 0).all()
        v0 = as_f64(to_device(inp.v, "bf16"))[1, :, :1]
        np.testing.assert_array_equal(got[1], np.broadcast_to(v0, got[1].shape))


@pytest.mark.parametrize("scale", [0.0, 1.0, 0.01, 0.35])
def test_other_scales(orc, scale):
    w = Workload("scales", "bf16", 2, 2, 160, 160, 64, MASK_CAUSAL, scale, 99)
    for kern in kernels_for(w):
        check_full(orc, w, kern)


def test_fp32_path_shapes(orc):
    for (m, n, d, mask) in [(16, 16, 64, 0), (33, 70, 17, 1), (50, 50, 64, 3), (5, 200, 2, 0)]:
        w = Workload("fp32", "fp32", 2, 2, m, n, d, mask, d ** -0.5, 5, (0, n))
        check_full(orc, w, K_SIMT)


def test_worked_example_on_every_kernel():
    """The primer's 2x2 example (scale 1) with d_k = 2 zero-padded to 64: zero
    columns leave every score unchanged.  bf16 holds 1, -1, 5 exactly."""
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_sdpa_2x2.json")))
    for dtype, kernels in (("bf16", [K_FLASH, K_SHORT, K_RESIDENT, K_SIMT]), ("fp32", [K_SIMT])):
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        q = torch.zeros(1, 1, 2, 64, dtype=tdt, device="cuda")
        k, v = torch.zeros_like(q), torch.zeros_like(q)
        q[0, 0, :, :2] = torch.tensor(g["Q"], dtype=tdt)
        k[0, 0, :, :2] = torch.tensor(g["K"], dtype=tdt)
        v[0, 0, :, :2] = torch.tensor(g["V"], dtype=tdt)
        for kern in kernels:
            out = attn.attn_fwd(q, k, v, None, 0, 1.0, kernel=kern).float().cpu().numpy()[0, 0]
            # printed precision 0.005 plus bf16 output rounding of 4.4 (half-ulp 0.0156)
            tol = 0.005 + (0.016 if dtype == "bf16" else 1e-4)
            np.testing.assert_allclose(out[:, :2], g["printed"]["output"], atol=tol)
            assert (out[:, 2:] == 0).all()


JUMP_CASES = [
    # name, B, h, m, n, mask, lengths, rows whose scores jump by ~20, by > 128 (log2 units)
    ("cross_split_mode", 3, 1, 128, 512, MASK_NONE, None, [5, 77, 127], [6, 100]),
    ("cross_pair_mode", 2, 2, 384, 512, MASK_KEY_PADDING, (380, 512), [5, 200, 383], [6, 301]),
    ("self_causal", 2, 2, 512, 512, MASK_CAUSAL, None, [300, 450, 511], [420, 509]),
]


def jump_inputs(name, B, h, m, n, mask, lengths, soft, hard, d=64):
    """Seeded inputs in which the listed rows' scores grow sharply after their first
    key tiles: by ~20 log2 units (exponentials against the running reference stay
    finite but leave the kept range) and by > 128 (they overflow fp32).  The two
    large keys also make most other rows peaked.  Any head width d (the dot products
    are the same: half the width carries the values)."""
    w = Workload(name, "bf16", B, h, m, n, d, mask, 0.125, 321, lengths)
    inp = draw(w)
    bits = lambda x: np.uint16(np.array(x, dtype=np.float32).view(np.uint32) >> 16)  # exact in bf16
    hd = d // 2
    inp.q[:, :, soft, :hd], inp.q[:, :, soft, hd:] = bits(1.0), bits(0.0)
    inp.q[:, :, hard, :hd], inp.q[:, :, hard, hd:] = bits(0.0), bits(1.0)
    inp.k[:, :, 260, :hd], inp.k[:, :, 260, hd:] = bits(128.0 / hd), bits(0.0)   # soft rows: q.k = 128
    inp.k[:, :, 400, :hd], inp.k[:, :, 400, hd:] = bits(0.0), bits(1024.0 / hd)  # hard rows: q.k = 1024
    return w, inp


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths,soft,hard", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_score_jumps_between_key_tiles(orc, name, B, h, m, n, mask, lengths, soft, hard):
    """Tolerance 1e-2 with value rows in [-1, 1].  A row dominated by one key carries
    that key's bf16 weight rounding (up to 2^-8 relative) into the output, plus the
    output's own rounding; with |v| <= 1 both together stay below 6e-3, so an error
    above 1e-2 here means a wrong reference, rescale or recomputation."""
    w, inp = jump_inputs(name, B, h, m, n, mask, lengths, soft, hard)
    rng = np.random.default_rng(5)
    vals = rng.uniform(-1.0, 1.0, size=inp.v.shape).astype(np.float32)
    inp.v[...] = (vals.view(np.uint32) >> 16).astype(np.uint16)  # truncation keeps |v| <= 1
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    for kern in kernels_for(w):
        got = as_f64(run(inp, kern))
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() <= 1e-2, f"kernel {kern}: " + report(got, ref, 1e-2)


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths,soft,hard", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_score_jumps_narrow_heads(orc, name, B, h, m, n, mask, lengths, soft, hard):
    """The score jumps with d_k = 32 on the tensor-core kernels: the rescale and the
    score recomputation (which reads Q and K rows of the true width) stay exact."""
    w, inp = jump_inputs(name, B, h, m, n, mask, lengths, soft, hard, d=32)
    rng = np.random.default_rng(6)
    vals = rng.uniform(-1.0, 1.0, size=inp.v.shape).astype(np.float32)
    inp.v[...] = (vals.view(np.uint32) >> 16).astype(np.uint16)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    kern = K_SHORT if m <= 128 else K_FLASH
    got = as_f64(run(inp, kern))
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths,soft,hard", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_score_jumps_wide_heads(orc, name, B, h, m, n, mask, lengths, soft, hard):
    """The score jumps with d_k = 128 on the wide kernel: its fixed per-row reference,
    the power-of-two rescale and the score recomputation (of 128-wide rows).  Its row
    sum adds the weights as rounded, so every output is a weighted mean of exactly
    the weights applied.  Standard normal values: 1e-2 plus only the output's own
    half-ulp where |out| >= 4, on every row.  Values of standard deviation 4: the
    same bound on the rows dominated by one key (the jumped rows); on rows that two
    or three keys share, each weight's own bf16 rounding (2^-8 relative) moves the
    mean by up to 2^-8 times the spread of their values, which wider values push
    past 1e-2."""
    w, inp = jump_inputs(name, B, h, m, n, mask, lengths, soft, hard, d=128)
    for sigma, rows in ((1.0, slice(None)), (4.0, soft + hard)):
        v = sigma * np.random.default_rng(7).standard_normal(inp.v.shape).astype(np.float32)
        inp.v[...] = round_to_bf16_bits(v)
        ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)[:, :, rows]
        got = as_f64(run(inp, K_WIDE))[:, :, rows]
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) - rounding_bound(ref)).max() <= 0, f"sd {sigma}: " + report(got, ref, 1e-2)


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths,soft,hard", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_peaked_rows_error_bound(orc, name, B, h, m, n, mask, lengths, soft, hard):
    """The same peaked rows with standard normal values, against the error bound of
    bf16 weights: per element |err| <= 2^-8 max|v| (weight rounding) + half an
    output ulp + 1e-3 (fp32 accumulation)."""
    w, inp = jump_inputs(name, B, h, m, n, mask, lengths, soft, hard)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    vmax = np.abs(as_f64(to_device(inp.v, "bf16"))).max(axis=(2, 3), keepdims=True)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
    bound = 2.0 ** -8 * vmax + half_ulp + 1e-3
    for kern in kernels_for(w):
        got = as_f64(run(inp, kern))
        assert np.isfinite(got).all()
        excess = np.abs(got - ref) - bound
        assert excess.max() <= 0, f"kernel {kern}: " + report(got, ref, float(bound.max()))


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths,soft,hard", JUMP_CASES, ids=[c[0] for c in JUMP_CASES])
def test_jumped_rows_are_weighted_means(orc, name, B, h, m, n, mask, lengths, soft, hard):
    """The rows whose scores jump, each dominated by one key of a later tile, with
    values of standard deviation 4: the tile that rescales (or recomputes) its
    weights adds them to the row sum as rounded, so these outputs are weighted means
    of exactly the weights applied (had the sum missed the dominant weight's
    rounding, the error would reach 2^-8 * 16 = 0.06): 1e-2 plus the output's own
    half-ulp where |out| >= 4."""
    w, inp = jump_inputs(name, B, h, m, n, mask, lengths, soft, hard)
    v = 4.0 * np.random.default_rng(8).standard_normal(inp.v.shape).astype(np.float32)
    inp.v[...] = round_to_bf16_bits(v)
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)[:, :, soft + hard]
    for kern in kernels_for(w):
        got = as_f64(run(inp, kern))[:, :, soft + hard]
        assert np.isfinite(got).all()
        assert (np.abs(got - ref) - rounding_bound(ref)).max() <= 0, f"kernel {kern}: " + report(got, ref, 1e-2)


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_masked_keys_do_not_matter_bitwise(cfg):
    """Changing K/V rows that the mask hides leaves the output bit-identical."""
    w = WORKLOADS[cfg].with_(B=8)
    inp = draw(w)
    for kern in kernels_for(w):
        base = run(inp, kern).clone()
        k2, v2 = inp.k.copy(), inp.v.copy()
        rng = np.random.default_rng(1)
        for b in range(w.B):
            if w.padded:
                L = inp.key_lengths[b]
                k2[b, :, L:] = rng.integers(0, 2 ** 14, size=k2[b, :, L:].shape, dtype=np.uint16)
                v2[b, :, L:] = rng.integers(0, 2 ** 14, size=v2[b, :, L:].shape, dtype=np.uint16)
        if w.causal:
            # for causal, perturb keys after a query row: compare rows up to it
            cut = 37
            k2[:, :, cut + 1:] ^= 0x0101
            v2[:, :, cut + 1:] ^= 0x0101
        inp2 = type(inp)(w, inp.q, k2, v2, inp.key_lengths)
        got = run(inp2, kern)
        if w.causal:
            assert torch.equal(got[:, :, :cut + 1], base[:, :, :cut + 1])
            assert not torch.equal(got, base)
        else:
            assert torch.equal(got, base)


def test_rows_sum_to_one_on_gpu():
    """With V = 1 everywhere every output is 1 (bf16: within 4e-3)."""
    w = WORKLOADS[3].with_(B=4, m=300, n=300)
    inp = draw(w)
    one = np.uint16(0x3F80)  # bf16 1.0
    inp.v[...] = one
    for kern in kernels_for(w):
        got = as_f64(run(inp, kern))
        assert np.abs(got - 1.0).max() <= 4e-3


def test_deterministic_bitwise():
    for cfg in (3, 4):
        w = WORKLOADS[cfg]
        inp = draw(w)
        for kern in kernels_for(w):
            a = run(inp, kern).clone()
            b = run(inp, kern)
            assert torch.equal(a, b)


def test_no_writes_outside_out():
    """Guard bands around `out` keep their sentinel bytes."""
    w = WORKLOADS[4].with_(B=3, m=100)
    inp = draw(w)
    for kern in kernels_for(w):
        n_out = w.B * w.h * w.m * w.d
        guard = 4096
        buf = torch.full((n_out + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
        out = buf[guard:guard + n_out].view(w.B, w.h, w.m, w.d)
        run(inp, kern, out=out)
        assert (buf[:guard] == -7.0).all() and (buf[guard + n_out:] == -7.0).all()


# ---------------------------------------------------------------- other head widths
WIDTHS = [
    # the model variants that change d_k (h * d_k = 512): h=4 d_k=128, h=16 d_k=32, h=32 d_k=16
    ("h4_d128_padding", "bf16", 4, 4, 100, 100, 128, MASK_KEY_PADDING, (10, 100)),
    ("h16_d32_causal", "bf16", 4, 16, 128, 128, 32, MASK_CAUSAL, None),
    ("h32_d16_cross", "bf16", 2, 32, 60, 90, 16, MASK_KEY_PADDING, (0, 90)),
    ("fp32_d128_causal", "fp32", 2, 2, 70, 70, 128, MASK_CAUSAL, None),
    ("fp32_d100_ragged", "fp32", 2, 3, 33, 47, 100, MASK_KEY_PADDING, (0, 47)),
]


@pytest.mark.parametrize("name,dtype,B,h,m,n,d,mask,lengths", WIDTHS, ids=[c[0] for c in WIDTHS])
def test_head_widths(orc, name, dtype, B, h, m, n, d, mask, lengths):
    """bf16 heads narrower than 64 run zero-padded on the tensor-core kernels (and still
    on the CUDA-core one when asked); other widths and fp32 on the CUDA cores."""
    w = Workload(name, dtype, B, h, m, n, d, mask, d ** -0.5, 61, lengths)
    auto = attn.select_kernel(B, h, m, n, d, 0 if dtype == "bf16" else 1, mask)
    if dtype == "bf16" and d <= 64:
        assert auto == auto_for(m, n)
        check_full(orc, w, K_SIMT)
    elif dtype == "bf16" and d == 128:
        assert auto == K_WIDE
        check_full(orc, w, K_SIMT)
    else:
        assert auto == K_SIMT
    check_full(orc, w, K_AUTO)


WIDE_CASES = [
    # d_k = 128 on the tensor-core kernel: ragged query and key tiles, padding (with
    # empty rows), causal, cross-attention, a long sequence, a single query
    ("causal_ragged", 2, 3, 300, 300, MASK_CAUSAL, None),
    ("padding_with_empty", 3, 2, 200, 200, MASK_KEY_PADDING, (0, 200)),
    ("cross_padding", 2, 4, 100, 333, MASK_KEY_PADDING, (1, 333)),
    ("long_causal", 1, 2, 2048, 2048, MASK_CAUSAL, None),
    ("no_mask_long_keys", 1, 3, 128, 1000, MASK_NONE, None),
    ("causal_padding", 2, 2, 260, 260, MASK_CAUSAL | MASK_KEY_PADDING, (0, 260)),
    ("single_query", 4, 2, 1, 77, MASK_NONE, None),
    # m, n <= 128: two heads per CTA; an odd head count leaves the last CTA's second
    # slot without a head, and zero key lengths leave whole slots without keys
    ("head_pairs_odd_padding", 3, 1, 100, 100, MASK_KEY_PADDING, (0, 100)),
    ("head_pairs_causal", 2, 3, 128, 128, MASK_CAUSAL, None),
    ("head_pairs_cross", 5, 3, 37, 128, MASK_KEY_PADDING, (1, 128)),
]


@pytest.mark.parametrize("name,B,h,m,n,mask,lengths", WIDE_CASES, ids=[c[0] for c in WIDE_CASES])
def test_wide_heads_tensor_cores(orc, name, B, h, m, n, mask, lengths):
    w = Workload(name, "bf16", B, h, m, n, 128, mask, 128 ** -0.5, 64, lengths)
    assert attn.select_kernel(B, h, m, n, 128, 0, mask) == K_WIDE
    check_full(orc, w, K_WIDE)


@pytest.mark.parametrize("B,h,m", [(2, 3, 200), (3, 1, 100)], ids=["query_tile_pairs", "head_pairs_odd"])
def test_wide_heads_lse_and_bounds(orc, B, h, m):
    """The log-sum-exp output of the wide kernel, and that it writes exactly its output
    (guard regions on both sides untouched), with two query tiles per CTA and with two
    heads per CTA (an odd head count: the last CTA's second slot has no head)."""
    w = Workload("wide_lse", "bf16", B, h, m, m, 128, MASK_CAUSAL | MASK_KEY_PADDING, 0.09, 65, (0, m))
    inp = draw(w)
    q, k, v = (to_device(x, "bf16") for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).cuda()
    out, lse = attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale)
    torch.cuda.synchronize()
    ref = orc.attn_lse(inp.q, inp.k, inp.key_lengths, w.mask, w.scale)
    got = lse.double().cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - ref[fin]).max() <= 2e-3
    n_out = w.B * w.h * w.m * w.d
    guard = 4096
    buf = torch.full((n_out + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
    o2 = buf[guard:guard + n_out].view(w.B, w.h, w.m, w.d)
    run(inp, K_WIDE, out=o2)
    assert (buf[:guard] == -7.0).all() and (buf[guard + n_out:] == -7.0).all()
    np.testing.assert_array_equal(as_f64(o2), as_f64(out))


NARROW = [
    # tensor-core kernels with zero-padded heads: pair mode, windows, padding, ragged tails
    ("d8_pair_causal", 1, 3, 300, 300, 8, MASK_CAUSAL, None),
    ("d16_pair_padding", 2, 2, 400, 400, 16, MASK_KEY_PADDING, (0, 400)),
    ("d24_cross_split", 3, 2, 100, 230, 24, MASK_KEY_PADDING, (1, 230)),
    ("d32_long_causal", 1, 2, 2048, 2048, 32, MASK_CAUSAL, None),
    ("d48_pair_padding_causal", 2, 2, 333, 333, 48, MASK_CAUSAL | MASK_KEY_PADDING, (0, 333)),
    ("d56_split_causal", 4, 2, 128, 128, 56, MASK_CAUSAL, None),
]


@pytest.mark.parametrize("name,B,h,m,n,d,mask,lengths", NARROW, ids=[c[0] for c in NARROW])
def test_narrow_heads_tensor_cores(orc, name, B, h, m, n, d, mask, lengths):
    w = Workload(name, "bf16", B, h, m, n, d, mask, d ** -0.5, 62, lengths)
    kern = auto_for(m, n)
    assert attn.select_kernel(B, h, m, n, d, 0, mask) == kern
    check_full(orc, w, kern)
    if kern == K_RESIDENT:
        check_full(orc, w, K_SHORT)


def test_narrow_heads_output_stays_in_bounds():
    """A d_k = 16 launch writes exactly its [B, h, m, 16] output: the TMA store clips the
    zero-padded columns (guard regions on both sides stay untouched)."""
    w = Workload("guard16", "bf16", 2, 3, 300, 300, 16, MASK_CAUSAL, 0.25, 63)
    inp = draw(w)
    n_out = w.B * w.h * w.m * w.d
    guard = 4096
    buf = torch.full((n_out + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n_out].view(w.B, w.h, w.m, w.d)
    run(inp, K_FLASH, out=out)
    assert (buf[:guard] == -7.0).all() and (buf[guard + n_out:] == -7.0).all()


# ---------------------------------------------------------------- whole-head-resident kernel
@pytest.mark.parametrize("scale", [0.0, 1.0, 0.01, 0.35])
def test_resident_other_scales(orc, scale):
    """Scale 1 with d_k = 64 makes most rows peaked (score spread ~8): there the bound
    adds the output's own half-ulp where |out| >= 4."""
    w = Workload("resident_scales", "bf16", 2, 2, 128, 128, 64, MASK_CAUSAL, scale, 99)
    inp = draw(w)
    got = as_f64(run(inp, K_RESIDENT))
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    assert (np.abs(got - ref) - rounding_bound(ref)).max() <= 0, report(got, ref, 1e-2)


def test_resident_rows_sum_to_one():
    """With V = 1 everywhere every output is exactly 1: the row sum adds the same
    rounded weights the P V product applies."""
    w = WORKLOADS[4].with_(B=4)
    inp = draw(w)
    inp.v[...] = np.uint16(0x3F80)  # bf16 1.0
    got = as_f64(run(inp, K_RESIDENT))
    assert np.abs(got - 1.0).max() <= 2.0 ** -8


def test_resident_peaked_rows_standard_values(orc):
    """Rows whose scores jump far above the rest (by ~20 and by > 128 in log2 units),
    with standard normal values.  The resident kernel takes each row's exact maximum
    and sums the rounded weights, so the output is a weighted mean with the weights
    applied: 1e-2, plus the output's own half-ulp where |out| >= 4 (bf16 spacing)."""
    B, h, m, n, d = 3, 2, 128, 160, 64
    w = Workload("resident_peaked", "bf16", B, h, m, n, d, MASK_KEY_PADDING, 0.125, 322, (100, 160))
    inp = draw(w)
    bits = lambda x: np.uint16(np.array(x, dtype=np.float32).view(np.uint32) >> 16)
    soft, hard = [5, 77, 127], [6, 100]
    inp.q[:, :, soft, :32], inp.q[:, :, soft, 32:] = bits(1.0), bits(0.0)
    inp.q[:, :, hard, :32], inp.q[:, :, hard, 32:] = bits(0.0), bits(1.0)
    inp.k[:, :, 60, :32], inp.k[:, :, 60, 32:] = bits(4.0), bits(0.0)    # soft rows: q.k = 128
    inp.k[:, :, 90, :32], inp.k[:, :, 90, 32:] = bits(0.0), bits(32.0)   # hard rows: q.k = 1024
    ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    got = as_f64(run(inp, K_RESIDENT))
    assert np.isfinite(got).all()
    assert (np.abs(got - ref) - rounding_bound(ref)).max() <= 0, report(got, ref, 1e-2)


@pytest.mark.parametrize("mask,m,n", [(MASK_KEY_PADDING, 100, 150), (MASK_CAUSAL | MASK_KEY_PADDING, 128, 128),
                                      (MASK_KEY_PADDING, 200, 256), (MASK_CAUSAL | MASK_KEY_PADDING, 250, 250)],
                         ids=["padding", "causal_padding", "padding_256_keys_two_tiles", "causal_250"])
def test_resident_lse_and_bounds(orc, mask, m, n):
    """The log-sum-exp output of the resident kernel (rows with no allowed key: -inf),
    and that it writes exactly its output (guard regions on both sides untouched), with
    one and two query tiles per head and up to 256 keys."""
    B, h = 3, 3
    w = Workload("resident_lse", "bf16", B, h, m, n, 64, mask, 0.125, 66, (0, n))
    inp = draw(w)
    inp.key_lengths[0] = 0
    q, k, v = (to_device(x, "bf16") for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).cuda()
    assert attn.select_kernel(B, h, m, n, 64, 0, mask) == K_RESIDENT
    out, lse = attn.attn_fwd_lse(q, k, v, lens, w.mask, w.scale)
    torch.cuda.synchronize()
    ref = orc.attn_lse(inp.q, inp.k, inp.key_lengths, w.mask, w.scale)
    got = lse.double().cpu().numpy()
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.abs(got[fin] - ref[fin]).max() <= 2e-3
    n_out = w.B * w.h * w.m * w.d
    guard = 4096
    buf = torch.full((n_out + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
    o2 = buf[guard:guard + n_out].view(w.B, w.h, w.m, w.d)
    run(inp, K_RESIDENT, out=o2)
    assert (buf[:guard] == -7.0).all() and (buf[guard + n_out:] == -7.0).all()
    np.testing.assert_array_equal(as_f64(o2), as_f64(out))


@pytest.mark.parametrize("d", [8, 16, 24, 32, 40, 48, 56])
def test_resident_narrow_heads(orc, d):
    """Every narrower head width on the resident kernel (zero-padded 64-wide tiles,
    d_k-column stores): padding with empty rows, causal with padding, and the
    log-sum-exp; guard regions around the output stay untouched."""
    for name, m, n, mask in (("pad", 100, 170, MASK_KEY_PADDING), ("causal_pad", 128, 128, MASK_CAUSAL | MASK_KEY_PADDING)):
        w = Workload(f"resident_d{d}_{name}", "bf16", 3, 2, m, n, d, mask, d ** -0.5, 70 + d, (0, n))
        inp = draw(w)
        inp.key_lengths[0] = 0
        assert attn.select_kernel(w.B, w.h, m, n, d, 0, mask) == K_RESIDENT
        q, k, v = (to_device(x, "bf16") for x in (inp.q, inp.k, inp.v))
        lens = torch.from_numpy(inp.key_lengths).cuda()
        n_out = w.B * w.h * m * d
        guard = 4096
        buf = torch.full((n_out + 2 * guard,), -7.0, dtype=torch.bfloat16, device="cuda")
        out = buf[guard:guard + n_out].view(w.B, w.h, m, d)
        lse = torch.empty((w.B, w.h, m), dtype=torch.float32, device="cuda")
        attn.attn_fwd_lse(q, k, v, lens, mask, w.scale, out=out, lse=lse)
        torch.cuda.synchronize()
        assert attn.device_status() == (0, 0)
        assert (buf[:guard] == -7.0).all() and (buf[guard + n_out:] == -7.0).all()
        ref = orc.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, mask, w.scale)
        got = as_f64(out)
        assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)
        ref_lse = orc.attn_lse(inp.q, inp.k, inp.key_lengths, mask, w.scale)
        g = lse.double().cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(g), fin)
        assert np.abs(g[fin] - ref_lse[fin]).max() <= 2e-3
