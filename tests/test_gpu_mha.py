"""Multi-head attention with projections (attn_mha_fwd) against the fp64 MultiHead oracle.

Tolerance 2e-2 absolute, from the arithmetic: Q, K, V and the heads' outputs are
rounded to bf16 (2^-8 relative each) and the attention stays within its own
1e-2 bar; W^O is drawn with variance 1/(h*64), so the output projection carries
the per-feature errors over with unit gain (they add in quadrature over its
h*64 inputs), plus the output's own bf16 rounding.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import mha
import transformer_scaled_dot_masked_gb300 as attn
from workloads import MASK_CAUSAL, MASK_KEY_PADDING, MASK_NONE, draw_mha

from gpu_helpers import as_f64, report

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


CASES = [
    # name, B, h, m, n, d_model, mask, self-attention, lengths (lo, hi)
    ("base_encoder_padding", 3, 8, 100, 100, 512, MASK_KEY_PADDING, True, (10, 100)),
    ("base_decoder_causal", 2, 8, 130, 130, 512, MASK_CAUSAL, True, None),
    ("big_cross_padding", 2, 16, 128, 160, 1024, MASK_KEY_PADDING, False, (40, 160)),
    ("two_heads_long", 1, 2, 700, 700, 128, MASK_NONE, True, None),
    ("six_heads_odd_column_tiles", 2, 6, 300, 300, 384, MASK_CAUSAL, True, None),
    # the projections' CTA pairs on tiny and ragged row counts: a pair tile of 256 rows
    # with one valid row (the second CTA's rows all past L, never stored), and 17 / 33
    ("one_position", 1, 2, 1, 1, 128, MASK_NONE, True, None),
    ("ragged_cross_17_33", 3, 2, 17, 33, 128, MASK_KEY_PADDING, False, (1, 33)),
]


@pytest.mark.parametrize("name,B,h,m,n,dm,mask,selfattn,lengths", CASES, ids=[c[0] for c in CASES])
def test_mha_matches_oracle(orc, name, B, h, m, n, dm, mask, selfattn, lengths):
    xq, xkv, wq, wk, wv, wo = draw_mha(B, h, m, n, dm, seed=81, self_attention=selfattn)
    lens = np.full(B, n, dtype=np.int32)
    if lengths is not None:
        lens = np.random.default_rng(82).integers(lengths[0], lengths[1] + 1, size=B).astype(np.int32)
    out = attn.attn_mha_fwd(dev(xq), dev(xkv), dev(wq), dev(wk), dev(wv), dev(wo), h,
                            torch.from_numpy(lens).cuda(), mask, 64 ** -0.5)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    ref = mha.mha_fwd(orc, xq, xkv, wq, wk, wv, wo, h, lens, mask, 64 ** -0.5)
    got = as_f64(out)
    assert np.abs(got - ref).max() <= 2e-2, report(got, ref, 2e-2)


WIDE_CASES = [
    # heads of width 128: the model-variant table's h = 4 row (d_model 512) and a wider
    # model; the attention runs on the d_k = 128 kernel, each head spans two 64-column
    # blocks of the projections
    ("h4_d128_encoder_padding", 3, 4, 100, 100, 512, MASK_KEY_PADDING, True, (10, 100)),
    ("h4_d128_decoder_causal", 2, 4, 300, 300, 512, MASK_CAUSAL, True, None),
    ("h8_d128_cross_padding", 2, 8, 128, 200, 1024, MASK_KEY_PADDING, False, (40, 200)),
    ("h1_d128_long", 1, 1, 700, 700, 256, MASK_NONE, True, None),
]


@pytest.mark.parametrize("name,B,h,m,n,dm,mask,selfattn,lengths", WIDE_CASES, ids=[c[0] for c in WIDE_CASES])
def test_mha_wide_heads(orc, name, B, h, m, n, dm, mask, selfattn, lengths):
    xq, xkv, wq, wk, wv, wo = draw_mha(B, h, m, n, dm, seed=83, self_attention=selfattn, d_k=128)
    lens = np.full(B, n, dtype=np.int32)
    if lengths is not None:
        lens = np.random.default_rng(84).integers(lengths[0], lengths[1] + 1, size=B).astype(np.int32)
    out = attn.attn_mha_fwd(dev(xq), dev(xkv), dev(wq), dev(wk), dev(wv), dev(wo), h,
                            torch.from_numpy(lens).cuda(), mask)  # default scale: 1/sqrt(128)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    ref = mha.mha_fwd(orc, xq, xkv, wq, wk, wv, wo, h, lens, mask, 128 ** -0.5)
    got = as_f64(out)
    assert np.abs(got - ref).max() <= 2e-2, report(got, ref, 2e-2)


NARROW_CASES = [
    # the model-variant table's narrower heads at d_model 512: h = 16 with d_k = 32 and
    # h = 32 with d_k = 16 (projections through the concatenated layout), and d_k = 48
    ("h16_d32_encoder_padding", 2, 16, 100, 100, 512, MASK_KEY_PADDING, True, (10, 100)),
    ("h32_d16_decoder_causal", 2, 32, 130, 130, 512, MASK_CAUSAL, True, None),
    ("h16_d32_cross_padding", 2, 16, 128, 200, 512, MASK_KEY_PADDING, False, (40, 200)),
    ("h8_d48_long", 1, 8, 300, 300, 384, MASK_NONE, True, None),
    ("h4_d32_five_causal", 1, 4, 5, 5, 128, MASK_CAUSAL, True, None),
]


@pytest.mark.parametrize("name,B,h,m,n,dm,mask,selfattn,lengths", NARROW_CASES, ids=[c[0] for c in NARROW_CASES])
def test_mha_narrow_heads(orc, name, B, h, m, n, dm, mask, selfattn, lengths):
    dk = int(name.split("_d")[1].split("_")[0])
    xq, xkv, wq, wk, wv, wo = draw_mha(B, h, m, n, dm, seed=85, self_attention=selfattn, d_k=dk)
    lens = np.full(B, n, dtype=np.int32)
    if lengths is not None:
        lens = np.random.default_rng(86).integers(lengths[0], lengths[1] + 1, size=B).astype(np.int32)
    out = attn.attn_mha_fwd(dev(xq), dev(xkv), dev(wq), dev(wk), dev(wv), dev(wo), h,
                            torch.from_numpy(lens).cuda(), mask)  # default scale: 1/sqrt(d_k)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    ref = mha.mha_fwd(orc, xq, xkv, wq, wk, wv, wo, h, lens, mask, dk ** -0.5)
    got = as_f64(out)
    assert np.abs(got - ref).max() <= 2e-2, report(got, ref, 2e-2)


def test_mha_benchmarked_size(orc):
    """The benchmarked call at full size and with its inputs: B32 sentences of 256
    positions, d_model 1024, h 16, key padding with lengths in [128, 256] (the same
    seeds as the benchmark), every output element against the oracle."""
    B, h, L, dm = 32, 16, 256, 1024
    xq, _, wq, wk, wv, wo = draw_mha(B, h, L, L, dm, seed=1007, self_attention=True)
    lens = np.random.default_rng(1008).integers(128, 257, size=B).astype(np.int32)
    x = dev(xq)
    out = attn.attn_mha_fwd(x, x, dev(wq), dev(wk), dev(wv), dev(wo), h, torch.from_numpy(lens).cuda(),
                            MASK_KEY_PADDING, 0.125)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    ref = mha.mha_fwd(orc, xq, xq, wq, wk, wv, wo, h, lens, MASK_KEY_PADDING, 0.125)
    got = as_f64(out)
    assert np.abs(got - ref).max() <= 2e-2, report(got, ref, 2e-2)
