"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics.

Each ``pin_*`` function takes an ``oracle.Oracle`` handle and raises
``AssertionError`` when the oracle disagrees with the fact it checks.  The
same functions run against the real oracle (``test_oracle_pins.py``) and
against deliberately broken copies of it (``test_oracle_mutants.py``), which
shows that a plausible mistake anywhere in the oracle fails at least one pin.

Sources:
* worked 2x2 example and two-head example: "Attention Is All You Need --
  Paper Primer" (paperglide), worked examples of scaled dot-product and
  multi-head attention (golden files under ``tests/golden/``);
* mask semantics: "Paper Deep Reading: Attention Is All You Need", §03
  "Decoder layer" (future connections set to -inf before the softmax) and §04
  (M masks padding in the encoder, future positions in the decoder);
* softmax normalisation and the weighted sum of values: the attention
  equation on the slide deck ("Scaled Dot-Product Attention") and §04;
* a library routine: torch's fp64 CPU ``scaled_dot_product_attention``.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PAD, CAUSAL = 1, 2


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _as4(x):
    return np.asarray(x, dtype=np.float64)[None, None]


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def pin_worked_example_printed(o):
    """Scale 1 reproduces the printed softmax rows and output to printed precision."""
    g = _golden("worked_sdpa_2x2.json")
    tol = g["printed"]["printed_precision"]
    Q, K, V = _as4(g["Q"]), _as4(g["K"]), _as4(g["V"])
    np.testing.assert_allclose((Q[0, 0] @ K[0, 0].T), g["printed"]["QKt"], atol=0)
    out = o.attn_fwd(Q, K, V, None, 0, 1.0)[0, 0]
    np.testing.assert_allclose(out, g["printed"]["output"], atol=tol)
    # V = I turns the output into the softmax weights themselves
    w = o.attn_fwd(Q, K, _as4(np.eye(2)), None, 0, 1.0)[0, 0]
    np.testing.assert_allclose(w, g["printed"]["softmax_rows"], atol=tol)


def pin_worked_example_closed_form(o):
    """At the stated scale 1/sqrt(2): row 2 weights are 1/(1+e^-sqrt2) and 1 - that."""
    g = _golden("worked_sdpa_2x2.json")
    Q, K, V = _as4(g["Q"]), _as4(g["K"]), _as4(g["V"])
    p = 1.0 / (1.0 + math.exp(-math.sqrt(2.0)))
    out = o.attn_fwd(Q, K, V, None, 0, g["printed"]["stated_scale"])[0, 0]
    np.testing.assert_allclose(out, [[2.5, 2.5], [5 * p, 5 * (1 - p)]], rtol=0, atol=1e-12)
    w = o.attn_fwd(Q, K, _as4(np.eye(2)), None, 0, 1 / math.sqrt(2))[0, 0]
    np.testing.assert_allclose(w, [[0.5, 0.5], [p, 1 - p]], rtol=0, atol=1e-12)


def pin_two_head_layout(o):
    """Two heads with swapped features, concatenated along features (head 1 first)."""
    g1 = _golden("worked_sdpa_2x2.json")
    g = _golden("worked_mha_2head.json")
    tol = g["printed"]["printed_precision"]
    P = np.array([[0.0, 1.0], [1.0, 0.0]])
    Q1, K1, V1 = (np.asarray(g1[x], dtype=np.float64) for x in ("Q", "K", "V"))
    Q = np.stack([Q1, Q1 @ P])[None]  # [B=1, h=2, m=2, d=2]
    K = np.stack([K1, K1 @ P])[None]
    V = np.stack([V1, V1 @ P])[None]
    out = o.attn_fwd(Q, K, V, None, 0, 1.0)[0]  # [h, m, d]
    np.testing.assert_allclose(out[0], g["printed"]["O1"], atol=tol)
    np.testing.assert_allclose(out[1], g["printed"]["O2"], atol=tol)
    concat = out.transpose(1, 0, 2).reshape(2, 4)  # [m, h*d]
    np.testing.assert_allclose(concat, g["printed"]["concat"], atol=tol)


def pin_rows_sum_to_one(o):
    """With every value row equal to 1, every output with an allowed key is exactly 1."""
    rng = np.random.default_rng(11)
    B, h, m, n, d = 2, 3, 9, 9, 5
    Q, K = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d)
    V = np.ones((B, h, n, d))
    lens = np.array([4, 9], dtype=np.int32)
    for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
        out = o.attn_fwd(Q, K, V, lens, mk, 0.7)
        np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


def pin_causal_future_independence(o):
    """Row i does not change when keys/values j > i change; row 0 is V[0] exactly."""
    rng = np.random.default_rng(12)
    B, h, n, d = 1, 2, 7, 4
    Q, K, V = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    base = o.attn_fwd(Q, K, V, None, CAUSAL, 0.5)
    np.testing.assert_array_equal(base[:, :, 0], V[:, :, 0])
    for i in range(n - 1):
        K2, V2 = K.copy(), V.copy()
        K2[:, :, i + 1:] = _rand(rng, B, h, n - i - 1, d) * 3
        V2[:, :, i + 1:] = _rand(rng, B, h, n - i - 1, d) * 3
        out = o.attn_fwd(Q, K2, V2, None, CAUSAL, 0.5)
        np.testing.assert_array_equal(out[:, :, : i + 1], base[:, :, : i + 1])
        assert not np.array_equal(out[:, :, i + 1:], base[:, :, i + 1:])


def pin_padding_independence(o):
    """Padded keys (j >= len_b) do not matter; len_b = 1 gives V[b, :, 0] on every row."""
    rng = np.random.default_rng(13)
    B, h, m, n, d = 3, 2, 5, 8, 4
    Q, K, V = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([3, 8, 1], dtype=np.int32)
    base = o.attn_fwd(Q, K, V, lens, PAD, 0.4)
    K2, V2 = K.copy(), V.copy()
    for b in range(B):
        K2[b, :, lens[b]:] += 5.0
        V2[b, :, lens[b]:] -= 7.0
    np.testing.assert_array_equal(o.attn_fwd(Q, K2, V2, lens, PAD, 0.4), base)
    np.testing.assert_array_equal(base[2], np.broadcast_to(V[2, :, :1], (h, m, d)))
    # the padded rows do matter once the length covers them
    assert not np.array_equal(o.attn_fwd(Q, K2, V2, np.full(B, n, np.int32), PAD, 0.4),
                              o.attn_fwd(Q, K, V, np.full(B, n, np.int32), PAD, 0.4))


def pin_uniform_scores_mean(o):
    """Q = 0 makes every allowed key equally weighted: the mean of the allowed values."""
    rng = np.random.default_rng(14)
    B, h, n, d = 2, 2, 6, 3
    Q = np.zeros((B, h, n, d))
    K, V = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([6, 2], dtype=np.int32)
    np.testing.assert_allclose(o.attn_fwd(Q, K, V, None, 0, 1.0),
                               np.broadcast_to(V.mean(axis=2, keepdims=True), V.shape), atol=1e-14)
    cum = np.cumsum(V, axis=2) / np.arange(1, n + 1)[None, None, :, None]
    np.testing.assert_allclose(o.attn_fwd(Q, K, V, None, CAUSAL, 1.0), cum, atol=1e-14)
    out = o.attn_fwd(Q, K, V, lens, PAD, 1.0)
    for b in range(B):
        np.testing.assert_allclose(out[b], np.broadcast_to(V[b, :, : lens[b]].mean(axis=1, keepdims=True),
                                                           (h, n, d)), atol=1e-14)


def pin_one_hot_limit(o):
    """Orthogonal keys with a large scale: each query picks the value of its own key."""
    rng = np.random.default_rng(15)
    n = 6
    Q = _as4(np.eye(n))
    K = _as4(np.eye(n))
    V = _as4(_rand(rng, n, n))
    out = o.attn_fwd(Q, K, V, None, 0, 80.0)
    np.testing.assert_allclose(out, V, rtol=0, atol=1e-12)


def pin_fully_masked_row_is_zero(o):
    """len_b = 0 leaves no allowed key; the output row is 0 (reading of 0/0)."""
    rng = np.random.default_rng(16)
    Q, K, V = _rand(rng, 2, 1, 3, 4), _rand(rng, 2, 1, 5, 4), _rand(rng, 2, 1, 5, 4)
    out = o.attn_fwd(Q, K, V, np.array([0, 5], np.int32), PAD, 1.0)
    np.testing.assert_array_equal(out[0], 0.0)
    assert np.abs(out[1]).sum() > 0
    out = o.attn_fwd(Q, K, V, np.array([0, 5], np.int32), PAD | CAUSAL, 1.0)
    np.testing.assert_array_equal(out[0], 0.0)


def pin_lengths_clamped(o):
    """Lengths outside [0, n] act as n (no padding) and 0 (nothing allowed)."""
    rng = np.random.default_rng(21)
    B, h, m, n, d = 2, 2, 4, 6, 3
    Q, K, V = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    out = o.attn_fwd(Q, K, V, np.array([n + 3, -2], np.int32), PAD, 0.5)
    np.testing.assert_array_equal(out[0], o.attn_fwd(Q, K, V, None, 0, 0.5)[0])
    np.testing.assert_array_equal(out[1], 0.0)


def pin_key_permutation(o):
    """Without a mask, permuting key rows and value rows together changes nothing."""
    rng = np.random.default_rng(17)
    B, h, m, n, d = 1, 2, 4, 7, 5
    Q, K, V = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    perm = rng.permutation(n)
    a = o.attn_fwd(Q, K, V, None, 0, 0.6)
    b = o.attn_fwd(Q, K[:, :, perm], V[:, :, perm], None, 0, 0.6)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)
    # ...but permuting only the values does change it
    c = o.attn_fwd(Q, K, V[:, :, perm], None, 0, 0.6)
    assert np.abs(a - c).max() > 1e-3


def pin_lengths_indexed_by_batch(o):
    """key_lengths[b] applies to every head of batch b and to no other batch."""
    rng = np.random.default_rng(18)
    B, h, m, n, d = 3, 2, 4, 6, 3
    Q, K, V = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([2, 6, 4], dtype=np.int32)
    full = o.attn_fwd(Q, K, V, lens, PAD | CAUSAL, 0.8)
    for b in range(B):
        one = o.attn_fwd(Q[b:b + 1], K[b:b + 1], V[b:b + 1], lens[b:b + 1], PAD | CAUSAL, 0.8)
        np.testing.assert_array_equal(full[b:b + 1], one)
        for head in range(h):
            ref = brute.attention(Q[b:b + 1, head:head + 1], K[b:b + 1, head:head + 1],
                                  V[b:b + 1, head:head + 1], lens[b:b + 1], PAD | CAUSAL, 0.8)
            np.testing.assert_allclose(full[b:b + 1, head:head + 1], ref, rtol=0, atol=1e-13)


def pin_brute_force(o):
    """The full-matrix formula (oracle/brute.py) on every tiny shape and mask kind."""
    rng = np.random.default_rng(19)
    for d in (1, 2, 3, 64):
        for m in range(1, 8):
            for n in range(1, 8):
                B, h = 2, 2
                Q, K, V = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
                lens = rng.integers(0, n + 1, size=B).astype(np.int32)
                scale = 1.0 / math.sqrt(d)
                for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
                    got = o.attn_fwd(Q, K, V, lens, mk, scale)
                    ref = brute.attention(Q, K, V, lens, mk, scale)
                    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13,
                                               err_msg=f"d={d} m={m} n={n} mask={mk}")


def pin_torch_sdpa(o):
    """torch's fp64 CPU scaled_dot_product_attention with a boolean mask (rows with an allowed key)."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(20)
    B, h, m, n, d = 2, 3, 11, 13, 16
    Q, K, V = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([5, 13], dtype=np.int32)
    for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
        allow = np.ones((B, 1, m, n), dtype=bool)
        if mk & CAUSAL:
            allow &= ~(np.arange(n)[None, None, None, :] > np.arange(m)[None, None, :, None])
        if mk & PAD:
            allow &= np.arange(n)[None, None, None, :] < lens[:, None, None, None]
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q), torch.from_numpy(K),
                                             torch.from_numpy(V), attn_mask=torch.from_numpy(allow),
                                             scale=0.3).numpy()
        got = o.attn_fwd(Q, K, V, lens, mk, 0.3)
        live = np.broadcast_to(allow.any(axis=3, keepdims=True), got.shape)
        np.testing.assert_allclose(got[live], ref[live], rtol=0, atol=1e-12)


ALL_PINS = [
    pin_worked_example_printed,
    pin_worked_example_closed_form,
    pin_two_head_layout,
    pin_rows_sum_to_one,
    pin_causal_future_independence,
    pin_padding_independence,
    pin_uniform_scores_mean,
    pin_one_hot_limit,
    pin_fully_masked_row_is_zero,
    pin_lengths_clamped,
    pin_key_permutation,
    pin_lengths_indexed_by_batch,
    pin_brute_force,
    pin_torch_sdpa,
]
