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
    """The full-matrix formula (oracle/brute.py) on every tiny shape and mask kind, at
    the head widths the kernels take (16, 32, 64, 128) and odd ones."""
    rng = np.random.default_rng(19)
    for d in (1, 2, 3, 16, 32, 64, 128):
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


# ---------------------------------------------------------------- backward and lse
# The gradients are the chain rule of the attention equation (the pages train the
# model but do not write the backward pass out).  They are pinned by the forward
# oracle itself through finite differences of sum(dO * out), by exact identities
# that follow from the softmax, and by torch's fp64 autograd.

def _bwd_case(rng, B, h, m, n, d):
    return (_rand(rng, B, h, m, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d),
            _rand(rng, B, h, m, d))


def _loss(o, Q, K, V, dO, lens, mk, scale):
    return float((dO * o.attn_fwd(Q, K, V, lens, mk, scale)).sum())


def pin_bwd_elementwise_finite_differences(o):
    """Every element of dQ, dK, dV against a central difference of sum(dO * out)."""
    rng = np.random.default_rng(31)
    eps = 1e-6
    for mk, (m, n), lens in ((0, (3, 4), None), (PAD, (3, 5), [0, 3]), (CAUSAL, (4, 4), None),
                             (PAD | CAUSAL, (4, 4), [2, 9])):
        B, h, d = 2, 2, 3
        Q, K, V, dO = _bwd_case(rng, B, h, m, n, d)
        lens_a = None if lens is None else np.array(lens, dtype=np.int32)
        grads = o.attn_bwd(Q, K, V, dO, lens_a, mk, 0.9)
        for x, g, name in zip((Q, K, V), grads, "QKV"):
            for idx in np.ndindex(x.shape):
                keep = x[idx]
                x[idx] = keep + eps
                up = _loss(o, Q, K, V, dO, lens_a, mk, 0.9)
                x[idx] = keep - eps
                down = _loss(o, Q, K, V, dO, lens_a, mk, 0.9)
                x[idx] = keep
                fd = (up - down) / (2 * eps)
                assert abs(fd - g[idx]) <= 1e-7 * (1 + abs(fd)), (name, mk, idx, fd, g[idx])


def pin_bwd_directional_finite_differences(o):
    """Larger shapes (several heads, ragged lengths): directional derivatives along random
    directions against central differences."""
    rng = np.random.default_rng(32)
    B, h, m, n, d = 3, 2, 19, 19, 8
    eps = 1e-6
    lens = np.array([19, 7, 0], dtype=np.int32)
    for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
        Q, K, V, dO = _bwd_case(rng, B, h, m, n, d)
        grads = o.attn_bwd(Q, K, V, dO, lens, mk, 0.35)
        for which in range(3):
            xs = [Q, K, V]
            Dir = rng.standard_normal(xs[which].shape)
            up = list(xs)
            up[which] = xs[which] + eps * Dir
            down = list(xs)
            down[which] = xs[which] - eps * Dir
            fd = (_loss(o, *up, dO, lens, mk, 0.35) - _loss(o, *down, dO, lens, mk, 0.35)) / (2 * eps)
            an = float((grads[which] * Dir).sum())
            assert abs(fd - an) <= 1e-6 * (1 + abs(fd)), ("QKV"[which], mk, fd, an)


def pin_bwd_softmax_identities(o):
    """Exact consequences of the softmax, per (batch, head):
    sum_j dK_j = 0 (shifting every key by one vector shifts a row's scores by a constant);
    sum_j dV_j = sum of dO over rows with an allowed key (each row's weights sum to one);
    sum_i q_i . dQ_i = sum_j k_j . dK_j (Q and K enter only through their products)."""
    rng = np.random.default_rng(33)
    B, h, m, n, d = 2, 3, 9, 12, 5
    lens = np.array([0, 8], dtype=np.int32)
    for mk in (0, PAD, PAD | CAUSAL):
        mm = n if mk & CAUSAL else m
        Q, K, V, dO = _bwd_case(rng, B, h, mm, n, d)
        dQ, dK, dV = o.attn_bwd(Q, K, V, dO, lens, mk, 0.6)
        np.testing.assert_allclose(dK.sum(axis=2), 0.0, atol=1e-12)
        live = np.ones((B, 1, mm, 1), dtype=bool)
        if mk & PAD:
            live[lens == 0] = False
        np.testing.assert_allclose(dV.sum(axis=2), (dO * live).sum(axis=2), atol=1e-12)
        np.testing.assert_allclose((Q * dQ).sum(axis=(2, 3)), (K * dK).sum(axis=(2, 3)), atol=1e-12)


def pin_bwd_uniform_scores(o):
    """Q = 0: every allowed key has weight 1/len, so dV_j is the mean of dO over the rows
    that see key j, and dQ_i = scale * sum_j (1/len)(dP_ij - mean dP_i.) k_j."""
    rng = np.random.default_rng(34)
    B, h, n, d = 1, 1, 6, 4
    Q = np.zeros((B, h, n, d))
    K, V, dO = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    dQ, dK, dV = o.attn_bwd(Q, K, V, dO, None, CAUSAL, 0.5)
    for j in range(n):
        ref = sum(dO[0, 0, i] / (i + 1) for i in range(j, n))
        np.testing.assert_allclose(dV[0, 0, j], ref, atol=1e-13)
    for i in range(n):
        dp = V[0, 0, :i + 1] @ dO[0, 0, i]
        ds = (dp - dp.mean()) / (i + 1)
        np.testing.assert_allclose(dQ[0, 0, i], 0.5 * ds @ K[0, 0, :i + 1], atol=1e-13)
    np.testing.assert_allclose(dK, 0.0, atol=1e-15)  # dS is multiplied by q_i = 0


def pin_lse(o):
    """lse against the full-matrix formula: exp(scale*QK^T + M - lse) has unit row sums,
    and uniform scores give log(len)."""
    rng = np.random.default_rng(35)
    for d in (3, 128):
        _lse_unit_row_sums(o, rng, d)
    zero = np.zeros((1, 1, 5, 3))
    K = _rand(rng, 1, 1, 5, 3)
    np.testing.assert_allclose(o.attn_lse(zero, K, None, CAUSAL, 1.0)[0, 0],
                               np.log(np.arange(1, 6)), atol=1e-14)


def _lse_unit_row_sums(o, rng, d):
    B, h, m, n = 2, 2, 7, 7
    Q, K = _rand(rng, B, h, m, d), _rand(rng, B, h, n, d)
    lens = np.array([0, 5], dtype=np.int32)
    scale = 0.7 / math.sqrt(d / 3.0)
    for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
        lse = o.attn_lse(Q, K, lens, mk, scale)
        for b in range(B):
            M = brute.additive_mask(m, n, mk, int(lens[b]))
            for head in range(h):
                S = Q[b, head] @ K[b, head].T * scale + M
                for i in range(m):
                    if np.isfinite(S[i]).any():
                        assert abs(np.exp(S[i] - lse[b, head, i]).sum() - 1.0) <= 1e-13
                    else:
                        assert lse[b, head, i] == -np.inf


def pin_bwd_torch_autograd(o):
    """torch fp64 autograd through its scaled_dot_product_attention (rows with an allowed key)."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(36)
    B, h, m, n, d = 2, 2, 10, 10, 8
    lens = np.array([4, 10], dtype=np.int32)
    for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
        Q, K, V, dO = _bwd_case(rng, B, h, m, n, d)
        allow = np.ones((B, 1, m, n), dtype=bool)
        if mk & CAUSAL:
            allow &= ~(np.arange(n)[None, None, None, :] > np.arange(m)[None, None, :, None])
        if mk & PAD:
            allow &= np.arange(n)[None, None, None, :] < lens[:, None, None, None]
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (Q, K, V))
        out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(allow), scale=0.4)
        out.backward(torch.from_numpy(dO))
        for got, ref in zip(o.attn_bwd(Q, K, V, dO, lens, mk, 0.4), (tq.grad, tk.grad, tv.grad)):
            np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- restricted attention
# Restricted self-attention: the deep-reading page's §04 complexity table lists it as
# O(r n d) with path length O(n / r); the slide deck lists local, restricted attention
# under "Limitations and Future Work".  Reading: keys with |i - j| <= w stay.
WIN = 4


def pin_window_brute_force(o):
    """The full-matrix formula with the banded mask, every tiny shape, window and mask,
    at head widths 3 and 128 (the widths windows run at on tensor cores include 128)."""
    rng = np.random.default_rng(41)
    for d in (3, 128):
        scale = 0.7 / math.sqrt(d / 3.0)
        for n in range(1, 8):
            for w in (0, 1, 2, 3, 9):
                B, h = 2, 2
                Q, K, V = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
                lens = rng.integers(0, n + 1, size=B).astype(np.int32)
                for mk in (WIN, WIN | PAD, WIN | CAUSAL, WIN | PAD | CAUSAL):
                    got = o.attn_fwd(Q, K, V, lens, mk, scale, window=w)
                    ref = brute.attention(Q, K, V, lens, mk, scale, window=w)
                    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13,
                                               err_msg=f"d={d} n={n} w={w} mask={mk}")


def pin_window_zero_copies_values(o):
    """w = 0: each query sees only its own position, so its output is that value row."""
    rng = np.random.default_rng(42)
    Q, K, V = _rand(rng, 2, 3, 9, 5), _rand(rng, 2, 3, 9, 5), _rand(rng, 2, 3, 9, 5)
    for mk in (WIN, WIN | CAUSAL):
        np.testing.assert_allclose(o.attn_fwd(Q, K, V, None, mk, 0.9, window=0), V, rtol=0, atol=1e-15)


def pin_window_wide_equals_full(o):
    """A window covering every key changes nothing (bit for bit)."""
    rng = np.random.default_rng(43)
    Q, K, V = _rand(rng, 2, 2, 11, 4), _rand(rng, 2, 2, 11, 4), _rand(rng, 2, 2, 11, 4)
    lens = np.array([5, 11], dtype=np.int32)
    for mk in (0, PAD, CAUSAL, PAD | CAUSAL):
        np.testing.assert_array_equal(o.attn_fwd(Q, K, V, lens, mk | WIN, 0.5, window=10),
                                      o.attn_fwd(Q, K, V, lens, mk, 0.5))


def pin_window_locality(o):
    """Row i is bitwise unchanged when keys and values outside [i - w, i + w] change."""
    rng = np.random.default_rng(44)
    n, w, i = 16, 3, 7
    Q, K, V = _rand(rng, 1, 1, n, 4), _rand(rng, 1, 1, n, 4), _rand(rng, 1, 1, n, 4)
    base = o.attn_fwd(Q, K, V, None, WIN, 0.8, window=w)
    K2, V2 = K.copy(), V.copy()
    far = [j for j in range(n) if abs(j - i) > w]
    K2[0, 0, far] = rng.standard_normal((len(far), 4)) * 5
    V2[0, 0, far] = rng.standard_normal((len(far), 4)) * 5
    moved = o.attn_fwd(Q, K2, V2, None, WIN, 0.8, window=w)
    np.testing.assert_array_equal(moved[0, 0, i], base[0, 0, i])
    assert not np.array_equal(moved, base)


def pin_window_torch_sdpa(o):
    """torch's fp64 scaled_dot_product_attention with a banded boolean mask."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(45)
    B, h, n, d, w = 2, 2, 13, 8, 2
    Q, K, V = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([6, 13], dtype=np.int32)
    for mk in (WIN, WIN | CAUSAL, WIN | PAD):
        allow = np.abs(np.arange(n)[None, :] - np.arange(n)[:, None]) <= w
        allow = np.broadcast_to(allow, (B, 1, n, n)).copy()
        if mk & CAUSAL:
            allow &= ~(np.arange(n)[None, None, None, :] > np.arange(n)[None, None, :, None])
        if mk & PAD:
            allow &= np.arange(n)[None, None, None, :] < lens[:, None, None, None]
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V),
                                             attn_mask=torch.from_numpy(allow), scale=0.4).numpy()
        got = o.attn_fwd(Q, K, V, lens, mk, 0.4, window=w)
        live = np.broadcast_to(allow.any(axis=3, keepdims=True), got.shape)
        np.testing.assert_allclose(got[live], ref[live], rtol=0, atol=1e-12)



def pin_window_rows(o):
    """Selected rows through the windowed row entry point equal the same rows of the
    full-matrix formula with the banded mask, for every mask kind and w in {0, 2, 9}."""
    rng = np.random.default_rng(46)
    B, h, n, d = 2, 2, 12, 5
    Q, K, V = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([7, 12], dtype=np.int32)
    rows = rng.choice(B * h * n, size=17, replace=False).astype(np.int64)
    for w in (0, 2, 9):
        for mk in (WIN, WIN | PAD, WIN | CAUSAL, WIN | PAD | CAUSAL):
            ref = brute.attention(Q, K, V, lens, mk, 0.6, window=w).reshape(B * h * n, d)[rows]
            got = o.attn_rows(Q, K, V, lens, mk, 0.6, rows, window=w)
            np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13, err_msg=f"w={w} mask={mk}")


def pin_window_lse(o):
    """Windowed log-sum-exp against the banded full-matrix formula: exp(scale*QK^T + M - lse)
    has unit row sums; with Q = 0 every allowed key scores 0, so lse = log(number of keys
    in the row's window)."""
    rng = np.random.default_rng(47)
    B, h, n, d = 2, 2, 9, 4
    Q, K = _rand(rng, B, h, n, d), _rand(rng, B, h, n, d)
    lens = np.array([0, 6], dtype=np.int32)
    for w in (0, 2, 9):
        for mk in (WIN, WIN | PAD, WIN | CAUSAL, WIN | PAD | CAUSAL):
            lse = o.attn_lse(Q, K, lens, mk, 0.7, window=w)
            for b in range(B):
                M = brute.additive_mask(n, n, mk, int(lens[b]), w)
                for head in range(h):
                    S = Q[b, head] @ K[b, head].T * 0.7 + M
                    for i in range(n):
                        if np.isfinite(S[i]).any():
                            assert abs(np.exp(S[i] - lse[b, head, i]).sum() - 1.0) <= 1e-13
                        else:
                            assert lse[b, head, i] == -np.inf
    zero = np.zeros((1, 1, n, d))
    for w in (0, 1, 3):
        got = o.attn_lse(zero, K[:1, :1], None, WIN, 1.0, window=w)[0, 0]
        count = np.array([min(n - 1, i + w) - max(0, i - w) + 1 for i in range(n)], dtype=np.float64)
        np.testing.assert_allclose(got, np.log(count), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- multi-head projections
def pin_mha_two_head_example(o):
    """The primer's two-head example through the projections: X_q = X_kv = I, head 1's
    projections give the worked 2x2 example (Q = I, K = [[1,1],[1,-1]], V = [[5,0],[0,5]]),
    head 2's are the same followed by the feature swap P, W^O = I: the output is the
    printed concatenation (scale 1, printed precision)."""
    from oracle import mha
    g = _golden("worked_mha_2head.json")
    I2, P = np.eye(2), np.array([[0.0, 1.0], [1.0, 0.0]])
    K1, V1 = np.array([[1.0, 1.0], [1.0, -1.0]]), np.array([[5.0, 0.0], [0.0, 5.0]])
    wq = np.hstack([I2, P])
    wk = np.hstack([K1, K1 @ P])
    wv = np.hstack([V1, V1 @ P])
    out = mha.mha_fwd(o, I2[None], I2[None], wq, wk, wv, np.eye(4), 2, None, 0, 1.0)
    np.testing.assert_allclose(out[0], g["printed"]["concat"], atol=g["printed"]["printed_precision"])


def pin_mha_torch(o):
    """torch's fp64 multi_head_attention_forward (separate projection weights, no biases,
    boolean mask), against the same inputs."""
    import torch
    import torch.nn.functional as F
    from oracle import mha

    rng = np.random.default_rng(71)
    B, m, n, h, dk = 2, 7, 9, 3, 4
    dm = h * dk  # d_k = d_model / h, as on the pages (and as torch requires)
    xq, xkv = rng.standard_normal((B, m, dm)), rng.standard_normal((B, n, dm))
    wq, wk, wv = (rng.standard_normal((dm, h * dk)) / np.sqrt(dm) for _ in range(3))
    wo = rng.standard_normal((h * dk, dm)) / np.sqrt(h * dk)
    lens = np.array([4, 9], dtype=np.int32)
    for mk in (0, PAD):
        allow = np.ones((B, m, n), dtype=bool)
        if mk & PAD:
            allow &= np.arange(n)[None, None, :] < lens[:, None, None]
        got = mha.mha_fwd(o, xq, xkv, wq, wk, wv, wo, h, lens, mk, dk ** -0.5)
        for b in range(B):
            t = lambda x: torch.from_numpy(np.ascontiguousarray(x))
            ref, _ = F.multi_head_attention_forward(
                t(xq[b][:, None]), t(xkv[b][:, None]), t(xkv[b][:, None]), dm, h,
                in_proj_weight=None, in_proj_bias=None, bias_k=None, bias_v=None, add_zero_attn=False,
                dropout_p=0.0, out_proj_weight=t(wo.T), out_proj_bias=None, training=False, need_weights=False,
                attn_mask=t(~allow[b]), use_separate_proj_weight=True, q_proj_weight=t(wq.T),
                k_proj_weight=t(wk.T), v_proj_weight=t(wv.T))
            np.testing.assert_allclose(got[b], ref[:, 0].numpy(), rtol=0, atol=1e-12)


def pin_mha_identity_projections(o):
    """Identity projections and W^O: each head attends over its own column block of the
    inputs, and the output is those heads side by side."""
    from oracle import mha

    rng = np.random.default_rng(72)
    B, n, h, dk = 2, 6, 2, 3
    x = rng.standard_normal((B, n, h * dk))
    I = np.eye(h * dk)
    out = mha.mha_fwd(o, x, x, I, I, I, I, h, None, CAUSAL, 0.6)
    for head in range(h):
        xs = x[:, None, :, head * dk:(head + 1) * dk]
        np.testing.assert_allclose(out[:, :, head * dk:(head + 1) * dk],
                                   brute.attention(xs, xs, xs, None, CAUSAL, 0.6)[:, 0], atol=1e-13)


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
    pin_bwd_elementwise_finite_differences,
    pin_bwd_directional_finite_differences,
    pin_bwd_softmax_identities,
    pin_bwd_uniform_scores,
    pin_lse,
    pin_bwd_torch_autograd,
    pin_window_brute_force,
    pin_window_zero_copies_values,
    pin_window_wide_equals_full,
    pin_window_locality,
    pin_window_torch_sdpa,
    pin_window_rows,
    pin_window_lse,
    pin_mha_two_head_example,
    pin_mha_torch,
    pin_mha_identity_projections,
]
