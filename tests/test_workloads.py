"""The seeded input generator: determinism, shapes, bf16 encoding, statistics."""
import numpy as np
import torch

from workloads import WORKLOADS, draw, round_to_bf16_bits, bf16_bits_to_float32, sample_rows


def test_deterministic_and_shaped():
    w = WORKLOADS[2].with_(B=4)
    a, b = draw(w), draw(w)
    for x, y in ((a.q, b.q), (a.k, b.k), (a.v, b.v), (a.key_lengths, b.key_lengths)):
        np.testing.assert_array_equal(x, y)
    assert a.q.shape == (4, 8, 100, 64) and a.q.dtype == np.uint16
    assert a.key_lengths.min() >= 10 and a.key_lengths.max() <= 100


def test_length_ranges_inclusive():
    w = WORKLOADS[4].with_(B=4000)
    lens = draw(w.with_(h=1, m=1, n=160, d=1)).key_lengths
    assert lens.min() == 40 and lens.max() == 160


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(1).standard_normal(100000).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0]  # ties to even
    ours = round_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    np.testing.assert_array_equal(bf16_bits_to_float32(ours),
                                  torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_dot_product_variance_is_dk():
    """iid unit-variance q, k give var(q.k) = d_k, so scale 1/sqrt(d_k) restores unit
    variance ("Paper Deep Reading", §04, why divide by sqrt(d_k))."""
    w = WORKLOADS[3].with_(B=8)
    inp = draw(w)
    q = bf16_bits_to_float32(inp.q).astype(np.float64)
    k = bf16_bits_to_float32(inp.k).astype(np.float64)
    dots = np.einsum("bhid,bhjd->bhij", q, k).ravel()
    assert abs(dots.var() / w.d - 1.0) < 0.03
    assert abs((dots * w.scale).var() - 1.0) < 0.03


def test_sample_rows_cover_tile_edges():
    w = WORKLOADS[5]
    rows = sample_rows(w, 3000)
    assert len(rows) == 3000 and rows.max() < w.B * w.h * w.m
    assert 127 in rows and 128 in rows and w.B * w.h * w.m - 1 in rows
