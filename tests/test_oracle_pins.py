"""The fp64 oracle against the pages' worked examples, closed forms and invariants."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_widening_is_exact(oracle_lib):
    import numpy as np
    from workloads import round_to_bf16_bits, bf16_bits_to_float32
    x = np.random.default_rng(3).standard_normal(1000).astype(np.float32)
    bits = round_to_bf16_bits(x)
    np.testing.assert_array_equal(oracle_lib.widen(bits), bf16_bits_to_float32(bits).astype(np.float64))
    np.testing.assert_array_equal(oracle_lib.widen(x), x.astype(np.float64))


def test_rows_match_full(oracle_lib):
    import numpy as np
    from workloads import WORKLOADS, draw, sample_rows
    w = WORKLOADS[4].with_(B=2, h=3)
    inp = draw(w)
    full = oracle_lib.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    rows = sample_rows(w, 40)
    part = oracle_lib.attn_rows(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale, rows)
    np.testing.assert_array_equal(part, full.reshape(-1, w.d)[rows])


def test_bwd_heads_subset_matches_full(oracle_lib):
    import numpy as np
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((2, 3, 9, 4)) for _ in range(4))
    lens = np.array([4, 9], dtype=np.int32)
    full = oracle_lib.attn_bwd(q, k, v, do, lens, 3, 0.5)
    heads = np.array([1, 4])
    part = oracle_lib.attn_bwd(q, k, v, do, lens, 3, 0.5, heads=heads)
    for f, g in zip(full, part):
        f, g = f.reshape(6, 9, 4), g.reshape(6, 9, 4)
        np.testing.assert_array_equal(g[heads], f[heads])
        assert np.isnan(np.delete(g, heads, axis=0)).all()

