"""Plant plausible mistakes in a copy of the oracle; the pins must catch every one.

Each mutant is the oracle's C source with one edit (an off-by-one mask, a
dropped scale, a flipped sign, a wrong index...).  It is compiled on the CPU
into a temporary library and run against every pin; at least one pin must
fail.  The committed oracle itself is never modified.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "causal_includes_diagonal": ("j > i) return 0", "j >= i) return 0"),
    "padding_off_by_one": ("j >= len_b) return 0", "j > len_b) return 0"),
    "scale_dropped": ("w[j] = scale * dot;", "w[j] = dot;"),
    "exponent_sign_flipped": ("w[j] = exp(w[j] - mu);", "w[j] = exp(mu - w[j]);"),
    "not_normalised": ("double p = w[j] / Z;", "double p = w[j];"),
    "keys_reversed": ("dot += q[c] * Kh[j * d + c];", "dot += q[c] * Kh[(n - 1 - j) * d + c];"),
    "values_reversed": ("o[c] += p * Vh[j * d + c];", "o[c] += p * Vh[(n - 1 - j) * d + c];"),
    "query_row_of_first_position": ("const double *q = Q + r * d;", "const double *q = Q + bh * m * d;"),
    "length_of_wrong_batch": ("int64_t b = bh / h;", "int64_t b = (bh / h + 1) % B;"),
    "length_not_clamped": ("if (len > n) len = n;", "if (len > n) len = n - 1;"),
    # backward and lse
    "bwd_dq_drops_row_term": ("double ds = exp(scale * dot - mx) / z * (dp - Di);",
                              "double ds = exp(scale * dot - mx) / z * dp;"),
    "bwd_dk_drops_row_term": ("double ds = p * (dp - D[i]);", "double ds = p * dp;"),
    "bwd_row_term_unweighted": ("Di += exp(scale * dot - mx) / z * dp;", "Di += dp;"),
    "bwd_dv_uses_score_gradient": ("dv[c] += p * g[c];", "dv[c] += ds * g[c];"),
    "bwd_dk_missing_scale": ("dk[c] += scale * ds * q[c];", "dk[c] += ds * q[c];"),
    "bwd_dq_uses_values": ("dq[c] += scale * ds * kj[c];", "dq[c] += scale * ds * vj[c];"),
    "bwd_key_pass_ignores_mask": ("if (mu[i] == -INFINITY || !key_allowed(mask_kind, i, j, len_b)) continue;",
                                  "if (mu[i] == -INFINITY) continue;"),
    "bwd_upstream_of_wrong_head": ("const double *dOh = dO + bh * m * d;",
                                   "const double *dOh = dO + (bh + 1) % (B * h) * m * d;"),
    "bwd_normaliser_dropped_in_key_pass": ("double p = exp(scale * dot - mu[i]) / Z[i];",
                                           "double p = exp(scale * dot - mu[i]);"),
    "lse_missing_max": ("lse[r] = mu + log(Z);", "lse[r] = log(Z);"),
    # restricted attention
    "window_off_by_one": ("(i - j > g_window || j - i > g_window)", "(i - j >= g_window || j - i > g_window)"),
    "window_one_sided": ("(i - j > g_window || j - i > g_window)", "(i - j > g_window)"),
    "window_rows_ignores_window": ("g_window = window;\n    int rc = oracle_attn_rows(",
                                   "int rc = oracle_attn_rows("),
    "window_lse_ignores_window": ("g_window = window;\n    int rc = oracle_attn_lse(",
                                  "int rc = oracle_attn_lse("),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor {old!r} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(path), str(tmp_path / "libmutant.so"), openmp=False)
    mutant = oracle.load(lib)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"


# Mistakes planted in the multi-head oracle (oracle/mha.py): the mutated function
# replaces oracle.mha.mha_fwd while the multi-head pins run.
MHA_MUTANTS = {
    "interleaved_head_split": (".reshape(B, L, h, dk).transpose(0, 2, 1, 3)", ".reshape(B, L, dk, h).transpose(0, 3, 1, 2)"),
    "output_projection_transposed": ("return concat @ wo", "return concat @ wo.T"),
    "concat_in_head_order": ("concat = O.transpose(0, 2, 1, 3).reshape(B, m, hd)", "concat = O.reshape(B, m, hd)"),
    "keys_projected_with_value_weights": ("K, V = heads(xq, wq, m), heads(xkv, wk, n), heads(xkv, wv, n)",
                                          "K, V = heads(xq, wq, m), heads(xkv, wv, n), heads(xkv, wv, n)"),
}


@pytest.mark.parametrize("name", sorted(MHA_MUTANTS))
def test_mha_mutant_is_caught(name, monkeypatch, oracle_lib):
    import oracle.mha as mha
    old, new = MHA_MUTANTS[name]
    src = open(mha.__file__).read()
    assert src.count(old) == 1, f"mutation anchor {old!r} not found exactly once"
    ns = {}
    exec(compile(src.replace(old, new), "mha_mutant", "exec"), ns)
    monkeypatch.setattr(mha, "mha_fwd", ns["mha_fwd"])
    caught = []
    for pin in (oracle_pins.pin_mha_two_head_example, oracle_pins.pin_mha_torch,
                oracle_pins.pin_mha_identity_projections):
        try:
            pin(oracle_lib)
        except Exception:  # a wrong shape is as much a catch as a wrong value
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
