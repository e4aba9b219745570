"""bench.py's check of the timed buffers, on CPU: the oracle outputs its CPU-baseline
leg computes are compared with the outputs the timed launches wrote, for every
short workload by name, at the tests' bars.  Here the "timed outputs" are the
oracle's own (every check passes with error 0) except one workload with a planted
error just above its bar, which the check must report."""
import numpy as np

import bench
from workloads import WORKLOADS, draw


def test_timed_outputs_are_checked_by_name(oracle_lib):
    outs = {}
    for cfg in (1, 2, 3, 4):
        w = WORKLOADS[cfg]
        inp = draw(w)
        outs[w.name] = oracle_lib.attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    bad = WORKLOADS[3]
    planted = outs[bad.name].copy()
    planted.reshape(-1)[12345] += 1.5 * bench.parity_tol(bad)
    outs[bad.name] = planted
    parity = {}
    bench.cpu_per_config({"tflops_useful": 0.0}, outs, parity)
    assert set(parity) == {WORKLOADS[c].name for c in (1, 2, 3, 4)}
    for cfg in (1, 2, 4):
        entry = parity[WORKLOADS[cfg].name]
        assert entry["ok"] and entry["max_abs_err"] == 0.0, entry
        assert entry["elements"] == outs[WORKLOADS[cfg].name].size
    entry = parity[bad.name]
    assert not entry["ok"]
    assert np.isclose(entry["max_abs_err"], 1.5 * bench.parity_tol(bad))


def test_parity_bars():
    assert bench.parity_tol(WORKLOADS[1]) == 1e-4  # fp32
    for cfg in (2, 3, 4, 5):
        assert bench.parity_tol(WORKLOADS[cfg]) == 1e-2  # bf16
