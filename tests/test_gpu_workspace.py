"""attn_fwd_ws (dynamic tile schedule through a caller-owned workspace) on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from workloads import WORKLOADS, MASK_CAUSAL, MASK_KEY_PADDING, Workload, draw, sample_rows

from gpu_helpers import as_f64, report, to_device

pytestmark = pytest.mark.gpu


def _dev(inp):
    w = inp.workload
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    return q, k, v, torch.from_numpy(inp.key_lengths).cuda()


@pytest.mark.parametrize("cfg,shape", [
    (5, dict(B=1, h=3, m=1000, n=1000)),
    (4, dict(B=5)),
    (2, dict(B=7)),
    (3, dict()),
])
def test_workspace_matches_static_schedule_bitwise(cfg, shape):
    w = WORKLOADS[cfg].with_(**shape)
    inp = draw(w)
    q, k, v, lens = _dev(inp)
    ws = attn.make_workspace()
    static = attn.attn_fwd(q, k, v, lens, w.mask, w.scale)
    for _ in range(3):  # the workspace is reused: each call must leave it zeroed
        dyn = attn.attn_fwd(q, k, v, lens, w.mask, w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert attn.device_status()[0] == 0
        assert torch.equal(dyn, static)
        assert int(ws.count_nonzero()) == 0
    ref = oracle.load().attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    got = as_f64(dyn)
    assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)


def test_workspace_full_size_long_causal():
    w = WORKLOADS[5]
    inp = draw(w)
    q, k, v, lens = _dev(inp)
    ws = attn.make_workspace()
    out = attn.attn_fwd(q, k, v, lens, w.mask, w.scale, workspace=ws)
    torch.cuda.synchronize()
    assert attn.device_status()[0] == 0 and int(ws.count_nonzero()) == 0
    rows = sample_rows(w, 768, seed=11)
    ref = oracle.load().attn_rows(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale, rows)
    got = as_f64(out).reshape(-1, w.d)[rows]
    assert np.abs(got - ref).max() <= 1e-2, report(got, ref, 1e-2)
