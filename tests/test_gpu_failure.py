"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every mbarrier wait of the tensor-core kernels gives up after a time limit, records
the time-out in a device status word, lets the kernel drain its own copies and MMAs,
free its TMEM and exit, and leaves the CUDA context usable.  The test hook
attn_test_withheld_arrival runs the whole-head-resident kernel with a 20 ms limit and
the barrier of the first chunk of weights waiting for one arrival more than the row
threads make, so the MMA issuer's wait for that chunk runs out (no other wait can:
each completes in microseconds).  Its
long-key variant (above 192 keys, the held chunks) and query tiles are covered too.
"""
import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_masked_gb300 as attn
from transformer_scaled_dot_masked_gb300 import _native as N
from workloads import WORKLOADS, draw

from gpu_helpers import BF16_TOL, as_f64, report, to_device

pytestmark = pytest.mark.gpu

SITE_RESIDENT_WEIGHTS = 403  # 400 + the resident kernel's weights-wait site


def _withheld(inp, out, wait_ns):
    w = inp.workload
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).cuda()
    dims = N.make_dims(w.B, w.h, w.m, w.n, w.d, N.DTYPE_BF16)
    st = N.test_withheld_arrival_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), lens.data_ptr(), w.mask, w.scale,
                                     out.data_ptr(), dims, wait_ns, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("cfg,shape", [(3, dict(B=1, h=1)), (4, dict(B=2, h=2)),
                                       (4, dict(B=2, h=2, m=200, n=256, lengths=(200, 256)))],
                         ids=["causal_128", "cross_160", "two_query_tiles_256_keys"])
def test_wait_runs_out_and_context_survives(cfg, shape):
    w = WORKLOADS[cfg].with_(**shape)
    inp = draw(w)
    assert attn.device_status() == (0, 0)
    out = torch.full((w.B, w.h, w.m, w.d), 7.0, dtype=torch.bfloat16, device="cuda")
    assert _withheld(inp, out, 20_000_000) == N.ATTN_OK
    st, info = attn.device_status()
    assert st == N.ATTN_ERR_DEVICE_TIMEOUT and info == SITE_RESIDENT_WEIGHTS, (st, info)
    assert (out == 7.0).all(), "a kernel that gave up must not store its output"
    assert attn.device_status() == (0, 0), "the record is cleared once read"
    # the same context runs the next call normally, on the same kernel
    got = as_f64(attn.attn_fwd(*(to_device(x, "bf16") for x in (inp.q, inp.k, inp.v)),
                               torch.from_numpy(inp.key_lengths).cuda(), w.mask, w.scale))
    torch.cuda.synchronize()
    assert attn.device_status() == (0, 0)
    ref = oracle.load().attn_fwd(inp.q, inp.k, inp.v, inp.key_lengths, w.mask, w.scale)
    assert np.abs(got - ref).max() <= BF16_TOL, report(got, ref, BF16_TOL)


def test_hook_rejects_what_it_cannot_run():
    w = WORKLOADS[5].with_(B=1, h=1, m=300, n=300)  # more than 256 keys: not the resident kernel
    inp = draw(w)
    out = torch.empty((w.B, w.h, w.m, w.d), dtype=torch.bfloat16, device="cuda")
    assert _withheld(inp, out, 20_000_000) == 6  # ATTN_ERR_UNSUPPORTED
    w = WORKLOADS[3].with_(B=1, h=1)
    inp = draw(w)
    out = torch.empty((w.B, w.h, w.m, w.d), dtype=torch.bfloat16, device="cuda")
    assert _withheld(inp, out, 10) == 9      # wait limit out of range: ATTN_ERR_VALUE
    assert attn.device_status() == (0, 0)
