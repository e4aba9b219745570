"""Shared helpers for the GPU parity tests: move seeded inputs to the device,
run one kernel through the C ABI, compare with the fp64 oracle."""
import numpy as np
import torch

import transformer_scaled_dot_masked_gb300 as attn

BF16_TOL = 1e-2   # max abs error, bf16 inputs/outputs
FP32_TOL = 1e-4   # max abs error, fp32 path


def to_device(x: np.ndarray, dtype: str):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def run(inp, kernel=attn.KERNEL_AUTO, scale=None, out=None):
    w = inp.workload
    q, k, v = (to_device(x, w.dtype) for x in (inp.q, inp.k, inp.v))
    lens = torch.from_numpy(inp.key_lengths).cuda()
    res = attn.attn_fwd(q, k, v, lens, w.mask, w.scale if scale is None else scale, out=out, kernel=kernel)
    torch.cuda.synchronize()
    st, info = attn.device_status()
    assert st == 0, f"device status {st} (info {info})"
    return res


def as_f64(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def tol_for(w):
    return BF16_TOL if w.dtype == "bf16" else FP32_TOL


def rounding_bound(ref, tol=BF16_TOL):
    """Per-element bound for bf16 outputs: tol, plus the output's own half-ulp where
    |ref| >= 4 (the spacing of bf16 there is 2^-5, so a correctly rounded output can be
    up to 0.0156 from the exact value, beyond 1e-2 by its rounding alone)."""
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 8)
    return tol + np.where(np.abs(ref) >= 4.0, half_ulp, 0.0)


def report(got, ref, tol):
    err = np.abs(got - ref)
    worst = np.unravel_index(int(err.argmax()), err.shape)
    return (f"max abs err {err.max():.3e} (tol {tol}) at {worst}: got {got[worst]:.6f} "
            f"ref {ref[worst]:.6f}")
