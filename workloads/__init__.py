"""Seeded synthetic inputs for masked scaled dot-product attention.

This module only *draws* inputs: query/key/value tensors of iid N(0, 1) values
and per-sequence valid key lengths.  It holds none of the attention arithmetic,
so that both the CUDA path and the CPU oracle can be fed the exact same bytes
without sharing any of the method's code.

Workloads stand in for the activations the Transformer's attention sub-layers
see (there is no dataset here):

* base model width, d_model = 512 with h = 8 heads of d_k = 64
  ("Paper Deep Reading: Attention Is All You Need", §03 Architecture, "dimensions");
* big model width, d_model = 1024 with h = 16 heads;
* sentences batched by similar length, so a batch holds a spread of valid
  lengths below the padded length ("Attention Is All You Need" slide deck,
  "Training Details").

Random draws (order matters for reproducibility): with
``rng = numpy.random.default_rng(seed)``, first the key lengths
(``rng.integers(lo, hi + 1, size=B)``, inclusive range) when the workload has a
key-padding mask, then Q ``[B,h,m,d]``, K ``[B,h,n,d]`` and V ``[B,h,n,d]`` from
``rng.standard_normal(dtype=float32)``.  bf16 workloads round those float32
values to bf16 with round-to-nearest-even; the resulting 16-bit patterns are
what both sides receive.  Padded key/value rows keep their random values so a
masking bug cannot hide behind zeros.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple

import numpy as np

# Mask kinds are bit flags; 3 = key padding AND causal.
MASK_NONE = 0
MASK_KEY_PADDING = 1
MASK_CAUSAL = 2


@dataclass(frozen=True)
class Workload:
    """Shape, mask and seed of one attention forward call."""

    name: str
    dtype: str  # "bf16" or "fp32"
    B: int
    h: int
    m: int  # number of queries
    n: int  # number of keys / values
    d: int  # d_k == d_v
    mask: int
    scale: float
    seed: int
    lengths: Optional[Tuple[int, int]] = None  # inclusive [lo, hi] for key padding
    description: str = field(default="", compare=False)

    @property
    def causal(self) -> bool:
        return bool(self.mask & MASK_CAUSAL)

    @property
    def padded(self) -> bool:
        return bool(self.mask & MASK_KEY_PADDING)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five reference workloads.  Seeds are 1000 + workload number.
WORKLOADS = {
    1: Workload("sdpa_fp32_single_head", "fp32", 1, 1, 16, 16, 64, MASK_NONE, 0.125, 1001,
                description="single-head SDPA, fp32, B=1 h=1 n=m=16 d_k=64, no mask"),
    2: Workload("encoder_self_attention_padding", "bf16", 64, 8, 100, 100, 64, MASK_KEY_PADDING,
                0.125, 1002, (10, 100),
                description="encoder self-attention, bf16, B=64 h=8 n=m=100 d_k=64, "
                            "key padding with lengths uniform in [10,100]"),
    3: Workload("decoder_self_attention_causal", "bf16", 32, 8, 128, 128, 64, MASK_CAUSAL,
                0.125, 1003,
                description="decoder masked self-attention, bf16, B=32 h=8 n=m=128 d_k=64, causal"),
    4: Workload("cross_attention_padding", "bf16", 32, 16, 128, 160, 64, MASK_KEY_PADDING,
                0.125, 1004, (40, 160),
                description="encoder-decoder cross-attention, bf16, B=32 h=16 m=128 n=160 d_k=64, "
                            "key padding with lengths uniform in [40,160]"),
    5: Workload("long_causal_self_attention", "bf16", 4, 16, 8192, 8192, 64, MASK_CAUSAL,
                0.125, 1005,
                description="long causal self-attention, bf16, B=4 h=16 n=m=8192 d_k=64"),
}


# One incremental-decoding step against a key/value cache: 16 sentences x beam 4,
# the big model's 16 heads, one new query row each, caches of capacity 4096 holding
# 1024..4096 positions.  Same draw order as the others (lengths, then Q, K, V).
DECODE = Workload("decode_step_kv_cache", "bf16", 64, 16, 1, 4096, 64, MASK_KEY_PADDING, 0.125, 1006,
                  (1024, 4096),
                  description="decode step, bf16, B=64 (16 x beam 4) h=16 m=1 against K/V caches of "
                              "capacity 4096 holding 1024..4096 rows, d_k=64")


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even.

    Inputs are finite by construction (normal draws), so NaN handling is not
    needed.  This is input *encoding* only: the kernels read these bits as
    bf16 and the oracle widens them itself.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for inspection in tests)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass
class Inputs:
    """One draw of a workload.  For bf16, q/k/v hold uint16 bit patterns."""

    workload: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    key_lengths: np.ndarray  # int32 [B]; all n when the workload has no padding


def draw(w: Workload, seed: Optional[int] = None) -> Inputs:
    """Draw Q, K, V (and key lengths) for workload ``w`` in the documented order."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    if w.padded:
        lo, hi = w.lengths if w.lengths is not None else (0, w.n)
        lens = rng.integers(lo, hi + 1, size=w.B).astype(np.int32)
    else:
        lens = np.full(w.B, w.n, dtype=np.int32)
    q = rng.standard_normal(size=(w.B, w.h, w.m, w.d), dtype=np.float32)
    k = rng.standard_normal(size=(w.B, w.h, w.n, w.d), dtype=np.float32)
    v = rng.standard_normal(size=(w.B, w.h, w.n, w.d), dtype=np.float32)
    if w.dtype == "bf16":
        q, k, v = round_to_bf16_bits(q), round_to_bf16_bits(k), round_to_bf16_bits(v)
    elif w.dtype != "fp32":
        raise ValueError(f"unknown dtype {w.dtype!r}")
    return Inputs(w, q, k, v, lens)


def draw_dout(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """An upstream gradient dO for workload ``w``: standard normal [B, h, m, d] from its
    own generator (seed 2000 + the workload's seed unless given), rounded like the inputs."""
    rng = np.random.default_rng(2000 + w.seed if seed is None else seed)
    g = rng.standard_normal(size=(w.B, w.h, w.m, w.d), dtype=np.float32)
    return round_to_bf16_bits(g) if w.dtype == "bf16" else g


def draw_mha(B: int, h: int, m: int, n: int, d_model: int, seed: int, self_attention: bool, d_k: int = 64):
    """Inputs of one multi-head call: Xq [B, m, d_model], Xkv [B, n, d_model] (Xq itself for
    self-attention) standard normal, and W^Q, W^K, W^V [d_model, h*d_k], W^O [h*d_k, d_model]
    normal with variance 1/fan_in (so projected values stay of order one); all rounded to
    bf16, drawn in that order from default_rng(seed)."""
    rng = np.random.default_rng(seed)
    xq = rng.standard_normal((B, m, d_model), dtype=np.float32)
    xkv = xq if self_attention else rng.standard_normal((B, n, d_model), dtype=np.float32)
    ws = [rng.standard_normal((d_model, h * d_k), dtype=np.float32) / np.float32(np.sqrt(d_model))
          for _ in range(3)]
    wo = rng.standard_normal((h * d_k, d_model), dtype=np.float32) / np.float32(np.sqrt(h * d_k))
    r = round_to_bf16_bits
    return r(xq), r(xkv), r(ws[0]), r(ws[1]), r(ws[2]), r(wo)


def sample_rows(w: Workload, count: int, seed: int = 7) -> np.ndarray:
    """Linear output-row ids ``((b*h + head)*m + i)`` spread over a workload.

    Always includes the first and last row of every 128-row query tile of the
    first and last (b, head) pair, then fills up with uniform random rows.
    Used to check full-size outputs one row at a time.
    """
    rows = set()
    for bh in {0, w.B * w.h - 1}:
        for t0 in range(0, w.m, 128):
            for i in (t0, min(t0 + 127, w.m - 1)):
                rows.add(bh * w.m + i)
    rng = np.random.default_rng(seed)
    total = w.B * w.h * w.m
    while len(rows) < min(count, total):
        rows.add(int(rng.integers(0, total)))
    return np.array(sorted(rows), dtype=np.int64)
