"""fp64 multi-head attention with its projections (test infrastructure only).

NOT part of the product path: only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import it.

The MultiHead equation of "Paper Deep Reading: Attention Is All You Need", §04
(and the slide deck's "Multi-Head Attention" slide):

    head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V),
    MultiHead(Q, K, V) = Concat(head_1, ..., head_h) W^O,

with d_k = d_v = d_model / h and no bias terms (the formula has none).  The
per-head matrices are stored stacked as column blocks: W^Q, W^K, W^V are
[d_model, h * d_k] with head i in columns i * d_k .. (i + 1) * d_k, and W^O is
[h * d_k, d_model]; Concat puts head 1 first along the feature axis.  The
attention step is the pinned C oracle (``oracle.Oracle.attn_fwd``); the
projections are plain matrix products (numpy, float64).
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def mha_fwd(orc, xq, xkv, wq, wk, wv, wo, h: int, key_lengths: Optional[np.ndarray], mask_kind: int,
            scale: float, window: Optional[int] = None) -> np.ndarray:
    """xq [B, m, d_model], xkv [B, n, d_model] (bf16 bits, float32 or float64); returns
    MultiHead(xq, xkv, xkv) as float64 [B, m, d_model]."""
    xq, xkv, wq, wk, wv, wo = (orc.widen(x) for x in (xq, xkv, wq, wk, wv, wo))
    B, m, dm = xq.shape
    n = xkv.shape[1]
    hd = wq.shape[1]
    if hd % h or wk.shape != wq.shape or wv.shape != wq.shape or wo.shape != (hd, wo.shape[1]):
        raise ValueError("projection shapes do not match h")
    dk = hd // h
    # the h projections at once: column block i of the product is the i-th head's
    heads = lambda x, w, L: (x @ w).reshape(B, L, h, dk).transpose(0, 2, 1, 3)
    Q, K, V = heads(xq, wq, m), heads(xkv, wk, n), heads(xkv, wv, n)
    O = orc.attn_fwd(np.ascontiguousarray(Q), np.ascontiguousarray(K), np.ascontiguousarray(V), key_lengths,
                     mask_kind, scale, window=window)
    concat = O.transpose(0, 2, 1, 3).reshape(B, m, hd)
    return concat @ wo
