"""Second, independent statement of masked attention for tiny inputs (test infrastructure).

Written the way the formula is printed in "Paper Deep Reading: Attention Is All
You Need", §04 Attention mechanics: build the whole additive mask matrix M
(0 where attention is allowed, -inf where it is not), form
softmax(Q K^T * scale + M) row by row over the full n x n score matrix, and
multiply by V.  It shares no code with ``attn_oracle.c``; the two are compared
on tiny cases in the oracle's pin tests.  Only for sizes where the full score
matrix is small.
"""
from __future__ import annotations

import numpy as np

MASK_KEY_PADDING = 1
MASK_CAUSAL = 2
MASK_WINDOW = 4


def additive_mask(m: int, n: int, mask_kind: int, length: int, window: int = 0) -> np.ndarray:
    """M for one (batch, head): -inf for future keys (causal), padded keys, and keys
    further than `window` positions from the query (restricted attention)."""
    M = np.zeros((m, n), dtype=np.float64)
    if mask_kind & MASK_WINDOW:
        far = np.abs(np.arange(n)[None, :] - np.arange(m)[:, None]) > window
        M[far] = -np.inf
    if mask_kind & MASK_CAUSAL:
        future = np.arange(n)[None, :] > np.arange(m)[:, None]
        M[future] = -np.inf
    if mask_kind & MASK_KEY_PADDING:
        M[:, max(0, min(length, n)):] = -np.inf
    return M


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, key_lengths, mask_kind: int,
              scale: float, window: int = 0) -> np.ndarray:
    """q [B,h,m,d], k/v [B,h,n,d] float64 -> [B,h,m,d]; rows with no allowed key are 0."""
    B, h, m, d = q.shape
    n = k.shape[2]
    out = np.zeros((B, h, m, d), dtype=np.float64)
    for b in range(B):
        length = n if key_lengths is None else int(key_lengths[b])
        M = additive_mask(m, n, mask_kind, length, window)
        for head in range(h):
            S = (q[b, head] @ k[b, head].T) * scale + M
            top = S.max(axis=1, keepdims=True)
            live = np.isfinite(top[:, 0])
            E = np.zeros_like(S)
            E[live] = np.exp(S[live] - top[live])
            P = np.zeros_like(S)
            P[live] = E[live] / E[live].sum(axis=1, keepdims=True)
            out[b, head] = P @ v[b, head]
    return out
