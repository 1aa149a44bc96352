"""Textbook dense attention in numpy matrix form, used only to pin the oracle.

It is written independently of the oracle: whole score matrices, scipy's softmax
and logsumexp, an explicit mask matrix, numpy matmuls.  Tiny sizes only.
"""
import numpy as np
from scipy.special import logsumexp, softmax


def dense_attention(q, k, v, scale, causal=False, window=None):
    """q [Lq, D], k/v [Lk, D] -> (o [Lq, D], lse [Lq]).  ``window`` = (left,
    right): query i sees keys i-left .. i+right (None: that side open)."""
    s = scale * (q @ k.T)
    lq, lk = s.shape
    row, col = np.arange(lq)[:, None], np.arange(lk)[None, :]
    hidden = np.zeros((lq, lk), dtype=bool)
    if causal:
        hidden |= col > row
    if window is not None:
        left, right = window
        if left is not None:
            hidden |= col < row - left
        if right is not None:
            hidden |= col > row + right
    s = np.where(hidden, -np.inf, s)
    return softmax(s, axis=1) @ v, logsumexp(s, axis=1)


def packed_dense(q, k, v, offsets, scale, causal=False, nq=0, window=None):
    """Loop over sequences and heads of packed [rows, H, D] buffers, calling
    dense_attention on each unpacked piece (GQA: head h reads kv head h // (H/Hkv))."""
    H, Hkv = q.shape[1], k.shape[1]
    G = H // Hkv
    B = len(offsets) - 1
    rows = B * nq if nq else int(offsets[-1])
    o = np.zeros((rows, H, q.shape[2]))
    lse = np.zeros((H, rows))
    for b in range(B):
        a, e = int(offsets[b]), int(offsets[b + 1])
        for h in range(H):
            if nq:
                if e == a:
                    o[b * nq:(b + 1) * nq, h] = 0.0
                    lse[h, b * nq:(b + 1) * nq] = -np.inf
                    continue
                ob, lb = dense_attention(q[:, h], k[a:e, h // G], v[a:e, h // G], scale)
                o[b * nq:(b + 1) * nq, h] = ob
                lse[h, b * nq:(b + 1) * nq] = lb
            else:
                if e == a:
                    continue
                ob, lb = dense_attention(q[a:e, h], k[a:e, h // G], v[a:e, h // G], scale, causal, window)
                o[a:e, h] = ob
                lse[h, a:e] = lb
    return o, lse
