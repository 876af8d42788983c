"""Contiguous-KV brute force in NumPy fp64, used only to pin the oracle.

It never looks at the paged pool or the block table: it takes each sequence's
logical K/V ([ctx, n_kv, d], as the workload generator drew them), repeats the
KV heads G times along the head axis exactly as the GQA module on the page
"注意力演进与推理流程" (section 3.2) does with repeat_interleave, and evaluates
softmax(Q K^T * scale + M) V with the causal rule M_ij = 0 for j <= i, -inf
otherwise (section 1.1 of the same page), row by row, as a dense matrix product.
"""
from __future__ import annotations

import numpy as np


def _widen(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def dense_attention(q_bits, cu_q_lens, logical_k, logical_v, scale, n_q):
    """Attention of every query row against its sequence's contiguous K/V."""
    rows = []
    for b in range(len(logical_k)):
        K = _widen(logical_k[b])  # [ctx, n_kv, d]
        V = _widen(logical_v[b])
        ctx, n_kv, d = K.shape
        G = n_q // n_kv
        Kr = np.repeat(K, G, axis=1)  # [ctx, n_q, d]; head h <- KV head h // G
        Vr = np.repeat(V, G, axis=1)
        r0, r1 = int(cu_q_lens[b]), int(cu_q_lens[b + 1])
        Q = _widen(q_bits[r0:r1])  # [q_len, n_q, d]
        q_len = r1 - r0
        c = ctx - q_len
        # scores[h, i, j]
        S = np.einsum("ihd,jhd->hij", Q, Kr) * float(scale)
        i = np.arange(q_len)[:, None]
        j = np.arange(ctx)[None, :]
        S = np.where(j <= c + i, S, -np.inf)
        S = S - S.max(axis=-1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=-1, keepdims=True)
        O = np.einsum("hij,jhd->ihd", P, Vr)
        rows.append(O)
    return np.concatenate(rows, axis=0)
