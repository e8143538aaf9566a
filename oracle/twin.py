"""NumPy float64 twin of the oracle (O2): contiguous dense attention.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

It does not walk the block table row by row as the C oracle does.  Instead it
  1. gathers every row of sequence b into a dense [L, Hkv, D] array
     (logical block n of the sequence is physical block block_table[b, n];
     "Inference part 1", brunomaga, section "PagedAttention"),
  2. repeats each KV head over its group of consecutive query heads
     (``np.repeat`` along the head axis is ``repeat_interleave``, as in
     MultiHeadAttention_GQA of "Inference part 1", section "Smaller KV
     caches: MQA, GQA and MLA", and gqa_forward of "Efficient Inference"),
  3. computes dense scores Q K^T * scale, masks them with the shifted causal
     mask tril(diagonal = Sk - Sq) of scaled_dot_product_attention_kv_cache
     ("Inference part 1", section "KV cache"), and applies a row softmax
     followed by the product with V.
A query row with no visible key (Sk - Sq + j < 0) returns zeros, the same
reading the C oracle takes.
"""
from __future__ import annotations

import numpy as np


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 value of stored elements (uint16 bit patterns for the
    16-bit types, float32 otherwise)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return a.view(np.float16).astype(np.float64)
    raise ValueError(dtype)


def gather_sequence(cache: np.ndarray, table_row: np.ndarray,
                    length: int) -> np.ndarray:
    """Rows 0..length-1 of one sequence as a dense [length, Hkv, D] array."""
    NB, Hkv, bs, D = cache.shape
    n_blocks = -(-length // bs)
    blocks = cache[np.asarray(table_row[:n_blocks], dtype=np.int64)]
    # [n_blocks, Hkv, bs, D] -> [n_blocks, bs, Hkv, D] -> [n_blocks*bs, Hkv, D]
    dense = blocks.transpose(0, 2, 1, 3).reshape(n_blocks * bs, Hkv, D)
    return dense[:length]


def contiguous_attention(q: np.ndarray, k_cache: np.ndarray,
                         v_cache: np.ndarray, block_table: np.ndarray,
                         context_lens: np.ndarray, scale: float,
                         dtype: str) -> np.ndarray:
    """Float64 output [B, Q, Hq, D] of dense attention on gathered rows."""
    if q.ndim == 3:
        q = q[:, None]
    B, Q, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    out = np.zeros((B, Q, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        if L <= 0:
            continue
        k = widen(gather_sequence(k_cache, block_table[b], L), dtype)
        v = widen(gather_sequence(v_cache, block_table[b], L), dtype)
        k = np.repeat(k, group, axis=1)  # [L, Hq, D]
        v = np.repeat(v, group, axis=1)
        qb = widen(q[b], dtype)  # [Q, Hq, D]
        scores = np.einsum("jhd,ihd->hji", qb, k) * scale  # [Hq, Q, L]
        mask = np.tril(np.ones((Q, L), dtype=bool), k=L - Q)
        scores = np.where(mask[None], scores, -np.inf)
        for j in range(Q):
            if not mask[j].any():
                continue  # no visible key: output row stays zero
            s = scores[:, j, :]
            w = np.exp(s - s.max(axis=-1, keepdims=True))
            w /= w.sum(axis=-1, keepdims=True)
            out[b, j] = np.einsum("hi,ihd->hd", w, v)
    return out


def tree_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                   block_table: np.ndarray, context_lens: np.ndarray, scale: float,
                   dtype: str, tree_mask: np.ndarray) -> np.ndarray:
    """Dense twin of tree verification: the boolean visibility matrix of the
    Q tree nodes over the L rows is built from the bitmasks (every cached row
    visible; tree row k visible to node j iff bit k of mask[j] is set) and
    applied to dense scores, as in contiguous_attention."""
    B, Q, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    masks = np.broadcast_to(np.asarray(tree_mask, dtype=np.uint64), (B, Q))
    out = np.zeros((B, Q, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        if L <= 0:
            continue
        k = np.repeat(widen(gather_sequence(k_cache, block_table[b], L), dtype), group, axis=1)
        v = np.repeat(widen(gather_sequence(v_cache, block_table[b], L), dtype), group, axis=1)
        qb = widen(q[b], dtype)
        scores = np.einsum("jhd,ihd->hji", qb, k) * scale
        vis = np.zeros((Q, L), dtype=bool)
        base = L - Q
        vis[:, :max(base, 0)] = True
        for j in range(Q):
            for kk in range(Q):
                if base + kk >= 0 and (int(masks[b, j]) >> kk) & 1:
                    vis[j, base + kk] = True
        scores = np.where(vis[None], scores, -np.inf)
        for j in range(Q):
            if not vis[j].any():
                continue
            s = scores[:, j, :]
            w = np.exp(s - s.max(axis=-1, keepdims=True))
            w /= w.sum(axis=-1, keepdims=True)
            out[b, j] = np.einsum("hi,ihd->hd", w, v)
    return out


def e4m3_values() -> np.ndarray:
    """Value of each of the 256 FP8 E4M3 codes from the format's definition
    (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0 is
    subnormal; S.1111.111 is NaN), computed with NumPy."""
    c = np.arange(256)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    v = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    v = np.where((e == 15) & ((c & 7) == 7), np.nan, v)
    return sign * v


def contiguous_attention_fp8(q, k_codes, v_codes, block_table, context_lens, scale, q_dtype,
                             k_scale, v_scale):
    """contiguous_attention over an e4m3 cache: dequantise every code to
    code value * tensor scale in float64, then the dense computation."""
    table = e4m3_values()
    B = q.shape[0]
    kf = (table[k_codes] * k_scale)
    vf = (table[v_codes] * v_scale)
    # reuse the dense path on float64 caches
    if q.ndim == 3:
        q = q[:, None]
    Bq, Q, Hq, D = q.shape
    Hkv = k_codes.shape[1]
    group = Hq // Hkv
    out = np.zeros((Bq, Q, Hq, D))
    for b in range(B):
        L = int(context_lens[b])
        if L <= 0:
            continue
        k = np.repeat(gather_sequence(kf, block_table[b], L), group, axis=1)
        v = np.repeat(gather_sequence(vf, block_table[b], L), group, axis=1)
        qb = widen(q[b], q_dtype)
        s = np.einsum("jhd,ihd->hji", qb, k) * scale
        mask = np.tril(np.ones((Q, L), dtype=bool), k=L - Q)
        s = np.where(mask[None], s, -np.inf)
        for j in range(Q):
            if not mask[j].any():
                continue
            w = np.exp(s[:, j] - s[:, j].max(axis=-1, keepdims=True))
            w /= w.sum(axis=-1, keepdims=True)
            out[b, j] = np.einsum("hi,ihd->hd", w, v)
    return out
