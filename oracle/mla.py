"""Float64 oracle of multi-head latent attention (MLA) decode over a paged
latent cache.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): the product path never
imports it, and it shares no code with the CUDA path.

What MLA computes ("Inference part 1", brunomaga, section "Smaller KV caches:
MQA, GQA and MLA"): every token's keys and values are compressed into one
small latent vector c, and only c is cached.  Per-head keys and values are
linear up-projections of c (K_h = W_uk,h c, V_h = W_uv,h c); those matrices
can be absorbed into the query and output projections, so that attention
runs directly over the cached latents, which play the part of both keys and
values: multi-query attention with one large shared head.  Rotary position
embeddings do not commute with the absorption, so MLA keeps a small separate
key part that carries the position, cached beside c ("KV cache, prefill va
decode", section 04 on MLA: d_c = 512 latent values and d_h^R = 64 rotary
values per token and layer).

Readings taken here (the pages give the algebra, not a kernel interface):
  * a cache row is [c (d_c values) ; k_rope (d_r values)], one row per token,
    paged like the other caches: row i of sequence b is row i % bs of
    physical block block_table[b][i // bs] ("Inference part 1", section
    "PagedAttention");
  * the absorbed query of head h is [q_c,h ; q_r,h] with q_c,h = W_uk,h^T
    q_nope,h (d_c values) and q_r,h the rotated query part (d_r values);
  * score_{h,i} = scale (<q_c,h, c_i> + <q_r,h, k_rope_i>), one dot product
    over the whole d_c + d_r row;
  * the output of head h is the latent sum_i softmax_i(score_h) c_i (d_c
    values); the caller applies W_uv,h (and the output projection) to it.
The softmax is the two-pass textbook form (maximum, then exponentials and
their sum), as in the other oracles here.
"""
from __future__ import annotations

import numpy as np

from .twin import widen


def _values(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements; "f64" arrays are taken as is."""
    return a.astype(np.float64) if dtype == "f64" else widen(a, dtype)


def gather_latents(cache: np.ndarray, table_row: np.ndarray, length: int) -> np.ndarray:
    """Rows 0..length-1 of one sequence of a [NB, bs, W] latent cache as a
    dense [length, W] array."""
    NB, bs, W = cache.shape
    n_blocks = -(-length // bs)
    rows = cache[np.asarray(table_row[:n_blocks], dtype=np.int64)].reshape(n_blocks * bs, W)
    return rows[:length]


def mla_decode(q: np.ndarray, ckv_cache: np.ndarray, block_table: np.ndarray,
               context_lens: np.ndarray, d_c: int, scale: float, dtype: str) -> np.ndarray:
    """Absorbed MLA decode, float64.

    q [B, H, d_c + d_r] and ckv_cache [NB, bs, d_c + d_r] in storage form
    (uint16 bit patterns for bf16 / f16, float32 for f32, float64 for
    "f64"); block_table [B, max_blocks]; context_lens [B].  Returns out
    [B, H, d_c]: for head h of sequence b, sum_i softmax_i(scale q[b, h] .
    row_i) row_i[:d_c] over the rows i < L_b.  A sequence with L_b = 0
    gives zeros."""
    B, H, W = q.shape
    assert ckv_cache.shape[2] == W and 0 < d_c <= W
    out = np.zeros((B, H, d_c), dtype=np.float64)
    for b in range(B):
        L = int(context_lens[b])
        if L <= 0:
            continue
        rows = _values(gather_latents(ckv_cache, block_table[b], L), dtype)  # [L, W]
        qb = _values(q[b], dtype)                                              # [H, W]
        s = (qb @ rows.T) * scale                                             # [H, L]
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        out[b] = w @ rows[:, :d_c]
    return out


# ---- the same attention before absorption (for the pins) ------------------
def absorb_query(q_nope: np.ndarray, q_rope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """[q_c ; q_r] per head: q_c,h = W_uk,h^T q_nope,h.

    q_nope [H, dh], q_rope [H, d_r], w_uk [H, dh, d_c] -> [H, d_c + d_r]."""
    q_c = np.einsum("hd,hdc->hc", q_nope, w_uk)
    return np.concatenate([q_c, q_rope], axis=1)


def expand_output(out_latent: np.ndarray, w_uv: np.ndarray) -> np.ndarray:
    """Per-head outputs from latent outputs: o_h = W_uv,h out_latent,h.

    out_latent [H, d_c], w_uv [H, dv, d_c] -> [H, dv]."""
    return np.einsum("hdc,hc->hd", w_uv, out_latent)


def attention_recomputed(q_nope: np.ndarray, q_rope: np.ndarray, c: np.ndarray,
                         k_rope: np.ndarray, w_uk: np.ndarray, w_uv: np.ndarray,
                         scale: float) -> np.ndarray:
    """Multi-head attention with every head's keys and values recomputed from
    the latents (no absorption): k_h,i = [W_uk,h c_i ; k_rope_i], v_h,i =
    W_uv,h c_i, out_h = sum_i softmax_i(scale q_h . k_h,i) v_h,i with
    q_h = [q_nope,h ; q_rope,h].  c [L, d_c], k_rope [L, d_r] -> [H, dv]."""
    H = q_nope.shape[0]
    outs = []
    for h in range(H):
        k = np.concatenate([c @ w_uk[h].T, k_rope], axis=1)       # [L, dh + d_r]
        v = c @ w_uv[h].T                                           # [L, dv]
        qh = np.concatenate([q_nope[h], q_rope[h]])
        s = (k @ qh) * scale
        w = np.exp(s - s.max())
        w /= w.sum()
        outs.append(w @ v)
    return np.stack(outs)
