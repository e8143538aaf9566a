"""Byte accounting of the paged decode-attention path.

The KV bytes per token follow the formula of "KV cache, prefill va decode"
(truongducdung, section 03: 2 x layers x kv_heads x head_dim x bytes per
value, the 2 being K and V) and of "Inference part 1" (brunomaga, section
"KV cache"); for latent (MLA) caches one latent of kv_lora_rank + rope dims
is stored per token and layer (same section 03, DeepSeek-V3 row).

``attention_bytes`` is the algorithmic HBM traffic of one attention call:
every valid K and V row once, q once, the output once, the block-table
entries and context lengths, plus the split-K partials written and read back.
"""
from __future__ import annotations

from typing import Sequence


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int,
                       bytes_per_value: int, latent: bool = False) -> int:
    """KV-cache bytes one token occupies across all layers."""
    if latent:  # one shared latent vector (K and V derived from it)
        return layers * head_dim * bytes_per_value
    return 2 * layers * kv_heads * head_dim * bytes_per_value


def attention_bytes(context_lens: Sequence[int], num_queries: int,
                    num_heads: int, num_kv_heads: int, head_dim: int,
                    block_size: int, elt_bytes: int, num_splits_per_seq=None,
                    fused_append: bool = False, q_elt_bytes=None) -> dict:
    """Algorithmic bytes of one paged attention call, by component.  With
    ``fused_append`` the call also reads the new K/V rows and writes them into
    the cache (the rows it then reads are already counted in ``kv``).
    ``q_elt_bytes`` is the element size of q and out when it differs from the
    cache's (an FP8 cache read with bf16 queries)."""
    lens = [max(0, int(x)) for x in context_lens]
    B = len(lens)
    kv = 2 * sum(lens) * num_kv_heads * head_dim * elt_bytes
    qe = elt_bytes if q_elt_bytes is None else q_elt_bytes
    qo = B * num_queries * num_heads * head_dim * qe
    table = sum(-(-L // block_size) for L in lens) * 4 + B * 4
    partials = 0
    if num_splits_per_seq is not None:
        rows = num_queries * num_heads
        # fp32 O (head_dim) + one fp32 LSE per split and row, written then read
        partials = 2 * sum(int(s) for s in num_splits_per_seq) * rows * (head_dim + 1) * 4
    new_rows = 0
    if fused_append:
        new_rows = 2 * 2 * B * num_queries * num_kv_heads * head_dim * elt_bytes
    return {"kv": kv, "q": qo, "out": qo, "table": table, "partials": partials,
            "append": new_rows, "total": kv + 2 * qo + table + partials + new_rows}


def append_bytes(num_tokens: int, num_kv_heads: int, head_dim: int,
                 elt_bytes: int) -> int:
    """kv_append: read k_new and v_new, write them into the cache, + slots."""
    rows = 2 * num_tokens * num_kv_heads * head_dim * elt_bytes
    return 2 * rows + 8 * num_tokens


MIN_DEVICE_SPLIT = 16  # smallest split of the device partition, in blocks


def device_split_counts(context_lens: Sequence[int], block_size: int, units: int,
                        target: int, max_context_len: int, max_blocks_per_seq: int) -> list:
    """Splits per sequence of the split-K partition the decode kernels make
    on the device from the real lengths (pkv_plan.split_target = target > 0;
    units = KV heads x row chunks per sequence): the smallest split length
    S >= MIN_DEVICE_SPLIT blocks with units * sum_b ceil(n_b / S) <= target,
    each sequence getting max(1, ceil(n_b / S)) splits.  For the byte
    accounting of the partials; the kernels compute it themselves."""
    nb = []
    for L in context_lens:
        L = min(max(0, int(L)), max_context_len)
        nb.append(min(-(-L // block_size), max_blocks_per_seq))
    cap = max(target // units, 1)
    lo = max(MIN_DEVICE_SPLIT, -(-sum(nb) // cap))
    hi = max(lo, max(nb) if nb else lo)
    while lo < hi:
        mid = (lo + hi) // 2
        if sum(max(1, -(-n // mid)) for n in nb) <= cap:
            hi = mid
        else:
            lo = mid + 1
    return [max(1, -(-n // lo)) for n in nb]


STREAM_K_WEIGHT = 24  # the balanced partition's per-unit weight, in blocks (as the library's)


def stream_k_splits(context_lens: Sequence[int], block_size: int, units: int, ctas: int,
                    max_context_len: int, max_blocks_per_seq: int,
                    weight: int = STREAM_K_WEIGHT) -> list:
    """Splits per unit, averaged over each sequence's units, of the balanced
    partition (pkv_plan.stream_k = 1, ctas = grid_x): the units laid end to end
    as one list, a unit with n blocks taking weight + n places (the weight
    first, then its blocks), CTA c taking places floor(c T / ctas) ..
    floor((c + 1) T / ctas) - 1 of T, and a unit split wherever a CTA
    boundary falls among its blocks (with fewer places than CTAs some CTAs
    take none).  For the byte accounting of the partials; the kernel computes
    the partition itself."""
    nb = []
    for L in context_lens:
        L = min(max(0, int(L)), max_context_len)
        nb.append(min(-(-L // block_size), max_blocks_per_seq))
    total = units * sum(n + weight for n in nb if n > 0)
    cta_of = lambda x: ((x + 1) * ctas - 1) // total  # noqa: E731
    begin = lambda c: total * c // ctas  # noqa: E731
    out, start = [], 0
    for n in nb:
        pieces = 0
        vlen = n + weight if n > 0 else 0
        for u in range(units):
            if n > 0:  # the CTAs from the first block's to the last's, empty ranges aside
                s = start + u * vlen + weight
                pieces += sum(1 for c in range(cta_of(s), cta_of(s + n - 1) + 1)
                              if begin(c + 1) > begin(c))
        out.append(pieces / units)
        start += units * vlen
    return out
