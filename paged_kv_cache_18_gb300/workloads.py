"""Seeded synthetic inputs for paged decode attention.

This module is the only code that both the CUDA path's tests/benchmark and the
float64 oracle consume.  It holds none of the attention arithmetic: it draws
random values, rounds them to the storage type, builds a shuffled block
table (a host stand-in for the free-block pool of PagedAttention, where
"logical blocks map to physical blocks anywhere in GPU memory"), assigns the
cache slots of the new tokens, and poisons every cache row that no sequence
owns with NaN so that a read outside the context shows up in the output.

Workload recipe (all five named workloads use it):
  * q, K, V ~ N(0, 1) drawn in float32 from NumPy's PCG64 with a fixed seed,
    then rounded to nearest-even into the storage dtype;
  * sequence b owns ceil(L_b / block_size) blocks; the physical ids are a
    random permutation of range(NB) with NB = owned + ceil(10 %) slack;
  * the last Q rows of every sequence are the "new" tokens: their K/V rows
    are returned separately (k_new, v_new) together with their slots, and
    their cache slots start out poisoned, so the step appends them first.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

STORAGE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16}
ELT_BYTES = {"f32": 4, "bf16": 2, "f16": 2}
NAN_BITS16 = {"bf16": 0x7FC0, "f16": 0x7E00}


def round_f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (finite x)."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((bits >> 16) & 1) + np.uint32(0x7FFF)
    return ((bits + bias) >> 16).astype(np.uint16)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values into the storage representation of ``dtype``."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return round_f32_to_bf16_bits(x)
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
    raise ValueError(dtype)


def _normal_storage(rng: np.random.Generator, shape, dtype: str,
                    chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) values in storage form, drawn in chunks to bound host memory."""
    out = np.empty(int(np.prod(shape)), dtype=STORAGE[dtype])
    for lo in range(0, out.size, chunk):
        hi = min(out.size, lo + chunk)
        out[lo:hi] = to_storage(rng.standard_normal(hi - lo, dtype=np.float32), dtype)
    return out.reshape(shape)


def _poison_value(dtype: str):
    return np.float32(np.nan) if dtype == "f32" else np.uint16(NAN_BITS16[dtype])


@dataclasses.dataclass
class Workload:
    """Shape of one paged-attention call (and the append before it)."""
    name: str
    batch: int
    num_heads: int          # Hq
    num_kv_heads: int       # Hkv
    head_dim: int           # D
    dtype: str              # "f32" | "bf16" | "f16"
    context_lens: Optional[Sequence[int]] = None   # fixed lengths, or
    len_range: Optional[tuple] = None               # (lo, hi) inclusive uniform
    num_queries: int = 1    # Q: 1 = decode, K+1 = speculative verify
    block_size: int = 16
    scale: Optional[float] = None                   # None -> 1/sqrt(D)
    seed: int = 0
    slack: float = 0.10
    tree_parents: Optional[Sequence[int]] = None    # tree verification: parent of each node

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    def lengths(self) -> np.ndarray:
        if self.context_lens is not None:
            lens = np.asarray(self.context_lens, dtype=np.int32)
            if lens.size == 1 and self.batch > 1:
                lens = np.full(self.batch, int(lens[0]), dtype=np.int32)
            return lens
        lo, hi = self.len_range
        rng = np.random.Generator(np.random.PCG64(self.seed + 7919))
        return rng.integers(lo, hi, size=self.batch, endpoint=True).astype(np.int32)


# The five named workloads (seed = 1000 + index).
WORKLOADS = {
    "tiny": Workload("tiny GPTlite-scale decode", 4, 6, 6, 64, "f32",
                     context_lens=[17, 64, 100, 256], seed=1001),
    "llama2_13b": Workload("Llama-2-13B-shaped decode layer", 32, 40, 40, 128,
                           "bf16", context_lens=[2048], seed=1002),
    "llama3_8b_gqa": Workload("Llama-3-8B-shaped GQA decode", 128, 32, 8, 128,
                              "bf16", len_range=(128, 4096), seed=1003),
    "long_splitk": Workload("long-context small-batch split-K", 2, 32, 8, 128,
                            "bf16", context_lens=[32768, 65536], seed=1004),
    "spec_verify": Workload("speculative verify K=4", 16, 32, 8, 128, "bf16",
                            len_range=(512, 8192), num_queries=5, seed=1005),
}


def medusa_parents(branching: Sequence[int]) -> list:
    """Parents of a candidate tree in breadth-first order ("Inference part 2",
    section "Medusa": the top candidates of each extra head are combined into
    a tree of continuations): node 0 is the last accepted token, and every
    node of depth d has branching[d] children.  parents[0] = -1."""
    parents, level = [-1], [0]
    for k in branching:
        nxt = []
        for p in level:
            for _ in range(k):
                parents.append(p)
                nxt.append(len(parents) - 1)
        level = nxt
    return parents


def tree_mask_bits(parents: Sequence[int]) -> np.ndarray:
    """Visibility bitmask of each tree node: bit k of mask[j] is set when node
    k is node j or one of its ancestors (parents[j] < j)."""
    masks = np.zeros(len(parents), dtype=np.uint64)
    for j, p in enumerate(parents):
        masks[j] = (masks[p] if p >= 0 else np.uint64(0)) | np.uint64(1 << j)
    return masks


# Tree verification on the speculative-verify shape: two extra heads, top-3
# and top-2 candidates (1 + 3 + 6 = 10 nodes).
TREE_WORKLOADS = {
    "medusa_tree": Workload("Medusa tree verify, 10 nodes (top-3 x top-2)", 16, 32, 8, 128,
                            "bf16", len_range=(512, 8192), num_queries=10, seed=1008,
                            tree_parents=medusa_parents((3, 2))),
}


@dataclasses.dataclass
class PagedBatch:
    """Host arrays of one step: append Q new rows per sequence, then attend."""
    wl: Workload
    q: np.ndarray             # [B, Q, Hq, D] storage dtype
    k_cache: np.ndarray       # [NB, Hkv, bs, D] storage dtype (new slots poisoned)
    v_cache: np.ndarray
    k_new: np.ndarray         # [B*Q, Hkv, D]
    v_new: np.ndarray
    slot_mapping: np.ndarray  # [B*Q] int64
    block_table: np.ndarray   # [B, max_blocks] int32 (unused entries = -1)
    context_lens: np.ndarray  # [B] int32 (includes the Q new rows)
    num_blocks: int

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    def kv_bytes(self) -> int:
        """Bytes of the valid K and V rows one attention call reads."""
        wl = self.wl
        return int(2 * int(self.context_lens.clip(min=0).sum()) * wl.num_kv_heads
                   * wl.head_dim * ELT_BYTES[wl.dtype])


def make_batch(wl: Workload, poison: bool = True) -> PagedBatch:
    """Build the seeded host arrays of ``wl``."""
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, Q, Hq, Hkv, D, bs = (wl.batch, wl.num_queries, wl.num_heads,
                            wl.num_kv_heads, wl.head_dim, wl.block_size)
    lens = wl.lengths()
    assert lens.shape == (B,)
    owned = [max(0, -(-int(L) // bs)) for L in lens]
    total = sum(owned)
    NB = max(1, total + int(math.ceil(wl.slack * total)))
    perm = rng.permutation(NB).astype(np.int32)
    max_blocks = max(1, max(owned) if owned else 1)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :owned[b]] = perm[pos:pos + owned[b]]
        pos += owned[b]

    k_cache = _normal_storage(rng, (NB, Hkv, bs, D), wl.dtype)
    v_cache = _normal_storage(rng, (NB, Hkv, bs, D), wl.dtype)
    q = _normal_storage(rng, (B, Q, Hq, D), wl.dtype)

    # New rows: the last Q positions of each sequence (those that exist).
    new_rows = []
    for b in range(B):
        for j in range(Q):
            i = int(lens[b]) - Q + j
            new_rows.append((b, i))
    slots = np.full(len(new_rows), -1, dtype=np.int64)
    k_new = np.empty((len(new_rows), Hkv, D), dtype=STORAGE[wl.dtype])
    v_new = np.empty_like(k_new)
    bad = _poison_value(wl.dtype)
    for t, (b, i) in enumerate(new_rows):
        if i < 0:
            k_new[t] = bad
            v_new[t] = bad
            continue
        phys = int(table[b, i // bs])
        slots[t] = phys * bs + i % bs
        k_new[t] = k_cache[phys, :, i % bs, :]
        v_new[t] = v_cache[phys, :, i % bs, :]

    if poison:
        used = np.zeros(NB, dtype=bool)
        used[perm[:total]] = True
        k_cache[~used] = bad
        v_cache[~used] = bad
        for b in range(B):
            L = int(lens[b])
            if owned[b] and L % bs:
                last = int(table[b, owned[b] - 1])
                k_cache[last, :, L % bs:, :] = bad
                v_cache[last, :, L % bs:, :] = bad
        for t, (b, i) in enumerate(new_rows):
            if slots[t] >= 0:
                phys, off = divmod(int(slots[t]), bs)
                k_cache[phys, :, off, :] = bad
                v_cache[phys, :, off, :] = bad

    return PagedBatch(wl, q, k_cache, v_cache, k_new, v_new, slots, table,
                      lens.astype(np.int32), NB)


# ---- chunked prefill ----------------------------------------------------------------
@dataclasses.dataclass
class PrefillWorkload:
    """One chunked-prefill call: each sequence has `prefix` cached rows and
    brings a chunk of `chunk` new rows (appended first, then attending)."""
    name: str
    batch: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str
    chunk_lens: Optional[Sequence[int]] = None      # fixed chunk lengths (or one for all)
    chunk_range: Optional[tuple] = None             # (lo, hi) inclusive uniform
    prefix_lens: Optional[Sequence[int]] = None
    prefix_range: Optional[tuple] = None
    block_size: int = 16
    scale: Optional[float] = None
    seed: int = 0
    slack: float = 0.10

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.head_dim)

    def _draw(self, fixed, rng_range, salt):
        if fixed is not None:
            a = np.asarray(fixed, dtype=np.int32)
            return np.full(self.batch, int(a[0]), np.int32) if a.size == 1 else a
        lo, hi = rng_range
        rng = np.random.Generator(np.random.PCG64(self.seed + salt))
        return rng.integers(lo, hi, size=self.batch, endpoint=True).astype(np.int32)

    def chunks(self) -> np.ndarray:
        return self._draw(self.chunk_lens, self.chunk_range, 7907)

    def prefixes(self) -> np.ndarray:
        return self._draw(self.prefix_lens, self.prefix_range, 7919)

    def flops(self) -> int:
        """Multiply-adds x 2 of both products, over the keys each row sees."""
        tot = 0
        for P, C in zip(self.prefixes().tolist(), self.chunks().tolist()):
            tot += C * P + C * (C + 1) // 2           # sum over rows of visible keys
        return 4 * self.num_heads * self.head_dim * tot


PREFILL_WORKLOADS = {
    "prefill_llama3_8b": PrefillWorkload(
        "Llama-3-8B-shaped chunked prefill, 512-token chunks", 8, 32, 8, 128, "bf16",
        chunk_lens=[512], prefix_range=(0, 3584), seed=1006),
}


@dataclasses.dataclass
class PrefillBatch:
    wl: PrefillWorkload
    q: np.ndarray             # [total_q, Hq, D] storage dtype
    k_cache: np.ndarray       # [NB, Hkv, bs, D] (the chunk's slots poisoned)
    v_cache: np.ndarray
    k_new: np.ndarray         # [total_q, Hkv, D]: the chunk rows to append
    v_new: np.ndarray
    slot_mapping: np.ndarray  # [total_q] int64
    block_table: np.ndarray   # [B, max_blocks] int32 (unused = -1)
    context_lens: np.ndarray  # [B] int32: prefix + chunk
    query_start: np.ndarray   # [B + 1] int32
    num_blocks: int

    @property
    def max_query_len(self) -> int:
        d = np.diff(self.query_start)
        return int(d.max()) if d.size else 0

    @property
    def total_q(self) -> int:
        return int(self.query_start[-1])


def make_prefill_batch(wl: PrefillWorkload, poison: bool = True) -> PrefillBatch:
    """Seeded host arrays of one chunked-prefill step: random block tables
    over a shuffled pool, N(0, 1) q/K/V, NaN in every unused row."""
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, Hq, Hkv, D, bs = wl.batch, wl.num_heads, wl.num_kv_heads, wl.head_dim, wl.block_size
    chunks, prefixes = wl.chunks(), wl.prefixes()
    lens = (chunks + prefixes).astype(np.int32)
    owned = [-(-int(L) // bs) for L in lens]
    total = sum(owned)
    NB = max(1, total + int(math.ceil(wl.slack * total)))
    perm = rng.permutation(NB).astype(np.int32)
    table = np.full((B, max(1, max(owned) if owned else 1)), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :owned[b]] = perm[pos:pos + owned[b]]
        pos += owned[b]
    k_cache = _normal_storage(rng, (NB, Hkv, bs, D), wl.dtype)
    v_cache = _normal_storage(rng, (NB, Hkv, bs, D), wl.dtype)
    qs = np.zeros(B + 1, dtype=np.int32)
    qs[1:] = np.cumsum(chunks)
    q = _normal_storage(rng, (int(qs[-1]), Hq, D), wl.dtype)
    slots = np.empty(int(qs[-1]), dtype=np.int64)
    for b in range(B):
        for j in range(int(chunks[b])):
            i = int(prefixes[b]) + j
            slots[qs[b] + j] = int(table[b, i // bs]) * bs + i % bs
    phys, off = slots // bs, slots % bs
    k_new = np.ascontiguousarray(k_cache[phys, :, off, :])
    v_new = np.ascontiguousarray(v_cache[phys, :, off, :])
    if poison:
        bad = _poison_value(wl.dtype)
        used = np.zeros(NB, dtype=bool)
        used[perm[:total]] = True
        k_cache[~used] = bad
        v_cache[~used] = bad
        for b in range(B):
            L = int(lens[b])
            if owned[b] and L % bs:
                last = int(table[b, owned[b] - 1])
                k_cache[last, :, L % bs:, :] = bad
                v_cache[last, :, L % bs:, :] = bad
        k_cache[phys, :, off, :] = bad
        v_cache[phys, :, off, :] = bad
    return PrefillBatch(wl, q, k_cache, v_cache, k_new, v_new, slots, table, lens, qs, NB)


def storage_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of stored elements (for comparing outputs)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.view(np.float16).astype(np.float64)


def fp8_caches(b: PagedBatch, k_scale: float, v_scale: float):
    """e4m3 code caches (uint8) of a batch's float caches: every stored value
    divided by the tensor scale in float32 and cast to FP8 E4M3 (round to
    nearest even); NaN-filled rows become the NaN code.  The new rows stay in
    b.k_new / b.v_new for a quantising append."""
    import torch

    def codes(cache, scale):
        f = storage_to_f64(cache, b.wl.dtype).astype(np.float32) / np.float32(scale)
        return torch.from_numpy(np.ascontiguousarray(f)).to(torch.float8_e4m3fn).view(
            torch.uint8).numpy()

    return codes(b.k_cache, k_scale), codes(b.v_cache, v_scale)


# ---- multi-head latent attention (MLA) decode -------------------------------------
@dataclasses.dataclass
class MlaWorkload:
    """One MLA decode step over a paged latent cache: each sequence appends
    its newest latent row [c ; k_rope], then every query head attends over
    the sequence's rows with the absorbed query [q_c ; q_r]."""
    name: str
    batch: int
    num_heads: int
    rope_dim: int                                   # 0 or 64
    dtype: str                                      # "bf16" | "f16"
    context_lens: Optional[Sequence[int]] = None
    len_range: Optional[tuple] = None
    latent_dim: int = 512
    head_dim: int = 128                             # per-head dim before absorption
    block_size: int = 16
    scale: Optional[float] = None                   # None -> 1/sqrt(head_dim + rope_dim)
    seed: int = 0
    slack: float = 0.10

    @property
    def width(self) -> int:
        return self.latent_dim + self.rope_dim

    @property
    def softmax_scale(self) -> float:
        if self.scale is not None:
            return self.scale
        return 1.0 / math.sqrt(self.head_dim + self.rope_dim)

    def lengths(self) -> np.ndarray:
        if self.context_lens is not None:
            lens = np.asarray(self.context_lens, dtype=np.int32)
            if lens.size == 1 and self.batch > 1:
                lens = np.full(self.batch, int(lens[0]), dtype=np.int32)
            return lens
        lo, hi = self.len_range
        rng = np.random.Generator(np.random.PCG64(self.seed + 7919))
        return rng.integers(lo, hi, size=self.batch, endpoint=True).astype(np.int32)


# DeepSeek-V2's latent sizes (d_c 512, d_h^R 64) with 16 query heads per GPU.
MLA_WORKLOADS = {
    "mla_deepseek_v2": MlaWorkload("DeepSeek-V2-shaped MLA decode, 16 heads", 64, 16, 64,
                                   "bf16", len_range=(1024, 8192), seed=1007),
}


@dataclasses.dataclass
class MlaBatch:
    wl: MlaWorkload
    q: np.ndarray             # [B, H, W] storage dtype
    ckv_cache: np.ndarray     # [NB, bs, W] storage dtype (the new slots poisoned)
    ckv_new: np.ndarray       # [B, W]: the newest row of each sequence
    slot_mapping: np.ndarray  # [B] int64 (-1: the sequence is empty)
    block_table: np.ndarray   # [B, max_blocks] int32 (unused entries = -1)
    context_lens: np.ndarray  # [B] int32 (includes the new row)
    num_blocks: int

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.context_lens.size else 0

    def kv_bytes(self) -> int:
        """Bytes of the valid latent rows one decode call reads (each once)."""
        return int(int(self.context_lens.clip(min=0).sum()) * self.wl.width
                   * ELT_BYTES[self.wl.dtype])


def make_mla_batch(wl: MlaWorkload, poison: bool = True) -> MlaBatch:
    """Seeded host arrays of ``wl``: latent and rotary values ~ N(0, 1) in the
    storage dtype, physical blocks a random permutation with 10% spare, rows
    past each context and spare blocks NaN-filled (poison), and each
    sequence's newest row held back as the step's append."""
    rng = np.random.Generator(np.random.PCG64(wl.seed))
    B, H, W, bs = wl.batch, wl.num_heads, wl.width, wl.block_size
    lens = wl.lengths()
    assert lens.shape == (B,)
    owned = [max(0, -(-int(L) // bs)) for L in lens]
    total = sum(owned)
    NB = max(1, total + int(math.ceil(wl.slack * total)))
    perm = rng.permutation(NB).astype(np.int32)
    table = np.full((B, max(1, max(owned) if owned else 1)), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :owned[b]] = perm[pos:pos + owned[b]]
        pos += owned[b]
    cache = _normal_storage(rng, (NB, bs, W), wl.dtype)
    q = _normal_storage(rng, (B, H, W), wl.dtype)
    slots = np.full(B, -1, dtype=np.int64)
    new = np.empty((B, W), dtype=STORAGE[wl.dtype])
    bad = _poison_value(wl.dtype)
    for b in range(B):
        i = int(lens[b]) - 1
        if i < 0:
            new[b] = bad
            continue
        phys = int(table[b, i // bs])
        slots[b] = phys * bs + i % bs
        new[b] = cache[phys, i % bs]
    if poison:
        used = np.zeros(NB, dtype=bool)
        used[perm[:total]] = True
        cache[~used] = bad
        for b in range(B):
            L = int(lens[b])
            if owned[b] and L % bs:
                cache[int(table[b, owned[b] - 1]), L % bs:] = bad
            if slots[b] >= 0:
                phys, off = divmod(int(slots[b]), bs)
                cache[phys, off] = bad
    return MlaBatch(wl, q, cache, new, slots, table, lens.astype(np.int32), NB)
