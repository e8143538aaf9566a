"""Reference model of the paged cache's block bookkeeping: on-demand blocks,
reference counts, copy-on-write, and the prefix hash chain.

TEST INFRASTRUCTURE ONLY: the test suite compares the library's native block
manager with this model; nothing in the product path imports it.

What it follows:

* "KV cache, prefill và decode" (truongducdung), section 05, "Block table":
  a sequence sees a run of logical blocks mapped to physical ones anywhere in
  the pool, and receives a new block only once its last one is full.
* Same page, "Chia sẻ block và copy-on-write": every physical block carries a
  reference count; samples drawn from one prompt share its blocks, and a
  sample that must write into a shared block first gets its own copy.
* Same page, "Prefix caching": a full block is named by a hash of its own
  tokens together with its parent block's hash, that is, of the whole prefix
  up to it; a new request that finds the hash takes the block (count + 1) and
  skips that part of the prefill.
* "Inference part 1" (brunomaga), section "Prefix caching": matching is on
  token ids, prefixes only; the lookup walks the prompt's blocks from the
  start and stops at the first miss; a finished request's blocks stay
  reusable until the memory is needed; generated tokens are cached too.
* "Efficient Inference" (obvix), section on PagedAttention: a finished
  request's blocks go back to the free pool.
* Least-recently-used eviction of cached blocks that nobody holds, as the
  pages describe for RadixAttention's cached prefixes.

Readings where the pages are silent (the same ones the native manager takes):

* free (never cached) blocks are taken last-freed first, and before any
  cached block is evicted; at the start the lowest id comes first;
* a block is registered in the cache the moment it becomes full; a second
  full block with a hash already registered is not merged and stays private;
* eviction takes, among cached blocks held by nobody, the one with the
  oldest use, ties to the lower id; taking, releasing or allocating a block
  counts as a use, on one counter that every such event advances;
* the hash is 64-bit FNV-1a (the published Fowler-Noll-Vo algorithm: xor the
  byte, then multiply by the 64-bit FNV prime) over the parent hash as 8
  little-endian bytes (0 for the first block) followed by the block's token
  ids as 4 little-endian bytes each;
* an operation that the pool cannot serve fails and changes nothing.

The hash chain here is recomputed from each sequence's own token list, not
carried block to block.
"""
from __future__ import annotations

import numpy as np

FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3
_MASK64 = (1 << 64) - 1

OK, INVALID, FULL = "ok", "invalid", "full"


def fnv1a_64(data: bytes, h: int = FNV64_OFFSET) -> int:
    """64-bit FNV-1a of a byte string."""
    for byte in data:
        h = ((h ^ byte) * FNV64_PRIME) & _MASK64
    return h


def block_hash(parent: int, tokens) -> int:
    """Hash of one full block given its parent block's hash (0 for none)."""
    data = int(parent).to_bytes(8, "little") + np.asarray(tokens, dtype="<i4").tobytes()
    return fnv1a_64(data)


def chain_hashes(tokens, block_size: int):
    """Hashes of every full block of a token sequence, first block first."""
    out, parent = [], 0
    for i in range(len(tokens) // block_size):
        parent = block_hash(parent, tokens[i * block_size:(i + 1) * block_size])
        out.append(parent)
    return out


class BlockPoolModel:
    """The pool and every sequence's block list, as plain Python lists and
    dicts; each public method returns (status, result)."""

    def __init__(self, num_blocks: int, block_size: int):
        self.bs = block_size
        self.n = num_blocks
        self.ref = [0] * num_blocks
        self.used_at = [0] * num_blocks
        self.hash_of = [None] * num_blocks     # set once the block is full
        self.registered = {}                   # hash -> block, cached blocks only
        self.free_list = list(range(num_blocks))  # position 0 is taken next
        self.time = 0
        self.seq_blocks = {}
        self.seq_tokens = {}

    # -- pool ---------------------------------------------------------------
    def _tick(self, b):
        self.time += 1
        self.used_at[b] = self.time

    def _is_cached(self, b):
        return self.hash_of[b] is not None and self.registered.get(self.hash_of[b]) == b

    def _evictable(self):
        return [b for b in range(self.n) if self.ref[b] == 0 and self._is_cached(b)]

    def _spare(self):
        return len(self.free_list) + len(self._evictable())

    def _victim(self):
        return min(self._evictable(), key=lambda x: (self.used_at[x], x))

    def _take_new(self):
        if self.free_list:
            b = self.free_list.pop(0)
        else:
            b = self._victim()
            del self.registered[self.hash_of[b]]
        self.hash_of[b] = None
        self.ref[b] = 1
        self._tick(b)
        return b

    def _hold(self, b):
        self.ref[b] += 1
        self._tick(b)

    def _drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self._tick(b)
            if not self._is_cached(b):
                self.free_list.insert(0, b)

    # -- sequences ----------------------------------------------------------
    def add_sequence(self, sid, tokens, prefix_cache=True):
        """-> (status, (cached_tokens, slots of the uncached tokens))."""
        tokens = [int(t) for t in tokens]
        if sid in self.seq_blocks:
            return INVALID, None
        hits = self._lookup(tokens) if prefix_cache else []
        cached = len(hits) * self.bs
        rest = len(tokens) - cached
        spare = self._spare() - sum(1 for b in hits if self.ref[b] == 0)
        if -(-rest // self.bs) > spare:
            return FULL, None
        for b in hits:
            self._hold(b)
        self.seq_blocks[sid] = list(hits)
        self.seq_tokens[sid] = tokens[:cached]
        status, (slots, _) = self.append(sid, tokens[cached:])
        assert status == OK
        return OK, (cached, slots)

    def _lookup(self, tokens):
        """Cached blocks of the prompt's leading full blocks, up to the first miss."""
        hits = []
        for h in chain_hashes(tokens, self.bs):
            if h not in self.registered:
                break
            hits.append(self.registered[h])
        return hits

    def _tail_is_shared(self, blocks, length):
        """The last block is partly filled and held by another sequence too."""
        return length % self.bs != 0 and self.ref[blocks[-1]] > 1

    def append(self, sid, tokens):
        """-> (status, (slots, [(copy_from, copy_to)]))."""
        if sid not in self.seq_blocks:
            return INVALID, None
        tokens = [int(t) for t in tokens]
        blocks, toks = self.seq_blocks[sid], self.seq_tokens[sid]
        length = len(toks)
        shared_tail = bool(tokens) and self._tail_is_shared(blocks, length)
        grow = max(0, -(-(length + len(tokens)) // self.bs) - len(blocks))
        if grow + int(shared_tail) > self._spare():
            return FULL, None
        copies = []
        if shared_tail:
            old = blocks[-1]
            new = self._take_new()
            self._drop(old)
            blocks[-1] = new
            copies.append((old, new))
        slots = []
        for t in tokens:
            pos = len(toks)
            if pos % self.bs == 0:
                blocks.append(self._take_new())
            slots.append(blocks[pos // self.bs] * self.bs + pos % self.bs)
            toks.append(t)
            if len(toks) % self.bs == 0:
                self._seal(sid, len(toks) // self.bs - 1)
        return OK, (slots, copies)

    def _seal(self, sid, i):
        b = self.seq_blocks[sid][i]
        if self.hash_of[b] is not None:
            return
        h = chain_hashes(self.seq_tokens[sid][:(i + 1) * self.bs], self.bs)[i]
        self.hash_of[b] = h
        if h not in self.registered:
            self.registered[h] = b

    def fork(self, parent, child):
        if parent not in self.seq_blocks or child in self.seq_blocks:
            return INVALID, None
        for b in self.seq_blocks[parent]:
            self._hold(b)
        self.seq_blocks[child] = list(self.seq_blocks[parent])
        self.seq_tokens[child] = list(self.seq_tokens[parent])
        return OK, None

    def free(self, sid):
        if sid not in self.seq_blocks:
            return INVALID, None
        for b in self.seq_blocks.pop(sid):
            self._drop(b)
        del self.seq_tokens[sid]
        return OK, None

    # -- views --------------------------------------------------------------
    def sequence(self, sid):
        return list(self.seq_blocks[sid]), len(self.seq_tokens[sid])

    def block_table(self, sids, width):
        table = np.full((len(sids), width), -1, dtype=np.int32)
        lens = np.zeros(len(sids), dtype=np.int32)
        for r, s in enumerate(sids):
            blocks = self.seq_blocks[s]
            table[r, :len(blocks)] = blocks
            lens[r] = len(self.seq_tokens[s])
        return table, lens

    def stats(self):
        return {"free": len(self.free_list), "cached": len(self.registered),
                "sequences": len(self.seq_blocks)}

    def block_info(self, b):
        return self.ref[b], self._is_cached(b), self.hash_of[b] or 0
