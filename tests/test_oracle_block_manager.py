"""Pins of the block-bookkeeping model (oracle/block_manager.py) against the
published FNV-1a test vectors, the pages' rules for paged blocks, sharing,
copy-on-write and prefix caching, and brute force on token lists.

A content check carries most of the weight: every slot the model hands out is
written with the token id it stands for, every copy it asks for is applied,
and after each operation every live sequence, read back through its block
table, must give exactly its own token list.
"""
import random

import numpy as np
import pytest

from oracle import block_manager as M


# --- the hash -----------------------------------------------------------------
@pytest.mark.parametrize("text,expected", [
    (b"", 0xCBF29CE484222325),
    (b"a", 0xAF63DC4C8601EC8C),
    (b"foobar", 0x85944171F73967E8),
])
def test_fnv1a_published_vectors(text, expected):
    # the Fowler-Noll-Vo reference test vectors for 64-bit FNV-1a
    assert M.fnv1a_64(text) == expected


def test_chain_hash_names_the_whole_prefix():
    rng = np.random.default_rng(0)
    a = rng.integers(0, 1000, 48).tolist()
    b = list(a)
    b[3] = a[3] + 1                       # differs in block 0 only
    ha, hb = M.chain_hashes(a, 16), M.chain_hashes(b, 16)
    assert len(ha) == 3
    assert all(x != y for x, y in zip(ha, hb))    # every later block differs too
    c = a[:16] + a[32:48] + a[16:32]      # same blocks, other order
    hc = M.chain_hashes(c, 16)
    assert hc[0] == ha[0] and hc[1] != ha[2] and hc[2] != ha[1]
    assert M.chain_hashes(a[:47], 16) == ha[:2]   # only full blocks are named


# --- a checker that replays every operation on a token-id "cache" --------------
class Checked:
    """The model plus a flat array of token ids, one per cache slot."""

    def __init__(self, num_blocks, bs, model_cls=M.BlockPoolModel):
        self.m = model_cls(num_blocks, bs)
        self.bs = bs
        self.cache = np.full(num_blocks * bs, -1, dtype=np.int64)
        self.history = []                 # token lists of every sequence ever made

    def _write(self, slots, tokens, copies):
        for src, dst in copies:
            self.cache[dst * self.bs:(dst + 1) * self.bs] = \
                self.cache[src * self.bs:(src + 1) * self.bs]
        for s, t in zip(slots, tokens):
            self.cache[s] = t

    def add(self, sid, tokens, prefix_cache=True):
        st, res = self.m.add_sequence(sid, tokens, prefix_cache)
        if st == M.OK:
            cached, slots = res
            self._write(slots, tokens[cached:], [])
        self.check()
        return st, res

    def append(self, sid, tokens):
        st, res = self.m.append(sid, tokens)
        if st == M.OK:
            self._write(res[0], tokens, res[1])
        self.check()
        return st, res

    def fork(self, parent, child):
        st, _ = self.m.fork(parent, child)
        self.check()
        return st

    def free(self, sid):
        if sid in self.m.seq_tokens:
            self.history.append(list(self.m.seq_tokens[sid]))
        st, _ = self.m.free(sid)
        self.check()
        return st

    def check(self):
        m, bs = self.m, self.bs
        held = {}
        for sid, blocks in m.seq_blocks.items():
            toks = m.seq_tokens[sid]
            # a new block only when the last one is full
            assert len(blocks) == -(-len(toks) // bs)
            for b in blocks:
                held[b] = held.get(b, 0) + 1
            # every live sequence reads back its own tokens through its table
            got = [int(self.cache[blocks[p // bs] * bs + p % bs]) for p in range(len(toks))]
            assert got == toks, f"sequence {sid} reads {got[:8]}... not {toks[:8]}..."
        # reference counts are the number of tables holding the block
        for b in range(m.n):
            assert m.ref[b] == held.get(b, 0), f"block {b}"
        # every block is held, cached-and-idle, or free, and only one of these
        free = set(m.free_list)
        assert len(free) == len(m.free_list)
        idle_cached = {b for b in range(m.n) if m.ref[b] == 0 and m._is_cached(b)}
        assert not free & set(held) and not free & idle_cached
        assert len(free) + len(idle_cached) + len(held) == m.n
        # cached blocks hold the tokens their hash names
        for h, b in m.registered.items():
            assert m.hash_of[b] == h


def toks(rng, n, vocab=50):
    return rng.integers(0, vocab, n).tolist()


# --- the pages' scenarios -----------------------------------------------------
def test_parallel_sampling_shares_the_prompt_and_copies_on_write():
    c = Checked(16, 16)
    rng = np.random.default_rng(1)
    prompt = toks(rng, 20)
    assert c.add(0, prompt)[0] == M.OK
    for child in (1, 2, 3):
        assert c.fork(0, child) == M.OK
    assert c.free(0) == M.OK
    b0, b1 = c.m.seq_blocks[1]
    assert c.m.ref[b0] == 3 and c.m.ref[b1] == 3
    _, (_, cow1) = c.append(1, [7])
    _, (_, cow2) = c.append(2, [8])
    _, (_, cow3) = c.append(3, [9])
    # the first two samples copy the shared, partly filled block; the last one
    # holds it alone by then and writes in place
    assert len(cow1) == 1 and cow1[0][0] == b1
    assert len(cow2) == 1 and cow2[0][0] == b1
    assert cow3 == []
    assert c.m.seq_blocks[3] == [b0, b1]
    # the full prompt block stays shared: 4 blocks instead of 6
    assert c.m.ref[b0] == 3
    assert len({b for s in (1, 2, 3) for b in c.m.seq_blocks[s]}) == 4


def test_full_shared_block_needs_no_copy():
    c = Checked(16, 4)
    c.add(0, [1, 2, 3, 4])
    c.fork(0, 1)
    _, (slots, cow) = c.append(1, [5])
    assert cow == [] and slots[0] // 4 != c.m.seq_blocks[0][0]


def test_prefix_cache_hit_stops_at_first_miss_and_matches_prefixes_only():
    c = Checked(32, 16)
    rng = np.random.default_rng(2)
    a = toks(rng, 48, vocab=1000)
    x = toks(rng, 16, vocab=1000)
    c.add(0, a)
    c.free(0)
    assert c.m.stats()["cached"] == 3
    # same first two blocks, new third block
    st, (cached, slots) = c.add(1, a[:32] + x)
    assert st == M.OK and cached == 32 and len(slots) == 16
    # block 2 equals a's block 2 but block 1 differs: the walk stops at block 1
    _, (cached, _) = c.add(2, a[:16] + x + a[32:48])
    assert cached == 16
    # the same blocks after a different first block: nothing reused
    _, (cached, _) = c.add(3, x + a[16:48])
    assert cached == 0
    # a prompt that is only a part of a cached block reuses nothing of it
    _, (cached, _) = c.add(4, a[:10])
    assert cached == 0
    # prefix caching off
    _, (cached, _) = c.add(5, list(a), prefix_cache=False)
    assert cached == 0


def test_a_block_matched_only_under_another_prefix_is_not_reused():
    # y + a1 must not hit: one sequence holds [y, z], another [a0, a1], and
    # no sequence starts with [y, a1]
    c = Checked(32, 8)
    rng = np.random.default_rng(3)
    a0, a1, y, z = (toks(rng, 8, vocab=10**6) for _ in range(4))
    c.add(0, a0 + a1)
    c.add(1, y + z)
    _, (cached, _) = c.add(2, y + a1 + [5])
    assert cached == 8


def test_generated_tokens_are_cached_too():
    c = Checked(16, 16)
    rng = np.random.default_rng(4)
    prompt = toks(rng, 10)
    answer = toks(rng, 22)
    c.add(0, prompt)
    for t in answer:
        c.append(0, [t])
    c.free(0)
    _, (cached, _) = c.add(1, prompt + answer + toks(rng, 5))
    assert cached == 32


def test_cached_blocks_stay_until_needed_then_least_recently_used_go_first():
    c = Checked(4, 4)
    a, b = [1, 2, 3, 4, 5, 6, 7, 8], [11, 12, 13, 14, 15, 16, 17, 18]
    c.add(0, a)
    c.free(0)
    assert c.m.stats() == {"free": 2, "cached": 2, "sequences": 0}
    c.add(1, b)                 # takes the two free blocks; a's stay cached
    assert c.m.stats()["cached"] == 4
    c.free(1)
    _, (cached, _) = c.add(2, [21, 22, 23, 24])    # pool dry: evict the oldest
    assert cached == 0
    assert c.m.stats()["cached"] == 4
    c.free(2)
    # b's blocks were used after a's: still reusable
    _, (cached, _) = c.add(3, b)
    assert cached == 8
    # a's first block went: a's prompt misses at once, although its second
    # block is still cached
    ha = M.chain_hashes(a, 4)
    assert ha[0] not in c.m.registered and ha[1] in c.m.registered
    _, (cached, _) = c.add(4, a)
    assert cached == 0


def snapshot(m):
    return (list(m.ref), list(m.used_at), m.time, list(m.free_list), dict(m.registered),
            list(m.hash_of), {k: list(v) for k, v in m.seq_blocks.items()},
            {k: list(v) for k, v in m.seq_tokens.items()})


def test_a_call_the_pool_cannot_serve_changes_nothing():
    c = Checked(3, 4)
    c.add(0, list(range(9)))              # 3 blocks, the last partly filled
    s0 = snapshot(c.m)
    assert c.append(0, list(range(4)))[0] == M.FULL
    assert c.add(1, list(range(5)))[0] == M.FULL   # a hit, but the last token has no block
    assert snapshot(c.m) == s0
    assert c.add(1, list(range(4)))[0] == M.OK     # the hit alone needs no new block
    c.fork(0, 2)
    s1 = snapshot(c.m)
    assert c.append(2, [1])[0] == M.FULL      # the copy of the shared block needs one
    assert snapshot(c.m) == s1


def test_unknown_and_duplicate_ids_are_invalid():
    c = Checked(8, 4)
    assert c.append(9, [1])[0] == M.INVALID
    assert c.free(9) == M.INVALID
    c.add(0, [1])
    assert c.add(0, [1])[0] == M.INVALID
    assert c.fork(0, 0) == M.INVALID
    assert c.fork(5, 6) == M.INVALID


# --- random scripts -------------------------------------------------------------
def brute_force_cached(history, prompt, bs):
    """Longest run of leading full blocks of `prompt` that some sequence ever
    held, on token lists alone (no hashing), for a pool that never evicts."""
    best = 0
    for h in history:
        k = 0
        while (k + 1) * bs <= min(len(h), len(prompt)) and \
                h[k * bs:(k + 1) * bs] == prompt[k * bs:(k + 1) * bs]:
            k += 1
        best = max(best, k * bs)
    return best


def run_script(c, seed, steps, vocab, check_prefix):
    rng = random.Random(seed)
    bs = c.bs
    next_id, live = 0, []
    base = [rng.randrange(vocab) for _ in range(4 * bs)]
    for _ in range(steps):
        op = rng.random()
        if op < 0.3 or not live:
            n = rng.randrange(0, 3 * bs)
            cut = rng.randrange(0, 4) * bs
            prompt = base[:cut] + [rng.randrange(vocab) for _ in range(n)]
            expect = None
            if check_prefix:
                everything = c.history + [list(v) for v in c.m.seq_tokens.values()]
                expect = brute_force_cached(everything, prompt, bs)
            st, res = c.add(next_id, prompt)
            if st == M.OK:
                if expect is not None:
                    assert res[0] == expect
                live.append(next_id)
            next_id += 1
        elif op < 0.7:
            sid = rng.choice(live)
            c.append(sid, [rng.randrange(vocab) for _ in range(rng.choice([1, 1, 1, 3, 5]))])
        elif op < 0.85:
            if c.fork(rng.choice(live), next_id) == M.OK:
                live.append(next_id)
            next_id += 1
        else:
            sid = rng.choice(live)
            c.free(sid)
            live.remove(sid)


@pytest.mark.parametrize("seed", range(6))
def test_random_scripts_without_eviction_match_brute_force_prefixes(seed):
    c = Checked(4000, 4)    # more blocks than 250 steps can take: no eviction
    run_script(c, seed, 250, vocab=3, check_prefix=True)


@pytest.mark.parametrize("seed", range(6))
def test_random_scripts_under_memory_pressure_keep_every_invariant(seed):
    c = Checked(24, 4)
    run_script(c, 100 + seed, 400, vocab=3, check_prefix=False)


# --- planted mistakes: each must fail one of the pins above ------------------------
class SkipsCopyOnWrite(M.BlockPoolModel):
    def _tail_is_shared(self, blocks, length):
        return False


class WalksPastAMiss(M.BlockPoolModel):
    def _lookup(self, tokens):
        return [self.registered[h] for h in M.chain_hashes(tokens, self.bs)
                if h in self.registered]


class EvictsMostRecent(M.BlockPoolModel):
    def _victim(self):
        return max(self._evictable(), key=lambda x: (self.used_at[x], x))


class ForgetsTheHit(M.BlockPoolModel):
    def _hold(self, b):
        self._tick(b)


def _expect_pin_failure(fn):
    with pytest.raises(AssertionError):
        fn()


def _with_model(cls, fn, monkeypatch):
    monkeypatch.setattr(M, "BlockPoolModel", cls)
    monkeypatch.setattr(Checked.__init__, "__defaults__", (cls,))
    fn()


@pytest.mark.parametrize("mutant,pin", [
    (SkipsCopyOnWrite, test_parallel_sampling_shares_the_prompt_and_copies_on_write),
    (WalksPastAMiss, test_cached_blocks_stay_until_needed_then_least_recently_used_go_first),
    (EvictsMostRecent, test_cached_blocks_stay_until_needed_then_least_recently_used_go_first),
    (ForgetsTheHit, test_prefix_cache_hit_stops_at_first_miss_and_matches_prefixes_only),
])
def test_planted_mistakes_are_caught(mutant, pin, monkeypatch):
    _expect_pin_failure(lambda: _with_model(mutant, pin, monkeypatch))


def test_a_hash_without_the_parent_is_caught(monkeypatch):
    monkeypatch.setattr(M, "block_hash",
                        lambda parent, tokens: M.fnv1a_64(np.asarray(tokens, "<i4").tobytes()))
    _expect_pin_failure(test_a_block_matched_only_under_another_prefix_is_not_reused)
