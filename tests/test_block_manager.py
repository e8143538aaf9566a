"""The library's native block manager (pkv_bm_*, host code, no GPU needed)
against the block-bookkeeping model of the oracle: the same operation
scripts must give the same statuses, slots, copy pairs, cached-token counts,
block tables, reference counts, hashes and pool statistics."""
import random

import numpy as np
import pytest

from oracle import block_manager as M
from paged_kv_cache_18_gb300 import binding, build


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.lib()


STATUS = {0: M.OK, 1: M.INVALID, 3: M.FULL}


def call(fn, *args):
    try:
        return M.OK, fn(*args)
    except binding.PkvError as e:
        return STATUS[e.status], None


class Pair:
    """One native manager and one model, driven in lockstep."""

    def __init__(self, num_blocks, bs):
        self.c = binding.BlockManager(num_blocks, bs)
        self.m = M.BlockPoolModel(num_blocks, bs)
        self.bs, self.n = bs, num_blocks

    def add(self, sid, tokens, prefix_cache=True):
        st, res = call(self.c.add_sequence, sid, tokens, prefix_cache)
        mst, mres = self.m.add_sequence(sid, tokens, prefix_cache)
        assert st == mst
        if st == M.OK:
            assert res[0] == mres[0]
            assert res[1].tolist() == mres[1]
        return st

    def append(self, sid, tokens):
        st, res = call(self.c.append, sid, tokens)
        mst, mres = self.m.append(sid, tokens)
        assert st == mst
        if st == M.OK:
            assert res[0].tolist() == mres[0] and res[1] == mres[1]
        return st

    def fork(self, parent, child):
        st, _ = call(self.c.fork, parent, child)
        assert st == self.m.fork(parent, child)[0]
        return st

    def free(self, sid):
        st, _ = call(self.c.free, sid)
        assert st == self.m.free(sid)[0]
        return st

    def compare(self):
        assert self.c.stats() == self.m.stats()
        for b in range(self.n):
            assert self.c.block_info(b) == self.m.block_info(b), f"block {b}"
        sids = sorted(self.m.seq_blocks)
        for s in sids:
            assert self.c.sequence(s) == self.m.sequence(s)
        if sids:
            width = max(len(self.m.seq_blocks[s]) for s in sids) + 2
            t, l = self.c.block_table(sids, width)
            mt, ml = self.m.block_table(sids, width)
            assert np.array_equal(t, mt) and np.array_equal(l, ml)


def test_hash_matches_the_model():
    rng = np.random.default_rng(0)
    for n in (0, 1, 16, 33):
        toks = rng.integers(-2**31, 2**31, n).tolist()
        parent = int(rng.integers(0, 2**63))
        assert binding.bm_hash(parent, toks) == M.block_hash(parent, toks)
    # a first block: the parent counts as eight zero bytes
    assert binding.bm_hash(0, []) == M.fnv1a_64(bytes(8))


def test_scenario_parallel_sampling_and_prefix_reuse():
    p = Pair(16, 16)
    rng = random.Random(1)
    prompt = [rng.randrange(1000) for _ in range(20)]
    assert p.add(0, prompt) == M.OK
    for child in (1, 2, 3):
        p.fork(0, child)
    p.free(0)
    for s in (1, 2, 3):
        p.append(s, [s])
    p.compare()
    p.free(1)
    assert p.add(4, prompt[:16] + [5, 6]) == M.OK
    assert p.m.seq_tokens[4][:16] == prompt[:16]
    p.compare()


def test_errors_match():
    p = Pair(3, 4)
    assert p.append(7, [1]) == M.INVALID
    assert p.free(7) == M.INVALID
    assert p.add(0, list(range(9))) == M.OK
    assert p.add(0, [1]) == M.INVALID
    assert p.append(0, list(range(4))) == M.FULL
    assert p.fork(0, 0) == M.INVALID
    assert p.fork(0, 1) == M.OK
    assert p.append(1, [3]) == M.FULL
    p.compare()
    with pytest.raises(binding.PkvError):
        p.c.block_table([0], 1)                      # too narrow for 3 blocks
    with pytest.raises(binding.PkvError):
        p.c.block_info(3)


def test_create_rejects_bad_sizes():
    L = binding.lib()
    assert not L.pkv_bm_create(0, 16)
    assert not L.pkv_bm_create(16, 0)
    assert L.pkv_bm_stats(None, None, None, None) == 1


@pytest.mark.parametrize("seed,num_blocks,bs,vocab", [
    (0, 4000, 4, 3), (1, 24, 4, 3), (2, 40, 8, 2), (3, 64, 16, 2), (4, 12, 2, 4),
    (5, 200, 16, 2)])
def test_random_scripts_agree(seed, num_blocks, bs, vocab):
    p = Pair(num_blocks, bs)
    rng = random.Random(seed)
    base = [rng.randrange(vocab) for _ in range(4 * bs)]
    next_id, live = 0, []
    for step in range(300):
        op = rng.random()
        if op < 0.3 or not live:
            cut = rng.randrange(0, 4) * bs
            prompt = base[:cut] + [rng.randrange(vocab) for _ in range(rng.randrange(0, 3 * bs))]
            if p.add(next_id, prompt, prefix_cache=rng.random() < 0.9) == M.OK:
                live.append(next_id)
            next_id += 1
        elif op < 0.7:
            p.append(rng.choice(live),
                     [rng.randrange(vocab) for _ in range(rng.choice([0, 1, 1, 1, 3, 5]))])
        elif op < 0.85:
            if p.fork(rng.choice(live), next_id) == M.OK:
                live.append(next_id)
            next_id += 1
        else:
            sid = rng.choice(live)
            p.free(sid)
            live.remove(sid)
        if step % 10 == 0:
            p.compare()
    p.compare()
