"""A tiny random-weight decoder whose attention is the float64 oracle.

Test infrastructure for the greedy speculative-decoding pin: "Inference part
2" (brunomaga, section "Speculative decoding", generate_speculative) states
that greedy verification reproduces plain greedy decoding of the target.
The model has no trained weights: embeddings, projections and the LM head
are seeded N(0, 1/sqrt(d)) matrices.  K, V and q are stored in float32 (the
oracle's storage type) and attention runs through the paged cache with the
oracle's append and attention calls, so a wrong shifted-causal mask would
change the verify logits.
"""
import numpy as np

import oracle


class ToyDecoder:
    def __init__(self, vocab=48, d_model=32, num_heads=4, num_kv_heads=2,
                 head_dim=16, max_len=96, block_size=16, seed=0):
        rng = np.random.default_rng(seed)
        s = 1.0 / np.sqrt(d_model)
        self.vocab, self.H, self.Hkv, self.D = vocab, num_heads, num_kv_heads, head_dim
        self.emb = rng.standard_normal((vocab, d_model))
        self.pos = rng.standard_normal((max_len, d_model)) * 0.5
        self.wq = rng.standard_normal((d_model, num_heads * head_dim)) * s
        self.wk = rng.standard_normal((d_model, num_kv_heads * head_dim)) * s
        self.wv = rng.standard_normal((d_model, num_kv_heads * head_dim)) * s
        self.wo = rng.standard_normal((num_heads * head_dim, d_model)) * s
        self.head = rng.standard_normal((d_model, vocab)) * s
        self.bs = block_size
        nblocks = -(-max_len // block_size)
        # one sequence; physical blocks deliberately shuffled
        self.table = rng.permutation(nblocks + 2)[:nblocks].astype(np.int32)[None]
        self.k_cache = np.zeros((nblocks + 2, num_kv_heads, block_size, head_dim), np.float32)
        self.v_cache = np.zeros_like(self.k_cache)

    def forward(self, tokens, start):
        """Logits [n, vocab] of ``tokens`` at positions start.. ; their K/V are
        written at those positions (overwriting whatever was there)."""
        n = len(tokens)
        x = self.emb[tokens] + self.pos[start:start + n]
        q = (x @ self.wq).reshape(n, self.H, self.D).astype(np.float32)
        k = (x @ self.wk).reshape(n, self.Hkv, self.D).astype(np.float32)
        v = (x @ self.wv).reshape(n, self.Hkv, self.D).astype(np.float32)
        pos = np.arange(start, start + n)
        slots = self.table[0, pos // self.bs].astype(np.int64) * self.bs + pos % self.bs
        oracle.kv_append(self.k_cache, self.v_cache, np.ascontiguousarray(k),
                         np.ascontiguousarray(v), slots, "f32")
        att = oracle.paged_attention(np.ascontiguousarray(q[None]), self.k_cache,
                                     self.v_cache, self.table,
                                     np.array([start + n], np.int32),
                                     1.0 / np.sqrt(self.D), "f32")[0]
        h = x + att.reshape(n, self.H * self.D) @ self.wo
        return h @ self.head


def greedy(model, prompt, n_tokens):
    tokens = list(prompt)
    logits = model.forward(np.array(tokens), 0)
    for _ in range(n_tokens):
        nxt = int(np.argmax(logits[-1]))
        tokens.append(nxt)
        logits = model.forward(np.array([nxt]), len(tokens) - 1)
    return tokens[:len(prompt) + n_tokens]


def speculative(model, prompt, n_tokens, propose, n_drafts):
    """Greedy speculative decoding: the cache holds every accepted token but
    the last; each pass scores [last, drafts...] and accepts drafts while
    they equal the target's argmax, then appends the target's own token."""
    tokens = list(prompt)
    if len(prompt) > 1:
        model.forward(np.array(prompt[:-1]), 0)
    passes = accepted_total = 0
    while len(tokens) < len(prompt) + n_tokens:
        drafts = list(propose(tokens, n_drafts))
        logits = model.forward(np.array([tokens[-1]] + drafts), len(tokens) - 1)
        pred = np.argmax(logits, axis=-1)
        n_acc = 0
        while n_acc < len(drafts) and drafts[n_acc] == pred[n_acc]:
            n_acc += 1
        tokens += drafts[:n_acc] + [int(pred[n_acc])]
        # truncating the cache = the next pass starts writing at len(tokens)-1
        passes += 1
        accepted_total += n_acc
    return tokens[:len(prompt) + n_tokens], passes, accepted_total


def ancestor_masks(parents):
    """Bit k of mask[j] set iff node k is node j or one of its ancestors
    (parents[0] = -1 for the root; parents[j] < j)."""
    masks = []
    for j, par in enumerate(parents):
        masks.append((1 << j) | (masks[par] if par >= 0 else 0))
    return np.array(masks, dtype=np.uint64)


def forward_tree(model, tokens, parents, start):
    """Logits of the tree nodes: node j sits at position start + depth(j) but
    in cache slot start + j; it attends to the cache and its ancestors."""
    n = len(tokens)
    depth = [0] * n
    for j in range(1, n):
        depth[j] = depth[parents[j]] + 1
    pos = start + np.array(depth)
    x = model.emb[tokens] + model.pos[pos]
    q = (x @ model.wq).reshape(n, model.H, model.D).astype(np.float32)
    k = (x @ model.wk).reshape(n, model.Hkv, model.D).astype(np.float32)
    v = (x @ model.wv).reshape(n, model.Hkv, model.D).astype(np.float32)
    rows = np.arange(start, start + n)
    slots = model.table[0, rows // model.bs].astype(np.int64) * model.bs + rows % model.bs
    oracle.kv_append(model.k_cache, model.v_cache, np.ascontiguousarray(k),
                     np.ascontiguousarray(v), slots, "f32")
    att = oracle.tree_attention(np.ascontiguousarray(q[None]), model.k_cache, model.v_cache,
                                model.table, np.array([start + n], np.int32),
                                1.0 / np.sqrt(model.D), "f32", ancestor_masks(parents))[0]
    h = x + att.reshape(n, model.H * model.D) @ model.wo
    return h @ model.head, depth


def _move_row(model, src, dst):
    """Copy cache row `src` of the sequence to row `dst` (K and V)."""
    bs = model.bs
    for cache in (model.k_cache, model.v_cache):
        cache[model.table[0, dst // bs], :, dst % bs] = cache[model.table[0, src // bs], :, src % bs]


def tree_speculative(model, prompt, n_tokens, propose_tree):
    """Greedy verification of a candidate tree per pass: the longest path
    whose tokens match the target's argmax is kept, plus the target's own
    next token; the accepted nodes' K/V rows are moved to their positions."""
    tokens = list(prompt)
    if len(prompt) > 1:
        model.forward(np.array(prompt[:-1]), 0)
    passes = 0
    while len(tokens) < len(prompt) + n_tokens:
        cand_tokens, cand_parents = propose_tree(tokens)
        node_tokens = [tokens[-1]] + cand_tokens
        parents = [-1] + cand_parents
        start = len(tokens) - 1
        logits, depth = forward_tree(model, np.array(node_tokens), parents, start)
        pred = np.argmax(logits, axis=-1)
        path, node = [0], 0
        while True:
            nxt = [c for c in range(1, len(node_tokens))
                   if parents[c] == node and node_tokens[c] == pred[node]]
            if not nxt:
                break
            node = nxt[0]
            path.append(node)
        for d, idx in enumerate(path):
            _move_row(model, start + idx, start + d)
        tokens += [node_tokens[i] for i in path[1:]] + [int(pred[path[-1]])]
        passes += 1
    return tokens[:len(prompt) + n_tokens], passes
