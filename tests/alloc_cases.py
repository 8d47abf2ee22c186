"""Pre-step states of a paged cache for the block-allocation checks: block
tables with shared prompt blocks (full and partially filled), private
suffixes, empty sequences, consistent reference counts and a shuffled free
stack of every unreferenced block."""
from __future__ import annotations

import numpy as np


def make_state(seed: int, B: int = 4, NB: int = 64, Hkv: int = 2, D: int = 8, elem=np.uint16,
               extra_free: int | None = None):
    """Lengths are set relative to the block size B, so the same situations
    arise for any B >= 4."""
    rng = np.random.default_rng(seed)
    order = list(rng.permutation(NB))
    seqs = []  # (tokens already cached, shared prompt blocks)
    # group A: share a prompt of one full and one partial block, each about to
    # append its first own token into the partial (shared) block
    prompt_a = [order.pop(), order.pop()]
    for _ in range(3):
        seqs.append((B + B // 2, list(prompt_a)))
    # group B: share a prompt of two full blocks plus private suffixes
    prompt_b = [order.pop(), order.pop()]
    for extra in (0, 1, 3, B + 1):
        seqs.append((2 * B + extra, list(prompt_b)))
    # private sequences of assorted lengths, and an empty one
    for n in (1, 3, B, B + 3, 3 * B, 0):
        seqs.append((n, []))
    S = len(seqs)
    MB = 8
    tables = np.full((S, MB), -1, np.int32)
    for s, (pre, shared) in enumerate(seqs):
        row = list(shared)
        need = (pre + B - 1) // B
        while len(row) < need:
            row.append(order.pop())
        tables[s, :need] = row[:need]
    refc = np.zeros(NB, np.int32)
    for s, (pre, _) in enumerate(seqs):
        for j in range((pre + B - 1) // B):
            refc[tables[s, j]] += 1
    free = np.array(order, np.int32)
    if extra_free is not None:
        free = free[:extra_free]
    # every non-empty sequence appends one token this step
    ctx = np.array([pre + 1 if pre > 0 else 0 for pre, _ in seqs], np.int32)
    g = np.random.default_rng(seed + 1)
    kc = g.integers(0, 2**15, size=(NB, Hkv, B, D)).astype(elem)
    vc = g.integers(0, 2**15, size=(NB, Hkv, B, D)).astype(elem)
    return dict(tables=tables, ctx=ctx, free=free, free_count=len(free), refc=refc, k=kc, v=vc,
                B=B, NB=NB)


def make_chunk_state(seed, chunks, NB=128, **kw):
    """A pre-step state from make_state in which sequence s brings
    chunks[s % len(chunks)] new tokens (empty sequences bring none):
    ctx counts them, qs holds the chunk offsets, pre the cached lengths."""
    st = make_state(seed, NB=NB, **kw)
    pre = np.where(st["ctx"] > 0, st["ctx"] - 1, 0)
    c = np.array([chunks[i % len(chunks)] if pre[i] > 0 else 0 for i in range(len(pre))], np.int32)
    st["ctx"] = (pre + c).astype(np.int32)
    st["qs"] = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
    st["pre"] = pre.astype(np.int32)
    return st


def gather_rows(tables, n, s, cache, B):
    """Logical rows [0, n) of sequence s through its table (all heads)."""
    return np.stack([cache[tables[s, t // B], :, t % B] for t in range(n)]) if n else None
