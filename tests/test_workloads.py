"""The seeded workload generator: shapes, table validity, sharing, poison."""
import numpy as np
import pytest
import torch

from paged_kv_cache_193_gb300 import workloads as W


def _check_tables(wl):
    B = wl.shape.block_size
    seen = {}
    for s in range(wl.shape.num_seqs):
        n = int(wl.context_lens[s])
        need = (n + B - 1) // B
        row = wl.block_tables[s]
        assert np.all(row[:need] >= 0) and np.all(row[:need] < wl.num_blocks)
        assert np.all(row[need:] == -1)
        assert len(set(row[:need].tolist())) == need
        for j, b in enumerate(row[:need]):
            seen.setdefault(int(b), set()).add((s, j))
    return seen


def test_tiny_matches_its_description():
    wl = W.make("tiny")
    assert wl.context_lens.tolist() == [1, 17, 100, 255]
    assert (wl.shape.num_q_heads, wl.shape.num_kv_heads, wl.shape.head_dim) == (8, 2, 64)
    assert wl.num_blocks == 64
    seen = _check_tables(wl)
    assert len(seen) == 26  # 1 + 2 + 7 + 16 blocks, none shared
    assert wl.softmax_scale == 1 / 8


@pytest.mark.parametrize("name,S,lo,hi", [("llama8b", 256, 512, 2048), ("long70b", 64, 4096, 32768)])
def test_uniform_contexts_and_pool(name, S, lo, hi):
    wl = W.make(name, fill_cache=False)
    assert wl.shape.num_seqs == S
    assert wl.context_lens.min() >= lo and wl.context_lens.max() <= hi
    B = wl.shape.block_size
    need = sum((int(c) + B - 1) // B for c in wl.context_lens)
    assert wl.num_blocks == int(np.ceil(1.2 * need))
    seen = _check_tables(wl)
    assert all(len(v) == 1 for v in seen.values())
    # shuffled: consecutive logical blocks are not consecutive physical blocks
    row = wl.block_tables[0][:8]
    assert not np.all(np.diff(row) == 1)


def test_prefix_sharing_layout():
    wl = W.make("prefix_fp8", fill_cache=False)
    seen = _check_tables(wl)
    prefix = wl.block_tables[:, :128]
    assert np.all(prefix == prefix[0])
    assert all(len(seen[int(b)]) == 256 for b in prefix[0])
    suf = wl.context_lens - 2048
    assert suf.min() >= 64 and suf.max() <= 512
    assert wl.shape.kv_dtype == W.KV_FP8_E4M3
    assert wl.unique_kv_bytes() < wl.kv_bytes() / 5


def test_ctx128k_shape():
    wl = W.make("ctx128k", fill_cache=False, extra_steps=3)
    assert wl.context_lens.tolist() == [131072] * 8
    assert (wl.shape.num_q_heads, wl.shape.num_kv_heads) == (128, 8)
    assert wl.block_tables.shape[1] == (131072 + 3 + 15) // 16
    _check_tables(wl)


def test_kv_bytes_per_layer_formula():
    wl = W.make("tiny")
    assert wl.kv_bytes() == (1 + 17 + 100 + 255) * 2 * 64 * 2 * 2


def test_poison_marks_only_dead_rows():
    wl = W.make("tiny")
    W.poison(wl, pending=True)
    k = W.bits(wl.k_cache)
    nan = k == W.BF16_NAN_BITS
    B = 16
    for s, n in enumerate(wl.context_lens):
        for t in range(n):
            b = wl.block_tables[s, t // B]
            assert nan[b, :, t % B].all() == (t == n - 1)


def test_allocator_refcounts():
    a = W.BlockAllocator(4, np.random.default_rng(0))
    x = a.allocate(3)
    a.share(x[:1])
    a.free(x)
    assert a.num_free() == 3
    a.free(x[:1])
    assert a.num_free() == 4
    with pytest.raises(MemoryError):
        a.allocate(5)


def test_seeded_reproducible():
    a, b = W.make("tiny"), W.make("tiny")
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    assert np.array_equal(a.block_tables, b.block_tables)


def test_prefill_workload_shapes():
    """The chunked-prefill step: chunk offsets are the prefix sums of the
    chunks, each context is its prefix plus its chunk, and the query / new
    K/V rows are the chunk rows."""
    chunks, prefixes = [0, 5, 130, 1, 64], [40, 0, 77, 300, 16]
    wl = W.make_prefill("cpu", seed=3, num_seqs=5, chunk=chunks, prefixes=prefixes, num_q_heads=8,
                        num_kv_heads=2, head_dim=128, block_size=16)
    assert wl.query_start.tolist() == [0, 0, 5, 135, 136, 200]
    assert wl.context_lens.tolist() == [p + c for p, c in zip(prefixes, chunks)]
    assert wl.max_query_len == 130
    assert tuple(wl.q.shape) == (200, 8, 128) and tuple(wl.k_new.shape) == (200, 2, 128)
    assert wl.q.dtype == torch.bfloat16
    seen = _check_tables(wl)
    assert all(len(v) == 1 for v in seen.values())  # no block is shared between sequences


def test_prefill_default_is_the_8192_token_step():
    wl = W.make_prefill("cpu")
    assert wl.shape.num_seqs == 16 and int(wl.query_start[-1]) == 8192
    assert np.all(np.diff(wl.query_start) == 512)
    prefixes = wl.context_lens - 512
    assert prefixes.min() >= 0 and prefixes.max() <= 2048
    assert (wl.shape.num_q_heads, wl.shape.num_kv_heads, wl.shape.head_dim) == (32, 8, 128)


def test_prefill_flops_count_the_causal_pairs():
    """4 * D * Hq multiply-adds x 2 per (query, key) pair the causal mask
    keeps, against a brute-force walk over every chunk row and every key."""
    wl = W.make_prefill("cpu", seed=4, num_seqs=3, chunk=[7, 1, 20], prefixes=[0, 33, 5],
                        num_q_heads=4, num_kv_heads=1, head_dim=64, block_size=16)
    pairs = 0
    for s in range(3):
        n = int(wl.context_lens[s])
        c = int(wl.query_start[s + 1] - wl.query_start[s])
        for i in range(c):
            pos = n - c + i
            pairs += sum(1 for t in range(n) if t <= pos)
    assert wl.attention_flops() == 4 * 64 * 4 * pairs


def test_prefill_poison_marks_only_rows_outside_the_prefixes():
    """After poisoning, exactly the cached-prefix rows of every sequence are
    finite: the chunk rows (which the append writes) and unused rows hold NaN."""
    wl = W.make_prefill("cpu", seed=6, num_seqs=3, chunk=[10, 3, 40], prefixes=[20, 0, 47],
                        num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16)
    W.poison_prefill(wl)
    B = wl.shape.block_size
    finite = torch.isfinite(wl.k_cache.float()).all(dim=3).all(dim=1).numpy()  # [NB, B]
    expect = np.zeros_like(finite)
    for s in range(3):
        n = int(wl.context_lens[s])
        c = int(wl.query_start[s + 1] - wl.query_start[s])
        for t in range(n - c):
            expect[wl.block_tables[s, t // B], t % B] = True
    assert np.array_equal(finite, expect)
    assert np.array_equal(torch.isfinite(wl.v_cache.float()).all(dim=3).all(dim=1).numpy(), expect)
