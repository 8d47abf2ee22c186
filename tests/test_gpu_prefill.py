"""Chunked prefill through the C ABI: chunk slots and the chunk's append bit
for bit, attention within tolerance of the oracle's causal definition."""
import numpy as np
import pytest
import torch

from gpu_helpers import Guarded, compare
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _dev(wl, device):
    return (torch.from_numpy(wl.block_tables).to(device), torch.from_numpy(wl.context_lens).to(device),
            torch.from_numpy(wl.query_start).to(device))


def _oracle_step(oracle, wl):
    kc, vc = W.bits(wl.k_cache).copy(), W.bits(wl.v_cache).copy()
    slots = oracle.chunk_slot_mapping(wl.block_tables, wl.context_lens, wl.query_start,
                                      wl.shape.block_size)
    oracle.cache_append(W.bits(wl.k_new), W.bits(wl.v_new), slots, kc, vc, wl.shape.block_size, 0, 1.0)
    out = oracle.prefill(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens, wl.query_start,
                         wl.shape.num_kv_heads, wl.shape.block_size, wl.softmax_scale)
    return slots, kc, vc, out


def _gpu_step(api, wl, device, kernel="auto"):
    bt, cl, qs = _dev(wl, device)
    g_slots = Guarded((int(wl.query_start[-1]),), torch.int32, device, fill=-7)
    g_out = Guarded(wl.q.shape, torch.bfloat16, device, fill=float("nan"))
    slots = api.chunk_slot_mapping(bt, cl, qs, wl.shape.block_size, out=g_slots.tensor)
    api.cache_append(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache)
    out = api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len, wl.softmax_scale,
                      out=g_out.tensor, kernel=kernel)
    torch.cuda.synchronize()
    g_slots.check(f"prefill {kernel} chunk slots")
    g_out.check(f"prefill {kernel} out")
    return slots.cpu().numpy(), out


@pytest.mark.parametrize("kernel", ["auto", "mma"])
@pytest.mark.parametrize("D,B,G,Hkv", [(128, 16, 4, 2), (128, 32, 8, 1), (64, 16, 16, 1),
                                       (64, 32, 1, 3), (128, 16, 2, 2), (128, 16, 16, 1),
                                       (128, 32, 1, 2)])
def test_prefill_matches_oracle(api, oracle, cuda_device, D, B, G, Hkv, kernel):
    wl = W.make_prefill(cuda_device, seed=D + B + G, num_seqs=5, chunk=[1, 7, 64, 300, 33],
                        prefixes=[0, 5, 33, 300, 16], num_q_heads=G * Hkv, num_kv_heads=Hkv,
                        head_dim=D, block_size=B)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    slots_ref, kc_ref, vc_ref, ref = _oracle_step(oracle, wl)
    slots, out = _gpu_step(api, wl, cuda_device, kernel)
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref) and np.array_equal(W.bits(wl.v_cache), vc_ref)
    compare(out, ref, what=f"prefill {kernel} D{D} B{B} G{G}")
    assert api.device_errors() == 0


@pytest.mark.parametrize("G,Hkv,B,D", [(4, 2, 16, 128), (16, 1, 32, 128), (1, 4, 16, 128), (4, 2, 16, 64),
                                       (1, 4, 32, 64)])
def test_prefill_many_items_matches_oracle(api, oracle, cuda_device, G, Hkv, B, D):
    """Several waves of (query-tile pair, KV head, sequence) blocks over 48
    sequences with ragged chunks and prefixes: blocks with no rows, with one
    tile, with a partial tile and with a partial last key block, all checked
    against the oracle element by element."""
    rng = np.random.default_rng(100 + G + B)
    S = 48
    chunks = rng.integers(1, 200, size=S, endpoint=True).tolist()
    prefixes = rng.integers(16, 300, size=S, endpoint=True).tolist()
    wl = W.make_prefill(cuda_device, seed=G + Hkv + B + D, num_seqs=S, chunk=chunks, prefixes=prefixes,
                        num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=D, block_size=B)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    slots_ref, kc_ref, vc_ref, ref = _oracle_step(oracle, wl)
    slots, out = _gpu_step(api, wl, cuda_device, "auto")
    assert np.array_equal(slots, slots_ref)
    compare(out, ref, what=f"prefill many items G{G} B{B} D{D}")
    assert api.device_errors() == 0


@pytest.mark.parametrize("S,ties", [(8, True), (32, False), (33, False), (32, True)])
def test_prefill_sequence_order(api, oracle, cuda_device, S, ties):
    """Grids of under two waves run their sequences longest context first,
    ranked inside the kernel (up to 32 sequences; 33 keep the launch order).
    Equal contexts rank by index.  Every sequence is computed exactly once,
    so each output row matches the oracle."""
    rng = np.random.default_rng(200 + S)
    chunks = [40] * S if ties else rng.integers(1, 90, size=S, endpoint=True).tolist()
    prefixes = [100] * S if ties else rng.integers(0, 400, size=S, endpoint=True).tolist()
    if ties and S > 8:
        prefixes[S // 2] = 300  # one longer among equal ones
    wl = W.make_prefill(cuda_device, seed=300 + S, num_seqs=S, chunk=chunks, prefixes=prefixes,
                        num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    slots_ref, kc_ref, vc_ref, ref = _oracle_step(oracle, wl)
    slots, out = _gpu_step(api, wl, cuda_device, "auto")
    assert np.array_equal(slots, slots_ref)
    compare(out, ref, what=f"prefill sequence order S{S} ties={ties}")
    assert api.device_errors() == 0


def make_e4m3_prefill(oracle, device, **kw):
    """A prefill workload whose pool is E4M3: the bf16 pool's codes of
    x / kv_scale by the oracle's encoder (token i of the pool -> slot i),
    kv_scale = the largest magnitude / 448.  Returns (workload, kv_scale)."""
    wl = W.make_prefill(device, **kw)
    scale = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
    kb, vb = W.bits(wl.k_cache), W.bits(wl.v_cache)
    NB, Hkv, B, D = kb.shape
    kc = np.zeros((NB, Hkv, B, D), np.uint8)
    vc = np.zeros_like(kc)
    oracle.cache_append(kb.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D),
                        vb.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D),
                        np.arange(NB * B, dtype=np.int32), kc, vc, B, 1, scale)
    wl.k_cache = torch.from_numpy(kc).to(device)
    wl.v_cache = torch.from_numpy(vc).to(device)
    return wl, scale


def e4m3_prefill_step(api, oracle, wl, scale, device):
    """Oracle and library of one E4M3 prefill step: chunk slots, the chunk's
    E4M3 append (bit for bit), attention.  Returns (oracle out, library out)."""
    kc, vc = W.bits(wl.k_cache).copy(), W.bits(wl.v_cache).copy()
    slots_ref = oracle.chunk_slot_mapping(wl.block_tables, wl.context_lens, wl.query_start,
                                          wl.shape.block_size)
    oracle.cache_append(W.bits(wl.k_new), W.bits(wl.v_new), slots_ref, kc, vc, wl.shape.block_size, 1, scale)
    ref = oracle.prefill(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens, wl.query_start,
                         wl.shape.num_kv_heads, wl.shape.block_size, wl.softmax_scale, kv_dtype=1,
                         kv_scale=scale)
    bt, cl, qs = _dev(wl, device)
    g_out = Guarded(wl.q.shape, torch.bfloat16, device, fill=float("nan"))
    slots = api.chunk_slot_mapping(bt, cl, qs, wl.shape.block_size)
    api.cache_append(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache, scale=scale)
    out = api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len, wl.softmax_scale,
                      out=g_out.tensor, kv_scale=scale)
    torch.cuda.synchronize()
    g_out.check("prefill E4M3 out")
    assert np.array_equal(slots.cpu().numpy(), slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc) and np.array_equal(W.bits(wl.v_cache), vc)
    return ref, out


@pytest.mark.parametrize("G,Hkv,B", [(4, 2, 16), (1, 4, 32), (16, 1, 16), (8, 1, 32)])
def test_prefill_e4m3_matches_oracle(api, oracle, cuda_device, G, Hkv, B):
    """E4M3 cache (one scale for K and V): the pages widen to fp16 in
    shared memory and the products run in fp16; against the oracle fed the
    same E4M3 bytes, with NaN codes in every row outside the contexts."""
    wl, scale = make_e4m3_prefill(oracle, cuda_device, seed=70 + G + B, num_seqs=5,
                                  chunk=[1, 7, 64, 300, 33], prefixes=[0, 5, 33, 300, 16],
                                  num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=128, block_size=B)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    ref, out = e4m3_prefill_step(api, oracle, wl, scale, cuda_device)
    compare(out, ref, what=f"prefill E4M3 G{G} B{B}")
    assert api.device_errors() == 0


@pytest.mark.parametrize("G,Hkv,B", [(4, 2, 16), (1, 4, 32), (16, 1, 16)])
def test_prefill_scaled_matches_oracle(api, oracle, cuda_device, G, Hkv, B):
    """E4M3 cache with a K and a V scale per KV head: the pool encoded by
    the oracle with each head's scales, the chunk appended by the library's
    per-head append (bit for bit), attention against the oracle."""
    wl = W.make_prefill(cuda_device, seed=90 + G + B, num_seqs=5, chunk=[1, 7, 64, 300, 33],
                        prefixes=[0, 5, 33, 300, 16], num_q_heads=G * Hkv, num_kv_heads=Hkv,
                        head_dim=128, block_size=B)
    base = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
    ks = np.array([base * (1.0 + 0.37 * h) for h in range(Hkv)], np.float32)
    vs = np.array([base * (1.6 - 0.21 * h) for h in range(Hkv)], np.float32)
    kb, vb = W.bits(wl.k_cache), W.bits(wl.v_cache)
    NB, _, _, D = kb.shape
    kc = np.zeros((NB, Hkv, B, D), np.uint8)
    vc = np.zeros_like(kc)
    oracle.cache_append_scaled(kb.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D),
                               vb.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D),
                               np.arange(NB * B, dtype=np.int32), kc, vc, B, ks, vs)
    wl.k_cache = torch.from_numpy(kc).to(cuda_device)
    wl.v_cache = torch.from_numpy(vc).to(cuda_device)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    kc, vc = W.bits(wl.k_cache).copy(), W.bits(wl.v_cache).copy()
    slots_ref = oracle.chunk_slot_mapping(wl.block_tables, wl.context_lens, wl.query_start, B)
    oracle.cache_append_scaled(W.bits(wl.k_new), W.bits(wl.v_new), slots_ref, kc, vc, B, ks, vs)
    ref = oracle.prefill_scaled(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens, wl.query_start,
                                Hkv, B, wl.softmax_scale, ks, vs)
    bt, cl, qs = _dev(wl, cuda_device)
    ks_d, vs_d = torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device)
    g_out = Guarded(wl.q.shape, torch.bfloat16, cuda_device, fill=float("nan"))
    slots = api.chunk_slot_mapping(bt, cl, qs, B)
    api.cache_append_scaled(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache, ks_d, vs_d)
    out = api.prefill_scaled(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len, ks_d, vs_d,
                             wl.softmax_scale, out=g_out.tensor)
    torch.cuda.synchronize()
    g_out.check("prefill scaled out")
    assert np.array_equal(slots.cpu().numpy(), slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc) and np.array_equal(W.bits(wl.v_cache), vc)
    compare(out, ref, what=f"prefill per-head scales G{G} B{B}")
    assert api.device_errors() == 0


@pytest.mark.parametrize("G,Hkv,B", [(4, 2, 16), (1, 4, 32)])
def test_prefill_e4m3_many_items(api, oracle, cuda_device, G, Hkv, B):
    """48 ragged sequences over several waves of blocks, E4M3 cache."""
    rng = np.random.default_rng(400 + G + B)
    S = 48
    wl, scale = make_e4m3_prefill(oracle, cuda_device, seed=80 + G + B, num_seqs=S,
                                  chunk=rng.integers(1, 200, size=S, endpoint=True).tolist(),
                                  prefixes=rng.integers(16, 300, size=S, endpoint=True).tolist(),
                                  num_q_heads=G * Hkv, num_kv_heads=Hkv, head_dim=128, block_size=B)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    ref, out = e4m3_prefill_step(api, oracle, wl, scale, cuda_device)
    compare(out, ref, what=f"prefill E4M3 many items G{G} B{B}")
    assert api.device_errors() == 0


@pytest.mark.parametrize("kernel", ["auto", "mma"])
def test_prefill_empty_chunks(api, oracle, cuda_device, kernel):
    """Sequences that bring no chunk rows sit between ones that do: their
    blocks have nothing to compute and nothing of theirs is written."""
    wl = W.make_prefill(cuda_device, seed=31, num_seqs=6, chunk=[0, 5, 0, 130, 1, 0],
                        prefixes=[40, 0, 300, 77, 16, 9], num_q_heads=8, num_kv_heads=2,
                        head_dim=128, block_size=16)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    slots_ref, kc_ref, vc_ref, ref = _oracle_step(oracle, wl)
    slots, out = _gpu_step(api, wl, cuda_device, kernel)
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref) and np.array_equal(W.bits(wl.v_cache), vc_ref)
    compare(out, ref, what=f"prefill empty chunks {kernel}")
    assert api.device_errors() == 0


@pytest.mark.parametrize("B", [16, 32])
def test_prefill_long_context(api, oracle, cuda_device, B):
    """A 64-token chunk at the end of a 32,768-token context: 512 key blocks
    per tile pair, so every stage of the page ring is reused many times."""
    wl = W.make_prefill(cuda_device, seed=40 + B, num_seqs=2, chunk=[64, 40],
                        prefixes=[32768 - 64, 20000], num_q_heads=4, num_kv_heads=1,
                        head_dim=128, block_size=B)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    _, _, _, ref = _oracle_step(oracle, wl)
    _, out = _gpu_step(api, wl, cuda_device, "auto")
    compare(out, ref, what=f"prefill long context B{B}")
    assert api.device_errors() == 0


def test_prefill_last_row_is_decode(api, cuda_device):
    """The last chunk token of every sequence computes what the decode
    kernel computes for that context."""
    wl = W.make_prefill(cuda_device, seed=2, num_seqs=6, chunk=48, max_prefix=700)
    bt, cl, qs = _dev(wl, cuda_device)
    slots = api.chunk_slot_mapping(bt, cl, qs, 16)
    api.cache_append(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache)
    out = api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len)
    last = torch.from_numpy(wl.query_start[1:] - 1).long().to(cuda_device)
    dec = api.decode(wl.q[last].contiguous(), wl.k_cache, wl.v_cache, bt, cl)
    diff = (out[last].float() - dec.float()).abs().max().item()
    assert diff <= 1e-2


@pytest.mark.slow
def test_prefill_workload_sampled(api, oracle, cuda_device):
    """The 8192-token chunked-prefill workload: every row of three sequences
    against the oracle."""
    wl = W.make_prefill(cuda_device)
    W.poison_prefill(wl)
    pick = [0, 7, 15]
    # oracle on those sequences only (compacted), before the GPU append
    B = wl.shape.block_size
    rows = [wl.block_tables[s, : (int(wl.context_lens[s]) + B - 1) // B] for s in pick]
    used = np.unique(np.concatenate(rows))
    remap = {int(b): i for i, b in enumerate(used)}
    tables = np.full((len(pick), wl.block_tables.shape[1]), -1, np.int32)
    for i, row in enumerate(rows):
        tables[i, : len(row)] = [remap[int(b)] for b in row]
    idx = torch.from_numpy(used.astype(np.int64)).to(cuda_device)
    kc = W.bits(wl.k_cache.index_select(0, idx))
    vc = W.bits(wl.v_cache.index_select(0, idx))
    ctx = wl.context_lens[pick]
    qs_all = wl.query_start
    spans = [(int(qs_all[s]), int(qs_all[s + 1])) for s in pick]
    qs = np.concatenate([[0], np.cumsum([b - a for a, b in spans])]).astype(np.int32)
    sel = np.concatenate([np.arange(a, b) for a, b in spans])
    slots = oracle.chunk_slot_mapping(tables, ctx, qs, B)
    oracle.cache_append(W.bits(wl.k_new)[sel], W.bits(wl.v_new)[sel], slots, kc, vc, B, 0, 1.0)
    ref = oracle.prefill(W.bits(wl.q)[sel], kc, vc, tables, ctx, qs, wl.shape.num_kv_heads, B,
                         wl.softmax_scale)
    _, out = _gpu_step(api, wl, cuda_device)
    compare(out[torch.from_numpy(sel).to(cuda_device)], ref, what="prefill workload")
    bt, cl, qsd = _dev(wl, cuda_device)
    out2 = api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qsd, wl.max_query_len,
                       wl.softmax_scale, kernel="mma")
    compare(out2[torch.from_numpy(sel).to(cuda_device)], ref, what="prefill workload (mma)")
    assert api.device_errors() == 0
