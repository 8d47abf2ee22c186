"""GPU parity of every kernel against the oracle on small seeded cases that
still span several tiles, partitions and ragged tails.  Calls go through the
C ABI (via the thin binding)."""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import bf16_to_f64, compare, device_tables, guard_step, quantize_with_oracle
from paged_cases import bits_to_f64
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _random_case(seed, S, Hq, Hkv, D, B, ctx_list, kv_dtype, oracle, device, nb_extra=7):
    """Random pool + shuffled tables for the given contexts (contexts include
    the token appended this step)."""
    rng = np.random.default_rng(seed)
    ctx = np.array(ctx_list, np.int64)
    need = sum((int(c) + B - 1) // B for c in ctx)
    nb = need + nb_extra
    tables, _ = W.build_tables(ctx, B, nb, rng)
    shape = W.Shape(S, Hq, Hkv, D, B, kv_dtype=kv_dtype)
    wl = W._finish("case", shape, ctx, tables, nb, device, seed)
    if kv_dtype == W.KV_FP8_E4M3:
        quantize_with_oracle(oracle, wl)
    return wl


def _oracle_step(oracle, wl, partition_size=0):
    """Oracle's view of one step: append the new tokens into a host copy of
    the caches, then attend.  Returns (slots, k_cache_after, v_cache_after, out)."""
    kc = W.bits(wl.k_cache).copy()
    vc = W.bits(wl.v_cache).copy()
    slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, wl.shape.block_size)
    oracle.cache_append(W.bits(wl.k_new), W.bits(wl.v_new), slots, kc, vc, wl.shape.block_size,
                        wl.shape.kv_dtype, wl.kv_scale)
    out = oracle.decode(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens,
                        wl.shape.num_kv_heads, wl.shape.block_size, wl.softmax_scale,
                        kv_dtype=wl.shape.kv_dtype, kv_scale=wl.kv_scale)
    return slots, kc, vc, out


def _gpu_step(api, wl, partition_size, fused=True):
    bt, cl = device_tables(wl, wl.k_cache.device)
    step = api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, wl.shape.num_q_heads,
                          wl.softmax_scale, wl.kv_scale, partition_size, fused=fused)
    check_guards = guard_step(step)
    out = step(wl.q, wl.k_new, wl.v_new).clone()
    torch.cuda.synchronize()
    check_guards(f"decode step ps={partition_size} fused={fused}")
    return step.slots.cpu().numpy(), out


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "separate"])
@pytest.mark.parametrize("partition_size", [0, 16, 32, 64, 512])
def test_tiny_step_matches_oracle(api, oracle, cuda_device, partition_size, fused):
    wl = W.make("tiny", device=cuda_device)
    W.poison(wl, pending=True)
    api.device_errors(clear=True)
    slots_ref, kc_ref, vc_ref, out_ref = _oracle_step(oracle, wl)
    slots, out = _gpu_step(api, wl, partition_size, fused)
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref)
    assert np.array_equal(W.bits(wl.v_cache), vc_ref)
    compare(out, out_ref, what=f"tiny ps={partition_size}")
    assert api.device_errors() == 0


CASES = []
for D in (64, 128):
    for B in (16, 32):
        for G, Hkv in ((1, 2), (4, 2), (8, 1), (16, 1), (6, 2)):
            for kv in (W.KV_BF16, W.KV_FP8_E4M3):
                CASES.append((D, B, G, Hkv, kv))


@pytest.mark.parametrize("D,B,G,Hkv,kv", CASES)
def test_shapes_match_oracle(api, oracle, cuda_device, D, B, G, Hkv, kv):
    ctx = [1, B - 1, B, B + 1, 3 * B + 5, 700]
    wl = _random_case(D * 7 + B * 3 + G + kv, len(ctx), G * Hkv, Hkv, D, B, ctx, kv, oracle,
                      cuda_device)
    W.poison(wl, pending=True)
    slots_ref, kc_ref, vc_ref, out_ref = _oracle_step(oracle, wl)
    for ps, fused in ((0, True), (4 * B, True), (256, False), (0, False)):
        # poison the pending slots again so each call's append is checked
        W.poison(wl, pending=True)
        slots, out = _gpu_step(api, wl, ps, fused)
        assert np.array_equal(slots, slots_ref)
        assert np.array_equal(W.bits(wl.k_cache), kc_ref)
        assert np.array_equal(W.bits(wl.v_cache), vc_ref)
        compare(out, out_ref, what=f"D{D} B{B} G{G} kv{kv} ps{ps}")
    assert api.device_errors() == 0


def test_slot_mapping_bitexact(api, oracle, cuda_device):
    rng = np.random.default_rng(5)
    for B in (16, 32):
        ctx = np.array([0, 1, B - 1, B, B + 1, 5 * B, 333, 4096], np.int32)
        mb = int(max((c + B - 1) // B for c in ctx)) + 3
        tables, _ = W.build_tables(ctx, B, int(sum((c + B - 1) // B for c in ctx)) + 10, rng, mb)
        bt = torch.from_numpy(tables).to(cuda_device)
        cl = torch.from_numpy(ctx).to(cuda_device)
        got = api.slot_mapping(bt, cl, B).cpu().numpy()
        assert np.array_equal(got, oracle.slot_mapping(tables, ctx, B))


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8_E4M3])
@pytest.mark.parametrize("D,B", [(64, 16), (128, 32)])
def test_append_bitexact(api, oracle, cuda_device, kv, D, B):
    rng = np.random.default_rng(11)
    NB, Hkv, T = 40, 3, 57
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int32)
    slots[::7] = -1
    g = torch.Generator().manual_seed(3)
    k = torch.randn(T, Hkv, D, generator=g).mul(3).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).mul(3).to(torch.bfloat16)
    dt = torch.bfloat16 if kv == W.KV_BF16 else torch.uint8
    kc0 = torch.randint(0, 255, (NB, Hkv, B, D * (2 if kv == W.KV_BF16 else 1)), dtype=torch.uint8, generator=g)
    kc0 = kc0.view(dt) if kv == W.KV_BF16 else kc0
    vc0 = kc0.clone()
    scale = 0.0123
    kc_ref, vc_ref = W.bits(kc0).copy(), W.bits(vc0).copy()
    oracle.cache_append(W.bits(k), W.bits(v), slots, kc_ref, vc_ref, B, kv, scale)
    kc, vc = kc0.to(cuda_device), vc0.to(cuda_device)
    api.cache_append(k.to(cuda_device), v.to(cuda_device), torch.from_numpy(slots).to(cuda_device),
                     kc, vc, scale)
    assert np.array_equal(W.bits(kc), kc_ref)
    assert np.array_equal(W.bits(vc), vc_ref)


@pytest.mark.parametrize("scale", [1.0, 4.5 / 448.0, 0.37, 1e-3])
def test_fp8_encode_exhaustive(api, oracle, cuda_device, scale):
    """Every bf16 bit pattern through the GPU append vs the oracle's encoder
    (NaN inputs compared as 'some NaN code')."""
    D, B, Hkv = 128, 16, 1
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    T = 65536 // D
    k = allbits.reshape(T, Hkv, D)
    slots = np.arange(T, dtype=np.int32)
    NB = T // B
    kc_ref = np.zeros((NB, Hkv, B, D), np.uint8)
    vc_ref = np.zeros_like(kc_ref)
    oracle.cache_append(k, k, slots, kc_ref, vc_ref, B, 1, scale)
    kt = W.from_bits(k, cuda_device)
    kc = torch.zeros(NB, Hkv, B, D, dtype=torch.uint8, device=cuda_device)
    vc = torch.zeros_like(kc)
    api.cache_append(kt, kt, torch.from_numpy(slots).to(cuda_device), kc, vc, scale)
    got = W.bits(kc).reshape(-1)
    ref = kc_ref.reshape(-1)
    x = bits_to_f64(allbits).astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        isnan = np.isnan(x / np.float32(scale))
    assert np.all((got[isnan] & 0x7F) == 0x7F)
    bad = np.flatnonzero((got != ref) & ~isnan)
    assert bad.size == 0, [(hex(allbits[i]), hex(got[i]), hex(ref[i])) for i in bad[:8]]


def test_fp8_decode_lanes(api, oracle, cuda_device):
    """Every E4M3 code as K and V of a one-token context: the output row is
    V itself, so the decode's E4M3->fp16 widening and its permuted head-dim
    order are checked code by code."""
    D, B, Hkv, Hq = 128, 16, 1, 1
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]  # finite codes only
    n = codes.size
    reps = (n + D - 1) // D
    pad = np.concatenate([codes, np.zeros(reps * D - n, np.uint8)]).reshape(reps, D)
    S = reps
    kc = np.zeros((S, Hkv, B, D), np.uint8)
    vc = np.zeros_like(kc)
    kc[:, 0, 0, :] = pad
    vc[:, 0, 0, :] = pad[:, ::-1]
    tables = np.arange(S, dtype=np.int32).reshape(S, 1)
    ctx = np.ones(S, np.int32)
    q = torch.randn(S, Hq, D, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    out = api.decode(q.to(cuda_device), torch.from_numpy(kc).to(cuda_device),
                     torch.from_numpy(vc).to(cuda_device), torch.from_numpy(tables).to(cuda_device),
                     torch.from_numpy(ctx).to(cuda_device), 0.1, kv_scale=0.5)
    ref = oracle.decode(W.bits(q), kc, vc, tables, ctx, Hkv, B, 0.1, kv_dtype=1, kv_scale=0.5)
    # a one-token softmax is exactly 1, so out = bf16(V * 0.5)
    compare(out, ref, max_abs=0.0, mean_abs=0.0, what="fp8 code lanes", ulp_rel=0.0)


@pytest.mark.parametrize("D,MB,PS", [(128, 40, 64), (64, 40, 64), (128, 40, 32), (64, 70, 16),
                                     (128, 200, 16), (64, 300, 16)])
def test_reduce_alone(api, oracle, cuda_device, D, MB, PS):
    """The merge alone on random partials: 10, 20, 70, 200 and 300
    partitions per row cover one, four and eight warps per row."""
    rng = np.random.default_rng(21 + MB + D)
    S, Hq, B = 5, 6, 16
    P = api.max_partitions(MB, B, PS)
    ctx = np.array([0, 1, PS, PS + 1, MB * B], np.int32)
    o = rng.standard_normal((S, Hq, P, D)).astype(np.float32)
    m = (rng.standard_normal((S, Hq, P)) * 4).astype(np.float32)
    l = rng.uniform(1, 50, (S, Hq, P)).astype(np.float32)
    ws = torch.zeros(api.workspace_size(S, Hq, D, MB, B, PS), dtype=torch.uint8, device=cuda_device)
    wo, wm, wl_ = api.workspace_views(ws, S, Hq, D, P)
    wo.copy_(torch.from_numpy(o))
    wm.copy_(torch.from_numpy(m))
    wl_.copy_(torch.from_numpy(l))
    out = torch.full((S, Hq, D), float("nan"), dtype=torch.bfloat16, device=cuda_device)
    api.decode_reduce(ws, torch.from_numpy(ctx).to(cuda_device), Hq, D, MB, B, PS, out)
    ref = oracle.merge_partitions(o, m, l, ctx, PS)
    got = bf16_to_f64(out)
    # fp32 merge then one bf16 rounding: within one bf16 ulp of the fp64 value
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0**-8 + 1e-6)
    assert np.array_equal(got[0], np.zeros_like(got[0]))


def test_partitions_match_oracle(api, oracle, cuda_device):
    wl = _random_case(3, 4, 16, 2, 128, 16, [1, 100, 512, 1300], W.KV_BF16, oracle, cuda_device)
    W.poison(wl)
    PS = 256
    bt, cl = device_tables(wl, cuda_device)
    P = api.max_partitions(bt.shape[1], 16, PS)
    ws = torch.zeros(api.workspace_size(4, 16, 128, bt.shape[1], 16, PS), dtype=torch.uint8, device=cuda_device)
    api.decode_partitions(wl.q, wl.k_cache, wl.v_cache, bt, cl, wl.softmax_scale, 1.0, PS, ws)
    o_ref, m_ref, l_ref = oracle.decode_partitions(W.bits(wl.q), W.bits(wl.k_cache), W.bits(wl.v_cache),
                                                   wl.block_tables, wl.context_lens, 2, 16,
                                                   wl.softmax_scale, PS, P)
    wo, wm, wl_ = [t.cpu().numpy().astype(np.float64) for t in api.workspace_views(ws, 4, 16, 128, P)]
    for s, n in enumerate(wl.context_lens):
        np_ = (int(n) + PS - 1) // PS
        assert np.abs(wm[s, :, :np_] - m_ref[s, :, :np_]).max() < 1e-4 * max(1, np.abs(m_ref).max())
        assert np.all(np.abs(wl_[s, :, :np_] / l_ref[s, :, :np_] - 1) < 2e-3)
        assert np.abs(wo[s, :, :np_] - o_ref[s, :, :np_]).max() < 5e-3


def test_permutation_and_prefix_bitwise(api, oracle, cuda_device):
    """The same logical K/V under different physical block assignments, and
    with a prefix shared through the same physical blocks, give bit-identical
    output (the kernel's arithmetic depends only on the logical sequence)."""
    from paged_cases import LogicalCase
    D, B, Hq, Hkv = 128, 16, 32, 8
    c = LogicalCase((200, 64, 97, 80), Hq, Hkv, D, seed=9)
    # equal 64-token prefixes for the sharing check
    for s in range(1, 4):
        c.k[s][:, :64] = c.k[0][:, :64]
        c.v[s][:, :64] = c.v[0][:, :64]
    q = W.from_bits(c.q, cuda_device)
    ctx = torch.tensor(c.ctx, dtype=torch.int32, device=cuda_device)
    outs = []
    for seed, share in ((1, 0), (2, 0), (3, 64)):
        tables, kc, vc = c.paged(B, 60, np.random.default_rng(seed), share_prefix_tokens=share)
        for ps in (0, 64):
            out = api.decode(q, W.from_bits(kc, cuda_device), W.from_bits(vc, cuda_device),
                             torch.from_numpy(tables).to(cuda_device), ctx, 0.09, partition_size=ps)
            outs.append((ps, W.bits(out)))
    for ps in (0, 64):
        same = [o for p, o in outs if p == ps]
        assert all(np.array_equal(same[0], o) for o in same[1:])
    ref = c.sdpa(0.09)
    compare(W.from_bits(outs[0][1]), ref, what="permutation case vs SDPA")


def test_determinism(api, cuda_device):
    wl = W.make("llama8b", device=cuda_device, num_seqs=16)
    bt, cl = device_tables(wl, cuda_device)
    a = api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl, partition_size=512)
    b = api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl, partition_size=512)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_bad_block_and_context_flags(api, cuda_device):
    wl = W.make("tiny", device=cuda_device)
    tables = wl.block_tables.copy()
    tables[3, 2] = wl.num_blocks + 5  # outside the pool
    bt = torch.from_numpy(tables).to(cuda_device)
    cl = torch.from_numpy(wl.context_lens).to(cuda_device)
    api.device_errors(clear=True)
    out = api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl)
    torch.cuda.synchronize()
    assert api.device_errors() & 0x1
    assert torch.isfinite(out.float()).all()
    cl2 = cl.clone()
    cl2[0] = 10_000  # longer than the table
    api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl2)
    assert api.device_errors() & 0x2
    assert api.device_errors() == 0


def test_host_validation(api, cuda_device):
    wl = W.make("tiny", device=cuda_device)
    bt, cl = device_tables(wl, cuda_device)
    with pytest.raises(api.PagedAttentionError) as e:
        api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl, partition_size=24)  # not a multiple of 16
    assert e.value.status == 2
    with pytest.raises(api.PagedAttentionError) as e:
        ws = torch.empty(16, dtype=torch.uint8, device=cuda_device)
        api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl, partition_size=32, workspace=ws)
    assert e.value.status == 3


def test_empty_batch_and_zero_context(api, oracle, cuda_device):
    wl = _random_case(4, 3, 8, 2, 64, 16, [0, 5, 0], W.KV_BF16, oracle, cuda_device)
    bt, cl = device_tables(wl, cuda_device)
    for ps in (0, 16):
        out = api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl, partition_size=ps)
        ref = oracle.decode(W.bits(wl.q), W.bits(wl.k_cache), W.bits(wl.v_cache), wl.block_tables,
                            wl.context_lens, 2, 16, wl.softmax_scale)
        compare(out, ref, what="zero contexts")
        assert np.all(bf16_to_f64(out)[[0, 2]] == 0)
