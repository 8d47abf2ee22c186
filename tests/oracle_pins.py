"""Checks that pin the oracle to things other than itself.

Each ``pin_*`` function takes an ``Oracle`` and raises AssertionError when the
oracle disagrees with what the pages or the mathematics fix:

* the KV-bytes formula's worked example printed in the tuning guide (golden);
* torch's own float8_e4m3fn conversions (a library implementation of the
  OCP E4M3 format the pages name);
* torch ``scaled_dot_product_attention`` in float64 over the LOGICAL K/V,
  repeated per query group (a library routine; the oracle instead walks the
  block table of a randomly permuted pool);
* invariants: any physical permutation gives the same result, shared prefix
  blocks equal private copies, a one-token context returns V, identical keys
  return the mean of V, a large softmax scale stays finite;
* brute-force enumeration of every slot of a sequence for the slot mapping;
* read-back of appended rows through the block table;
* the log-sum-exp identity: merging partition results equals one softmax
  over the union.

``tests/test_oracle.py`` runs them on the oracle; ``tests/test_oracle_mutants.py``
runs them on deliberately broken copies to show each plausible mistake trips
at least one of them.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

from paged_cases import LogicalCase, bits_to_f64

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _e4m3_torch(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _encode_many(o, xs_bits: np.ndarray, scale: float) -> np.ndarray:
    """Run the oracle's append over a one-element-per-token cache so the whole
    array is encoded in one call."""
    n = xs_bits.size
    k = xs_bits.reshape(n, 1, 1).astype(np.uint16)
    kc = np.zeros((n, 1, 1, 1), np.uint8)
    vc = np.zeros_like(kc)
    o.cache_append(k, k, np.arange(n, dtype=np.int32), kc, vc, 1, 1, scale)
    assert np.array_equal(kc, vc)
    return kc.reshape(n)


def pin_kv_formula(o):
    with open(os.path.join(GOLDEN, "kv_bytes_per_token.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        b = o.kv_bytes_per_token(c["num_layers"], c["num_kv_heads"], c["head_dim"], c["bytes_per_elem"])
        assert b == c["bytes_per_token"], b
        assert b // 1024 == c["kib_per_token"]
        assert b * c["context_tokens"] == c["bytes_per_sequence"]
        assert b * c["context_tokens"] == c["gib_per_sequence"] * 2**30


def pin_e4m3_decode(o):
    codes = np.arange(256)
    ref = _e4m3_torch(codes)
    got = np.array([o.e4m3_to_double(c) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert sorted(np.flatnonzero(nan).tolist()) == [0x7F, 0xFF]
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0**-9


def pin_e4m3_encode(o, exhaustive=True):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    if not exhaustive:
        allbits = allbits[::17]
    x = bits_to_f64(allbits).astype(np.float32)
    for scale in (1.0, float(np.float32(4.5) / np.float32(448.0)), 0.37):
        got = _encode_many(o, allbits, scale)
        with np.errstate(invalid="ignore", over="ignore"):
            y = x / np.float32(scale)
        isnan = np.isnan(y)
        assert np.all((got[isnan] & 0x7F) == 0x7F)
        big = ~isnan & (np.abs(y) > 448.0)
        want_big = np.where(np.signbit(y[big]), 0xFE, 0x7E)
        assert np.array_equal(got[big], want_big)
        fine = ~isnan & ~big
        want = torch.from_numpy(y[fine]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(got[fine], want), np.flatnonzero(got[fine] != want)[:8]


def pin_e4m3_roundtrip(o):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        assert o.e4m3_from_float(o.e4m3_to_double(c)) == c, c


def _case(ctx=(1, 5, 16, 17, 40), Hq=8, Hkv=2, D=16, seed=3, **kw):
    return LogicalCase(ctx, Hq, Hkv, D, seed, **kw)


def pin_attention_sdpa(o):
    rng = np.random.default_rng(7)
    for B, (Hq, Hkv) in ((16, (8, 2)), (4, (6, 3)), (32, (4, 4)), (8, (16, 1))):
        c = _case(Hq=Hq, Hkv=Hkv, seed=B + Hq)
        tables, kc, vc = c.paged(B, 40, rng)
        out = o.decode(c.q, kc, vc, tables, np.array(c.ctx), Hkv, B, 0.3)
        ref = c.sdpa(0.3)
        assert np.isfinite(out).all()
        assert np.abs(out - ref).max() < 1e-12, np.abs(out - ref).max()


def pin_attention_fp8(o):
    rng = np.random.default_rng(8)
    c = _case(seed=11)
    tables, _, _ = c.paged(16, 30, rng)
    scale = 0.02
    codes_k = [np.array([[[_byte(o, x, scale) for x in row] for row in h] for h in k]) for k in c.k]
    codes_v = [np.array([[[_byte(o, x, scale) for x in row] for row in h] for h in v]) for v in c.v]
    kc = np.full((30, c.Hkv, 16, c.D), 0x7F, np.uint8)
    vc = np.full_like(kc, 0x7F)
    for s, n in enumerate(c.ctx):
        for t in range(n):
            kc[tables[s, t // 16], :, t % 16, :] = codes_k[s][:, t, :]
            vc[tables[s, t // 16], :, t % 16, :] = codes_v[s][:, t, :]
    out = o.decode(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, 16, 0.25, kv_dtype=1, kv_scale=scale)
    c.k, c.v = codes_k, codes_v
    ref = c.sdpa(0.25, deq_k=lambda a: _e4m3_torch(a) * scale, deq_v=lambda a: _e4m3_torch(a) * scale)
    assert np.abs(out - ref).max() < 1e-12, np.abs(out - ref).max()


def _byte(o, bits, scale):
    x = np.float32(bits_to_f64(np.array([bits], np.uint16))[0])
    return o.e4m3_from_float(x / np.float32(scale))


def pin_extreme_scores(o):
    rng = np.random.default_rng(9)
    c = _case(ctx=(30, 64), seed=5)
    tables, kc, vc = c.paged(16, 12, rng)
    out = o.decode(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, 16, 400.0)
    ref = c.sdpa(400.0)
    assert np.isfinite(out).all()
    assert np.abs(out - ref).max() < 1e-9


def pin_permutation(o):
    c = _case(seed=13)
    outs = []
    for seed in (1, 2, 3):
        tables, kc, vc = c.paged(16, 50, np.random.default_rng(seed))
        outs.append(o.decode(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, 16, 0.2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def pin_prefix_sharing(o):
    def same_prefix(ks):
        ks = [k.copy() for k in ks]
        for k in ks[1:]:
            k[:, :32, :] = ks[0][:, :32, :]
        return ks
    c = _case(ctx=(40, 33, 64), seed=17)
    c.k = same_prefix(c.k)
    c.v = same_prefix(c.v)
    t_sh, k_sh, v_sh = c.paged(16, 20, np.random.default_rng(4), share_prefix_tokens=32)
    t_pr, k_pr, v_pr = c.paged(16, 20, np.random.default_rng(5))
    assert t_sh[0, 0] == t_sh[1, 0] == t_sh[2, 0]
    a = o.decode(c.q, k_sh, v_sh, t_sh, np.array(c.ctx), c.Hkv, 16, 0.2)
    b = o.decode(c.q, k_pr, v_pr, t_pr, np.array(c.ctx), c.Hkv, 16, 0.2)
    assert np.array_equal(a, b)


def pin_context_one(o):
    c = _case(ctx=(1, 1, 1), seed=19)
    tables, kc, vc = c.paged(16, 8, np.random.default_rng(6))
    out = o.decode(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, 16, 0.7)
    G = c.Hq // c.Hkv
    for s in range(3):
        for hq in range(c.Hq):
            assert np.array_equal(out[s, hq], bits_to_f64(c.v[s][hq // G, 0]))


def pin_identical_keys(o):
    def same_keys(ks):
        return [np.repeat(k[:, :1, :], k.shape[1], axis=1) for k in ks]
    c = _case(ctx=(7, 33), seed=23, k_override=same_keys)
    tables, kc, vc = c.paged(16, 10, np.random.default_rng(7))
    out = o.decode(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, 16, 0.9)
    G = c.Hq // c.Hkv
    for s, n in enumerate(c.ctx):
        for hq in range(c.Hq):
            mean = bits_to_f64(c.v[s][hq // G]).mean(axis=0)
            assert np.abs(out[s, hq] - mean).max() < 1e-12


def pin_empty_context(o):
    c = _case(ctx=(0, 3), seed=29)
    tables, kc, vc = c.paged(16, 4, np.random.default_rng(8))
    out = o.decode(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, 16, 0.5)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.isfinite(out[1]).all()


def pin_slot_mapping(o):
    rng = np.random.default_rng(10)
    for B in (1, 4, 16, 32):
        ctx = np.array([0, 1, B, B + 1, 3 * B - 1, 100], np.int32)
        mb = int(max((c + B - 1) // B for c in ctx))
        tables = np.full((len(ctx), mb), -1, np.int32)
        pool = list(rng.permutation(1000))
        for s, c in enumerate(ctx):
            for j in range((c + B - 1) // B):
                tables[s, j] = pool.pop()
        got = o.slot_mapping(tables, ctx, B)
        for s, c in enumerate(ctx):
            slots = [int(b) * B + off for b in tables[s] if b >= 0 for off in range(B)][:c]
            assert got[s] == (slots[-1] if c > 0 else -1), (B, s)


def pin_append_readback(o):
    rng = np.random.default_rng(11)
    B, Hkv, D, NB = 16, 2, 8, 12
    for kv_dtype in (0, 1):
        ctx = np.array([5, 16, 17, 1], np.int32)
        tables = np.full((4, 2), -1, np.int32)
        pool = list(rng.permutation(NB))
        for s, c in enumerate(ctx):
            for j in range((c + B - 1) // B):
                tables[s, j] = pool.pop()
        slots = np.array([tables[s, (c - 1) // B] * B + (c - 1) % B for s, c in enumerate(ctx)], np.int32)
        slots[3] = -1
        g = torch.Generator().manual_seed(kv_dtype)
        k = torch.randn(4, Hkv, D, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        v = torch.randn(4, Hkv, D, generator=g).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        dt = np.uint16 if kv_dtype == 0 else np.uint8
        fill = 0x7FC0 if kv_dtype == 0 else 0x7F
        kc = np.full((NB, Hkv, B, D), fill, dt)
        vc = np.full_like(kc, fill)
        before_k = kc.copy()
        o.cache_append(k, v, slots, kc, vc, B, kv_dtype, 0.01)
        changed = np.argwhere((kc != before_k).any(axis=(1, 3)))
        assert len(changed) == 3
        for s in range(3):
            b, off = divmod(int(slots[s]), B)
            if kv_dtype == 0:
                assert np.array_equal(kc[b, :, off, :], k[s]) and np.array_equal(vc[b, :, off, :], v[s])
            else:
                kd = _e4m3_torch(kc[b, :, off, :]) * 0.01
                assert np.abs(kd - bits_to_f64(k[s])).max() <= 0.01 * 16  # within half a step at 448
                for h in range(Hkv):
                    for d in range(D):
                        assert kc[b, h, off, d] == _byte(o, k[s, h, d], 0.01)


def pin_partition_merge(o):
    rng = np.random.default_rng(12)
    c = _case(ctx=(1, 16, 17, 70, 0), seed=31)
    tables, kc, vc = c.paged(16, 30, rng)
    ctx = np.array(c.ctx)
    full = o.decode(c.q, kc, vc, tables, ctx, c.Hkv, 16, 0.4)
    for P in (16, 32, 48, 128):
        n = int(np.ceil(ctx.max() / P))
        po, pm, pl = o.decode_partitions(c.q, kc, vc, tables, ctx, c.Hkv, 16, 0.4, P, n)
        merged = o.merge_partitions(po.astype(np.float32), pm.astype(np.float32),
                                    pl.astype(np.float32), ctx, P)
        assert np.abs(merged - full).max() < 1e-6, (P, np.abs(merged - full).max())
        if P >= ctx.max():
            assert np.array_equal(po[:, :, 0, :], full)


def pin_fp8_per_head_scales(o):
    """E4M3 cache with a different scale per KV head and for K vs V: the
    oracle's attention equals torch SDPA over values decoded by torch's
    float8_e4m3fn and multiplied by each head's own scale; the appended codes
    are the per-head encodings, and equal scales reduce to the one-scale
    append."""
    rng = np.random.default_rng(14)
    c = _case(Hq=12, Hkv=3, seed=41)
    B = 16
    tables, _, _ = c.paged(B, 30, rng)
    ks = np.array([0.011, 0.023, 0.007], np.float32)
    vs = np.array([0.019, 0.005, 0.031], np.float32)
    kc = np.full((30, c.Hkv, B, c.D), 0x7F, np.uint8)
    vc = np.full_like(kc, 0x7F)
    for s_, n in enumerate(c.ctx):
        slots = np.array([tables[s_, t // B] * B + t % B for t in range(n)], np.int32)
        o.cache_append_scaled(c.k[s_].transpose(1, 0, 2), c.v[s_].transpose(1, 0, 2), slots,
                              kc, vc, B, ks, vs)
    codes_k, codes_v = [], []
    for s_, n in enumerate(c.ctx):
        ck = np.zeros((c.Hkv, n, c.D), np.uint8)
        cv = np.zeros_like(ck)
        for t in range(n):
            ck[:, t] = kc[tables[s_, t // B], :, t % B]
            cv[:, t] = vc[tables[s_, t // B], :, t % B]
        for h in range(c.Hkv):
            for d in (0, 5, c.D - 1):
                assert ck[h, 0, d] == _byte(o, c.k[s_][h, 0, d], ks[h])
                assert cv[h, 0, d] == _byte(o, c.v[s_][h, 0, d], vs[h])
        codes_k.append(ck)
        codes_v.append(cv)
    out = o.decode_scaled(c.q, kc, vc, tables, np.array(c.ctx), c.Hkv, B, 0.21, ks, vs)
    c.k, c.v = codes_k, codes_v
    ref = c.sdpa(0.21, deq_k=lambda a: _e4m3_torch(a) * ks[:, None, None].astype(np.float64),
                 deq_v=lambda a: _e4m3_torch(a) * vs[:, None, None].astype(np.float64))
    assert np.abs(out - ref).max() < 1e-12, np.abs(out - ref).max()
    # one scale everywhere: the per-head functions agree with the one-scale ones
    same = np.full(c.Hkv, 0.013, np.float32)
    k1 = np.zeros((8, c.Hkv, B, c.D), np.uint8)
    v1, k2, v2 = k1.copy(), k1.copy(), k1.copy()
    kb = (np.arange(3 * c.Hkv * c.D, dtype=np.uint32) * 2654435761 % 65535).astype(np.uint16)
    kb = kb.reshape(3, c.Hkv, c.D) & 0x7FFF  # finite patterns only
    sl = np.array([1, 17, 40], np.int32)
    o.cache_append_scaled(kb, kb, sl, k1, v1, B, same, same)
    o.cache_append(kb, kb, sl, k2, v2, B, 1, float(same[0]))
    assert np.array_equal(k1, k2) and np.array_equal(v1, v2)



def pin_prefill_scaled(o):
    """Chunked prefill over an E4M3 cache with a scale per KV head for K and
    for V: every chunk's last row equals the per-head-scaled decode (pinned
    against torch) bit for bit; with one scale everywhere it equals the
    one-scale prefill bit for bit."""
    rng = np.random.default_rng(16)
    c = _case(Hq=12, Hkv=3, seed=42)
    B = 16
    tables, _, _ = c.paged(B, 30, rng)
    ks = np.array([0.011, 0.023, 0.007], np.float32)
    vs = np.array([0.019, 0.005, 0.031], np.float32)
    kc = np.full((30, c.Hkv, B, c.D), 0x7F, np.uint8)
    vc = np.full_like(kc, 0x7F)
    for s_, n in enumerate(c.ctx):
        slots = np.array([tables[s_, t // B] * B + t % B for t in range(n)], np.int32)
        o.cache_append_scaled(c.k[s_].transpose(1, 0, 2), c.v[s_].transpose(1, 0, 2), slots, kc, vc, B, ks, vs)
    ctx = np.array(c.ctx, np.int32)
    chunk = np.minimum(ctx, np.array([3, 1, 7, 2, 5, 4, 6, 8][:len(ctx)], np.int32))
    qs = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    g = torch.Generator().manual_seed(5)
    q = torch.randn(int(qs[-1]), c.Hq, c.D, generator=g).to(torch.bfloat16)
    qb = q.view(torch.int16).numpy().view(np.uint16)
    out = o.prefill_scaled(qb, kc, vc, tables, ctx, qs, c.Hkv, B, 0.21, ks, vs)
    live = np.flatnonzero(chunk > 0)
    last = qs[1:][live] - 1
    dec = o.decode_scaled(qb[last], kc, vc, tables[live], ctx[live], c.Hkv, B, 0.21, ks, vs)
    assert np.array_equal(out[last], dec)
    same = np.full(c.Hkv, 0.013, np.float32)
    one = o.prefill(qb, kc, vc, tables, ctx, qs, c.Hkv, B, 0.21, kv_dtype=1, kv_scale=float(same[0]))
    assert np.array_equal(o.prefill_scaled(qb, kc, vc, tables, ctx, qs, c.Hkv, B, 0.21, same, same), one)

def pin_block_alloc(o):
    """Allocation for the newest tokens: checked against invariants that any
    correct allocator with these rules keeps (conservation of blocks,
    reference counts equal to the references in the tables, exclusive
    ownership of every block about to be written, untouched sole owners,
    unchanged logical contents, fresh blocks from the top of the stack in
    sequence order, all-or-nothing when the stack is short)."""
    from alloc_cases import gather_rows, make_state
    for seed in (1, 2, 3):
        st = make_state(seed)
        B, NB = st["B"], st["NB"]
        t0, r0, f0 = st["tables"].copy(), st["refc"].copy(), st["free"].copy()
        k0, v0 = st["k"].copy(), st["v"].copy()
        tables, refc, free = st["tables"], st["refc"], np.concatenate([st["free"], np.zeros(NB, np.int32)])
        status, fc, cow = o.block_alloc(tables, st["ctx"], B, free, st["free_count"], refc,
                                        st["k"], st["v"])
        assert status == 0
        ctx = st["ctx"]
        S = len(ctx)
        # reference counts equal the references in the tables
        recount = np.zeros(NB, np.int32)
        for s_ in range(S):
            for j in range((ctx[s_] + B - 1) // B):
                assert 0 <= tables[s_, j] < NB
                recount[tables[s_, j]] += 1
        assert np.array_equal(recount, refc)
        # conservation: every block is either free or referenced, never both
        free_now = free[:fc]
        assert len(set(free_now.tolist())) == fc
        assert not (set(free_now.tolist()) & set(np.flatnonzero(recount).tolist()))
        assert fc + np.count_nonzero(recount) == NB
        need = 0
        for s_ in range(S):
            n = int(ctx[s_])
            if n <= 0:
                assert np.array_equal(tables[s_], t0[s_])
                continue
            pos, j = n - 1, (n - 1) // B
            # only entry j may change
            mask = np.ones(tables.shape[1], bool)
            mask[j] = False
            assert np.array_equal(tables[s_][mask], t0[s_][mask])
            assert refc[tables[s_, j]] == 1  # exclusive before the write
            shared_before = pos % B != 0 and r0[t0[s_, j]] > 1
            if pos % B != 0 and not shared_before:
                assert tables[s_, j] == t0[s_, j] and cow[s_] == -1  # sole owner: in place
            if pos % B == 0 or shared_before:
                assert tables[s_, j] == f0[st["free_count"] - 1 - need]  # stack top, in order
                need += 1
            assert cow[s_] == (t0[s_, j] if shared_before else -1)
            # the logical rows before the new token are unchanged
            for old, new in ((k0, st["k"]), (v0, st["v"])):
                a = gather_rows(t0, pos, s_, old, B)
                b = gather_rows(tables, pos, s_, new, B)
                assert (a is None and b is None) or np.array_equal(a, b)
        assert fc == st["free_count"] - need + len(set(int(c) for c in cow if c >= 0 and refc[c] == 0))
    # a short stack changes nothing
    st = make_state(4, extra_free=2)
    t0, r0 = st["tables"].copy(), st["refc"].copy()
    free = st["free"].copy()
    status, fc, cow = o.block_alloc(st["tables"], st["ctx"], st["B"], free, st["free_count"],
                                    st["refc"], st["k"], st["v"])
    assert status == 1 and fc == st["free_count"]
    assert np.array_equal(st["tables"], t0) and np.array_equal(st["refc"], r0)



def pin_block_alloc_chunk(o):
    """Allocation for a chunk of new tokens per sequence.  (1) One-token
    chunks give exactly what the single-token allocator gives.  (2) Any
    chunks keep the allocator's invariants: blocks conserved, reference
    counts equal to the references in the tables, every block the chunk
    writes owned by the sequence alone, earlier entries and logical rows
    unchanged, fresh blocks from the top of the stack in sequence order
    (a sequence's copy first).  (3) A chunk allocated at once and then
    written holds the same logical rows as its tokens allocated and written
    one at a time.  (4) A short stack changes nothing."""
    from alloc_cases import gather_rows, make_chunk_state, make_state
    # (1) one-token chunks
    for seed in (1, 2, 3):
        a, b = make_state(seed), make_state(seed)
        fa = np.concatenate([a["free"], np.zeros(a["NB"], np.int32)])
        fb = fa.copy()
        c = (b["ctx"] > 0).astype(np.int32)
        qs = np.concatenate([[0], np.cumsum(c)]).astype(np.int32)
        ra = o.block_alloc(a["tables"], a["ctx"], a["B"], fa, a["free_count"], a["refc"], a["k"], a["v"])
        rb = o.block_alloc_chunk(b["tables"], b["ctx"], qs, b["B"], fb, b["free_count"], b["refc"], b["k"], b["v"])
        assert ra[0] == rb[0] == 0 and ra[1] == rb[1] and np.array_equal(ra[2], rb[2])
        for x, y in ((a["tables"], b["tables"]), (fa, fb), (a["refc"], b["refc"]), (a["k"], b["k"]), (a["v"], b["v"])):
            assert np.array_equal(x, y)
    # (2) invariants, chunks crossing block boundaries from shared and private blocks
    for seed, chunks in ((1, [2, 7, 1, 4]), (2, [3, 9, 4, 13]), (3, [1, 5, 8, 12])):
        st = make_chunk_state(seed, chunks)
        B, NB = st["B"], st["NB"]
        t0, r0, f0 = st["tables"].copy(), st["refc"].copy(), st["free"].copy()
        k0, v0 = st["k"].copy(), st["v"].copy()
        tables, refc = st["tables"], st["refc"]
        free = np.concatenate([st["free"], np.zeros(NB, np.int32)])
        status, fc, cow = o.block_alloc_chunk(tables, st["ctx"], st["qs"], B, free, st["free_count"], refc,
                                              st["k"], st["v"])
        assert status == 0
        ctx, pre, S = st["ctx"], st["pre"], len(st["ctx"])
        recount = np.zeros(NB, np.int32)
        for s_ in range(S):
            for j in range((int(ctx[s_]) + B - 1) // B):
                assert 0 <= tables[s_, j] < NB
                recount[tables[s_, j]] += 1
        assert np.array_equal(recount, refc)
        free_now = free[:fc]
        assert len(set(free_now.tolist())) == fc
        assert not (set(free_now.tolist()) & set(np.flatnonzero(recount).tolist()))
        assert fc + np.count_nonzero(recount) == NB
        taken = 0
        for s_ in range(S):
            n, old = int(ctx[s_]), int(pre[s_])
            if n == old:
                assert np.array_equal(tables[s_], t0[s_]) and cow[s_] == -1
                continue
            j0, jl = old // B, (n - 1) // B
            shared = old % B != 0 and r0[t0[s_, j0]] > 1
            assert np.array_equal(tables[s_, :j0], t0[s_, :j0])      # earlier entries unchanged
            for j in range(j0 if old % B else old // B, jl + 1):
                assert refc[tables[s_, j]] == 1                      # written blocks owned alone
            if old % B != 0 and not shared:
                assert tables[s_, j0] == t0[s_, j0]                  # sole owner: in place
            assert cow[s_] == (t0[s_, j0] if shared else -1)
            first = j0 if (old % B == 0 or shared) else j0 + 1
            for j in range(first, jl + 1):
                assert tables[s_, j] == f0[st["free_count"] - 1 - taken]  # stack top, in order
                taken += 1
            for c0, c1 in ((k0, st["k"]), (v0, st["v"])):
                a_ = gather_rows(t0, old, s_, c0, B)
                b_ = gather_rows(tables, old, s_, c1, B)
                assert (a_ is None and b_ is None) or np.array_equal(a_, b_)
        assert fc == st["free_count"] - taken + len(set(int(c) for c in cow if c >= 0 and refc[c] == 0))
    # (3) at once vs token by token: the same logical rows once the chunk is written
    for seed, chunks in ((4, [3, 6, 9]), (5, [1, 4, 10, 2])):
        a, b = make_chunk_state(seed, chunks), make_chunk_state(seed, chunks)
        B = a["B"]
        rows = np.random.default_rng(seed + 7).integers(0, 2**15, size=(len(a["ctx"]), 64) + a["k"].shape[1:2]
                                                        + a["k"].shape[3:]).astype(a["k"].dtype)
        fa = np.concatenate([a["free"], np.zeros(a["NB"], np.int32)])
        st_, fca, _ = o.block_alloc_chunk(a["tables"], a["ctx"], a["qs"], B, fa, a["free_count"], a["refc"],
                                          a["k"], a["v"])
        assert st_ == 0
        for s_ in range(len(a["ctx"])):
            for t in range(int(a["pre"][s_]), int(a["ctx"][s_])):
                blk = a["tables"][s_, t // B]
                a["k"][blk, :, t % B] = rows[s_, t - a["pre"][s_]]
                a["v"][blk, :, t % B] = rows[s_, t - a["pre"][s_]] ^ 1
        fb = np.concatenate([b["free"], np.zeros(b["NB"], np.int32)])
        fcb = b["free_count"]
        cur = b["pre"].copy()
        for _ in range(int((b["ctx"] - b["pre"]).max())):
            grow = (cur < b["ctx"]).astype(np.int32)
            n1 = (cur + grow).astype(np.int32)
            qs1 = np.concatenate([[0], np.cumsum(grow)]).astype(np.int32)
            st1, fcb, _ = o.block_alloc_chunk(b["tables"], n1, qs1, B, fb, fcb, b["refc"], b["k"], b["v"])
            assert st1 == 0
            for s_ in np.flatnonzero(grow):
                t = int(cur[s_])
                blk = b["tables"][s_, t // B]
                b["k"][blk, :, t % B] = rows[s_, t - b["pre"][s_]]
                b["v"][blk, :, t % B] = rows[s_, t - b["pre"][s_]] ^ 1
            cur = n1
        assert fca == fcb
        for s_ in range(len(a["ctx"])):
            n = int(a["ctx"][s_])
            for x, y in ((a["k"], b["k"]), (a["v"], b["v"])):
                ga, gb = gather_rows(a["tables"], n, s_, x, B), gather_rows(b["tables"], n, s_, y, B)
                assert (ga is None and gb is None) or np.array_equal(ga, gb)
    # (4) a short stack changes nothing
    st = make_chunk_state(6, [5, 9])
    st["free"] = st["free"][:3]
    t0, r0, f0 = st["tables"].copy(), st["refc"].copy(), st["free"].copy()
    status, fc, cow = o.block_alloc_chunk(st["tables"], st["ctx"], st["qs"], st["B"], st["free"], 3, st["refc"],
                                          st["k"], st["v"])
    assert status == 1 and fc == 3 and np.all(cow == -1)
    assert np.array_equal(st["tables"], t0) and np.array_equal(st["refc"], r0) and np.array_equal(st["free"], f0)

def pin_prefill(o):
    """Chunked prefill: a chunk covering the whole sequence is causal
    attention (torch SDPA, is_causal); a chunk after a cached prefix is SDPA
    with the mask 'key position <= query position'; the last token of every
    chunk equals decode attention; chunk slots equal brute-force enumeration
    and their last entry equals the newest-token slot."""
    import torch.nn.functional as F
    rng = np.random.default_rng(15)
    for B, (Hq, Hkv) in ((16, (8, 2)), (4, (6, 3))):
        ctx = [5, 40, 33, 17]
        chunk = [5, 7, 1, 17]  # whole, after prefix, single token, whole (17 > B)
        c = LogicalCase(ctx, Hq, Hkv, 16, seed=B + Hq)
        tables, kc, vc = c.paged(B, 40, rng)
        qs = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
        g = torch.Generator().manual_seed(3)
        q = torch.randn(int(qs[-1]), Hq, 16, generator=g).to(torch.bfloat16)
        qb = q.view(torch.int16).numpy().view(np.uint16)
        out = o.prefill(qb, kc, vc, tables, np.array(ctx), qs, Hkv, B, 0.3)
        G = Hq // Hkv
        for s_, (n, ch) in enumerate(zip(ctx, chunk)):
            rows = slice(qs[s_], qs[s_ + 1])
            qq = torch.from_numpy(bits_to_f64(qb[rows])).permute(1, 0, 2)[None]   # [1, Hq, ch, D]
            k = torch.from_numpy(bits_to_f64(c.k[s_])).repeat_interleave(G, 0)[None]
            v = torch.from_numpy(bits_to_f64(c.v[s_])).repeat_interleave(G, 0)[None]
            qpos = torch.arange(n - ch, n)[:, None]
            mask = torch.arange(n)[None, :] <= qpos
            ref = F.scaled_dot_product_attention(qq, k, v, attn_mask=mask, scale=0.3)
            if ch == n:
                causal = F.scaled_dot_product_attention(qq, k, v, is_causal=True, scale=0.3)
                assert torch.allclose(ref, causal, atol=1e-12)
            got = out[rows].transpose(1, 0, 2)[None]
            assert np.abs(got - ref.numpy()).max() < 1e-12
        # the last chunk token is the decode token
        last = qs[1:] - 1
        dec = o.decode(qb[last], kc, vc, tables, np.array(ctx), Hkv, B, 0.3)
        assert np.array_equal(out[last], dec)
        # slots
        slots = o.chunk_slot_mapping(tables, np.array(ctx), qs, B)
        for s_, (n, ch) in enumerate(zip(ctx, chunk)):
            allslots = [int(b) * B + off for b in tables[s_] if b >= 0 for off in range(B)][:n]
            assert slots[qs[s_]:qs[s_ + 1]].tolist() == allslots[n - ch:]
        assert np.array_equal(slots[last], o.slot_mapping(tables, np.array(ctx), B))


def pin_fp8_qk(o):
    """E4M3 x E4M3 scores: the oracle equals torch SDPA over a query rounded
    by torch's float8_e4m3fn (x / q_scale, read back times q_scale) and an
    E4M3 cache decoded with each head's scales; a query already on the E4M3
    grid with q_scale 1 gives the per-head-scaled decode unchanged; a query
    element past the E4M3 range counts as +-448 q_scale."""
    rng = np.random.default_rng(16)
    c = _case(Hq=12, Hkv=3, seed=43)
    B = 16
    tables, _, _ = c.paged(B, 30, rng)
    ks = np.array([0.012, 0.021, 0.009], np.float32)
    vs = np.array([0.017, 0.006, 0.029], np.float32)
    kc = np.full((30, c.Hkv, B, c.D), 0x7F, np.uint8)
    vc = np.full_like(kc, 0x7F)
    for s_, n in enumerate(c.ctx):
        slots = np.array([tables[s_, t // B] * B + t % B for t in range(n)], np.int32)
        o.cache_append_scaled(c.k[s_].transpose(1, 0, 2), c.v[s_].transpose(1, 0, 2), slots,
                              kc, vc, B, ks, vs)
    ctx = np.array(c.ctx)
    qs = 0.0173  # N(0,1) queries stay far inside +-448 qs
    out = o.decode_fp8_qk(c.q, kc, vc, tables, ctx, c.Hkv, B, 0.21, qs, ks, vs)
    codes_k, codes_v = [], []
    for s_, n in enumerate(c.ctx):
        ck = np.zeros((c.Hkv, n, c.D), np.uint8)
        cv = np.zeros_like(ck)
        for t in range(n):
            ck[:, t] = kc[tables[s_, t // B], :, t % B]
            cv[:, t] = vc[tables[s_, t // B], :, t % B]
        codes_k.append(ck)
        codes_v.append(cv)
    plain = o.decode_scaled(c.q, kc, vc, tables, ctx, c.Hkv, B, 0.21, ks, vs)

    def round_q(bits):
        x = torch.from_numpy(bits_to_f64(bits).astype(np.float32) / np.float32(qs))
        return x.to(torch.float8_e4m3fn).to(torch.float64).numpy() * np.float64(np.float32(qs))

    logical = LogicalCase(c.ctx, c.Hq, c.Hkv, c.D, 43)
    logical.k, logical.v = codes_k, codes_v
    ref = logical.sdpa(0.21, deq_q=round_q,
                       deq_k=lambda a: _e4m3_torch(a) * ks[:, None, None].astype(np.float64),
                       deq_v=lambda a: _e4m3_torch(a) * vs[:, None, None].astype(np.float64))
    assert np.abs(out - ref).max() < 1e-12, np.abs(out - ref).max()
    assert np.abs(out - plain).max() > 1e-6  # the rounding of the query is visible
    # a query already on the E4M3 grid, q_scale 1: nothing changes
    grid = _e4m3_torch(rng.integers(0, 0x7F, size=c.q.shape).astype(np.uint8))
    grid *= np.where(rng.random(c.q.shape) < 0.5, -1.0, 1.0)
    qg = (torch.from_numpy(grid).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    a1 = o.decode_fp8_qk(qg, kc, vc, tables, ctx, c.Hkv, B, 0.21, 1.0, ks, vs)
    a2 = o.decode_scaled(qg, kc, vc, tables, ctx, c.Hkv, B, 0.21, ks, vs)
    assert np.array_equal(a1, a2)
    # saturation: 1000 becomes 448 (q_scale 1)
    big, sat = qg.copy(), qg.copy()
    big[:, :, 3] = 0x447A  # bf16 1000.0
    sat[:, :, 3] = 0x43E0  # bf16 448.0
    b1 = o.decode_fp8_qk(big, kc, vc, tables, ctx, c.Hkv, B, 0.21, 1.0, ks, vs)
    b2 = o.decode_scaled(sat, kc, vc, tables, ctx, c.Hkv, B, 0.21, ks, vs)
    assert np.array_equal(b1, b2)



def _pairs_for(S, Hq, rng):
    """Every (sequence, query head) pair in shuffled order, then a sampled
    run with repeats."""
    every = np.array([(s_, h) for s_ in range(S) for h in range(Hq)], np.int32)
    every = every[rng.permutation(len(every))]
    sampled = np.stack([rng.integers(0, S, 3 * S), rng.integers(0, Hq, 3 * S)], 1).astype(np.int32)
    return every, sampled


def pin_decode_pairs(o):
    """Decode attention for listed (sequence, query head) pairs -- the oracle
    of every sampled full-size comparison -- row for row against torch SDPA
    over the logical K/V (bf16 and E4M3 caches; groups 1, 4 and 16; page
    sizes 16 and 32; contexts 0 and 1 among them), and bit for bit against
    the whole-batch decode.  The per-head-scaled and E4M3-query variants'
    pair lists equal their whole-batch results row for row."""
    rng = np.random.default_rng(18)
    ctx = (0, 1, 5, 16, 17, 40)
    for B, (Hq, Hkv) in ((16, (8, 8)), (32, (8, 2)), (16, (16, 1))):
        c = _case(ctx=ctx, Hq=Hq, Hkv=Hkv, seed=B + 3 * Hq + Hkv)
        tables, kc, vc = c.paged(B, 24, rng)
        cl = np.array(c.ctx)
        G = Hq // Hkv
        ref = c.sdpa(0.3)
        full = o.decode(c.q, kc, vc, tables, cl, Hkv, B, 0.3)
        for pairs in _pairs_for(len(ctx), Hq, rng):
            got = o.decode_pairs(c.q, kc, vc, tables, cl, Hkv, B, 0.3, pairs)
            want = ref[pairs[:, 0], pairs[:, 1]]
            assert got.shape == want.shape
            assert np.abs(got - want).max() < 1e-12, np.abs(got - want).max()
            assert np.array_equal(got, full[pairs[:, 0], pairs[:, 1]])
            empty = cl[pairs[:, 0]] == 0
            assert np.array_equal(got[empty], np.zeros_like(got[empty]))
            one = cl[pairs[:, 0]] == 1
            for (s_, h), row in zip(pairs[one], got[one]):
                assert np.array_equal(row, bits_to_f64(c.v[s_][h // G, 0]))
        # E4M3 cache with one scale: decoded by torch's float8_e4m3fn
        scale = 0.021
        kq = np.full(kc.shape, 0x7F, np.uint8)
        vq = np.full_like(kq, 0x7F)
        codes_k, codes_v = [], []
        for s_, n in enumerate(c.ctx):
            ck = np.array([[[_byte(o, x, scale) for x in row] for row in h] for h in c.k[s_]],
                          np.uint8).reshape(Hkv, n, c.D)
            cv = np.array([[[_byte(o, x, scale) for x in row] for row in h] for h in c.v[s_]],
                          np.uint8).reshape(Hkv, n, c.D)
            for t in range(n):
                kq[tables[s_, t // B], :, t % B, :] = ck[:, t, :]
                vq[tables[s_, t // B], :, t % B, :] = cv[:, t, :]
            codes_k.append(ck)
            codes_v.append(cv)
        logical = LogicalCase(c.ctx, Hq, Hkv, c.D, B + 3 * Hq + Hkv)
        logical.k, logical.v = codes_k, codes_v
        ref8 = logical.sdpa(0.3, deq_k=lambda a: _e4m3_torch(a) * scale,
                            deq_v=lambda a: _e4m3_torch(a) * scale)
        every, sampled = _pairs_for(len(ctx), Hq, rng)
        for pairs in (every, sampled):
            got = o.decode_pairs(c.q, kq, vq, tables, cl, Hkv, B, 0.3, pairs, kv_dtype=1,
                                 kv_scale=scale)
            assert np.abs(got - ref8[pairs[:, 0], pairs[:, 1]]).max() < 1e-12
        # per-head scales and the E4M3 query: pair lists against whole batches
        ks = np.linspace(0.01, 0.03, Hkv).astype(np.float32)
        vs = np.linspace(0.02, 0.005, Hkv).astype(np.float32)
        whole = o.decode_scaled(c.q, kq, vq, tables, cl, Hkv, B, 0.3, ks, vs)
        whole_qk = o.decode_fp8_qk(c.q, kq, vq, tables, cl, Hkv, B, 0.3, 0.013, ks, vs)
        for pairs in (every, sampled):
            got = o.decode_scaled(c.q, kq, vq, tables, cl, Hkv, B, 0.3, ks, vs, pairs=pairs)
            assert np.array_equal(got, whole[pairs[:, 0], pairs[:, 1]])
            got = o.decode_fp8_qk(c.q, kq, vq, tables, cl, Hkv, B, 0.3, 0.013, ks, vs, pairs=pairs)
            assert np.array_equal(got, whole_qk[pairs[:, 0], pairs[:, 1]])


ALL = [pin_kv_formula, pin_e4m3_decode, pin_e4m3_encode, pin_e4m3_roundtrip, pin_attention_sdpa,
       pin_attention_fp8, pin_extreme_scores, pin_permutation, pin_prefix_sharing, pin_context_one,
       pin_identical_keys, pin_empty_context, pin_slot_mapping, pin_append_readback,
       pin_partition_merge, pin_fp8_per_head_scales, pin_prefill_scaled, pin_block_alloc, pin_block_alloc_chunk,
       pin_prefill,
       pin_fp8_qk,
       pin_decode_pairs]
