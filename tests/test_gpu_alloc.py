"""Device-side block allocation with copy-on-write: bit for bit against the
oracle (tables, free stack, counts, reference counts, copied rows), the
all-or-nothing refusal, and a device-driven decode loop (allocate with
advance, then the fused step) against the oracle step by step; the same for
a chunk of new tokens per sequence, and a device-driven chunked prefill."""
import numpy as np
import pytest
import torch

from alloc_cases import make_chunk_state, make_state
from gpu_helpers import compare
from paged_kv_cache_193_gb300 import _lib
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _run_both(api, oracle, dev, st, advance=False):
    B, NB = st["B"], st["NB"]
    ctx_dev = st["ctx"] - (st["ctx"] > 0) if advance else st["ctx"]
    pool = api.DeviceBlockPool(st["free"], st["refc"], dev)
    bt = torch.from_numpy(st["tables"].copy()).to(dev)
    cl = torch.from_numpy(ctx_dev.astype(np.int32)).to(dev)
    kc = W.from_bits(st["k"], dev)
    vc = W.from_bits(st["v"], dev)
    cow = pool.allocate(bt, cl, kc, vc, advance=advance)
    torch.cuda.synchronize()
    # oracle on host copies (its context lengths already include the token)
    tables, refc = st["tables"].copy(), st["refc"].copy()
    free = np.concatenate([st["free"], np.zeros(NB, np.int32)])[:NB].copy()
    k, v = st["k"].copy(), st["v"].copy()
    status, fc, cow_ref = oracle.block_alloc(tables, st["ctx"], B, free, st["free_count"], refc, k, v)
    return dict(pool=pool, bt=bt, cl=cl, kc=kc, vc=vc, cow=cow), dict(
        status=status, fc=fc, tables=tables, refc=refc, free=free, k=k, v=v, cow=cow_ref)


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("B", [16, 32])
@pytest.mark.parametrize("advance", [False, True])
def test_block_alloc_matches_oracle(api, oracle, cuda_device, seed, B, advance):
    st = make_state(seed, B=B, NB=96, Hkv=2, D=128)
    gpu, ref = _run_both(api, oracle, cuda_device, st, advance)
    assert ref["status"] == 0
    fc = int(gpu["pool"].free_count.item())
    assert fc == ref["fc"]
    assert np.array_equal(gpu["pool"].free_blocks.cpu().numpy()[:fc], ref["free"][:fc])
    assert np.array_equal(gpu["pool"].refcounts.cpu().numpy(), ref["refc"])
    assert np.array_equal(gpu["bt"].cpu().numpy(), ref["tables"])
    assert np.array_equal(gpu["cow"].cpu().numpy(), ref["cow"])
    assert np.array_equal(gpu["cl"].cpu().numpy(), st["ctx"])
    assert np.array_equal(W.bits(gpu["kc"]), ref["k"]) and np.array_equal(W.bits(gpu["vc"]), ref["v"])
    assert (ref["cow"] >= 0).sum() == 3  # the partially filled shared block was copied 3 times
    assert api.device_errors() == 0


def test_block_alloc_short_stack_changes_nothing(api, oracle, cuda_device):
    st = make_state(4, B=16, NB=96, Hkv=2, D=128, extra_free=2)
    api.device_errors(clear=True)
    gpu, ref = _run_both(api, oracle, cuda_device, st)
    assert ref["status"] == 1
    assert int(gpu["pool"].free_count.item()) == st["free_count"]
    assert np.array_equal(gpu["bt"].cpu().numpy(), st["tables"])
    assert np.array_equal(gpu["pool"].refcounts.cpu().numpy(), st["refc"])
    assert np.all(gpu["cow"].cpu().numpy() == -1)
    assert api.device_errors() & 0x10


def test_device_driven_decode_loop(api, oracle, cuda_device):
    """Sequences sharing a 40-token prompt (one full and one partial block of
    16 tokens) decode 20 steps: each step allocates on the device (advance),
    then runs the fused step; outputs, tables and caches follow the oracle."""
    B, Hkv, G, D, S, NB = 16, 2, 4, 64, 5, 48
    rng = np.random.default_rng(8)
    order = list(rng.permutation(NB))
    prompt = [order.pop() for _ in range(3)]  # 40 tokens: blocks of 16, 16, 8
    tables = np.full((S, 8), -1, np.int32)
    pre = np.array([40, 40, 40, 17, 0], np.int32)
    for s in range(S):
        if s < 3:
            tables[s, :3] = prompt
        elif pre[s]:
            tables[s, :2] = [order.pop(), order.pop()]
    refc = np.zeros(NB, np.int32)
    for s in range(S):
        for j in range((pre[s] + B - 1) // B):
            refc[tables[s, j]] += 1
    free = np.array(order, np.int32)
    g = torch.Generator().manual_seed(2)
    kc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, Hkv, B, D, generator=g).to(torch.bfloat16)
    # host (oracle) state
    h_tables, h_refc = tables.copy(), refc.copy()
    h_free = np.concatenate([free, np.zeros(NB, np.int32)])[:NB].copy()
    h_fc = len(free)
    h_k, h_v = W.bits(kc).copy(), W.bits(vc).copy()
    h_ctx = pre.copy()
    # device state
    pool = api.DeviceBlockPool(free, refc, cuda_device)
    bt = torch.from_numpy(tables.copy()).to(cuda_device)
    cl = torch.from_numpy(pre.copy()).to(cuda_device)
    dk, dv = kc.to(cuda_device), vc.to(cuda_device)
    ws = torch.zeros(api.workspace_size(S, Hkv * G, D, 8, B, 32), dtype=torch.uint8, device=cuda_device)
    for step in range(20):
        q = torch.randn(S, Hkv * G, D, generator=g).to(torch.bfloat16)
        kn = torch.randn(S, Hkv, D, generator=g).to(torch.bfloat16)
        vn = torch.randn(S, Hkv, D, generator=g).to(torch.bfloat16)
        # oracle: advance, allocate, append, attend
        h_ctx = np.where(h_ctx > 0, h_ctx + 1, 0).astype(np.int32)
        status, h_fc, _ = oracle.block_alloc(h_tables, h_ctx, B, h_free, h_fc, h_refc, h_k, h_v)
        assert status == 0
        slots = oracle.slot_mapping(h_tables, h_ctx, B)
        oracle.cache_append(W.bits(kn), W.bits(vn), slots, h_k, h_v, B, 0, 1.0)
        ref = oracle.decode(W.bits(q), h_k, h_v, h_tables, h_ctx, Hkv, B, 1 / 8)
        # device
        pool.allocate(bt, cl, dk, dv, advance=True)
        out = api.decode_step(q.to(cuda_device), kn.to(cuda_device), vn.to(cuda_device), dk, dv,
                              bt, cl, 1 / 8, 1.0, 32, ws)
        torch.cuda.synchronize()
        compare(out, ref, what=f"step {step}")
        assert np.array_equal(bt.cpu().numpy(), h_tables)
        assert np.array_equal(cl.cpu().numpy(), h_ctx)
        assert np.array_equal(W.bits(dk), h_k) and np.array_equal(W.bits(dv), h_v)
    assert api.device_errors() == 0


# ---------------------------------------------------------------------------
# a chunk of new tokens per sequence (chunked prefill)
# ---------------------------------------------------------------------------

def _chunk_both(api, oracle, dev, st):
    B, NB = st["B"], st["NB"]
    pool = api.DeviceBlockPool(st["free"], st["refc"], dev)
    bt = torch.from_numpy(st["tables"].copy()).to(dev)
    cl = torch.from_numpy(st["ctx"]).to(dev)
    qs = torch.from_numpy(st["qs"]).to(dev)
    kc = W.from_bits(st["k"], dev)
    vc = W.from_bits(st["v"], dev)
    cow = pool.allocate_chunk(bt, cl, qs, kc, vc)
    torch.cuda.synchronize()
    tables, refc = st["tables"].copy(), st["refc"].copy()
    free = np.concatenate([st["free"], np.zeros(NB, np.int32)])[:NB].copy()
    k, v = st["k"].copy(), st["v"].copy()
    status, fc, cow_ref = oracle.block_alloc_chunk(tables, st["ctx"], st["qs"], B, free, st["free_count"],
                                                   refc, k, v)
    return dict(pool=pool, bt=bt, cl=cl, qs=qs, kc=kc, vc=vc, cow=cow), dict(
        status=status, fc=fc, tables=tables, refc=refc, free=free, k=k, v=v, cow=cow_ref)


@pytest.mark.parametrize("seed,chunks", [(1, [2, 7, 1, 4]), (2, [3, 9, 4, 13]), (3, [1, 5, 8, 12]),
                                         (4, [17, 40, 33, 1])])
@pytest.mark.parametrize("B", [16, 32])
def test_block_alloc_chunk_matches_oracle(api, oracle, cuda_device, seed, chunks, B):
    """Chunks crossing block boundaries from shared (full and partly filled)
    and private blocks: tables, free stack, counts, reference counts,
    copy sources and copied rows bit for bit."""
    st = make_chunk_state(seed, chunks, B=B, NB=192, Hkv=2, D=128)
    gpu, ref = _chunk_both(api, oracle, cuda_device, st)
    assert ref["status"] == 0
    fc = int(gpu["pool"].free_count.item())
    assert fc == ref["fc"]
    assert np.array_equal(gpu["pool"].free_blocks.cpu().numpy()[:fc], ref["free"][:fc])
    assert np.array_equal(gpu["pool"].refcounts.cpu().numpy(), ref["refc"])
    assert np.array_equal(gpu["bt"].cpu().numpy(), ref["tables"])
    assert np.array_equal(gpu["cow"].cpu().numpy(), ref["cow"])
    assert np.array_equal(W.bits(gpu["kc"]), ref["k"]) and np.array_equal(W.bits(gpu["vc"]), ref["v"])
    assert api.device_errors() == 0


def test_block_alloc_chunk_short_stack_changes_nothing(api, oracle, cuda_device):
    st = make_chunk_state(6, [5, 9, 40], B=16, NB=192, Hkv=2, D=128)
    st["free"] = st["free"][:3]
    st["free_count"] = 3
    api.device_errors(clear=True)
    gpu, ref = _chunk_both(api, oracle, cuda_device, st)
    assert ref["status"] == 1
    assert int(gpu["pool"].free_count.item()) == 3
    assert np.array_equal(gpu["bt"].cpu().numpy(), st["tables"])
    assert np.array_equal(gpu["pool"].refcounts.cpu().numpy(), st["refc"])
    assert np.all(gpu["cow"].cpu().numpy() == -1)
    assert api.device_errors(clear=True) == _lib.PA_DEVERR_OUT_OF_BLOCKS


@pytest.mark.parametrize("B", [16, 32])
def test_device_driven_chunked_prefill(api, oracle, cuda_device, B):
    """Sequences sharing prompt blocks each bring a chunk: blocks allocated on
    the device, chunk slots, the chunk's append and the attention, against
    the oracle doing the same four steps."""
    st = make_chunk_state(7, [3, 21, 40, 9], B=B, NB=192, Hkv=2, D=128)
    S = len(st["ctx"])
    g = torch.Generator().manual_seed(B)
    # the pool's rows as N(0, 1) values (the allocation states carry raw bits)
    for name in ("k", "v"):
        st[name] = W.bits(torch.randn(st[name].shape, generator=g).to(torch.bfloat16))
    T = int(st["qs"][-1])
    q = torch.randn((T, 8, 128), generator=g).to(torch.bfloat16)
    k_new = torch.randn((T, 2, 128), generator=g).to(torch.bfloat16)
    v_new = torch.randn((T, 2, 128), generator=g).to(torch.bfloat16)
    gpu, ref = _chunk_both(api, oracle, cuda_device, st)
    assert ref["status"] == 0
    slots = api.chunk_slot_mapping(gpu["bt"], gpu["cl"], gpu["qs"], B)
    api.cache_append(k_new.to(cuda_device), v_new.to(cuda_device), slots, gpu["kc"], gpu["vc"])
    out = api.prefill(q.to(cuda_device), gpu["kc"], gpu["vc"], gpu["bt"], gpu["cl"], gpu["qs"],
                      int(np.diff(st["qs"]).max()), 1.0 / np.sqrt(128))
    torch.cuda.synchronize()
    slots_ref = oracle.chunk_slot_mapping(ref["tables"], st["ctx"], st["qs"], B)
    oracle.cache_append(W.bits(k_new), W.bits(v_new), slots_ref, ref["k"], ref["v"], B, 0, 1.0)
    out_ref = oracle.prefill(W.bits(q), ref["k"], ref["v"], ref["tables"], st["ctx"], st["qs"], 2, B,
                             1.0 / np.sqrt(128))
    assert np.array_equal(slots.cpu().numpy(), slots_ref)
    assert np.array_equal(W.bits(gpu["kc"]), ref["k"]) and np.array_equal(W.bits(gpu["vc"]), ref["v"])
    compare(out, out_ref, what=f"device-driven chunked prefill B{B}")
    assert api.device_errors() == 0
    assert S > 0
