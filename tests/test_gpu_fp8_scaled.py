"""E4M3 cache with a scale per KV head for K and for V: GPU append bit for
bit and the fused step within tolerance of the oracle's per-head variant."""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, device_tables
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _scales(Hkv, seed):
    rng = np.random.default_rng(seed)
    ks = (rng.uniform(0.5, 2.0, Hkv) * 4.5 / 448).astype(np.float32)
    vs = (rng.uniform(0.5, 2.0, Hkv) * 4.5 / 448).astype(np.float32)
    return ks, vs


def _case(oracle, device, D, B, G, Hkv, ctx, seed):
    rng = np.random.default_rng(seed)
    ctx = np.array(ctx, np.int64)
    nb = int(sum((int(c) + B - 1) // B for c in ctx)) + 5
    tables, _ = W.build_tables(ctx, B, nb, rng)
    wl = W._finish("scaled", W.Shape(len(ctx), G * Hkv, Hkv, D, B, kv_dtype=W.KV_FP8_E4M3), ctx,
                   tables, nb, device, seed)
    ks, vs = _scales(Hkv, seed)
    kb, vb = W.bits(wl.k_cache), W.bits(wl.v_cache)
    kc = np.zeros(kb.shape, np.uint8)
    vc = np.zeros_like(kc)
    tok = lambda a: a.transpose(0, 2, 1, 3).reshape(nb * B, Hkv, D)
    oracle.cache_append_scaled(tok(kb), tok(vb), np.arange(nb * B, dtype=np.int32), kc, vc, B, ks, vs)
    wl.k_cache = torch.from_numpy(kc).to(device)
    wl.v_cache = torch.from_numpy(vc).to(device)
    return wl, ks, vs


def test_append_scaled_bitexact(api, oracle, cuda_device):
    rng = np.random.default_rng(3)
    NB, Hkv, B, D, T = 30, 4, 16, 128, 41
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int32)
    slots[::9] = -1
    g = torch.Generator().manual_seed(5)
    k = (torch.randn(T, Hkv, D, generator=g) * 2).to(torch.bfloat16)
    v = (torch.randn(T, Hkv, D, generator=g) * 2).to(torch.bfloat16)
    ks, vs = _scales(Hkv, 9)
    kc0 = torch.randint(0, 255, (NB, Hkv, B, D), dtype=torch.uint8, generator=g)
    vc0 = kc0.clone()
    kr, vr = kc0.numpy().copy(), vc0.numpy().copy()
    oracle.cache_append_scaled(W.bits(k), W.bits(v), slots, kr, vr, B, ks, vs)
    kc, vc = kc0.to(cuda_device), vc0.to(cuda_device)
    api.cache_append_scaled(k.to(cuda_device), v.to(cuda_device),
                            torch.from_numpy(slots).to(cuda_device), kc, vc,
                            torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device))
    assert np.array_equal(kc.cpu().numpy(), kr) and np.array_equal(vc.cpu().numpy(), vr)


@pytest.mark.parametrize("D,B,G,Hkv", [(128, 16, 4, 4), (128, 32, 8, 2), (64, 16, 16, 1), (128, 16, 1, 3)])
@pytest.mark.parametrize("ps", [0, 64])
def test_step_scaled_matches_oracle(api, oracle, cuda_device, D, B, G, Hkv, ps):
    ctx = [1, B + 1, 3 * B, 300]
    wl, ks, vs = _case(oracle, cuda_device, D, B, G, Hkv, ctx, D + B + G + ps)
    W.poison(wl, pending=True)
    kc, vc = W.bits(wl.k_cache).copy(), W.bits(wl.v_cache).copy()
    slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, B)
    oracle.cache_append_scaled(W.bits(wl.k_new), W.bits(wl.v_new), slots, kc, vc, B, ks, vs)
    ref = oracle.decode_scaled(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens, Hkv, B,
                               wl.softmax_scale, ks, vs)
    bt, cl = device_tables(wl, cuda_device)
    dks, dvs = torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device)
    slot_out = torch.empty(len(ctx), dtype=torch.int32, device=cuda_device)
    out = api.decode_step_scaled(wl.q, wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, bt, cl, dks, dvs,
                                 wl.softmax_scale, ps, slot_mapping=slot_out)
    torch.cuda.synchronize()
    assert np.array_equal(slot_out.cpu().numpy(), slots)
    assert np.array_equal(W.bits(wl.k_cache), kc) and np.array_equal(W.bits(wl.v_cache), vc)
    compare(out, ref, what=f"per-head scales D{D} B{B} G{G} ps{ps}")
    # attention only (no append): same output from the now-complete cache
    out2 = api.decode_step_scaled(wl.q, None, None, wl.k_cache, wl.v_cache, bt, cl, dks, dvs,
                                  wl.softmax_scale, ps)
    compare(out2, ref, what="attention only")
    assert api.device_errors() == 0
