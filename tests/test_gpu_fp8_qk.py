"""E4M3 x E4M3 scores (pa_decode_step_fp8_qk): the fused step within
tolerance of the oracle's rounded-query variant, closer to it than to the
exact-query result, at small shapes and on the full E4M3 workloads."""
import numpy as np
import pytest
import torch

from gpu_helpers import bf16_to_f64, compact, compare, device_tables, quantize_with_torch
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _q_scale(q):
    """The query's own range on the E4M3 grid: amax |q| / 448 (host, fp32)."""
    return float(np.float32(q.float().abs().max().item()) / np.float32(448.0))


def _scaled_case(oracle, device, D, B, G, Hkv, ctx, seed):
    rng = np.random.default_rng(seed)
    ctx = np.array(ctx, np.int64)
    nb = int(sum((int(c) + B - 1) // B for c in ctx)) + 5
    tables, _ = W.build_tables(ctx, B, nb, rng)
    wl = W._finish("fp8qk", W.Shape(len(ctx), G * Hkv, Hkv, D, B, kv_dtype=W.KV_FP8_E4M3), ctx,
                   tables, nb, device, seed)
    ks = (rng.uniform(0.5, 2.0, Hkv) * 4.5 / 448).astype(np.float32)
    vs = (rng.uniform(0.5, 2.0, Hkv) * 4.5 / 448).astype(np.float32)
    kb, vb = W.bits(wl.k_cache), W.bits(wl.v_cache)
    kc = np.zeros(kb.shape, np.uint8)
    vc = np.zeros_like(kc)
    tok = lambda a: a.transpose(0, 2, 1, 3).reshape(nb * B, Hkv, D)
    oracle.cache_append_scaled(tok(kb), tok(vb), np.arange(nb * B, dtype=np.int32), kc, vc, B, ks, vs)
    wl.k_cache = torch.from_numpy(kc).to(device)
    wl.v_cache = torch.from_numpy(vc).to(device)
    return wl, ks, vs


def _closer(out, ref_qk, ref_exact, what):
    """The kernel rounds the query: its output is much nearer the
    rounded-query oracle than the exact-query one."""
    g = bf16_to_f64(out)
    e_qk, e_exact = np.abs(g - ref_qk).mean(), np.abs(g - ref_exact).mean()
    assert e_qk < 0.5 * e_exact, f"{what}: mean err {e_qk:.2e} vs rounded-query oracle, {e_exact:.2e} vs exact"


@pytest.mark.parametrize("D,B,G,Hkv", [(128, 16, 4, 4), (128, 32, 8, 2), (64, 16, 16, 1), (128, 16, 1, 3)])
@pytest.mark.parametrize("ps", [0, 64])
def test_step_fp8_qk_matches_oracle(api, oracle, cuda_device, D, B, G, Hkv, ps):
    ctx = [1, B + 1, 3 * B, 300]
    wl, ks, vs = _scaled_case(oracle, cuda_device, D, B, G, Hkv, ctx, 7 * D + B + G + ps)
    W.poison(wl, pending=True)
    qs = _q_scale(wl.q)
    kc, vc = W.bits(wl.k_cache).copy(), W.bits(wl.v_cache).copy()
    slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, B)
    oracle.cache_append_scaled(W.bits(wl.k_new), W.bits(wl.v_new), slots, kc, vc, B, ks, vs)
    ref = oracle.decode_fp8_qk(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens, Hkv, B,
                               wl.softmax_scale, qs, ks, vs)
    exact = oracle.decode_scaled(W.bits(wl.q), kc, vc, wl.block_tables, wl.context_lens, Hkv, B,
                                 wl.softmax_scale, ks, vs)
    bt, cl = device_tables(wl, cuda_device)
    dks, dvs = torch.from_numpy(ks).to(cuda_device), torch.from_numpy(vs).to(cuda_device)
    slot_out = torch.empty(len(ctx), dtype=torch.int32, device=cuda_device)
    api.device_errors(clear=True)
    out = api.decode_step_scaled(wl.q, wl.k_new, wl.v_new, wl.k_cache, wl.v_cache, bt, cl, dks, dvs,
                                 wl.softmax_scale, ps, slot_mapping=slot_out, q_scale=qs)
    torch.cuda.synchronize()
    assert np.array_equal(slot_out.cpu().numpy(), slots)
    assert np.array_equal(W.bits(wl.k_cache), kc) and np.array_equal(W.bits(wl.v_cache), vc)
    what = f"fp8 qk D{D} B{B} G{G} ps{ps}"
    compare(out, ref, what=what)
    _closer(out, ref, exact, what)
    assert api.device_errors() == 0


def test_fp8_qk_rejects_bad_query_scale(api, cuda_device):
    wl = W.make("tiny", device=cuda_device)
    wl.shape.kv_dtype = W.KV_FP8_E4M3
    kc = torch.zeros(wl.k_cache.shape, dtype=torch.uint8, device=cuda_device)
    vc = torch.zeros_like(kc)
    bt, cl = device_tables(wl, cuda_device)
    one = torch.ones(wl.shape.num_kv_heads, dtype=torch.float32, device=cuda_device)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(api.PagedAttentionError):
            api.decode_step_scaled(wl.q, None, None, kc, vc, bt, cl, one, one, q_scale=bad)


@pytest.mark.slow
@pytest.mark.parametrize("name,ps", [("prefix_fp8", 0), ("llama8b", 0), ("prefix_fp8", 512)])
def test_fp8_qk_full_workload_sampled(api, oracle, cuda_device, name, ps):
    """The full E4M3 workloads (one cache scale for every head), attention
    over the cache as it stands, sampled (sequence, query head) outputs."""
    wl = W.make(name, device=cuda_device)
    if wl.shape.kv_dtype != W.KV_FP8_E4M3:
        wl.shape.kv_dtype = W.KV_FP8_E4M3
    quantize_with_torch(wl)
    sh = wl.shape
    qs = _q_scale(wl.q)
    ks = np.full(sh.num_kv_heads, wl.kv_scale, np.float32)
    rng = np.random.default_rng(11)
    seqs = sorted({0, sh.num_seqs - 1} | {int(x) for x in rng.integers(0, sh.num_seqs, 4)})
    tables_c, ctx_c, kc_c, vc_c = compact(wl, seqs, wl.k_cache, wl.v_cache)
    pairs = np.array([[i, h] for i in range(len(seqs)) for h in (0, sh.num_q_heads // 2, sh.num_q_heads - 1)],
                     np.int32)
    ref = oracle.decode_fp8_qk(W.bits(wl.q)[seqs], kc_c, vc_c, tables_c, ctx_c, sh.num_kv_heads,
                               sh.block_size, wl.softmax_scale, qs, ks, ks, pairs)
    bt, cl = device_tables(wl, cuda_device)
    dks = torch.from_numpy(ks).to(cuda_device)
    api.device_errors(clear=True)
    out = api.decode_step_scaled(wl.q, None, None, wl.k_cache, wl.v_cache, bt, cl, dks, dks,
                                 wl.softmax_scale, ps, q_scale=qs)
    torch.cuda.synchronize()
    assert api.device_errors() == 0
    rows = torch.tensor([seqs[i] for i, _ in pairs], device=out.device)
    heads = torch.tensor(pairs[:, 1].astype(np.int64), device=out.device)
    compare(out[rows, heads], ref, what=f"fp8 qk {name} ps{ps}")
