"""Edge cases at the limits of the decode and prefill paths, against the oracle:

* degenerate softmax scales: 0 weighs every cached token equally (the step
  returns the mean of V, checked here without the oracle too), a negative
  scale reverses the preference;
* the largest grid a launch takes: 65,535 sequences (the grid's z limit), of
  0 to 40 tokens each, unsplit and in partitions of 16 tokens, and with the
  E4M3 cache;
* one context of 2^20 tokens (65,536 pages of one KV head, group 16) beside a
  short one, unsplit (one CTA walks the whole table), in 2,048 partitions of
  512 (the merge's widest shape), with 32-token pages and with the E4M3
  cache, checked on sampled heads;
* prefill: one 2,048-token chunk (32 tile pairs of one sequence), 2,000
  sequences of 1-3-token chunks, and chunks with no cached prefix.
Slots and appended rows are compared bit for bit, outputs within the
attention tolerance, all through guarded buffers."""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, device_tables, guard_step, quantize_with_torch
from paged_kv_cache_193_gb300 import workloads as W
from test_gpu_configs import _check_step
from test_gpu_kernels import _oracle_step, _random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _full_step(api, wl, ps):
    bt, cl = device_tables(wl, wl.k_cache.device)
    step = api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, wl.shape.num_q_heads, wl.softmax_scale,
                          wl.kv_scale, ps)
    check = guard_step(step)
    api.device_errors(clear=True)
    out = step(wl.q, wl.k_new, wl.v_new)
    torch.cuda.synchronize()
    check(f"ps={ps}")
    assert api.device_errors() == 0
    return step.slots.cpu().numpy(), out


def _bf16_rows(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("scale", [0.0, -0.3])
@pytest.mark.parametrize("ps", [0, 32])
@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8_E4M3])
def test_degenerate_softmax_scales(api, oracle, cuda_device, scale, ps, kv):
    ctx = [1, 15, 16, 17, 200]
    B, G = 16, 4
    D = 64 if kv == W.KV_BF16 else 128
    wl = _random_case(77, len(ctx), 8, 2, D, B, ctx, kv, oracle, cuda_device)
    wl.softmax_scale = scale
    W.poison(wl, pending=True)
    slots_ref, kc_ref, vc_ref, out_ref = _oracle_step(oracle, wl)
    if scale == 0.0 and kv == W.KV_BF16:
        # uniform weights: each output row is the mean of its KV head's V rows
        for s, n in enumerate(ctx):
            for hq in range(8):
                rows = [vc_ref[wl.block_tables[s, t // B], hq // G, t % B] for t in range(n)]
                mean = _bf16_rows(np.stack(rows)).mean(axis=0)
                assert np.abs(mean - out_ref[s, hq]).max() < 1e-9
    slots, out = _full_step(api, wl, ps)
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref) and np.array_equal(W.bits(wl.v_cache), vc_ref)
    compare(out, out_ref, what=f"softmax_scale {scale} ps={ps}")


@pytest.mark.parametrize("ps,kv", [(0, W.KV_BF16), (16, W.KV_BF16), (0, W.KV_FP8_E4M3)])
def test_largest_grid(api, oracle, cuda_device, ps, kv):
    S = 65535
    ctx = [0 if s % 97 == 0 else 1 + (s * 7919) % 40 for s in range(S)]
    B = 16
    need = sum(-(-c // B) for c in ctx)
    tables, _ = W.build_tables(np.array(ctx, np.int64), B, need + 64, np.random.default_rng(65535))
    wl = W._finish("grid", W.Shape(S, 8, 2, 64, B, kv_dtype=kv), np.array(ctx, np.int64), tables, need + 64,
                   cuda_device, 65535)
    if kv == W.KV_FP8_E4M3:
        quantize_with_torch(wl)  # a library conversion, only to make the E4M3 input pool
    W.poison(wl, pending=True)
    slots_ref, kc_ref, vc_ref, out_ref = _oracle_step(oracle, wl)
    slots, out = _full_step(api, wl, ps)
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref) and np.array_equal(W.bits(wl.v_cache), vc_ref)
    compare(out, out_ref, what=f"65535 sequences ps={ps}")


@pytest.mark.parametrize("ps,B,kv", [(0, 16, W.KV_BF16), (512, 16, W.KV_BF16), (0, 32, W.KV_BF16),
                                     (512, 16, W.KV_FP8_E4M3)])
def test_million_token_context(api, oracle, cuda_device, ps, B, kv):
    ctx = np.array([1 << 20, 37], np.int64)
    nb = sum(-(-int(c) // B) for c in ctx) + 8
    tables, _ = W.build_tables(ctx, B, nb, np.random.default_rng(20))
    wl = W._finish("million", W.Shape(2, 16, 1, 128, B, kv_dtype=kv), ctx, tables, nb, cuda_device, 20)
    if kv == W.KV_FP8_E4M3:
        quantize_with_torch(wl)  # a library conversion, only to make the E4M3 input pool
    _check_step(api, oracle, wl, ps, n_seqs=2, heads_per_seq=5, seed=20)


# ---------------------------------------------------------------------------
# chunked prefill at its limits
# ---------------------------------------------------------------------------

def _prefill_case(api, oracle, cuda_device, what, **kw):
    from test_gpu_prefill import _gpu_step as prefill_step, _oracle_step as prefill_oracle
    wl = W.make_prefill(cuda_device, **kw)
    W.poison_prefill(wl)
    api.device_errors(clear=True)
    slots_ref, kc_ref, vc_ref, ref = prefill_oracle(oracle, wl)
    slots, out = prefill_step(api, wl, cuda_device, "auto")
    assert np.array_equal(slots, slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref) and np.array_equal(W.bits(wl.v_cache), vc_ref)
    compare(out, ref, what=what)
    assert api.device_errors() == 0


def test_prefill_long_chunk(api, oracle, cuda_device):
    """One 2,048-token chunk after a 1,500-token prefix (32 tile pairs of one
    sequence, keys up to 3,548) beside a 5-token chunk."""
    _prefill_case(api, oracle, cuda_device, "prefill long chunk", seed=61, num_seqs=2, chunk=[2048, 5],
                  prefixes=[1500, 0], num_q_heads=4, num_kv_heads=1, head_dim=128, block_size=16)


def test_prefill_many_sequences(api, oracle, cuda_device):
    """2,000 sequences with chunks of 1-3 tokens after prefixes of 0-100:
    2,000 x 2 work items of one partial tile each."""
    rng = np.random.default_rng(62)
    S = 2000
    chunks = rng.integers(1, 3, size=S, endpoint=True).tolist()
    prefixes = rng.integers(0, 100, size=S, endpoint=True).tolist()
    _prefill_case(api, oracle, cuda_device, "prefill 2000 sequences", seed=62, num_seqs=S, chunk=chunks,
                  prefixes=prefixes, num_q_heads=16, num_kv_heads=2, head_dim=128, block_size=16)


@pytest.mark.parametrize("G,B", [(4, 16), (1, 32)])
def test_prefill_without_prefix(api, oracle, cuda_device, G, B):
    """Chunks that are the whole context (no cached prefix): causal
    self-attention, the first row attending to itself only."""
    _prefill_case(api, oracle, cuda_device, f"prefill no prefix G{G} B{B}", seed=63 + G, num_seqs=4,
                  chunk=[1, 64, 129, 300], prefixes=[0, 0, 0, 0], num_q_heads=2 * G, num_kv_heads=2,
                  head_dim=128, block_size=B)
