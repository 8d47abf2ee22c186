"""The five workloads at full size, in the launch configuration the
benchmark times, checked on sampled (sequence, query head) outputs that the
oracle computes one by one, plus bit-exact checks of the appended rows.

The oracle reads a compacted host copy of only the sampled sequences'
blocks, taken BEFORE the GPU append; it then runs its own slot mapping and
append on that copy, so no value it reads comes from the GPU kernels."""
import numpy as np
import pytest
import torch

from gpu_helpers import compact, compare, device_tables, guard_step, quantize_with_torch
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# name, block size, partition size (the benchmark's launch configuration
# for each workload is in bench.py: DEFAULT_PARTITION)
CONFIGS = [
    ("llama8b", 16, 0),
    ("llama8b", 16, 512),
    ("long70b", 16, 512),
    ("long70b", 32, 512),
    ("prefix_fp8", 16, 0),
    ("prefix_fp8", 16, 512),
    ("ctx128k", 16, 512),
]


def _bench_launches():
    import bench
    return [(name, bs, ps) for name, (bs, ps) in bench.DEFAULT_LAUNCH.items() if name != "tiny"]


CONFIGS += [c for c in _bench_launches() if c not in CONFIGS]


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _sample_seqs(S, n, seed):
    rng = np.random.default_rng(seed)
    picks = {0, S - 1}
    while len(picks) < min(n, S):
        picks.add(int(rng.integers(0, S)))
    return sorted(picks)


def _check_step(api, oracle, wl, partition_size, n_seqs=6, heads_per_seq=6, seed=0):
    sh = wl.shape
    seqs = _sample_seqs(sh.num_seqs, n_seqs, seed)
    W.poison(wl, pending=True)
    # oracle side, from the pre-append state
    tables_c, ctx_c, kc_c, vc_c = compact(wl, seqs, wl.k_cache, wl.v_cache)
    slots_c = oracle.slot_mapping(tables_c, ctx_c, sh.block_size)
    kn = W.bits(wl.k_new)[seqs]
    vn = W.bits(wl.v_new)[seqs]
    oracle.cache_append(kn, vn, slots_c, kc_c, vc_c, sh.block_size, sh.kv_dtype, wl.kv_scale)
    rng = np.random.default_rng(seed + 1)
    pairs_local = []
    for i in range(len(seqs)):
        heads = {0, sh.num_q_heads - 1}
        while len(heads) < min(heads_per_seq, sh.num_q_heads):
            heads.add(int(rng.integers(0, sh.num_q_heads)))
        pairs_local += [[i, h] for h in sorted(heads)]
    pairs_local = np.array(pairs_local, np.int32)
    ref = oracle.decode_pairs(W.bits(wl.q)[seqs], kc_c, vc_c, tables_c, ctx_c, sh.num_kv_heads,
                              sh.block_size, wl.softmax_scale, pairs_local,
                              kv_dtype=sh.kv_dtype, kv_scale=wl.kv_scale)
    # GPU side: the full step
    bt, cl = device_tables(wl, wl.k_cache.device)
    api.device_errors(clear=True)
    step = api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, sh.num_q_heads, wl.softmax_scale,
                          wl.kv_scale, partition_size)
    check_guards = guard_step(step)
    out = step(wl.q, wl.k_new, wl.v_new)
    torch.cuda.synchronize()
    check_guards(f"{wl.name} B{sh.block_size} ps{partition_size}")
    assert api.device_errors() == 0
    # slots and appended rows, bit for bit
    slots = step.slots.cpu().numpy()
    full_slots = oracle.slot_mapping(wl.block_tables, wl.context_lens, sh.block_size)
    assert np.array_equal(slots, full_slots)
    for i, s in enumerate(seqs):
        b, off = divmod(int(slots[s]), sh.block_size)
        bc, offc = divmod(int(slots_c[i]), sh.block_size)
        assert np.array_equal(W.bits(wl.k_cache[b, :, off]), kc_c[bc, :, offc])
        assert np.array_equal(W.bits(wl.v_cache[b, :, off]), vc_c[bc, :, offc])
    rows = torch.tensor([seqs[i] for i, _ in pairs_local], device=out.device)
    heads = torch.tensor(pairs_local[:, 1].astype(np.int64), device=out.device)
    got = out[rows, heads]
    return compare(got, ref, what=f"{wl.name} B{sh.block_size} ps{partition_size}")


@pytest.mark.parametrize("name,bs,ps", CONFIGS, ids=lambda x: str(x))
def test_config_sampled(api, oracle, cuda_device, name, bs, ps):
    wl = W.make(name, device=cuda_device, block_size=bs)
    if wl.shape.kv_dtype == W.KV_FP8_E4M3:
        quantize_with_torch(wl)
    _check_step(api, oracle, wl, ps)


@pytest.mark.parametrize("ps", [0, 512])
def test_llama8b_e4m3_sampled(api, oracle, cuda_device, ps):
    """The Llama-3-8B-shape layer with its cache in E4M3 (one per-tensor
    scale), as the benchmark also times it."""
    wl = W.make("llama8b", device=cuda_device)
    wl.shape.kv_dtype = W.KV_FP8_E4M3
    wl.kv_scale = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
    quantize_with_torch(wl)
    _check_step(api, oracle, wl, ps)


def test_ctx128k_growing_steps(api, oracle, cuda_device):
    """Long-context step sequence: each step appends one token per sequence
    (a fresh block from the host allocator when the position starts one),
    then attends over 131072+ tokens; three steps, crossing a block edge."""
    steps = 3
    wl = W.make("ctx128k", device=cuda_device, extra_steps=steps)
    alloc = wl.notes["allocator"]
    sh = wl.shape
    B = sh.block_size
    g = torch.Generator(device=cuda_device)
    for k in range(steps):
        if k > 0:
            wl.context_lens = wl.context_lens + 1
            for s in range(sh.num_seqs):
                pos = int(wl.context_lens[s]) - 1
                if pos % B == 0:
                    wl.block_tables[s, pos // B] = alloc.allocate(1)[0]
            g.manual_seed(100 + k)
            wl.q = torch.randn(wl.q.shape, generator=g, device=cuda_device).to(torch.bfloat16)
            wl.k_new = torch.randn(wl.k_new.shape, generator=g, device=cuda_device).to(torch.bfloat16)
            wl.v_new = torch.randn(wl.v_new.shape, generator=g, device=cuda_device).to(torch.bfloat16)
        _check_step(api, oracle, wl, 512, n_seqs=3, heads_per_seq=4, seed=k)
