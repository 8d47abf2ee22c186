"""Decode steps captured in a CUDA graph (one graph for several layers)
replay bit for bit like the same steps run eagerly, and read the context
lengths and block tables afresh at every replay."""
import numpy as np
import pytest
import torch

from gpu_helpers import device_tables
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _layers(name, n, device, ps, num_seqs=None, seed0=10):
    out = []
    for i in range(n):
        wl = W.make(name, device=device, num_seqs=num_seqs, data_seed=seed0 + i)
        W.poison(wl, pending=True)
        out.append(wl)
    return out


def _clone_caches(wls):
    return [(wl.k_cache.clone(), wl.v_cache.clone()) for wl in wls]


@pytest.mark.parametrize("name,num_seqs,ps", [("tiny", None, 0), ("tiny", None, 32),
                                              ("llama8b", 12, 512)])
def test_graph_matches_eager(api, cuda_device, name, num_seqs, ps):
    wls = _layers(name, 3, cuda_device, ps, num_seqs)
    fresh = _clone_caches(wls)
    # eager reference on copies of the caches
    ref_out, ref_caches, ref_slots = [], [], []
    for wl, (kc, vc) in zip(wls, fresh):
        bt, cl = device_tables(wl, cuda_device)
        st = api.DecodeStep(kc.clone(), vc.clone(), bt, cl, wl.shape.num_q_heads,
                            wl.softmax_scale, wl.kv_scale, ps)
        ref_out.append(st(wl.q, wl.k_new, wl.v_new).clone())
        ref_caches.append((st.k_cache, st.v_cache))
        ref_slots.append(st.slots.clone())
    # graph over all layers, on the original caches
    steps, inputs = [], []
    for wl in wls:
        bt, cl = device_tables(wl, cuda_device)
        steps.append(api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, wl.shape.num_q_heads,
                                    wl.softmax_scale, wl.kv_scale, ps))
        inputs.append((wl.q, wl.k_new, wl.v_new))
    g = api.StepGraph(steps, inputs)
    for i, (kc, vc) in enumerate(fresh):  # undo the eager warm-up's append
        steps[i].k_cache.copy_(kc)
        steps[i].v_cache.copy_(vc)
        steps[i].out.zero_()
    g.replay()
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(steps[i].out.view(torch.int16), ref_out[i].view(torch.int16))
        assert torch.equal(steps[i].slots, ref_slots[i])
        assert torch.equal(steps[i].k_cache.view(torch.uint8), ref_caches[i][0].view(torch.uint8))
        assert torch.equal(steps[i].v_cache.view(torch.uint8), ref_caches[i][1].view(torch.uint8))
    assert api.device_errors() == 0


def test_graph_reads_buffers_at_replay(api, oracle, cuda_device):
    """Grow the context by one token between replays (host updates the
    device buffers); each replay must equal an eager step on the same state."""
    wl = W.make("llama8b", device=cuda_device, num_seqs=8, seed=3, extra_steps=4)
    B = wl.shape.block_size
    alloc = wl.notes["allocator"]
    bt, cl = device_tables(wl, cuda_device)
    q = wl.q.clone()
    kn, vn = wl.k_new.clone(), wl.v_new.clone()
    step = api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, wl.shape.num_q_heads,
                          wl.softmax_scale, 1.0, 512)
    g = api.StepGraph([step], [(q, kn, vn)])
    gen = torch.Generator(device=cuda_device).manual_seed(7)
    for it in range(3):
        wl.context_lens = wl.context_lens + 1
        for s in range(wl.shape.num_seqs):
            pos = int(wl.context_lens[s]) - 1
            if pos % B == 0:
                wl.block_tables[s, pos // B] = alloc.allocate(1)[0]
        bt.copy_(torch.from_numpy(wl.block_tables))
        cl.copy_(torch.from_numpy(wl.context_lens))
        q.copy_(torch.randn(q.shape, generator=gen, device=cuda_device))
        kn.copy_(torch.randn(kn.shape, generator=gen, device=cuda_device))
        vn.copy_(torch.randn(vn.shape, generator=gen, device=cuda_device))
        kc0, vc0 = wl.k_cache.clone(), wl.v_cache.clone()
        g.replay()
        torch.cuda.synchronize()
        got = step.out.clone()
        got_slots = step.slots.clone()
        kc1, vc1 = wl.k_cache.clone(), wl.v_cache.clone()
        wl.k_cache.copy_(kc0)
        wl.v_cache.copy_(vc0)
        ref = api.decode_step(q, kn, vn, wl.k_cache, wl.v_cache, bt, cl, wl.softmax_scale, 1.0,
                              512)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(wl.k_cache.view(torch.int16), kc1.view(torch.int16))
        want = oracle.slot_mapping(wl.block_tables, wl.context_lens, B)
        assert np.array_equal(got_slots.cpu().numpy(), want)
