"""Decode steps captured in a CUDA graph (one graph for several layers):
every replayed layer's output, slots and appended cache rows match the
oracle, also on a later replay after the captured input buffers, the
context lengths and the block tables were overwritten; replays are also bit
for bit the same steps run eagerly."""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, device_tables, guard_step
from test_gpu_kernels import _oracle_step
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


def _grow_contexts(wls, bt, cl, gen):
    """Every sequence gains one token (a fresh block from the host allocator
    when the token starts one; all layers share the tables), and every
    layer's captured q / new K / new V buffers get fresh values in place."""
    lead = wls[0]
    B = lead.shape.block_size
    alloc = lead.notes["allocator"]
    ctx = lead.context_lens + 1
    tables = lead.block_tables.copy()
    for s in range(lead.shape.num_seqs):
        pos = int(ctx[s]) - 1
        if pos % B == 0:
            tables[s, pos // B] = alloc.allocate(1)[0]
    for wl in wls:
        wl.context_lens = ctx.copy()
        wl.block_tables = tables.copy()
        for t in (wl.q, wl.k_new, wl.v_new):
            t.copy_(torch.randn(t.shape, generator=gen, device=t.device))
        W.poison(wl, pending=True)
    bt.copy_(torch.from_numpy(tables))
    cl.copy_(torch.from_numpy(ctx))


@pytest.mark.parametrize("name,num_seqs,layers,ps", [("tiny", None, 4, 0), ("tiny", None, 4, 32),
                                                     ("llama8b", 16, 2, 0), ("llama8b", 16, 2, 512)])
def test_graph_replay_matches_oracle(api, oracle, cuda_device, name, num_seqs, layers, ps):
    wls = []
    for i in range(layers):
        wl = W.make(name, device=cuda_device, num_seqs=num_seqs, data_seed=20 + i, extra_steps=2)
        W.poison(wl, pending=True)
        wls.append(wl)
    bt, cl = device_tables(wls[0], cuda_device)  # one set of tables for all layers
    refs = [_oracle_step(oracle, wl) for wl in wls]
    before = [(wl.k_cache.clone(), wl.v_cache.clone()) for wl in wls]
    steps = [api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, wl.shape.num_q_heads, wl.softmax_scale,
                            wl.kv_scale, ps) for wl in wls]
    guards = [guard_step(st) for st in steps]
    g = api.StepGraph(steps, [(wl.q, wl.k_new, wl.v_new) for wl in wls])
    # the capture's eager warm-up appended once: go back to the state the
    # oracle saw
    for st, (kc, vc) in zip(steps, before):
        st.k_cache.copy_(kc)
        st.v_cache.copy_(vc)
        st.out.fill_(float("nan"))
        st.slots.fill_(-7)
    gen = torch.Generator(device=cuda_device).manual_seed(99)
    api.device_errors(clear=True)
    for replay in range(2):
        if replay:
            _grow_contexts(wls, bt, cl, gen)
            refs = [_oracle_step(oracle, wl) for wl in wls]
        g.replay()
        torch.cuda.synchronize()
        for i, (st, wl, (slots_ref, kc_ref, vc_ref, out_ref)) in enumerate(zip(steps, wls, refs)):
            what = f"{name} ps={ps} replay {replay} layer {i}"
            guards[i](what)
            assert np.array_equal(st.slots.cpu().numpy(), slots_ref), what
            assert np.array_equal(W.bits(st.k_cache), kc_ref), what
            assert np.array_equal(W.bits(st.v_cache), vc_ref), what
            compare(st.out, out_ref, what=what)
    assert api.device_errors() == 0
