"""The kernels' bounded waits give up cleanly.

Every wait of the decode kernel and of the tensor-memory prefill kernel has
a time limit; when it runs out the kernel sets PA_DEVERR_TIMEOUT, waits
(with the full 2 s limit) for the copies it has already issued, and
finishes (decode: with zeros for the rows it could not compute; prefill:
with an invalid output), so a lost copy can never hang the GPU.  Here the
test hook makes the first wait (decode: every warp's; prefill: the MMA
threads') go to a barrier that nothing ever completes, with a 1 ms limit:
nothing faults and nothing hangs, the call returns, the flag is raised, and
the next call at the default limit is correct against the oracle (the
context is still usable)."""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, device_tables
from paged_kv_cache_193_gb300 import _lib
from paged_kv_cache_193_gb300 import workloads as W
from test_gpu_kernels import _oracle_step
from test_gpu_prefill import _dev, _oracle_step as _oracle_prefill, e4m3_prefill_step, make_e4m3_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api(cuda_device):
    from paged_kv_cache_193_gb300 import api as a
    a._lib_handle()
    return a


def _stalled(lib, fn):
    assert lib.pa_test_set_wait(1_000_000, 1) == _lib.PA_OK
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        assert lib.pa_test_set_wait(0, 0) == _lib.PA_OK
    return out


@pytest.mark.parametrize("name,num_seqs,ps", [("tiny", None, 0), ("tiny", None, 32),
                                              ("llama8b", 24, 0), ("llama8b", 24, 512)])
def test_wait_runs_out_then_recovers(api, oracle, cuda_device, name, num_seqs, ps):
    lib = _lib.load()
    wl = W.make(name, device=cuda_device, num_seqs=num_seqs)
    W.poison(wl, pending=True)
    slots_ref, kc_ref, vc_ref, out_ref = _oracle_step(oracle, wl)
    bt, cl = device_tables(wl, cuda_device)
    api.device_errors(clear=True)
    step = api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, wl.shape.num_q_heads,
                          wl.softmax_scale, wl.kv_scale, ps)
    step.out.fill_(float("nan"))
    out = _stalled(lib, lambda: step(wl.q, wl.k_new, wl.v_new).clone())
    flags = api.device_errors(clear=True)
    assert flags & _lib.PA_DEVERR_TIMEOUT, hex(flags)
    assert flags & ~_lib.PA_DEVERR_TIMEOUT == 0, hex(flags)
    # every warp with pages gave up before reading one: all rows are zeros
    assert torch.count_nonzero(out) == 0
    # the append runs before any wait, so it happened all the same
    assert np.array_equal(W.bits(wl.k_cache), kc_ref)
    assert np.array_equal(W.bits(wl.v_cache), vc_ref)
    # the next call, at the default limit, is correct
    W.poison(wl, pending=True)
    out = step(wl.q, wl.k_new, wl.v_new).clone()
    torch.cuda.synchronize()
    assert np.array_equal(step.slots.cpu().numpy(), slots_ref)
    assert np.array_equal(W.bits(wl.k_cache), kc_ref)
    compare(out, out_ref, what=f"{name} ps={ps} after a timed-out call")
    assert api.device_errors() == 0


def test_wait_limit_is_validated():
    lib = _lib.load()
    assert lib.pa_test_set_wait(61 * 10**9, 0) == _lib.PA_ERR_INVALID_ARG
    assert lib.pa_test_set_wait(0, 0) == _lib.PA_OK


@pytest.mark.parametrize("G,Hkv,B,D", [(4, 2, 16, 128), (1, 4, 32, 128), (16, 1, 16, 128), (4, 2, 16, 64)])
def test_prefill_wait_runs_out_then_recovers(api, oracle, cuda_device, G, Hkv, B, D):
    lib = _lib.load()
    wl = W.make_prefill(cuda_device, seed=40 + G + B, num_seqs=5, chunk=[1, 7, 64, 300, 33],
                        prefixes=[0, 5, 33, 300, 16], num_q_heads=G * Hkv, num_kv_heads=Hkv,
                        head_dim=D, block_size=B)
    W.poison_prefill(wl)
    _, _, _, ref = _oracle_prefill(oracle, wl)
    bt, cl, qs = _dev(wl, cuda_device)
    slots = api.chunk_slot_mapping(bt, cl, qs, wl.shape.block_size)
    api.cache_append(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache)
    torch.cuda.synchronize()
    api.device_errors(clear=True)
    _stalled(lib, lambda: api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len,
                                      wl.softmax_scale))
    flags = api.device_errors(clear=True)
    assert flags & _lib.PA_DEVERR_TIMEOUT, hex(flags)
    assert flags & ~_lib.PA_DEVERR_TIMEOUT == 0, hex(flags)
    # the next call, at the default limit, is correct
    out = api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len, wl.softmax_scale)
    torch.cuda.synchronize()
    compare(out, ref, what=f"prefill G{G} B{B} D{D} after a timed-out call")
    assert api.device_errors() == 0


def test_prefill_e4m3_wait_runs_out_then_recovers(api, oracle, cuda_device):
    """The E4M3 prefill kernel (a loader warp and a converting warp) gives up
    the same way, and the next call is correct."""
    lib = _lib.load()
    wl, scale = make_e4m3_prefill(oracle, cuda_device, seed=45, num_seqs=5, chunk=[1, 7, 64, 300, 33],
                                  prefixes=[0, 5, 33, 300, 16], num_q_heads=8, num_kv_heads=2,
                                  head_dim=128, block_size=16)
    W.poison_prefill(wl)
    bt, cl, qs = _dev(wl, cuda_device)
    api.device_errors(clear=True)
    _stalled(lib, lambda: api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, wl.max_query_len,
                                      wl.softmax_scale, kv_scale=scale))
    flags = api.device_errors(clear=True)
    assert flags & _lib.PA_DEVERR_TIMEOUT, hex(flags)
    assert flags & ~_lib.PA_DEVERR_TIMEOUT == 0, hex(flags)
    ref, out = e4m3_prefill_step(api, oracle, wl, scale, cuda_device)
    compare(out, ref, what="prefill E4M3 after a timed-out call")
    assert api.device_errors() == 0
