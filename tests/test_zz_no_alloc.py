"""pa_decode_static_workspace: split-context decode for callers that cannot
allocate device memory (their device memory belongs to another framework's
pool, or their host forbids allocation once serving has started).  The entry
point keeps its scratch in a fixed array inside the library, so the call
allocates nothing.

Checked here through the C ABI: two calls in a row (with different partition
sizes, so the second reuses the shared array the first one filled) must give
bit for bit what pa_decode gives with a caller-owned workspace (the same
kernels run on the same inputs), and must match the fp64 oracle on sampled
(sequence, query head) pairs within the attention tolerance; a call whose
scratch would not fit must be refused before anything is launched.  This
file is collected last so a failure here leaves every other test already
run."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import compare, device_tables, oracle_sampled, quantize_with_torch
from paged_kv_cache_193_gb300 import _lib
from paged_kv_cache_193_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _static_call(lib, wl, bt, cl, ps, out, stream):
    sh = wl.shape
    return lib.pa_decode_static_workspace(
        _ptr(wl.q), _ptr(wl.k_cache), _ptr(wl.v_cache), _ptr(bt), bt.shape[1], _ptr(cl),
        sh.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, wl.num_blocks, sh.block_size,
        sh.kv_dtype, ctypes.c_float(wl.kv_scale), ctypes.c_float(wl.softmax_scale), ps, _ptr(out),
        ctypes.c_void_p(stream))


def _reference_call(lib, wl, bt, cl, ps, out, stream):
    sh = wl.shape
    n = lib.pa_decode_workspace_size(sh.num_seqs, sh.num_q_heads, sh.head_dim, bt.shape[1],
                                     sh.block_size, ps)
    ws = torch.empty(n, dtype=torch.uint8, device=out.device)
    st = lib.pa_decode(_ptr(wl.q), _ptr(wl.k_cache), _ptr(wl.v_cache), _ptr(bt), bt.shape[1],
                       _ptr(cl), sh.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim,
                       wl.num_blocks, sh.block_size, sh.kv_dtype, ctypes.c_float(wl.kv_scale),
                       ctypes.c_float(wl.softmax_scale), ps, _ptr(ws), n, _ptr(out),
                       ctypes.c_void_p(stream))
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("name,fp8,num_seqs,sizes", [
    ("llama8b", False, 48, (512, 256)),
    ("llama8b", True, 48, (512, 256)),          # E4M3 cache
    ("ctx128k", False, 1, (512, 1024)),        # group 16, 256 and 128 partitions
])
def test_static_workspace_matches_pa_decode(cuda_device, oracle, name, fp8, num_seqs, sizes):
    lib = _lib.load()
    wl = W.make(name, device=cuda_device, num_seqs=num_seqs)
    if fp8:
        wl.shape.kv_dtype = W.KV_FP8_E4M3
        wl.kv_scale = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
        quantize_with_torch(wl)  # a library conversion, only to make the E4M3 input pool
    W.poison(wl)
    bt, cl = device_tables(wl, cuda_device)
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(48)
    sh = wl.shape
    # every query head of up to four sequences (the shortest and longest
    # among them), plus 64 random (sequence, head) pairs
    order = np.argsort(wl.context_lens)
    seqs = sorted({int(order[0]), int(order[min(1, len(order) - 1)]), int(order[-2 if len(order) > 1 else -1]),
                   int(order[-1])})
    pairs = [(s, h) for s in seqs for h in range(sh.num_q_heads)]
    pairs += [(int(rng.integers(sh.num_seqs)), int(rng.integers(sh.num_q_heads))) for _ in range(64)]
    pairs = np.array(pairs, np.int32)
    want = oracle_sampled(oracle, wl, pairs, wl.k_cache, wl.v_cache, wl.q)
    for ps in sizes:
        ref = torch.empty_like(wl.q)
        assert _reference_call(lib, wl, bt, cl, ps, ref, stream) == 0
        out = torch.full_like(wl.q, float("nan"))
        st = _static_call(lib, wl, bt, cl, ps, out, stream)
        assert st == 0, lib.pa_last_error()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"ps={ps}: differs from pa_decode"
        sel = out[torch.from_numpy(pairs[:, 0]).long().to(cuda_device),
                  torch.from_numpy(pairs[:, 1]).long().to(cuda_device)]
        compare(sel, want, what=f"static scratch ps={ps} vs oracle")
    flags = ctypes.c_uint(0)
    assert lib.pa_device_errors(ctypes.byref(flags), 1) == 0 and flags.value == 0


def test_static_workspace_refuses_oversized_calls(cuda_device):
    lib = _lib.load()
    wl = W.make("tiny", device=cuda_device)
    bt, cl = device_tables(wl, cuda_device)
    # 4 sequences with a table of 40000 blocks at 16-token partitions need
    # 4 * 8 * 40000 * 66 * 4 bytes of scratch, far beyond the fixed array.
    big = torch.full((4, 40000), -1, dtype=torch.int32, device=cuda_device)
    big[:, : bt.shape[1]] = bt
    out = torch.zeros_like(wl.q)
    sh = wl.shape
    need = lib.pa_decode_workspace_size(4, sh.num_q_heads, sh.head_dim, 40000, 16, 16)
    assert need > _lib.PA_STATIC_WORKSPACE_BYTES
    st = _static_call(lib, wl, big, cl, 16, out, torch.cuda.current_stream().cuda_stream)
    assert st == _lib.PA_ERR_WORKSPACE
    assert b"static scratch" in lib.pa_last_error()
    assert torch.count_nonzero(out) == 0
