"""Thin PyTorch binding of the C ABI (``include/pa.h``).

Only argument marshalling lives here: tensors are checked for device, dtype
and layout, then their device pointers, sizes and the current CUDA stream are
passed to ``libpa.so``.  Every step of the computation runs in the library's
kernels; there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib
from ._lib import PA_KV_BF16, PA_KV_FP8_E4M3


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(message)


def _lib_handle():
    return _lib.load()


def _check(status: int) -> None:
    if status != _lib.PA_OK:
        lib = _lib_handle()
        what = lib.pa_status_string(status).decode()
        detail = lib.pa_last_error().decode()
        raise PagedAttentionError(status, f"{what}: {detail}")


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _need(t: torch.Tensor, name: str, dtypes, ndim: int | None = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}; expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions (got shape {tuple(t.shape)})")


_CACHE_DTYPES = {PA_KV_BF16: (torch.bfloat16,), PA_KV_FP8_E4M3: (torch.uint8, torch.float8_e4m3fn)}


def cache_dtype_of(cache: torch.Tensor) -> int:
    return PA_KV_BF16 if cache.dtype == torch.bfloat16 else PA_KV_FP8_E4M3


def slot_mapping(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int,
                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """int32 [S] slot of each sequence's newest token (-1 for empty ones)."""
    _need(block_tables, "block_tables", (torch.int32,), 2)
    _need(context_lens, "context_lens", (torch.int32,), 1)
    S, MB = block_tables.shape
    if out is None:
        out = torch.empty(S, dtype=torch.int32, device=block_tables.device)
    _need(out, "out", (torch.int32,), 1)
    _check(_lib_handle().pa_slot_mapping(block_tables.data_ptr(), MB, context_lens.data_ptr(), S,
                                         block_size, out.data_ptr(), _stream(stream)))
    return out


def cache_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float = 1.0,
                 stream=None) -> None:
    """Write token i's K/V rows (bf16 [T, Hkv, D]) into slot slot_mapping[i]
    of the caches ([NB, Hkv, B, D], bf16 or E4M3 bytes); in place."""
    _need(k, "k", (torch.bfloat16,), 3)
    _need(v, "v", (torch.bfloat16,), 3)
    _need(slot_mapping, "slot_mapping", (torch.int32,), 1)
    kv_dtype = cache_dtype_of(k_cache)
    _need(k_cache, "k_cache", _CACHE_DTYPES[kv_dtype], 4)
    _need(v_cache, "v_cache", _CACHE_DTYPES[kv_dtype], 4)
    T, Hkv, D = k.shape
    NB, Hkv2, B, D2 = k_cache.shape
    if (Hkv2, D2) != (Hkv, D) or v.shape != k.shape or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent K/V and cache shapes")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    _check(_lib_handle().pa_cache_append(k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                                         k_cache.data_ptr(), v_cache.data_ptr(), NB, Hkv, D, B,
                                         kv_dtype, float(scale), _stream(stream)))


def max_partitions(max_blocks_per_seq: int, block_size: int, partition_size: int) -> int:
    return int(_lib_handle().pa_decode_max_partitions(max_blocks_per_seq, block_size, partition_size))


def workspace_size(num_seqs: int, num_q_heads: int, head_dim: int, max_blocks_per_seq: int,
                   block_size: int, partition_size: int) -> int:
    return int(_lib_handle().pa_decode_workspace_size(num_seqs, num_q_heads, head_dim,
                                                      max_blocks_per_seq, block_size,
                                                      partition_size))


def alloc_workspace(q: torch.Tensor, block_tables: torch.Tensor, block_size: int,
                    partition_size: int) -> torch.Tensor | None:
    S, Hq, D = q.shape
    n = workspace_size(S, Hq, D, block_tables.shape[1], block_size, partition_size)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=q.device)


def _decode_common(q, k_cache, v_cache, block_tables, context_lens):
    _need(q, "q", (torch.bfloat16,), 3)
    kv_dtype = cache_dtype_of(k_cache)
    _need(k_cache, "k_cache", _CACHE_DTYPES[kv_dtype], 4)
    _need(v_cache, "v_cache", _CACHE_DTYPES[kv_dtype], 4)
    _need(block_tables, "block_tables", (torch.int32,), 2)
    _need(context_lens, "context_lens", (torch.int32,), 1)
    S, Hq, D = q.shape
    NB, Hkv, B, D2 = k_cache.shape
    if D2 != D or v_cache.shape != k_cache.shape:
        raise ValueError("inconsistent q / cache shapes")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables and context_lens need one row per sequence")
    return kv_dtype, S, Hq, D, NB, Hkv, B


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables: torch.Tensor, context_lens: torch.Tensor, softmax_scale: float | None = None,
           kv_scale: float = 1.0, partition_size: int = 0, workspace: torch.Tensor | None = None,
           out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Paged decode attention; returns bf16 [S, Hq, D].  ``partition_size``
    0 = one pass per (sequence, KV head); > 0 = split context + merge."""
    kv_dtype, S, Hq, D, NB, Hkv, B = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (torch.bfloat16,), 3)
    if partition_size and workspace is None:
        workspace = alloc_workspace(q, block_tables, B, partition_size)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib_handle().pa_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   block_tables.data_ptr(), block_tables.shape[1],
                                   context_lens.data_ptr(), S, Hq, Hkv, D, NB, B, kv_dtype,
                                   float(kv_scale), float(softmax_scale), int(partition_size),
                                   ws_ptr, ws_bytes, out.data_ptr(), _stream(stream)))
    return out


def decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor,
                v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                softmax_scale: float | None = None, kv_scale: float = 1.0, partition_size: int = 0,
                workspace: torch.Tensor | None = None, slot_mapping: torch.Tensor | None = None,
                out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One fused decode step: append each sequence's new K/V row at position
    ctx - 1, then attend over the ctx tokens.  Returns bf16 [S, Hq, D]."""
    kv_dtype, S, Hq, D, NB, Hkv, B = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    _need(k_new, "k_new", (torch.bfloat16,), 3)
    _need(v_new, "v_new", (torch.bfloat16,), 3)
    if tuple(k_new.shape) != (S, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs, num_kv_heads, head_dim]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", (torch.bfloat16,), 3)
    if slot_mapping is not None:
        _need(slot_mapping, "slot_mapping", (torch.int32,), 1)
    if partition_size and workspace is None:
        workspace = alloc_workspace(q, block_tables, B, partition_size)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(_lib_handle().pa_decode_step(
        q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
        block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), S, Hq, Hkv, D, NB,
        B, kv_dtype, float(kv_scale), float(softmax_scale), int(partition_size), ws_ptr, ws_bytes,
        slot_mapping.data_ptr() if slot_mapping is not None else None, out.data_ptr(),
        _stream(stream)))
    return out


def cache_append_scaled(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, k_scales: torch.Tensor,
                        v_scales: torch.Tensor, stream=None) -> None:
    """E4M3 append with a scale per KV head for K (``k_scales``) and for V
    (``v_scales``), float32 device tensors [num_kv_heads]; in place."""
    _need(k, "k", (torch.bfloat16,), 3)
    _need(v, "v", (torch.bfloat16,), 3)
    _need(slot_mapping, "slot_mapping", (torch.int32,), 1)
    _need(k_cache, "k_cache", _CACHE_DTYPES[PA_KV_FP8_E4M3], 4)
    _need(v_cache, "v_cache", _CACHE_DTYPES[PA_KV_FP8_E4M3], 4)
    T, Hkv, D = k.shape
    NB, Hkv2, B, D2 = k_cache.shape
    _need(k_scales, "k_scales", (torch.float32,), 1)
    _need(v_scales, "v_scales", (torch.float32,), 1)
    if (Hkv2, D2) != (Hkv, D) or k_scales.shape[0] != Hkv or v_scales.shape[0] != Hkv:
        raise ValueError("inconsistent shapes")
    _check(_lib_handle().pa_cache_append_scaled(
        k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T, k_cache.data_ptr(),
        v_cache.data_ptr(), NB, Hkv, D, B, k_scales.data_ptr(), v_scales.data_ptr(),
        _stream(stream)))


def decode_step_scaled(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, k_scales,
                       v_scales, softmax_scale=None, partition_size=0, workspace=None,
                       slot_mapping=None, out=None, stream=None, q_scale=None) -> torch.Tensor:
    """Fused decode step over an E4M3 cache with per-KV-head K and V scales.
    ``k_new``/``v_new`` may both be None: attention without an append.
    ``q_scale`` (a positive float) rounds the query to E4M3 with that scale
    and takes the scores as an E4M3 x E4M3 product (pa_decode_step_fp8_qk)."""
    kv_dtype, S, Hq, D, NB, Hkv, B = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    if kv_dtype != PA_KV_FP8_E4M3:
        raise TypeError("per-head scales need an E4M3 cache")
    _need(k_scales, "k_scales", (torch.float32,), 1)
    _need(v_scales, "v_scales", (torch.float32,), 1)
    if k_new is not None:
        _need(k_new, "k_new", (torch.bfloat16,), 3)
        _need(v_new, "v_new", (torch.bfloat16,), 3)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if partition_size and workspace is None:
        workspace = alloc_workspace(q, block_tables, B, partition_size)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    lead = (q.data_ptr(), k_new.data_ptr() if k_new is not None else None,
            v_new.data_ptr() if v_new is not None else None, k_cache.data_ptr(), v_cache.data_ptr(),
            block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(), S, Hq, Hkv, D,
            NB, B, k_scales.data_ptr(), v_scales.data_ptr())
    tail = (float(softmax_scale), int(partition_size), ws_ptr, ws_bytes,
            slot_mapping.data_ptr() if slot_mapping is not None else None, out.data_ptr(),
            _stream(stream))
    if q_scale is None:
        _check(_lib_handle().pa_decode_step_scaled(*lead, *tail))
    else:
        _check(_lib_handle().pa_decode_step_fp8_qk(*lead, float(q_scale), *tail))
    return out


def chunk_slot_mapping(block_tables, context_lens, query_start, block_size, out=None,
                       stream=None) -> torch.Tensor:
    """int32 slots of every chunk token (chunks end their contexts)."""
    _need(block_tables, "block_tables", (torch.int32,), 2)
    _need(context_lens, "context_lens", (torch.int32,), 1)
    _need(query_start, "query_start", (torch.int32,), 1)
    S, MB = block_tables.shape
    if out is None:
        out = torch.empty(int(query_start[-1].item()), dtype=torch.int32, device=block_tables.device)
    _check(_lib_handle().pa_chunk_slot_mapping(block_tables.data_ptr(), MB, context_lens.data_ptr(),
                                               query_start.data_ptr(), S, block_size,
                                               out.data_ptr(), _stream(stream)))
    return out


def prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, max_query_len,
            softmax_scale=None, out=None, stream=None, kernel="auto", kv_scale=1.0) -> torch.Tensor:
    """Chunked prefill attention: bf16 [T, Hq, D] for the chunk rows q.
    ``kernel`` "auto" (tensor-memory kernel) or "mma" (warp-level MMA
    kernel, bf16 caches only).  An E4M3 cache (uint8) holds x / kv_scale."""
    _need(q, "q", (torch.bfloat16,), 3)
    _need(query_start, "query_start", (torch.int32,), 1)
    kv_dtype = cache_dtype_of(k_cache)
    _need(k_cache, "k_cache", _CACHE_DTYPES[kv_dtype], 4)
    _need(v_cache, "v_cache", _CACHE_DTYPES[kv_dtype], 4)
    _need(block_tables, "block_tables", (torch.int32,), 2)
    _need(context_lens, "context_lens", (torch.int32,), 1)
    T, Hq, D = q.shape
    NB, Hkv, B, _ = k_cache.shape
    S = context_lens.shape[0]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    fn = _lib_handle().pa_prefill if kernel == "auto" else _lib_handle().pa_prefill_mma
    _check(fn(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
              block_tables.shape[1], context_lens.data_ptr(), query_start.data_ptr(), S, T,
              int(max_query_len), Hq, Hkv, D, NB, B, kv_dtype, float(kv_scale), float(softmax_scale),
              out.data_ptr(), _stream(stream)))
    return out


def prefill_scaled(q, k_cache, v_cache, block_tables, context_lens, query_start, max_query_len,
                   k_scales, v_scales, softmax_scale=None, out=None, stream=None) -> torch.Tensor:
    """Chunked prefill over an E4M3 cache (uint8) holding x / scale[h], with
    a K and a V scale per KV head (float32 device tensors [num_kv_heads])."""
    _need(q, "q", (torch.bfloat16,), 3)
    _need(query_start, "query_start", (torch.int32,), 1)
    _need(k_cache, "k_cache", (torch.uint8,), 4)
    _need(v_cache, "v_cache", (torch.uint8,), 4)
    _need(block_tables, "block_tables", (torch.int32,), 2)
    _need(context_lens, "context_lens", (torch.int32,), 1)
    _need(k_scales, "k_scales", (torch.float32,), 1)
    _need(v_scales, "v_scales", (torch.float32,), 1)
    T, Hq, D = q.shape
    NB, Hkv, B, _ = k_cache.shape
    S = context_lens.shape[0]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _check(_lib_handle().pa_prefill_scaled(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
        context_lens.data_ptr(), query_start.data_ptr(), S, T, int(max_query_len), Hq, Hkv, D, NB, B,
        k_scales.data_ptr(), v_scales.data_ptr(), float(softmax_scale), out.data_ptr(), _stream(stream)))
    return out


class DeviceBlockPool:
    """Device-side free stack and reference counts of a paged cache's blocks,
    driven by ``pa_block_alloc``.  Build it from the host state once
    (``free`` = the free block ids in stack order, ``refcounts`` per block);
    afterwards every step allocates on the device."""

    def __init__(self, free, refcounts, device):
        NB = len(refcounts)
        self.free_blocks = torch.zeros(NB, dtype=torch.int32, device=device)
        self.free_blocks[: len(free)] = torch.as_tensor(free, dtype=torch.int32)
        self.free_count = torch.tensor([len(free)], dtype=torch.int32, device=device)
        self.refcounts = torch.as_tensor(refcounts, dtype=torch.int32).to(device).contiguous()
        self.num_blocks = NB

    def allocate(self, block_tables, context_lens, k_cache, v_cache, advance=False, cow_src=None,
                 stream=None) -> torch.Tensor:
        """Fresh blocks / copy-on-write for each sequence's newest token (see
        pa_block_alloc); returns cow_src (int32 [S])."""
        _need(block_tables, "block_tables", (torch.int32,), 2)
        _need(context_lens, "context_lens", (torch.int32,), 1)
        kv_dtype = cache_dtype_of(k_cache)
        NB, Hkv, B, D = k_cache.shape
        S, MB = block_tables.shape
        if cow_src is None:
            cow_src = torch.empty(S, dtype=torch.int32, device=block_tables.device)
        _check(_lib_handle().pa_block_alloc(
            block_tables.data_ptr(), MB, context_lens.data_ptr(), S, B, 1 if advance else 0,
            self.free_blocks.data_ptr(), self.free_count.data_ptr(), self.refcounts.data_ptr(), NB,
            k_cache.data_ptr(), v_cache.data_ptr(), Hkv, D, kv_dtype, cow_src.data_ptr(),
            _stream(stream)))
        return cow_src

    def allocate_chunk(self, block_tables, context_lens, query_start, k_cache, v_cache, cow_src=None,
                       stream=None) -> torch.Tensor:
        """Fresh blocks / copy-on-write for a chunk of new tokens per sequence
        (see pa_block_alloc_chunk; context_lens counts the chunk); returns
        cow_src (int32 [S])."""
        _need(block_tables, "block_tables", (torch.int32,), 2)
        _need(context_lens, "context_lens", (torch.int32,), 1)
        _need(query_start, "query_start", (torch.int32,), 1)
        kv_dtype = cache_dtype_of(k_cache)
        NB, Hkv, B, D = k_cache.shape
        S, MB = block_tables.shape
        if cow_src is None:
            cow_src = torch.empty(S, dtype=torch.int32, device=block_tables.device)
        _check(_lib_handle().pa_block_alloc_chunk(
            block_tables.data_ptr(), MB, context_lens.data_ptr(), query_start.data_ptr(), S, B,
            self.free_blocks.data_ptr(), self.free_count.data_ptr(), self.refcounts.data_ptr(), NB,
            k_cache.data_ptr(), v_cache.data_ptr(), Hkv, D, kv_dtype, cow_src.data_ptr(),
            _stream(stream)))
        return cow_src


def decode_partitions(q, k_cache, v_cache, block_tables, context_lens, softmax_scale, kv_scale,
                      partition_size, workspace, stream=None) -> None:
    """Per-partition (o, m, l) into ``workspace`` (layout in include/pa.h)."""
    kv_dtype, S, Hq, D, NB, Hkv, B = _decode_common(q, k_cache, v_cache, block_tables, context_lens)
    _check(_lib_handle().pa_decode_partitions(
        q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], context_lens.data_ptr(), S, Hq, Hkv, D, NB, B, kv_dtype,
        float(kv_scale), float(softmax_scale), int(partition_size), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def decode_reduce(workspace: torch.Tensor, context_lens: torch.Tensor, num_q_heads: int,
                  head_dim: int, max_blocks_per_seq: int, block_size: int, partition_size: int,
                  out: torch.Tensor, stream=None) -> torch.Tensor:
    """Log-sum-exp merge of the workspace partitions into bf16 ``out``."""
    _need(context_lens, "context_lens", (torch.int32,), 1)
    _need(out, "out", (torch.bfloat16,), 3)
    S = context_lens.shape[0]
    _check(_lib_handle().pa_decode_reduce(workspace.data_ptr(),
                                          workspace.numel() * workspace.element_size(),
                                          context_lens.data_ptr(), S, num_q_heads, head_dim,
                                          max_blocks_per_seq, block_size, partition_size,
                                          out.data_ptr(), _stream(stream)))
    return out


def workspace_views(workspace: torch.Tensor, num_seqs: int, num_q_heads: int, head_dim: int,
                    parts: int):
    """(o, m, l) fp32 views of a workspace: [S,Hq,P,D], [S,Hq,P], [S,Hq,P]."""
    f = workspace.view(torch.float32)
    n = num_seqs * num_q_heads * parts
    o = f[: n * head_dim].view(num_seqs, num_q_heads, parts, head_dim)
    m = f[n * head_dim: n * head_dim + n].view(num_seqs, num_q_heads, parts)
    l = f[n * head_dim + n: n * head_dim + 2 * n].view(num_seqs, num_q_heads, parts)
    return o, m, l


def device_errors(clear: bool = True) -> int:
    """PA_DEVERR_* bits set by kernels since the last clear (synchronises)."""
    flags = ctypes.c_uint(0)
    _check(_lib_handle().pa_device_errors(ctypes.byref(flags), 1 if clear else 0))
    return int(flags.value)


class DecodeStep:
    """One decode step of one attention layer over a paged cache, with every
    buffer allocated up front: slot mapping of the newest tokens, append of
    their K/V, partitioned attention and (when split) the merge.  Calling it
    allocates nothing.  ``fused`` (default) runs ``pa_decode_step``: 1 kernel,
    2 when split; otherwise the separate entry points: 3 kernels, 4 when
    split."""

    def __init__(self, k_cache, v_cache, block_tables, context_lens, num_q_heads,
                 softmax_scale=None, kv_scale=1.0, partition_size=0, fused=True,
                 k_scales=None, v_scales=None, q_scale=None):
        self.fused = fused
        # q_scale: E4M3 query and E4M3 x E4M3 scores (pa_decode_step_fp8_qk);
        # with one cache scale, every head gets it
        self.q_scale = q_scale
        if q_scale is not None and k_scales is None:
            k_scales = torch.full((k_cache.shape[1],), float(kv_scale), dtype=torch.float32,
                                  device=k_cache.device)
            v_scales = k_scales
        # per-KV-head E4M3 scales (device float32 [Hkv]); fused path only
        self.k_scales, self.v_scales = k_scales, v_scales
        if k_scales is not None and not fused:
            raise ValueError("per-head scales run through the fused step")
        self.k_cache, self.v_cache = k_cache, v_cache
        self.block_tables, self.context_lens = block_tables, context_lens
        NB, self.Hkv, self.B, self.D = k_cache.shape
        self.S = block_tables.shape[0]
        self.Hq = num_q_heads
        self.softmax_scale = softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(self.D)
        self.kv_scale = kv_scale
        self.partition_size = partition_size
        dev = k_cache.device
        self.slots = torch.empty(self.S, dtype=torch.int32, device=dev)
        self.out = torch.empty(self.S, self.Hq, self.D, dtype=torch.bfloat16, device=dev)
        n = workspace_size(self.S, self.Hq, self.D, block_tables.shape[1], self.B, partition_size)
        self.workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)

    def append(self, k_new, v_new, stream=None):
        slot_mapping(self.block_tables, self.context_lens, self.B, out=self.slots, stream=stream)
        cache_append(k_new, v_new, self.slots, self.k_cache, self.v_cache, self.kv_scale, stream=stream)

    def attend(self, q, stream=None):
        if self.partition_size:
            decode_partitions(q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                              self.softmax_scale, self.kv_scale, self.partition_size,
                              self.workspace, stream=stream)
            decode_reduce(self.workspace, self.context_lens, self.Hq, self.D,
                          self.block_tables.shape[1], self.B, self.partition_size, self.out,
                          stream=stream)
        else:
            decode(q, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                   self.softmax_scale, self.kv_scale, 0, None, self.out, stream=stream)
        return self.out

    def launches(self) -> int:
        """Kernels one call launches."""
        return (1 if self.fused else 3) + (1 if self.partition_size else 0)

    def __call__(self, q, k_new, v_new, stream=None):
        if self.fused and self.k_scales is not None:
            return decode_step_scaled(q, k_new, v_new, self.k_cache, self.v_cache,
                                      self.block_tables, self.context_lens, self.k_scales,
                                      self.v_scales, self.softmax_scale, self.partition_size,
                                      self.workspace, self.slots, self.out, stream,
                                      q_scale=self.q_scale)
        if self.fused:
            return decode_step(q, k_new, v_new, self.k_cache, self.v_cache, self.block_tables,
                               self.context_lens, self.softmax_scale, self.kv_scale,
                               self.partition_size, self.workspace, self.slots, self.out, stream)
        self.append(k_new, v_new, stream)
        return self.attend(q, stream)


class StepGraph:
    """Several layers' decode steps captured into one CUDA graph.

    ``steps`` are ``DecodeStep`` objects (one per attention layer, each with
    its own cache) and ``inputs`` the matching ``(q, k_new, v_new)`` device
    buffers.  ``replay()`` re-runs every step with whatever those buffers, the
    context lengths and the block tables hold at that moment; nothing is
    re-encoded on the host, so the per-step host cost is one graph launch.
    One eager pass runs first (outside the capture) so that the library's
    once-per-device set-up never happens while a stream is being captured.
    """

    def __init__(self, steps, inputs):
        if len(steps) != len(inputs):
            raise ValueError("one (q, k_new, v_new) triple per step")
        self.steps = list(steps)
        self.inputs = list(inputs)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._run()

    def _run(self):
        for step, (q, k, v) in zip(self.steps, self.inputs):
            step(q, k, v)

    def launches(self) -> int:
        return sum(s.launches() for s in self.steps)

    def replay(self) -> None:
        self.graph.replay()
