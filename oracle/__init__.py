"""fp64 CPU oracle for paged decode attention and the KV-cache append step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference legs of ``bench.py`` may import this package.
The GPU library never calls it and it never calls the GPU library.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64); this module only
marshals numpy arrays through ctypes.  Every function states which passage
of the source pages it follows; see the C file's header for the readings
taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.  ``path`` selects
    another compiled copy, which the mutation tests use."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.pa_oracle_bf16_to_double.restype = D
    lib.pa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.pa_oracle_e4m3_to_double.restype = D
    lib.pa_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.pa_oracle_e4m3_from_float.restype = ctypes.c_uint8
    lib.pa_oracle_e4m3_from_float.argtypes = [ctypes.c_float]
    lib.pa_oracle_kv_bytes_per_token.restype = ctypes.c_int64
    lib.pa_oracle_kv_bytes_per_token.argtypes = [ctypes.c_int64] * 4
    lib.pa_oracle_slot_mapping.restype = None
    lib.pa_oracle_slot_mapping.argtypes = [P, I, P, I, I, P]
    lib.pa_oracle_cache_append.restype = None
    lib.pa_oracle_cache_append.argtypes = [P, P, P, I, P, P, I, I, I, I, ctypes.c_float]
    lib.pa_oracle_decode.restype = None
    lib.pa_oracle_decode.argtypes = [P, P, P, P, I, P, I, I, I, I, I, D, I, D, P]
    lib.pa_oracle_decode_pairs.restype = None
    lib.pa_oracle_decode_pairs.argtypes = [P, P, P, P, I, P, I, I, I, I, D, I, D, P, I, P]
    lib.pa_oracle_decode_partitions.restype = None
    lib.pa_oracle_decode_partitions.argtypes = [P, P, P, P, I, P, I, I, I, I, I, D, I, D,
                                                I, I, P, P, P]
    lib.pa_oracle_merge_partitions.restype = None
    lib.pa_oracle_merge_partitions.argtypes = [P, P, P, P, I, I, I, I, I, P]
    lib.pa_oracle_cache_append_scaled.restype = None
    lib.pa_oracle_cache_append_scaled.argtypes = [P, P, P, I, P, P, I, I, I, P, P]
    lib.pa_oracle_decode_scaled.restype = None
    lib.pa_oracle_decode_scaled.argtypes = [P, P, P, P, I, P, I, I, I, I, I, D, P, P, P, I, P]
    lib.pa_oracle_decode_fp8_qk.restype = None
    lib.pa_oracle_decode_fp8_qk.argtypes = [P, P, P, P, I, P, I, I, I, I, I, D, ctypes.c_float, P, P, P,
                                            I, P]
    lib.pa_oracle_block_alloc.restype = I
    lib.pa_oracle_block_alloc.argtypes = [P, I, P, I, I, P, P, P, I, P, P, I, I, I, P]
    lib.pa_oracle_prefill_scaled.restype = None
    lib.pa_oracle_prefill_scaled.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, D, P, P, P]
    lib.pa_oracle_block_alloc_chunk.restype = I
    lib.pa_oracle_block_alloc_chunk.argtypes = [P, I, P, P, I, I, P, P, P, I, P, P, I, I, I, P]
    lib.pa_oracle_chunk_slot_mapping.restype = None
    lib.pa_oracle_chunk_slot_mapping.argtypes = [P, I, P, P, I, I, P]
    lib.pa_oracle_prefill.restype = None
    lib.pa_oracle_prefill.argtypes = [P, P, P, P, I, P, P, I, I, I, I, I, D, I, D, P]
    lib.pa_oracle_set_threads.restype = None
    lib.pa_oracle_set_threads.argtypes = [I]
    lib.pa_oracle_get_threads.restype = I
    lib.pa_oracle_get_threads.argtypes = []
    return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """numpy front end over one compiled copy of the oracle."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    # -- number formats ----------------------------------------------------
    def bf16_to_double(self, bits: int) -> float:
        return self.lib.pa_oracle_bf16_to_double(int(bits) & 0xFFFF)

    def e4m3_to_double(self, code: int) -> float:
        """OCP E4M3 decoding (the FP8 format named in "Optimizing Llama 3.1 405B
        Inference with vLLM PagedAttention", section "Quantization Without
        Quality Loss")."""
        return self.lib.pa_oracle_e4m3_to_double(int(code) & 0xFF)

    def e4m3_from_float(self, x: float) -> int:
        """Round-to-nearest-even, saturating E4M3 encoding of a binary32."""
        return int(self.lib.pa_oracle_e4m3_from_float(float(np.float32(x))))

    def kv_bytes_per_token(self, num_layers, num_kv_heads, head_dim, bytes_per_elem) -> int:
        """Step 1 of the tuning guide: 2 * layers * KV heads * head_dim * bytes."""
        return int(self.lib.pa_oracle_kv_bytes_per_token(num_layers, num_kv_heads, head_dim,
                                                         bytes_per_elem))

    # -- the hot path --------------------------------------------------------
    def slot_mapping(self, block_tables: np.ndarray, context_lens: np.ndarray,
                     block_size: int) -> np.ndarray:
        """Slot of each sequence's newest token (position ctx - 1)."""
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        out = np.empty(cl.shape[0], np.int32)
        self.lib.pa_oracle_slot_mapping(_p(bt), bt.shape[1], _p(cl), cl.shape[0],
                                        block_size, _p(out))
        return out

    def cache_append(self, k_bits: np.ndarray, v_bits: np.ndarray, slot_mapping: np.ndarray,
                     k_cache: np.ndarray, v_cache: np.ndarray, block_size: int,
                     kv_dtype: int, scale: float) -> None:
        """In-place scatter of new K/V rows (bf16 bits [T, Hkv, D]) into the
        caches ([NB, Hkv, B, D] as uint16 for bf16 or uint8 for e4m3)."""
        k = _c(k_bits, np.uint16)
        v = _c(v_bits, np.uint16)
        sm = _c(slot_mapping, np.int32)
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        want = np.uint16 if kv_dtype == 0 else np.uint8
        assert k_cache.dtype == want and v_cache.dtype == want
        T, Hkv, D = k.shape
        self.lib.pa_oracle_cache_append(_p(k), _p(v), _p(sm), T, _p(k_cache), _p(v_cache),
                                        Hkv, D, block_size, kv_dtype, float(np.float32(scale)))

    def decode(self, q_bits, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
               block_size, softmax_scale, kv_dtype=0, kv_scale=1.0) -> np.ndarray:
        """fp64 [S, Hq, D] decode attention through the block table."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        S, Hq, D = q.shape
        out = np.zeros((S, Hq, D), np.float64)
        self.lib.pa_oracle_decode(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), S, Hq,
                                  num_kv_heads, D, block_size, float(softmax_scale), kv_dtype,
                                  float(kv_scale), _p(out))
        return out

    def decode_pairs(self, q_bits, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                     block_size, softmax_scale, pairs, kv_dtype=0, kv_scale=1.0) -> np.ndarray:
        """fp64 [n, D] outputs for the listed (sequence, query head) pairs."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        pr = _c(pairs, np.int32).reshape(-1, 2)
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        S, Hq, D = q.shape
        out = np.zeros((pr.shape[0], D), np.float64)
        self.lib.pa_oracle_decode_pairs(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), Hq,
                                        num_kv_heads, D, block_size, float(softmax_scale),
                                        kv_dtype, float(kv_scale), _p(pr), pr.shape[0], _p(out))
        return out

    def decode_partitions(self, q_bits, k_cache, v_cache, block_tables, context_lens,
                          num_kv_heads, block_size, softmax_scale, partition_size,
                          max_partitions, kv_dtype=0, kv_scale=1.0):
        """Per-partition (o, m, l), fp64, shapes [S,Hq,P,D], [S,Hq,P], [S,Hq,P]."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        S, Hq, D = q.shape
        o = np.zeros((S, Hq, max_partitions, D), np.float64)
        m = np.zeros((S, Hq, max_partitions), np.float64)
        l = np.zeros((S, Hq, max_partitions), np.float64)
        self.lib.pa_oracle_decode_partitions(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl),
                                             S, Hq, num_kv_heads, D, block_size,
                                             float(softmax_scale), kv_dtype, float(kv_scale),
                                             partition_size, max_partitions, _p(o), _p(m), _p(l))
        return o, m, l

    def merge_partitions(self, o, m, l, context_lens, partition_size) -> np.ndarray:
        """Log-sum-exp merge of fp32 partials -> fp64 [S, Hq, D]."""
        o = _c(o, np.float32)
        m = _c(m, np.float32)
        l = _c(l, np.float32)
        cl = _c(context_lens, np.int32)
        S, Hq, P, D = o.shape
        out = np.zeros((S, Hq, D), np.float64)
        self.lib.pa_oracle_merge_partitions(_p(o), _p(m), _p(l), _p(cl), S, Hq, D,
                                            partition_size, P, _p(out))
        return out

    # -- E4M3 with per-head K and V scales ---------------------------------------
    def cache_append_scaled(self, k_bits, v_bits, slot_mapping, k_cache, v_cache, block_size,
                            k_scales, v_scales) -> None:
        """In-place E4M3 append with scale k_scales[h] / v_scales[h] per KV head."""
        k = _c(k_bits, np.uint16)
        v = _c(v_bits, np.uint16)
        sm = _c(slot_mapping, np.int32)
        ks = _c(k_scales, np.float32)
        vs = _c(v_scales, np.float32)
        assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        T, Hkv, D = k.shape
        assert ks.shape == (Hkv,) and vs.shape == (Hkv,)
        self.lib.pa_oracle_cache_append_scaled(_p(k), _p(v), _p(sm), T, _p(k_cache), _p(v_cache),
                                               Hkv, D, block_size, _p(ks), _p(vs))

    def decode_scaled(self, q_bits, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                      block_size, softmax_scale, k_scales, v_scales, pairs=None) -> np.ndarray:
        """fp64 attention over an E4M3 cache with per-head scales: [S, Hq, D],
        or [n, D] for the given (sequence, query head) pairs."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
        ks = _c(k_scales, np.float32)
        vs = _c(v_scales, np.float32)
        S, Hq, D = q.shape
        if pairs is None:
            out = np.zeros((S, Hq, D), np.float64)
            self.lib.pa_oracle_decode_scaled(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), S,
                                             Hq, num_kv_heads, D, block_size, float(softmax_scale),
                                             _p(ks), _p(vs), None, 0, _p(out))
            return out
        pr = _c(pairs, np.int32).reshape(-1, 2)
        out = np.zeros((pr.shape[0], D), np.float64)
        self.lib.pa_oracle_decode_scaled(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), S, Hq,
                                         num_kv_heads, D, block_size, float(softmax_scale), _p(ks),
                                         _p(vs), _p(pr), pr.shape[0], _p(out))
        return out

    def decode_fp8_qk(self, q_bits, k_cache, v_cache, block_tables, context_lens, num_kv_heads,
                      block_size, softmax_scale, q_scale, k_scales, v_scales, pairs=None) -> np.ndarray:
        """As decode_scaled, with every query element first rounded to E4M3
        (e4m3(float(q) / q_scale), read back times q_scale)."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        kc = np.ascontiguousarray(k_cache, dtype=np.uint8)
        vc = np.ascontiguousarray(v_cache, dtype=np.uint8)
        ks = _c(k_scales, np.float32)
        vs = _c(v_scales, np.float32)
        S, Hq, D = q.shape
        if pairs is None:
            pr, n = None, S * Hq
            out = np.zeros((S, Hq, D), np.float64)
        else:
            pr = _c(pairs, np.int32).reshape(-1, 2)
            n = pr.shape[0]
            out = np.zeros((n, D), np.float64)
        self.lib.pa_oracle_decode_fp8_qk(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), S, Hq,
                                         num_kv_heads, D, block_size, float(softmax_scale),
                                         float(q_scale), _p(ks), _p(vs),
                                         _p(pr) if pr is not None else None, n if pr is not None else 0,
                                         _p(out))
        return out

    # -- chunked prefill ------------------------------------------------------
    def chunk_slot_mapping(self, block_tables, context_lens, query_start, block_size):
        """int32 [Tq] slots of every chunk token (the chunk ends the context)."""
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        qs = _c(query_start, np.int32)
        out = np.empty(int(qs[-1]), np.int32)
        self.lib.pa_oracle_chunk_slot_mapping(_p(bt), bt.shape[1], _p(cl), _p(qs), cl.shape[0],
                                              block_size, _p(out))
        return out

    def prefill(self, q_bits, k_cache, v_cache, block_tables, context_lens, query_start,
                num_kv_heads, block_size, softmax_scale, kv_dtype=0, kv_scale=1.0) -> np.ndarray:
        """fp64 [Tq, Hq, D]: causal attention of every chunk token over its
        sequence's cached tokens up to and including itself."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        qs = _c(query_start, np.int32)
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        T, Hq, D = q.shape
        out = np.zeros((T, Hq, D), np.float64)
        self.lib.pa_oracle_prefill(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), _p(qs),
                                   cl.shape[0], Hq, num_kv_heads, D, block_size,
                                   float(softmax_scale), kv_dtype, float(kv_scale), _p(out))
        return out

    def prefill_scaled(self, q_bits, k_cache, v_cache, block_tables, context_lens, query_start,
                       num_kv_heads, block_size, softmax_scale, k_scales, v_scales) -> np.ndarray:
        """fp64 [Tq, Hq, D]: chunked prefill over an E4M3 cache with a K and
        a V scale per KV head."""
        q = _c(q_bits, np.uint16)
        bt = _c(block_tables, np.int32)
        cl = _c(context_lens, np.int32)
        qs = _c(query_start, np.int32)
        kc = np.ascontiguousarray(k_cache)
        vc = np.ascontiguousarray(v_cache)
        ks = _c(k_scales, np.float32)
        vs = _c(v_scales, np.float32)
        T, Hq, D = q.shape
        out = np.zeros((T, Hq, D), np.float64)
        self.lib.pa_oracle_prefill_scaled(_p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), _p(qs),
                                          cl.shape[0], Hq, num_kv_heads, D, block_size, float(softmax_scale),
                                          _p(ks), _p(vs), _p(out))
        return out

    # -- block allocation with copy-on-write ------------------------------------
    def block_alloc(self, block_tables, context_lens, block_size, free_blocks, free_count,
                    refcounts, k_cache, v_cache):
        """In place on every array: fresh blocks for tokens that open a block,
        copy-on-write for tokens written into a shared block.  Returns
        (status, free_count, cow_src)."""
        for a, dt in ((block_tables, np.int32), (free_blocks, np.int32), (refcounts, np.int32)):
            assert a.dtype == dt and a.flags.c_contiguous
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        cl = _c(context_lens, np.int32)
        S, MB = block_tables.shape
        NB, Hkv, B, D = k_cache.shape
        elem = k_cache.dtype.itemsize
        fc = np.array([free_count], np.int32)
        cow = np.empty(S, np.int32)
        st = self.lib.pa_oracle_block_alloc(_p(block_tables), MB, _p(cl), S, block_size,
                                            _p(free_blocks), _p(fc), _p(refcounts), NB,
                                            _p(k_cache.view(np.uint8)), _p(v_cache.view(np.uint8)),
                                            Hkv, D, elem, _p(cow))
        return int(st), int(fc[0]), cow

    def block_alloc_chunk(self, block_tables, context_lens, query_start, block_size, free_blocks,
                          free_count, refcounts, k_cache, v_cache):
        """In place, for a chunk of new tokens per sequence (context_lens
        counts them): copy-on-write of a shared, partly filled last block,
        fresh blocks for every further block the chunk reaches.  Returns
        (status, free_count, cow_src)."""
        for a, dt in ((block_tables, np.int32), (free_blocks, np.int32), (refcounts, np.int32)):
            assert a.dtype == dt and a.flags.c_contiguous
        assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
        cl = _c(context_lens, np.int32)
        qs = _c(query_start, np.int32)
        S, MB = block_tables.shape
        NB, Hkv, B, D = k_cache.shape
        elem = k_cache.dtype.itemsize
        fc = np.array([free_count], np.int32)
        cow = np.empty(S, np.int32)
        st = self.lib.pa_oracle_block_alloc_chunk(_p(block_tables), MB, _p(cl), _p(qs), S, block_size,
                                                  _p(free_blocks), _p(fc), _p(refcounts), NB,
                                                  _p(k_cache.view(np.uint8)), _p(v_cache.view(np.uint8)),
                                                  Hkv, D, elem, _p(cow))
        return int(st), int(fc[0]), cow

    # -- threads -------------------------------------------------------------
    def set_threads(self, n: int) -> None:
        self.lib.pa_oracle_set_threads(int(n))

    def threads(self) -> int:
        return int(self.lib.pa_oracle_get_threads())
