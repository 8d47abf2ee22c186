"""Seeded synthetic inputs for paged decode attention.

This module is shared by the GPU tests, the benchmark and the oracle tests.
It holds no attention, softmax, quantisation or slot arithmetic: it draws
random numbers, builds block tables from a shuffled free list and poisons the
memory a correct kernel must never read.  Everything the method computes is
done either by the CUDA library or by the oracle, never here.

Workloads (seed = index unless given):
  0 ``tiny``        4 sequences, context lengths {1, 17, 100, 255}, 8 query / 2 KV
                    heads, head_dim 64, 16-token blocks, 64-block pool handed out
                    in a random permutation, bf16 N(0, 1) data.
  1 ``llama8b``     Llama-3-8B-shaped decode layer: 256 sequences, context
                    lengths uniform on [512, 2048], 32 / 8 heads, head_dim 128,
                    16-token blocks, pool of 1.2x the blocks needed, shuffled.
  2 ``long70b``     Llama-3.1-70B-head-shaped long decode: 64 sequences, context
                    uniform on [4096, 32768], 64 / 8 heads, head_dim 128,
                    16- or 32-token blocks, 512-token context partitions.
  3 ``prefix_fp8``  256 sequences sharing one 2048-token prefix (the same
                    physical blocks in every table) plus private suffixes
                    uniform on [64, 512], 32 / 8 heads, head_dim 128, 16-token
                    blocks, e4m3 KV with one per-tensor scale.
  4 ``ctx128k``     405B-head-shaped long context: 8 sequences at 131072 tokens,
                    128 / 8 heads (group 16), head_dim 128, 16-token blocks,
                    512-token partitions; each step appends one token per
                    sequence then attends.

Values are drawn N(0, 1) in fp32 and rounded to bf16 (torch generators: the
CPU generator for small pools, the CUDA generator for large ones; both sides
of a comparison are handed the same bits at run time).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0   # a quiet NaN in bfloat16
E4M3_NAN_CODE = 0x7F     # the E4M3 NaN code S.1111.111

KV_BF16 = 0
KV_FP8_E4M3 = 1

NAMES = ("tiny", "llama8b", "long70b", "prefix_fp8", "ctx128k")


@dataclass
class Shape:
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: int = KV_BF16
    partition_size: int = 0


@dataclass
class Workload:
    """One decode step's inputs.  ``context_lens`` already counts the token
    appended this step; its K/V rows are ``k_new``/``v_new`` and the caches
    hold every earlier token."""

    name: str
    shape: Shape
    num_blocks: int
    context_lens: np.ndarray          # int32 [S]
    block_tables: np.ndarray          # int32 [S, MB]; -1 past the context
    q: torch.Tensor                   # bf16 [S, Hq, D]
    k_new: torch.Tensor               # bf16 [S, Hkv, D]
    v_new: torch.Tensor               # bf16 [S, Hkv, D]
    k_cache: torch.Tensor             # bf16 or uint8 [NB, Hkv, B, D]
    v_cache: torch.Tensor
    softmax_scale: float
    kv_scale: float = 1.0
    seed: int = 0
    notes: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_bytes(self) -> int:
        """Algorithmic bytes one decode step reads: every live token's K and V
        once, for every KV head (the per-layer form of the tuning guide's
        Step 1 formula)."""
        elem = 2 if self.shape.kv_dtype == KV_BF16 else 1
        sh = self.shape
        return int(self.context_lens.astype(np.int64).sum()) * sh.num_kv_heads * sh.head_dim * 2 * elem

    def unique_kv_bytes(self) -> int:
        """Bytes of distinct cache rows referenced (a shared block counted once)."""
        sh = self.shape
        elem = 2 if sh.kv_dtype == KV_BF16 else 1
        rows_of = {}
        for s in range(sh.num_seqs):
            n = int(self.context_lens[s])
            for j in range((n + sh.block_size - 1) // sh.block_size):
                b = int(self.block_tables[s, j])
                used = min(sh.block_size, n - j * sh.block_size)
                rows_of[b] = max(rows_of.get(b, 0), used)
        return sum(rows_of.values()) * sh.num_kv_heads * sh.head_dim * 2 * elem


class BlockAllocator:
    """Host free list of physical blocks with reference counts.  Blocks are
    handed out in the order of a seeded shuffle, so consecutive logical blocks
    land on scattered physical blocks."""

    def __init__(self, num_blocks: int, rng: np.random.Generator | None):
        order = np.arange(num_blocks, dtype=np.int64)
        if rng is not None:
            order = rng.permutation(num_blocks)
        self._free = [int(b) for b in order[::-1]]
        self.refcount = np.zeros(num_blocks, np.int32)
        self.num_blocks = num_blocks

    def num_free(self) -> int:
        return len(self._free)

    def allocate(self, n: int = 1) -> list[int]:
        if n > len(self._free):
            raise MemoryError(f"block pool exhausted: want {n}, have {len(self._free)}")
        out = [self._free.pop() for _ in range(n)]
        for b in out:
            self.refcount[b] = 1
        return out

    def share(self, blocks) -> None:
        for b in blocks:
            assert self.refcount[b] > 0
            self.refcount[b] += 1

    def free(self, blocks) -> None:
        for b in blocks:
            assert self.refcount[b] > 0
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self._free.append(int(b))


def _blocks_for(n_tokens: int, block_size: int) -> int:
    return (n_tokens + block_size - 1) // block_size


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def build_tables(context_lens: np.ndarray, block_size: int, num_blocks: int,
                 rng: np.random.Generator | None, max_blocks_per_seq: int | None = None,
                 shared_prefix_blocks: int = 0):
    """Give each sequence ceil(ctx / B) blocks from a shuffled free list.
    With ``shared_prefix_blocks`` = n, the first n logical blocks of every
    sequence are the same n physical blocks.  Returns (tables, allocator)."""
    S = len(context_lens)
    need = [_blocks_for(int(c), block_size) for c in context_lens]
    mb = max_blocks_per_seq or max(1, max(need))
    tables = np.full((S, mb), -1, np.int32)
    alloc = BlockAllocator(num_blocks, rng)
    prefix = alloc.allocate(shared_prefix_blocks) if shared_prefix_blocks else []
    for s in range(S):
        row = []
        if shared_prefix_blocks:
            if s > 0:
                alloc.share(prefix)
            row = list(prefix)
        row += alloc.allocate(need[s] - len(row))
        tables[s, :len(row)] = row
    return tables, alloc


def poison(wl: Workload, pending: bool = False) -> None:
    """Fill every cache row a correct kernel must not read (blocks no table
    references, and the slots past the context in each sequence's last block)
    with NaN, in place.  With ``pending`` the newest token's slot (position
    ctx - 1, which this step's append must write) is poisoned too."""
    sh = wl.shape
    nan = BF16_NAN_BITS if sh.kv_dtype == KV_BF16 else E4M3_NAN_CODE
    used = np.zeros(wl.num_blocks, bool)
    live = np.zeros((wl.num_blocks, sh.block_size), bool)
    for s in range(sh.num_seqs):
        n = int(wl.context_lens[s])
        for j in range(_blocks_for(n, sh.block_size)):
            b = int(wl.block_tables[s, j])
            used[b] = True
            live[b, :min(sh.block_size, n - j * sh.block_size)] = True
        if pending and n > 0:
            b = int(wl.block_tables[s, (n - 1) // sh.block_size])
            live[b, (n - 1) % sh.block_size] = False
    dead = torch.from_numpy(~live).to(wl.k_cache.device)          # [NB, B]
    mask = dead[:, None, :, None].expand(-1, sh.num_kv_heads, -1, sh.head_dim)
    for c in (wl.k_cache, wl.v_cache):
        raw = c.view(torch.int16) if c.dtype == torch.bfloat16 else c
        fill = torch.tensor(nan if c.dtype != torch.bfloat16 else np.int16(np.uint16(nan).view(np.int16)),
                            dtype=raw.dtype, device=raw.device)
        raw.masked_fill_(mask, fill)
    wl.notes["poisoned"] = True


def bits(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a tensor's raw bits (uint16 for bf16, uint8 for bytes)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """Inverse of :func:`bits`."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)
    if a.dtype == np.uint8:
        return torch.from_numpy(a.copy()).to(device)
    raise TypeError(a.dtype)


def fp8_scale_from(*tensors: torch.Tensor) -> float:
    """Per-tensor scale: the largest magnitude of the data divided by the
    largest finite E4M3 value (448), as a float32."""
    amax = max(float(t.float().abs().max()) for t in tensors)
    return float(np.float32(amax) / np.float32(448.0))


def _finish(name, shape, ctx, tables, nb, device, seed, gen_device=None, kv_scale=None,
            fill_cache=True) -> Workload:
    gen_device = gen_device or device
    g = _generator(seed, gen_device)
    S, Hq, Hkv, D, B = shape.num_seqs, shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.block_size
    q = _randn_bf16((S, Hq, D), g, gen_device).to(device)
    k_new = _randn_bf16((S, Hkv, D), g, gen_device).to(device)
    v_new = _randn_bf16((S, Hkv, D), g, gen_device).to(device)
    if fill_cache:
        k_data = _randn_bf16((nb, Hkv, B, D), g, gen_device).to(device)
        v_data = _randn_bf16((nb, Hkv, B, D), g, gen_device).to(device)
    else:
        k_data = torch.zeros((nb, Hkv, B, D), dtype=torch.bfloat16, device=device)
        v_data = torch.zeros_like(k_data)
    wl = Workload(name=name, shape=shape, num_blocks=nb, context_lens=ctx.astype(np.int32),
                  block_tables=tables, q=q, k_new=k_new, v_new=v_new, k_cache=k_data,
                  v_cache=v_data, softmax_scale=1.0 / math.sqrt(D), seed=seed)
    if shape.kv_dtype == KV_FP8_E4M3:
        wl.kv_scale = kv_scale if kv_scale is not None else fp8_scale_from(k_data, v_data, k_new, v_new)
        # The bf16 values stay in k_cache/v_cache until a quantiser (the
        # oracle's encoder or the library's append) turns them into codes.
        wl.notes["fp8_source"] = "bf16 N(0,1) pool, quantised by the caller"
    return wl


def make(name: str, device="cpu", seed: int | None = None, block_size: int | None = None,
         num_seqs: int | None = None, fill_cache: bool = True, extra_steps: int = 0,
         data_seed: int | None = None) -> Workload:
    """Build workload ``name`` (see the module docstring).  ``num_seqs``
    shrinks a workload (same distributions) for quick tests or profiling;
    ``extra_steps`` reserves table capacity and pool blocks for that many more
    appended tokens per sequence (the long-context step workload).
    ``data_seed`` (default: ``seed``) seeds the values only, so several
    layers can share one set of contexts and block tables."""
    idx = NAMES.index(name)
    seed = idx if seed is None else seed
    rng = np.random.default_rng(seed)
    vseed = seed if data_seed is None else data_seed
    if name == "tiny":
        shape = Shape(num_seqs or 4, 8, 2, 64, block_size or 16)
        ctx = np.array([1, 17, 100, 255], np.int64)[: shape.num_seqs]
        nb = 64 + extra_steps * shape.num_seqs
        tables, alloc = build_tables(ctx, shape.block_size, nb, rng,
                                     _blocks_for(255 + extra_steps, shape.block_size))
        wl = _finish(name, shape, ctx, tables, nb, device, vseed, fill_cache=fill_cache)
        wl.notes["allocator"] = alloc
        return wl
    if name == "llama8b":
        shape = Shape(num_seqs or 256, 32, 8, 128, block_size or 16)
        ctx = rng.integers(512, 2048, size=shape.num_seqs, endpoint=True)
        mb = _blocks_for(2048 + extra_steps, shape.block_size)
    elif name == "long70b":
        shape = Shape(num_seqs or 64, 64, 8, 128, block_size or 16, partition_size=512)
        ctx = rng.integers(4096, 32768, size=shape.num_seqs, endpoint=True)
        mb = _blocks_for(32768 + extra_steps, shape.block_size)
    elif name == "prefix_fp8":
        shape = Shape(num_seqs or 256, 32, 8, 128, block_size or 16, kv_dtype=KV_FP8_E4M3)
        prefix = 2048
        suffix = rng.integers(64, 512, size=shape.num_seqs, endpoint=True)
        ctx = prefix + suffix
        mb = _blocks_for(prefix + 512 + extra_steps, shape.block_size)
        pb = prefix // shape.block_size
        need = pb + sum(_blocks_for(int(c) + extra_steps, shape.block_size) - pb for c in ctx)
        nb = math.ceil(1.2 * need)
        tables, alloc = build_tables(ctx, shape.block_size, nb, rng, mb, shared_prefix_blocks=pb)
        wl = _finish(name, shape, ctx, tables, nb, device, vseed, gen_device=device,
                     fill_cache=fill_cache)
        wl.notes["shared_prefix_tokens"] = prefix
        wl.notes["allocator"] = alloc
        return wl
    elif name == "ctx128k":
        shape = Shape(num_seqs or 8, 128, 8, 128, block_size or 16, partition_size=512)
        ctx = np.full(shape.num_seqs, 131072, np.int64)
        mb = _blocks_for(131072 + extra_steps, shape.block_size)
    else:
        raise KeyError(name)
    need = sum(_blocks_for(int(c) + extra_steps, shape.block_size) for c in ctx)
    nb = math.ceil(1.2 * need)
    tables, alloc = build_tables(ctx, shape.block_size, nb, rng, mb)
    wl = _finish(name, shape, ctx, tables, nb, device, vseed, fill_cache=fill_cache)
    wl.notes["allocator"] = alloc
    return wl


def sample_pairs(wl: Workload, n: int, seed: int = 1234) -> np.ndarray:
    """n distinct (sequence, query head) pairs, always including the first and
    last sequence and the last query head (the ragged tails)."""
    rng = np.random.default_rng(seed)
    S, Hq = wl.shape.num_seqs, wl.shape.num_q_heads
    total = S * Hq
    picks = set([0, total - 1, (S - 1) * Hq, Hq - 1])
    while len(picks) < min(n, total):
        picks.add(int(rng.integers(0, total)))
    flat = np.array(sorted(picks), np.int64)
    return np.stack([flat // Hq, flat % Hq], axis=1).astype(np.int32)


@dataclass
class PrefillWorkload:
    """One chunked-prefill step: sequence s brings the chunk rows
    [query_start[s], query_start[s+1]) at the end of its context; the cache
    holds the prefix, the chunk's own K/V are ``k_new``/``v_new``."""

    shape: Shape
    num_blocks: int
    context_lens: np.ndarray      # int32 [S], prefix + chunk
    query_start: np.ndarray       # int32 [S + 1]
    block_tables: np.ndarray      # int32 [S, MB]
    q: torch.Tensor               # bf16 [T, Hq, D]
    k_new: torch.Tensor           # bf16 [T, Hkv, D]
    v_new: torch.Tensor
    k_cache: torch.Tensor         # bf16 [NB, Hkv, B, D]
    v_cache: torch.Tensor
    softmax_scale: float
    seed: int = 0

    @property
    def max_query_len(self) -> int:
        return int(np.diff(self.query_start).max()) if len(self.context_lens) else 0

    def attention_flops(self) -> int:
        """Multiply-adds x2 of QK^T and PV over the (query, key) pairs the
        causal mask keeps: 4 * D * Hq per pair."""
        sh = self.shape
        pairs = 0
        for s in range(sh.num_seqs):
            n = int(self.context_lens[s])
            c = int(self.query_start[s + 1] - self.query_start[s])
            pairs += sum(n - c + i + 1 for i in range(c))
        return 4 * sh.head_dim * sh.num_q_heads * pairs


def make_prefill(device="cpu", seed: int = 5, num_seqs: int = 16, chunk: int | list = 512,
                 max_prefix: int = 2048, num_q_heads: int = 32, num_kv_heads: int = 8,
                 head_dim: int = 128, block_size: int = 16, prefixes=None) -> PrefillWorkload:
    """Chunked prefill of a Llama-3-8B-shaped layer: ``num_seqs`` sequences
    with cached prefixes uniform on [0, max_prefix] each bring a chunk of
    ``chunk`` new tokens (16 x 512 = 8192 tokens per step, the batched-token
    budget the pages suggest as a starting point)."""
    rng = np.random.default_rng(seed)
    S = num_seqs
    chunks = np.array(chunk if isinstance(chunk, (list, tuple)) else [chunk] * S, np.int64)
    pre = (np.array(prefixes, np.int64) if prefixes is not None
           else rng.integers(0, max_prefix, size=S, endpoint=True))
    ctx = pre + chunks
    B = block_size
    need = sum(_blocks_for(int(c), B) for c in ctx)
    nb = math.ceil(1.2 * need) + 4
    tables, _ = build_tables(ctx, B, nb, rng)
    shape = Shape(S, num_q_heads, num_kv_heads, head_dim, B)
    g = _generator(seed, device)
    T = int(chunks.sum())
    q = _randn_bf16((T, num_q_heads, head_dim), g, device)
    k_new = _randn_bf16((T, num_kv_heads, head_dim), g, device)
    v_new = _randn_bf16((T, num_kv_heads, head_dim), g, device)
    kc = _randn_bf16((nb, num_kv_heads, B, head_dim), g, device)
    vc = _randn_bf16((nb, num_kv_heads, B, head_dim), g, device)
    qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    return PrefillWorkload(shape=shape, num_blocks=nb, context_lens=ctx.astype(np.int32),
                           query_start=qs, block_tables=tables, q=q, k_new=k_new, v_new=v_new,
                           k_cache=kc, v_cache=vc, softmax_scale=1.0 / math.sqrt(head_dim),
                           seed=seed)


def poison_prefill(wl: PrefillWorkload) -> None:
    """NaN in every cache row outside the sequences' contexts, and in the
    chunk rows (which the step's append must write first)."""
    sh = wl.shape
    B = sh.block_size
    live = np.zeros((wl.num_blocks, B), bool)
    for s in range(sh.num_seqs):
        n = int(wl.context_lens[s])
        c = int(wl.query_start[s + 1] - wl.query_start[s])
        for t in range(n - c):
            live[wl.block_tables[s, t // B], t % B] = True
    dead = torch.from_numpy(~live).to(wl.k_cache.device)
    mask = dead[:, None, :, None].expand(-1, sh.num_kv_heads, -1, sh.head_dim)
    for c_ in (wl.k_cache, wl.v_cache):
        if c_.dtype == torch.uint8:  # an E4M3 pool
            c_.masked_fill_(mask, E4M3_NAN_CODE)
        else:
            fill = torch.tensor(np.int16(np.uint16(BF16_NAN_BITS).view(np.int16)), device=c_.device)
            c_.view(torch.int16).masked_fill_(mask, fill)
