"""Benchmark: paged decode attention on one GB300 (or N independent replicas).

One step = one decode step of one attention layer over the paged KV cache:
slot mapping of each sequence's newest token, append of its K/V, paged
attention (per context partition when split) and the log-sum-exp merge --
every row of the hot path, 3 or 4 kernel launches.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama8b]
    python bench.py --impl reference ...   # the fp64 CPU oracle, same metric

Prints ONE JSON line (rank 0).  ``value`` is KV GB/s of the whole step:
algorithmic KV bytes (every live token's K and V read once, per KV head)
divided by the device time of the step, summed over replicas.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_193_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s and % of GB300 HBM peak; decode tokens/s"
NOMINAL_HBM_GBS = 8000.0
# launch configuration per workload: (block size, partition size)
# (the long-context 70B-head workload is defined with 512-token partitions;
# the others are free and use the fastest measured setting)
DEFAULT_LAUNCH = {
    "tiny": (16, 0),
    "llama8b": (16, 0),
    "long70b": (16, 512),
    "prefix_fp8": (16, 0),
    "ctx128k": (16, 2048),
}
DESCRIPTION = {
    "tiny": "4 seqs, ctx {1,17,100,255}, 8q/2kv heads, head_dim 64, block 16, bf16",
    "llama8b": "Llama-3-8B-shape decode layer: 256 seqs, ctx U[512,2048], 32q/8kv heads, "
               "head_dim 128, block 16, bf16 KV, pool 1.2x need, shuffled blocks",
    "long70b": "Llama-3.1-70B-head long decode: 64 seqs, ctx U[4096,32768], 64q/8kv heads, "
               "head_dim 128, bf16 KV, 512-token partitions",
    "prefix_fp8": "256 seqs sharing a 2048-token prefix + suffixes U[64,512], 32q/8kv heads, "
                  "head_dim 128, block 16, e4m3 KV with per-tensor scale",
    "ctx128k": "405B-head 128K context: 8 seqs x 131072 tokens, 128q/8kv heads, head_dim 128, "
               "block 16, bf16 KV, split context + log-sum-exp merge",
}
# Workloads the default run times after the headline one, with the same
# protocol: (label, workload, block size, partition size, E4M3 cache).
SECONDARY = [
    ("long70b_B16_P512", "long70b", 16, 512, False),
    ("long70b_B32_P512", "long70b", 32, 512, False),
    ("ctx128k_P512", "ctx128k", 16, 512, False),
    ("ctx128k_P2048", "ctx128k", 16, 2048, False),
    ("prefix_fp8", "prefix_fp8", 16, 0, False),
    ("llama8b_e4m3", "llama8b", 16, 0, True),
]
DECODE_SOURCES = ["paged_kv_cache_193_gb300/csrc/pa_decode.cu",
                  "paged_kv_cache_193_gb300/csrc/pa_device.cuh"]
PREFILL_SOURCES = ["paged_kv_cache_193_gb300/csrc/pa_prefill_tc.cu",
                   "paged_kv_cache_193_gb300/csrc/pa_prefill.cuh",
                   "paged_kv_cache_193_gb300/csrc/pa_device.cuh"]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=W.NAMES, default="llama8b")
    ap.add_argument("--block-size", type=int, default=None)
    ap.add_argument("--partition-size", type=int, default=None)
    ap.add_argument("--num-seqs", type=int, default=None, help="shrink the workload (profiling)")
    ap.add_argument("--fp8", action="store_true",
                    help="store the workload's KV cache as E4M3 (one per-tensor scale)")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step(s) from one CUDA graph instead of launching eagerly")
    ap.add_argument("--layers", type=int, default=1,
                    help="attention layers per step, each with its own KV cache")
    ap.add_argument("--per-head-scales", action="store_true",
                    help="E4M3 cache with its own K and V scale per KV head")
    ap.add_argument("--fp8-qk", action="store_true",
                    help="E4M3 cache and E4M3 x E4M3 scores: the query is rounded to E4M3 with "
                         "q_scale = amax |q| / 448 (pa_decode_step_fp8_qk)")
    ap.add_argument("--device-alloc", action="store_true",
                    help="each step first advances every context by one token and allocates "
                         "blocks on the device (pa_block_alloc), then runs the step")
    ap.add_argument("--prefill", action="store_true",
                    help="time chunked prefill (16 sequences x 512-token chunks) instead of decode")
    ap.add_argument("--q-heads", type=int, default=32, help="prefill: query heads (default 32)")
    ap.add_argument("--kv-heads", type=int, default=8, help="prefill: KV heads (default 8)")
    ap.add_argument("--head-dim", type=int, default=128, choices=(64, 128),
                    help="prefill: head dim (default 128)")
    ap.add_argument("--separate", action="store_true",
                    help="time the unfused entry points (3-4 kernels per step)")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads the default run also times (long70b at "
                         "16/32-token pages, ctx128k at 512/2048-token partitions, prefix_fp8, "
                         "llama8b with the E4M3 cache)")
    ap.add_argument("--secondary-steps", type=int, default=200,
                    help="timed steps of each secondary workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--min-warmup-seconds", type=float, default=1.0,
                    help="keep warming up at least this long (clocks settle, sampler fills)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="wall-time budget of the oracle sample")
    return ap.parse_args()


# --------------------------------------------------------------------------
# distributed plumbing (independent replicas; only timing is exchanged)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# clocks
# --------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if ts < t0 or ts > t1:
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# workload
# --------------------------------------------------------------------------

def build_workload(args, device, data_seed=None):
    bs, ps = DEFAULT_LAUNCH[args.config]
    bs = args.block_size or bs
    ps = ps if args.partition_size is None else args.partition_size
    extra = args.warmup + args.steps + 1 if args.device_alloc else 0
    wl = W.make(args.config, device=device, block_size=bs, num_seqs=args.num_seqs,
                data_seed=data_seed, extra_steps=extra)
    if args.fp8 and wl.shape.kv_dtype != W.KV_FP8_E4M3:
        wl.shape.kv_dtype = W.KV_FP8_E4M3
        wl.kv_scale = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
    return wl, ps


def quantize_fp8_pool(api, wl):
    """Fill an FP8 pool with codes produced by the library's own append from
    the workload's bf16 values (every slot of the pool, in chunks)."""
    NB, Hkv, B, D = wl.k_cache.shape
    wl.notes["bf16_pool"] = (wl.k_cache, wl.v_cache)
    kc = torch.empty((NB, Hkv, B, D), dtype=torch.uint8, device=wl.k_cache.device)
    vc = torch.empty_like(kc)
    chunk = max(1, (1 << 20) // B)
    for b0 in range(0, NB, chunk):
        b1 = min(NB, b0 + chunk)
        ksrc = wl.k_cache[b0:b1].permute(0, 2, 1, 3).reshape(-1, Hkv, D).contiguous()
        vsrc = wl.v_cache[b0:b1].permute(0, 2, 1, 3).reshape(-1, Hkv, D).contiguous()
        slots = torch.arange(b0 * B, b1 * B, dtype=torch.int32, device=kc.device)
        api.cache_append(ksrc, vsrc, slots, kc, vc, wl.kv_scale)
    wl.k_cache, wl.v_cache = kc, vc


def quantize_fp8_pool_scaled(api, wl, k_scales, v_scales):
    """As quantize_fp8_pool, with the library's per-head-scale append."""
    NB, Hkv, B, D = wl.k_cache.shape
    wl.notes["bf16_pool"] = (wl.k_cache, wl.v_cache)
    kc = torch.empty((NB, Hkv, B, D), dtype=torch.uint8, device=wl.k_cache.device)
    vc = torch.empty_like(kc)
    chunk = max(1, (1 << 20) // B)
    for b0 in range(0, NB, chunk):
        b1 = min(NB, b0 + chunk)
        ksrc = wl.k_cache[b0:b1].permute(0, 2, 1, 3).reshape(-1, Hkv, D).contiguous()
        vsrc = wl.v_cache[b0:b1].permute(0, 2, 1, 3).reshape(-1, Hkv, D).contiguous()
        slots = torch.arange(b0 * B, b1 * B, dtype=torch.int32, device=kc.device)
        api.cache_append_scaled(ksrc, vsrc, slots, kc, vc, k_scales, v_scales)
    wl.k_cache, wl.v_cache = kc, vc


def config_of(wl, ps, args):
    sh = wl.shape
    pool_gb = (wl.k_cache.numel() * wl.k_cache.element_size() * 2) / 1e9
    return {
        "workload": f"{wl.name}: {DESCRIPTION[wl.name]}",
        "num_seqs": sh.num_seqs, "num_q_heads": sh.num_q_heads, "num_kv_heads": sh.num_kv_heads,
        "head_dim": sh.head_dim, "block_size": sh.block_size, "partition_size": ps,
        "kv_dtype": "bf16" if sh.kv_dtype == W.KV_BF16 else
                    ("fp8_e4m3, K and V scale per KV head" if args.per_head_scales else
                     "fp8_e4m3, one scale"),
        "scores": "E4M3 x E4M3 (query rounded to E4M3, q_scale = amax|q|/448)" if args.fp8_qk else
                  "query at full precision",
        "mean_context": float(np.mean(wl.context_lens)), "num_blocks": wl.num_blocks,
        "kv_bytes_per_step": wl.kv_bytes(), "unique_kv_bytes_per_step": wl.unique_kv_bytes(),
        "seed": wl.seed, "parallelism": "replicas", "layers": args.layers,
        "l2": f"inputs larger than L2: KV pool {pool_gb:.2f} GB vs 129 MB L2"
              + ("; the shared prefix is L2-resident by design" if wl.name == "prefix_fp8" else ""),
    }


# --------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# --------------------------------------------------------------------------

def oracle_sample_inputs(wl, seqs):
    """Host bits of q and of just the blocks of ``seqs`` (tables renumbered);
    for an FP8 workload, the bf16 pool kept from before quantisation."""
    B = wl.shape.block_size
    rows = [wl.block_tables[s, : (int(wl.context_lens[s]) + B - 1) // B] for s in seqs]
    used = np.unique(np.concatenate(rows))
    remap = np.full(wl.num_blocks, -1, np.int64)
    remap[used] = np.arange(used.size)
    tables = np.full((len(seqs), wl.block_tables.shape[1]), -1, np.int32)
    for i, row in enumerate(rows):
        tables[i, : row.size] = remap[row]
    kpool, vpool = wl.notes.get("bf16_pool", (wl.k_cache, wl.v_cache))
    idx = torch.from_numpy(used.astype(np.int64)).to(kpool.device)
    kc = W.bits(kpool.index_select(0, idx))
    vc = W.bits(vpool.index_select(0, idx))
    q = W.bits(wl.q)[seqs]
    ctx = wl.context_lens[seqs].astype(np.int32)
    return q, kc, vc, tables, ctx


def run_oracle_sample(oracle, wl, seqs):
    q, kc, vc, tables, ctx = oracle_sample_inputs(wl, seqs)
    if wl.shape.kv_dtype == W.KV_FP8_E4M3 and kc.dtype == np.uint16:
        # E4M3 codes of the sampled blocks from the oracle's own encoder
        NB, Hkv, B, D = kc.shape
        codes = [np.zeros((NB, Hkv, B, D), np.uint8) for _ in range(2)]
        tok = [a.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D) for a in (kc, vc)]
        oracle.cache_append(tok[0], tok[1], np.arange(NB * B, dtype=np.int32), codes[0], codes[1],
                            B, 1, wl.kv_scale)
        kc, vc = codes
    t0 = time.perf_counter()
    oracle.decode(q, kc, vc, tables, ctx, wl.shape.num_kv_heads, wl.shape.block_size,
                  wl.softmax_scale, kv_dtype=wl.shape.kv_dtype, kv_scale=wl.kv_scale)
    dt = time.perf_counter() - t0
    elem = 2 if wl.shape.kv_dtype == W.KV_BF16 else 1
    kv = int(ctx.astype(np.int64).sum()) * wl.shape.num_kv_heads * wl.shape.head_dim * 2 * elem
    return kv, dt


def cpu_baseline(wl, budget_s: float):
    """Time the oracle (as it stands) on growing batches of sequences,
    passing over the step's sequences again if one pass is shorter than the
    wall-time budget; KV GB/s over what it processed."""
    from oracle import Oracle
    o = Oracle()
    S = wl.shape.num_seqs
    done, kv_total, t_total, i = 0, 0, 0.0, 0
    n = 1
    while t_total < budget_s:
        seqs = [(i + j) % S for j in range(n)]
        kv, dt = run_oracle_sample(o, wl, seqs)
        kv_total += kv
        t_total += dt
        done += len(seqs)
        i = (i + n) % S
        n = min(n * 2, 64)
    return {"value": kv_total / t_total / 1e9, "unit": "GB/s", "cores": o.threads(),
            "kind": "oracle",
            "sample": f"{done} sequence-steps (all query heads; the step has {S} sequences, taken "
                      f"in turn), fp64 C oracle with OpenMP over (sequence, query head), "
                      f"{t_total:.1f} s wall"}


def cpu_baseline_prefill(wl, budget_s: float, kv_scale=None):
    """The oracle's chunked-prefill attention (as it stands) on growing
    subsets of the step's sequences until the wall-time budget is used;
    TFLOP/s over the causal pairs it processed."""
    from oracle import Oracle
    o = Oracle()
    sh = wl.shape
    qb = W.bits(wl.q)
    kc, vc = W.bits(wl.k_cache), W.bits(wl.v_cache)
    S = sh.num_seqs
    done, flops, t_total, i, n = 0, 0, 0.0, 0, 1
    while t_total < budget_s:
        seqs = [(i + j) % S for j in range(n)]
        rows = [np.arange(wl.query_start[s], wl.query_start[s + 1]) for s in seqs]
        chunks = np.array([len(r) for r in rows], np.int64)
        qs = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
        ctx = wl.context_lens[seqs].astype(np.int32)
        t0 = time.perf_counter()
        o.prefill(qb[np.concatenate(rows)], kc, vc, wl.block_tables[seqs], ctx, qs, sh.num_kv_heads,
                  sh.block_size, wl.softmax_scale, kv_dtype=0 if kv_scale is None else 1,
                  kv_scale=1.0 if kv_scale is None else kv_scale)
        t_total += time.perf_counter() - t0
        pairs = sum(int(c) - int(ch) + k + 1 for c, ch in zip(ctx, chunks) for k in range(int(ch)))
        flops += 4 * sh.head_dim * sh.num_q_heads * pairs
        done += len(seqs)
        i = (i + n) % S
        n = min(n * 2, S)
    return {"value": flops / t_total / 1e12, "unit": "TFLOP/s", "cores": o.threads(), "kind": "oracle",
            "sample": f"{done} sequence chunks (all query heads; the step has {S}, taken in turn), "
                      f"fp64 C oracle with OpenMP over chunk rows, {t_total:.1f} s wall"}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

def source_digest(sources=DECODE_SOURCES) -> str:
    h = hashlib.sha256()
    for p in sources:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(wl, ps, args):
    """DRAM bytes per decode launch from a committed ncu capture, if it was
    taken on the current decode kernel source for this workload, page size,
    partition size and KV type (bf16 records carry no type suffix)."""
    if args.device_alloc:  # contexts grow during the run: no single figure applies
        return None
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    key = f"{wl.name}/B{wl.shape.block_size}/P{ps}"
    if wl.shape.kv_dtype != W.KV_BF16:
        key += "/e4m3"
    entry = rec.get(key)
    if not entry or entry.get("source_digest") != source_digest():
        return None
    return entry.get("dram_bytes_per_launch")


def recorded_prefill_traffic(sh, mq, num_seqs, fp8=False):
    """DRAM bytes per tcgen05 prefill launch from a committed ncu capture of
    the same kernel source and workload shape, else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "prefill_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    key = f"S{num_seqs}/C{mq}/H{sh.num_q_heads}/KV{sh.num_kv_heads}/D{sh.head_dim}/B{sh.block_size}"
    if fp8:
        key += "/e4m3"
    entry = rec.get(key)
    if not entry or entry.get("source_digest") != source_digest(PREFILL_SOURCES):
        return None
    return entry.get("dram_bytes_per_launch")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0}, "fallback"


def run_ours(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    from paged_kv_cache_193_gb300 import api

    wl, ps = build_workload(args, device)
    # further layers share the contexts and block tables, with their own values
    layers = [wl] + [build_workload(args, device, data_seed=wl.seed + 1000 * i)[0]
                     for i in range(1, args.layers)]
    steps, inputs = [], []
    for lw in layers:
        ks = vs = None
        if args.per_head_scales:
            if lw.shape.kv_dtype != W.KV_FP8_E4M3:
                raise SystemExit("--per-head-scales needs an E4M3 cache (--fp8 or prefix_fp8)")
            # amax / 448 per KV head, for K and V separately
            ks = (lw.k_cache.float().abs().amax(dim=(0, 2, 3)) / 448.0).contiguous()
            vs = (lw.v_cache.float().abs().amax(dim=(0, 2, 3)) / 448.0).contiguous()
            quantize_fp8_pool_scaled(api, lw, ks, vs)
        elif lw.shape.kv_dtype == W.KV_FP8_E4M3:
            quantize_fp8_pool(api, lw)
        lbt = torch.from_numpy(lw.block_tables).to(device)
        lcl = torch.from_numpy(lw.context_lens).to(device)
        qs = None
        if args.fp8_qk:
            if lw.shape.kv_dtype != W.KV_FP8_E4M3:
                raise SystemExit("--fp8-qk needs an E4M3 cache (--fp8 or prefix_fp8)")
            qs = float(lw.q.float().abs().max().item()) / 448.0
        steps.append(api.DecodeStep(lw.k_cache, lw.v_cache, lbt, lcl, lw.shape.num_q_heads,
                                    lw.softmax_scale, lw.kv_scale, ps, fused=not args.separate,
                                    k_scales=ks, v_scales=vs, q_scale=qs))
        inputs.append((lw.q, lw.k_new, lw.v_new))
    sh = wl.shape
    step = steps[0]
    bt, cl = step.block_tables, step.context_lens
    stream = torch.cuda.current_stream()
    if args.device_alloc:
        if len(steps) != 1 or args.graph:
            raise SystemExit("--device-alloc runs one eager layer")
        args.min_warmup_seconds = 0.0
        alloc = wl.notes["allocator"]
        pool = api.DeviceBlockPool(alloc._free, alloc.refcount, device)
        # contexts currently include the token appended at step 0: start one lower
        cl.sub_(1)
        kv0 = wl.kv_bytes() - sh.num_seqs * sh.num_kv_heads * sh.head_dim * 2 * (
            2 if sh.kv_dtype == W.KV_BF16 else 1)
        per_token = sh.num_kv_heads * sh.head_dim * 2 * (2 if sh.kv_dtype == W.KV_BF16 else 1)
        cow = torch.empty(sh.num_seqs, dtype=torch.int32, device=device)
        calls = [0]

        def run_step():
            pool.allocate(bt, cl, wl.k_cache, wl.v_cache, advance=True, cow_src=cow)
            step(wl.q, wl.k_new, wl.v_new)
            calls[0] += 1
        launches_per_step = step.launches() + 2
    elif args.graph:
        graph = api.StepGraph(steps, inputs)
        run_step = graph.replay
        launches_per_step = graph.launches()
    else:
        def run_step():
            for st, (q, k, v) in zip(steps, inputs):
                st(q, k, v)
        launches_per_step = sum(st.launches() for st in steps)

    # warm-up: at least W steps and at least --min-warmup-seconds of load
    clocks = ClockSampler(local)
    clocks.start()
    api.device_errors(clear=True)
    t_w = time.time()
    done = 0
    while done < args.warmup or time.time() - t_w < args.min_warmup_seconds:
        run_step()
        done += 1
        if done % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert api.device_errors() == 0, "device error flags raised during warm-up"

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        run_step()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(total_ms, world, device)
    t_step = np.array([a.elapsed_time(b) for a, b in ev])
    assert api.device_errors() == 0, "device error flags raised during the timed steps"

    # The dominant kernel on its own.  Unsplit, the fused step IS one kernel
    # (the per-step events above).  Split, time the attention kernel and the
    # merge one launch each with events between them (this breaks the
    # overlap of the merge's launch with the attention tail, so it is kept
    # out of the timed steps).
    if ps == 0 and step.fused and len(steps) == 1 and not args.device_alloc:
        dec_ms, red_ms, kname = float(np.mean(t_step)), 0.0, "decode_kernel (fused step)"
    else:
        n2 = min(K, 200)
        e = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n2)]
        for i in range(n2):
            e[i][0].record(stream)
            if ps == 0 and step.fused:
                step(wl.q, wl.k_new, wl.v_new)
            elif ps:
                api.decode_partitions(wl.q, wl.k_cache, wl.v_cache, bt, cl, wl.softmax_scale,
                                      wl.kv_scale, ps, step.workspace)
            else:
                api.decode(wl.q, wl.k_cache, wl.v_cache, bt, cl, wl.softmax_scale, wl.kv_scale,
                           0, None, step.out)
            e[i][1].record(stream)
            if ps:
                api.decode_reduce(step.workspace, cl, sh.num_q_heads, sh.head_dim, bt.shape[1],
                                  sh.block_size, ps, step.out)
            e[i][2].record(stream)
        torch.cuda.synchronize()
        dec_ms = float(np.mean([x[0].elapsed_time(x[1]) for x in e]))
        red_ms = float(np.mean([x[1].elapsed_time(x[2]) for x in e]))
        kname = "decode_kernel (per-partition attention)" if ps else "decode_kernel"
    clocks.stop()

    kv = sum(lw.kv_bytes() for lw in layers)
    if args.device_alloc:
        # the timed steps saw contexts growing by one token per step
        first = calls[0] - K
        kv = kv0 + per_token * sh.num_seqs * (first + (K + 1) / 2.0)
        assert api.device_errors() == 0, "device errors during the allocating steps"
    ms_per_step = total_ms / K
    value = world * kv * K / (total_ms / 1e3) / 1e9
    peaks, peak_kind = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    kv_launch = wl.kv_bytes()
    if args.device_alloc:  # the kernel-only launches ran at the final contexts
        kv_launch = kv0 + per_token * sh.num_seqs * calls[0]
    achieved = kv_launch / (dec_ms / 1e3) / 1e9
    traffic = recorded_traffic(wl, ps, args)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if
        sh.kv_dtype == W.KV_BF16 else ("fp8_e4m3 KV and E4M3 x E4M3 scores, bf16 q/out, fp32 accumulate"
                                       if args.fp8_qk else "fp8_e4m3 KV, bf16 q/out, fp32 accumulate"),
        "data": "synthetic (seeded N(0,1) bf16, shuffled block tables)",
        "config": config_of(wl, ps, args),
        "tokens_per_s": round(world * sh.num_seqs * K / (total_ms / 1e3), 1),
        "layers_per_step": len(layers), "launch": "one CUDA graph per step" if args.graph else "eager",
        "device_alloc": bool(args.device_alloc),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        f"pct_of_{peak_kind}_hbm": round(100 * value / world / hbm, 2),
        "breakdown_ms": {"step_median": round(float(np.median(t_step)), 5),
                         "step_min": round(float(np.min(t_step)), 5),
                         "decode_kernel": round(dec_ms, 5), "merge_kernel": round(red_ms, 5)},
        "step_path": "pa_decode_step (slot mapping + append + attention fused; merge as a "
                     "programmatic dependent launch when split)" if step.fused else
                     "separate pa_slot_mapping, pa_cache_append, pa_decode[_partitions], "
                     "pa_decode_reduce",
        "gpu_launches": K * launches_per_step,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": round(achieved, 1),
                     "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "algorithmic_bytes_per_launch": kv_launch, "traffic": traffic,
                     "statistic": "algorithmic bytes / mean of the kernel's per-launch "
                                  "CUDA-event durations"},
    }
    result["clocks"] = clocks.summary(t_wall0 - 1.0, t_wall1)

    if not args.no_e2e and len(layers) == 1 and not args.device_alloc:
        result["e2e"] = run_e2e(api, wl, step, ps, K, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.device_alloc:
        result["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds)
    if default_run(args):
        del steps, inputs, layers, step, wl
        torch.cuda.empty_cache()
        result["secondary"] = {label: time_secondary(api, label, name, bs, ps, fp8, args, world, local,
                                                     device, hbm)
                               for label, name, bs, ps, fp8 in SECONDARY}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def default_run(args) -> bool:
    """The plain headline run (no variant flags): it also times SECONDARY."""
    return (not args.no_secondary and args.config == "llama8b" and not args.fp8 and not args.graph
            and args.layers == 1 and not args.per_head_scales and not args.fp8_qk
            and not args.device_alloc and not args.separate and args.num_seqs is None
            and args.block_size is None and args.partition_size is None)


def time_secondary(api, label, name, bs, ps, fp8, args, world, local, device, hbm):
    """One more workload with the headline's protocol: fused step (slot
    mapping + append + attention, merge when split), warm-up of at least
    0.3 s, then ``--secondary-steps`` steps timed with CUDA events between
    barriers; the attention kernel timed alone the same way as the
    headline's; clocks sampled over the timed region."""
    wl = W.make(name, device=device, block_size=bs)
    if fp8 and wl.shape.kv_dtype != W.KV_FP8_E4M3:
        wl.shape.kv_dtype = W.KV_FP8_E4M3
        wl.kv_scale = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
    if wl.shape.kv_dtype == W.KV_FP8_E4M3:
        quantize_fp8_pool(api, wl)
        wl.notes.pop("bf16_pool", None)
    sh = wl.shape
    bt = torch.from_numpy(wl.block_tables).to(device)
    cl = torch.from_numpy(wl.context_lens).to(device)
    step = api.DecodeStep(wl.k_cache, wl.v_cache, bt, cl, sh.num_q_heads, wl.softmax_scale,
                          wl.kv_scale, ps)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    api.device_errors(clear=True)
    t_w, done = time.time(), 0
    while done < args.warmup or time.time() - t_w < 0.3:
        step(wl.q, wl.k_new, wl.v_new)
        done += 1
        if done % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    K = args.secondary_steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        step(wl.q, wl.k_new, wl.v_new)
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    total_ms = max_over_ranks(start.elapsed_time(end), world, device)
    t_step = np.array([a.elapsed_time(b) for a, b in ev])
    if ps == 0:
        dec_ms, red_ms = float(np.mean(t_step)), 0.0
    else:
        e = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(min(K, 100))]
        for x in e:
            x[0].record(stream)
            api.decode_partitions(wl.q, wl.k_cache, wl.v_cache, bt, cl, wl.softmax_scale,
                                  wl.kv_scale, ps, step.workspace)
            x[1].record(stream)
            api.decode_reduce(step.workspace, cl, sh.num_q_heads, sh.head_dim, bt.shape[1],
                              sh.block_size, ps, step.out)
            x[2].record(stream)
        torch.cuda.synchronize()
        dec_ms = float(np.mean([x[0].elapsed_time(x[1]) for x in e]))
        red_ms = float(np.mean([x[1].elapsed_time(x[2]) for x in e]))
    clocks.stop()
    assert api.device_errors() == 0, f"device error flags raised on {label}"
    kv = wl.kv_bytes()
    value = world * kv * K / (total_ms / 1e3) / 1e9
    achieved = kv / (dec_ms / 1e3) / 1e9
    res = {
        "workload": f"{name}: {DESCRIPTION[name]}" + ("; E4M3 cache, one scale" if fp8 else ""),
        "block_size": sh.block_size, "partition_size": ps,
        "kv_dtype": "bf16" if sh.kv_dtype == W.KV_BF16 else "fp8_e4m3, one scale",
        "kv_bytes_per_step": kv, "unique_kv_bytes_per_step": wl.unique_kv_bytes(),
        "value": round(value, 2), "unit": "GB/s", "steps": K, "ms_per_step": round(total_ms / K, 5),
        "step_median_ms": round(float(np.median(t_step)), 5),
        "decode_kernel_ms": round(dec_ms, 5), "merge_kernel_ms": round(red_ms, 5),
        "decode_kernel_gbs": round(achieved, 1), "frac": round(achieved / hbm, 4),
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "tokens_per_s": round(world * sh.num_seqs * K / (total_ms / 1e3), 1),
        "gpu_launches": K * step.launches(),
        "clocks": clocks.summary(t0 - 1.0, t1),
    }
    if name == "prefix_fp8":
        res["note"] = "logical bytes; the 2048-token shared prefix is read from L2 by design"
    del step, wl, bt, cl
    torch.cuda.empty_cache()
    return res


def run_e2e(api, wl, step, ps, K, world, device):
    """Same metric through the public API with the per-step inputs in pinned
    host memory: every step copies q, the new K/V and the context lengths in,
    runs the step and copies the output back, all inside the timed region.
    The copies are pipelined the way a serving loop would: step i + 1's
    inputs go in on a copy stream while step i runs, and step i's output
    comes back on a third stream; inputs and outputs are double-buffered
    (two DecodeStep objects over the same cache and block tables)."""
    sh = wl.shape
    h_q = wl.q.cpu().pin_memory()
    h_k = wl.k_new.cpu().pin_memory()
    h_v = wl.v_new.cpu().pin_memory()
    h_cl = torch.from_numpy(wl.context_lens).pin_memory()
    h_out = [torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory() for _ in range(2)]
    bufs = []
    for _ in range(2):
        d_cl = torch.empty_like(step.context_lens)
        st = api.DecodeStep(step.k_cache, step.v_cache, step.block_tables, d_cl, sh.num_q_heads,
                            step.softmax_scale, step.kv_scale, ps, fused=step.fused,
                            k_scales=step.k_scales, v_scales=step.v_scales, q_scale=step.q_scale)
        bufs.append((torch.empty_like(wl.q), torch.empty_like(wl.k_new), torch.empty_like(wl.v_new),
                     d_cl, st))
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_done, step_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def copy_in(i):
        d_q, d_k, d_v, d_cl, _ = bufs[i & 1]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(step_done[i & 1])  # step i - 2 has read this buffer
            d_q.copy_(h_q, non_blocking=True)
            d_k.copy_(h_k, non_blocking=True)
            d_v.copy_(h_v, non_blocking=True)
            d_cl.copy_(h_cl, non_blocking=True)
            in_done[i & 1].record(s_in)

    def run(i, n):
        d_q, d_k, d_v, _, st = bufs[i & 1]
        if i + 1 < n:
            copy_in(i + 1)
        comp.wait_event(in_done[i & 1])
        if i >= 2:
            comp.wait_event(out_done[i & 1])  # step i - 2's output is back on the host
        st(d_q, d_k, d_v, stream=comp)
        step_done[i & 1].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(step_done[i & 1])
            h_out[i & 1].copy_(st.out, non_blocking=True)
            out_done[i & 1].record(s_out)

    def loop(n, start=None, end=None):
        if start is not None:
            start.record(comp)
        s_in.wait_stream(comp)
        copy_in(0)
        for i in range(n):
            run(i, n)
        comp.wait_stream(s_out)
        if end is not None:
            end.record(comp)

    n = max(10, min(K, 500))
    loop(6)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    loop(n, a, b)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, device)
    # the pipelined steps computed what the plain step computes from the same inputs
    step(wl.q, wl.k_new, wl.v_new)
    torch.cuda.synchronize()
    if not torch.equal(h_out[(n - 1) & 1], step.out.cpu()):
        raise RuntimeError("pipelined end-to-end output differs from the plain step's")
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_cl))
    d2h = h_out[0].numel() * h_out[0].element_size()
    return {"value": round(world * wl.kv_bytes() * n / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": round(ms / n, 5),
            "pipelining": "step i+1's inputs copied in on a second stream while step i runs, "
                          "outputs copied back on a third; double-buffered"}


def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    from oracle import Oracle
    o = Oracle()
    wl, ps = build_workload(args, device)
    S = wl.shape.num_seqs
    # one step = a bounded sample of sequences, sized to ~1 s of oracle time
    probe_kv, probe_t = run_oracle_sample(o, wl, [0])
    per_seq = max(probe_t, 1e-4)
    n = int(max(1, min(S, 1.0 / per_seq)))
    for i in range(args.warmup if args.warmup < 2 else 1):
        run_oracle_sample(o, wl, list(range(min(n, S))))
    kv_total, t_total = 0, 0.0
    K = max(1, min(args.steps, 10))
    for i in range(K):
        seqs = [(i * n + j) % S for j in range(n)]
        kv, dt = run_oracle_sample(o, wl, sorted(set(seqs)))
        kv_total += kv
        t_total += dt
    value = kv_total / t_total / 1e9
    result = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_total / K, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload)",
        "config": config_of(wl, ps, args),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": o.threads(),
                         "kind": "oracle",
                         "sample": f"{n} sequences (all query heads) per step of one decode "
                                   f"step; fp64 C oracle, OpenMP"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)


def run_prefill_e2e(api, wl, bt, K, world, device, kv_scale=1.0):
    """The prefill metric through the public API with the step's inputs in
    pinned host memory: the queries, the chunk's new K/V rows, the context
    lengths and the chunk offsets are copied in, the step runs (chunk slots,
    append, attention) and the output is copied back, all inside the timed
    region.  Pipelined and double-buffered as the decode's end-to-end loop:
    step i + 1's inputs go in on a copy stream while step i runs, step i's
    output comes back on a third stream."""
    sh = wl.shape
    T = int(wl.query_start[-1])
    mq = wl.max_query_len
    h_in = [wl.q.cpu().pin_memory(), wl.k_new.cpu().pin_memory(), wl.v_new.cpu().pin_memory(),
            torch.from_numpy(wl.context_lens).pin_memory(), torch.from_numpy(wl.query_start).pin_memory()]
    h_out = [torch.empty(wl.q.shape, dtype=wl.q.dtype).pin_memory() for _ in range(2)]
    bufs = [([torch.empty(t.shape, dtype=t.dtype, device=device) for t in h_in],
             torch.empty(T, dtype=torch.int32, device=device), torch.empty_like(wl.q)) for _ in range(2)]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_done, step_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def copy_in(i):
        d_in = bufs[i & 1][0]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(step_done[i & 1])  # step i - 2 has read this buffer
            for d, h in zip(d_in, h_in):
                d.copy_(h, non_blocking=True)
            in_done[i & 1].record(s_in)

    def step_on(d_in, d_slots, d_out):
        d_q, d_k, d_v, d_cl, d_qs = d_in
        api.chunk_slot_mapping(bt, d_cl, d_qs, sh.block_size, out=d_slots, stream=comp)
        api.cache_append(d_k, d_v, d_slots, wl.k_cache, wl.v_cache, scale=kv_scale, stream=comp)
        api.prefill(d_q, wl.k_cache, wl.v_cache, bt, d_cl, d_qs, mq, wl.softmax_scale, out=d_out,
                    stream=comp, kv_scale=kv_scale)

    def run(i, n):
        d_in, d_slots, d_out = bufs[i & 1]
        if i + 1 < n:
            copy_in(i + 1)
        comp.wait_event(in_done[i & 1])
        if i >= 2:
            comp.wait_event(out_done[i & 1])  # step i - 2's output is back on the host
        step_on(d_in, d_slots, d_out)
        step_done[i & 1].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(step_done[i & 1])
            h_out[i & 1].copy_(d_out, non_blocking=True)
            out_done[i & 1].record(s_out)

    def loop(n, start=None, end=None):
        if start is not None:
            start.record(comp)
        s_in.wait_stream(comp)
        copy_in(0)
        for i in range(n):
            run(i, n)
        comp.wait_stream(s_out)
        if end is not None:
            end.record(comp)

    n = max(10, min(K, 200))
    loop(4)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    loop(n, a, b)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world, device)
    # the pipelined steps computed what a plain step computes from the same inputs
    d_slots = torch.empty(T, dtype=torch.int32, device=device)
    d_out = torch.empty_like(wl.q)
    step_on([wl.q, wl.k_new, wl.v_new, torch.from_numpy(wl.context_lens).to(device),
             torch.from_numpy(wl.query_start).to(device)], d_slots, d_out)
    torch.cuda.synchronize()
    if not torch.equal(h_out[(n - 1) & 1], d_out.cpu()):
        raise RuntimeError("pipelined end-to-end prefill output differs from the plain step's")
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out[0].numel() * h_out[0].element_size()
    return {"value": round(world * wl.attention_flops() * n / (ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": round(ms / n, 5),
            "pipelining": "step i+1's inputs copied in on a second stream while step i runs, "
                          "outputs copied back on a third; double-buffered"}


def run_prefill(args):
    """Chunked prefill step: chunk slots, append of the chunk's K/V, causal
    attention over the paged cache.  value = attention TFLOP/s (QK^T and PV
    over the (query, key) pairs the causal mask keeps)."""
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    from paged_kv_cache_193_gb300 import api
    wl = W.make_prefill(device, num_seqs=args.num_seqs or 16, block_size=args.block_size or 16,
                        num_q_heads=args.q_heads, num_kv_heads=args.kv_heads, head_dim=args.head_dim)
    sh = wl.shape
    kv_scale = 1.0
    if args.fp8:
        # an E4M3 pool of x / kv_scale (torch's conversion, only to make the
        # input pool; the step's own append writes the chunk with the library)
        kv_scale = W.fp8_scale_from(wl.k_cache, wl.v_cache, wl.k_new, wl.v_new)
        for name in ("k_cache", "v_cache"):
            x = getattr(wl, name)
            setattr(wl, name, (x.float() / kv_scale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous())
    bt = torch.from_numpy(wl.block_tables).to(device)
    cl = torch.from_numpy(wl.context_lens).to(device)
    qs = torch.from_numpy(wl.query_start).to(device)
    T = int(wl.query_start[-1])
    slots = torch.empty(T, dtype=torch.int32, device=device)
    out = torch.empty_like(wl.q)
    mq = wl.max_query_len
    stream = torch.cuda.current_stream()

    def step():
        api.chunk_slot_mapping(bt, cl, qs, sh.block_size, out=slots)
        api.cache_append(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache, scale=kv_scale)
        api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, mq, wl.softmax_scale, out=out, kv_scale=kv_scale)

    clocks = ClockSampler(local)
    clocks.start()
    t_w = time.time()
    done = 0
    while done < args.warmup or time.time() - t_w < args.min_warmup_seconds:
        step()
        done += 1
    torch.cuda.synchronize()
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    # the KV pool fits in L2: overwrite a buffer larger than L2 before every
    # timed step so no step starts with the previous one's lines resident
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        api.chunk_slot_mapping(bt, cl, qs, sh.block_size, out=slots)
        api.cache_append(wl.k_new, wl.v_new, slots, wl.k_cache, wl.v_cache, scale=kv_scale)
        kev[i][0].record(stream)
        api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, mq, wl.softmax_scale, out=out, kv_scale=kv_scale)
        kev[i][1].record(stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clocks.stop()
    assert api.device_errors() == 0
    step_ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])), world, device)
    kern_ms = float(np.mean([a.elapsed_time(b) for a, b in kev]))
    # the warp-level MMA kernel on the same inputs, for comparison (bf16 caches)
    mma_ms = None
    if not args.fp8:
        mev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(min(K, 50))]
        for a_, b_ in mev:
            a_.record(stream)
            api.prefill(wl.q, wl.k_cache, wl.v_cache, bt, cl, qs, mq, wl.softmax_scale, out=out,
                        kernel="mma")
            b_.record(stream)
        torch.cuda.synchronize()
        mma_ms = float(np.mean([a_.elapsed_time(b_) for a_, b_ in mev]))
    flops = wl.attention_flops()
    peaks, kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops / (kern_ms / 1e3) / 1e12
    res = {
        "metric": "paged chunked-prefill attention TFLOP/s", "value": round(world * flops / (step_ms / 1e3) / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 products on e4m3 KV" if args.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) bf16, shuffled block tables)",
        "config": {"workload": f"chunked prefill: {sh.num_seqs} seqs x {mq}-token chunks after "
                               f"cached prefixes U[0,2048], {sh.num_q_heads}q/{sh.num_kv_heads}kv heads, "
                               f"head_dim {sh.head_dim}, block {sh.block_size}, "
                               + ("e4m3 KV with per-tensor scale" if args.fp8 else "bf16"),
                   "chunk_tokens": T, "attention_flops_per_step": flops, "seed": wl.seed,
                   "l2": f"KV pool {2 * wl.k_cache.numel() * wl.k_cache.element_size() / 1e9:.2f} GB; "
                         "256 MB written between timed steps (L2 flush)"},
        "tokens_per_s": round(world * T / (step_ms / 1e3), 1),
        "breakdown_ms": {"prefill_kernel": round(kern_ms, 5),
                         "slots+append": round(step_ms - kern_ms, 5),
                         "prefill_kernel_warp_mma": None if mma_ms is None else round(mma_ms, 5)},
        "warp_mma_kernel_tflops": None if mma_ms is None else round(flops / (mma_ms / 1e3) / 1e12, 1),
        "gpu_launches": 3 * K,  # per timed step: chunk slots, append, attention
        "roofline": {"bound": "tensor", "kernel": "prefill_tc_kernel (tcgen05, TMEM accumulators)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4),
                     "peak_kind": f"{kind} cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops)",
                     "traffic": recorded_prefill_traffic(sh, mq, sh.num_seqs, fp8=args.fp8)},
        "clocks": clocks.summary(t0 - 1.0, t1),
    }
    if not args.no_e2e:
        res["e2e"] = run_prefill_e2e(api, wl, bt, K, world, device, kv_scale=kv_scale)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_prefill(wl, args.cpu_seconds, kv_scale if args.fp8 else None)
    if rank == 0:
        print(json.dumps(res), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill:
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
