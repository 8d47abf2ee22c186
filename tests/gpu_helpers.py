"""Helpers for the GPU parity tests: move workloads between host and device,
hand the oracle exactly the bits the GPU sees, and compare outputs.

Nothing here computes attention, softmax, slots or quantisation: the oracle
and the CUDA library do.  ``quantize_with_torch`` rounds large FP8 test pools
with torch's own float8_e4m3fn conversion (a library routine, used only to
make inputs; values are pre-scaled into the finite range so no saturation is
involved)."""
from __future__ import annotations

import numpy as np
import torch

from paged_kv_cache_193_gb300 import workloads as W

# Tolerance of bf16 attention outputs against the fp64 oracle: max-abs 1e-2
# and mean-abs 1e-3.  bf16 cannot hold every output to 1e-2: from |out| = 4
# up its spacing is 2^-5, so the nearest bf16 value can be 2^-6 away.  Where
# one unit in the last place of the exact value (at most 2^-7 |ref|) is
# larger than 1e-2 (|ref| > 1.28), that unit is the bound: half a unit for
# the output's own rounding, and under a quarter for the bf16 probabilities.
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
ULP_REL = 2.0 ** -7


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def compare(out: torch.Tensor, ref: np.ndarray, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what="",
            ulp_rel=ULP_REL):
    """Element-wise check of ``out`` against ``ref``: each error within
    max(max_abs, ulp_rel |ref|), the mean error within ``mean_abs``."""
    got = bf16_to_f64(out)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = np.maximum(max_abs, ulp_rel * np.abs(ref))
    excess = err - bound
    worst = np.unravel_index(int(np.argmax(excess)), err.shape) if err.size else ()
    assert not err.size or excess[worst] <= 0, (
        f"{what}: abs err {err[worst]:.3e} at {tuple(int(i) for i in worst)} (got {got[worst]:.6g}, "
        f"oracle {ref[worst]:.6g}) > bound {bound[worst]:.3e}; max abs err {err.max():.3e}")
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e} > {mean_abs}"
    return float(err.max()), float(err.mean())


# Bytes of margin before and after each guarded buffer, and their fill: 0xFF
# bytes read as NaN in bf16 and in fp32, and no kernel writes that pattern.
GUARD_BYTES = 4096
GUARD_FILL = 0xFF


class Guarded:
    """A device tensor of ``shape`` and ``dtype`` placed between two margins
    of GUARD_BYTES filled with GUARD_FILL.  ``check()`` asserts that no byte
    of either margin changed, i.e. that no kernel wrote before the start or
    past the end of the buffer it was given (a stand-in for a memory
    checker).  The tensor itself starts 16-byte aligned."""

    def __init__(self, shape, dtype, device, fill=None):
        self.shape = tuple(int(x) for x in shape)
        elem = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape, dtype=np.int64)) * elem
        body = (self.nbytes + 15) // 16 * 16
        self.raw = torch.full((GUARD_BYTES + body + GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8,
                              device=device)
        self.tail_start = GUARD_BYTES + self.nbytes
        self.tensor = self.raw[GUARD_BYTES:GUARD_BYTES + self.nbytes].view(dtype).view(self.shape)
        if fill is not None:
            self.tensor.fill_(fill)

    def check(self, what=""):
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[self.tail_start:]
        bad_head = int((head != GUARD_FILL).sum())
        bad_tail = int((tail != GUARD_FILL).sum())
        assert bad_head == 0, f"{what}: {bad_head} bytes written before the buffer"
        assert bad_tail == 0, f"{what}: {bad_tail} bytes written past the end of the buffer"


def guard_step(step):
    """Give a DecodeStep guarded output, slot and workspace buffers (the
    step writes through these views); returns a function that checks every
    margin."""
    dev = step.out.device
    g = {"out": Guarded(step.out.shape, step.out.dtype, dev, fill=float("nan")),
         "slots": Guarded(step.slots.shape, torch.int32, dev, fill=-7),
         "workspace": Guarded(step.workspace.shape, torch.uint8, dev)}
    step.out, step.slots, step.workspace = g["out"].tensor, g["slots"].tensor, g["workspace"].tensor

    def check(what=""):
        torch.cuda.synchronize()
        for name, buf in g.items():
            buf.check(f"{what} {name}")
    return check


def device_tables(wl: W.Workload, device):
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables)).to(device)
    cl = torch.from_numpy(np.ascontiguousarray(wl.context_lens)).to(device)
    return bt, cl


def quantize_with_oracle(oracle, wl: W.Workload) -> None:
    """Turn the bf16 pool of an FP8 workload into E4M3 codes with the
    oracle's encoder (small pools only), in place."""
    kb = W.bits(wl.k_cache)
    vb = W.bits(wl.v_cache)
    NB, Hkv, B, D = kb.shape
    kc = np.zeros((NB, Hkv, B, D), np.uint8)
    vc = np.zeros_like(kc)
    # the whole pool as NB*B tokens of [Hkv, D], token i -> slot i
    k_tok = kb.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D)
    v_tok = vb.transpose(0, 2, 1, 3).reshape(NB * B, Hkv, D)
    oracle.cache_append(k_tok, v_tok, np.arange(NB * B, dtype=np.int32), kc, vc, B, 1, wl.kv_scale)
    wl.k_cache = torch.from_numpy(kc).to(wl.k_cache.device)
    wl.v_cache = torch.from_numpy(vc).to(wl.v_cache.device)


def quantize_with_torch(wl: W.Workload) -> None:
    """E4M3 codes of x / kv_scale by torch's conversion (|x / scale| <= 448
    by the choice of scale), in place, on the pool's device."""
    s = torch.tensor(wl.kv_scale, dtype=torch.float32, device=wl.k_cache.device)
    for name in ("k_cache", "v_cache"):
        x = getattr(wl, name)
        y = (x.float() / s)
        assert float(y.abs().max()) <= 448.0
        setattr(wl, name, y.to(torch.float8_e4m3fn).view(torch.uint8).contiguous())


def compact(wl: W.Workload, seqs, k_cache: torch.Tensor, v_cache: torch.Tensor):
    """Host copy of just the blocks sequences ``seqs`` reference, with their
    tables renumbered to the compact pool.  Returns (tables [n, MB],
    context_lens [n], k [NBc, Hkv, B, D], v) as numpy bit arrays."""
    B = wl.shape.block_size
    rows = []
    for s in seqs:
        n = int(wl.context_lens[s])
        rows.append(wl.block_tables[s, : (n + B - 1) // B])
    used = np.unique(np.concatenate(rows)) if rows else np.zeros(0, np.int32)
    remap = {int(b): i for i, b in enumerate(used)}
    tables = np.full((len(seqs), wl.block_tables.shape[1]), -1, np.int32)
    for i, row in enumerate(rows):
        tables[i, : len(row)] = [remap[int(b)] for b in row]
    idx = torch.from_numpy(used.astype(np.int64)).to(k_cache.device)
    kc = W.bits(k_cache.index_select(0, idx))
    vc = W.bits(v_cache.index_select(0, idx))
    ctx = np.array([wl.context_lens[s] for s in seqs], np.int32)
    return tables, ctx, kc, vc


def oracle_sampled(oracle, wl: W.Workload, pairs: np.ndarray, k_cache, v_cache, q) -> np.ndarray:
    """Oracle outputs for (sequence, query head) pairs, reading only the
    sequences involved (through a compacted copy of their blocks)."""
    seqs = sorted(set(int(s) for s in pairs[:, 0]))
    pos = {s: i for i, s in enumerate(seqs)}
    tables, ctx, kc, vc = compact(wl, seqs, k_cache, v_cache)
    qb = W.bits(q)[seqs]
    local = np.array([[pos[int(s)], int(h)] for s, h in pairs], np.int32)
    return oracle.decode_pairs(qb, kc, vc, tables, ctx, wl.shape.num_kv_heads,
                               wl.shape.block_size, wl.softmax_scale, local,
                               kv_dtype=wl.shape.kv_dtype, kv_scale=wl.kv_scale)
