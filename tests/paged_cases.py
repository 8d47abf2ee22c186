"""Small paged cases built from LOGICAL (contiguous) K/V for the oracle pins.

The logical tensors are drawn first; a test then scatters them into a paged
pool under a chosen physical block assignment.  The oracle reads the pool
through the block table; the independent checks read the logical tensors
directly, so a wrong gather index in the oracle cannot cancel out.
"""
from __future__ import annotations

import numpy as np
import torch


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    return x.to(torch.bfloat16).contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (np.asarray(b).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class LogicalCase:
    """Per-sequence logical K/V [Hkv, ctx, D] (bf16 bits) and q [Hq, D]."""

    def __init__(self, ctx, Hq, Hkv, D, seed, k_override=None):
        g = torch.Generator().manual_seed(seed)
        self.ctx = [int(c) for c in ctx]
        self.Hq, self.Hkv, self.D = Hq, Hkv, D
        self.q = bf16_bits(torch.randn(len(ctx), Hq, D, generator=g))
        self.k = [bf16_bits(torch.randn(Hkv, c, D, generator=g)) for c in self.ctx]
        self.v = [bf16_bits(torch.randn(Hkv, c, D, generator=g)) for c in self.ctx]
        if k_override is not None:
            self.k = k_override(self.k)

    def paged(self, block_size, num_blocks, rng, share_prefix_tokens=0, elem=np.uint16):
        """Scatter into a pool of ``num_blocks`` blocks under a random block
        assignment.  With ``share_prefix_tokens`` (a multiple of the block size)
        all sequences' first blocks are ONE set of physical blocks filled from
        sequence 0 (the caller makes the logical prefixes equal).  Unused pool
        rows are NaN."""
        S, B = len(self.ctx), block_size
        need = [(c + B - 1) // B for c in self.ctx]
        mb = max(need)
        perm = list(rng.permutation(num_blocks))
        tables = np.full((S, mb), -1, np.int32)
        shared = []
        if share_prefix_tokens:
            shared = [perm.pop() for _ in range(share_prefix_tokens // B)]
        for s in range(S):
            row = list(shared) + [perm.pop() for _ in range(need[s] - len(shared))]
            tables[s, :need[s]] = row
        kc = np.full((num_blocks, self.Hkv, B, self.D), 0x7FC0, np.uint16)
        vc = np.full_like(kc, 0x7FC0)
        for s in range(S):
            for t in range(self.ctx[s]):
                b = tables[s, t // B]
                kc[b, :, t % B, :] = self.k[s][:, t, :]
                vc[b, :, t % B, :] = self.v[s][:, t, :]
        return tables, kc, vc

    def sdpa(self, softmax_scale, deq_k=None, deq_v=None, deq_q=None) -> np.ndarray:
        """torch scaled_dot_product_attention in float64 over the logical K/V,
        each KV head repeated for its G query heads (grouped-query attention)."""
        G = self.Hq // self.Hkv
        out = np.zeros((len(self.ctx), self.Hq, self.D))
        for s, c in enumerate(self.ctx):
            if c == 0:
                continue
            q = torch.from_numpy(deq_q(self.q[s]) if deq_q else bits_to_f64(self.q[s]))[None, :, None, :]
            k = torch.from_numpy(deq_k(self.k[s]) if deq_k else bits_to_f64(self.k[s]))
            v = torch.from_numpy(deq_v(self.v[s]) if deq_v else bits_to_f64(self.v[s]))
            k = k.repeat_interleave(G, dim=0)[None]
            v = v.repeat_interleave(G, dim=0)[None]
            o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=softmax_scale)
            out[s] = o[0, :, 0, :].numpy()
        return out
