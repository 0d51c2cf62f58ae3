"""Seeded synthetic decode-attention workloads.

This module only draws inputs: q, the paged K/V pool, the page table and the
sequence lengths.  It holds none of the attention arithmetic, so the CUDA
library and the f64 oracle can both be fed from it without sharing any of
the method's code.

Shapes follow the workloads the pages measure or that the benchmark names:
  * apache/tvm pull request 20426, sharded-nest commit: 3060 tokens of
    context, head_dim 64/128/256, Llama-3.1-8B shape (32 query heads, 8 KV
    heads, head_dim 128), and an accuracy sweep over 1..3060 positions;
  * the short-context path and its 256-token threshold (same page);
  * a batched serving mix and a long-context case with a sliding window.

Recipe (every workload): a ``torch.Generator`` seeded per workload; q, K and
V drawn N(0, 1) in fp32 and rounded to fp16; ``seq_lens`` fixed or drawn
uniformly; the physical pages of all sequences drawn without reuse from one
shared pool (plus unused decoy pages) by a random permutation, so a
sequence's pages are scattered; table entries past a sequence's last page
hold -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor            # [B, Hq, D] (or [B, T, Hq, D]) fp16 / bf16
    k_pages: torch.Tensor      # [P, PS, Hkv, D] fp16
    v_pages: torch.Tensor      # [P, PS, Hkv, D] fp16
    page_table: torch.Tensor   # [B, max_pages] int32
    seq_lens: torch.Tensor     # [B] int32
    scale: float
    window: int = 0
    seed: int = 0

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[-2]  # q is [B, Hq, D] or [B, T, Hq, D]

    @property
    def head_dim(self) -> int:
        return self.q.shape[-1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_pages.shape[2]

    @property
    def page_size(self) -> int:
        return self.k_pages.shape[1]

    def attended_tokens(self) -> int:
        """Total attended positions over the batch (after the window)."""
        L = self.seq_lens.to("cpu").to(torch.int64)
        if self.window > 0:
            L = torch.clamp(L, max=self.window)
        return int(torch.clamp(L, min=0).sum())

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes one decode step reads: every attended
        (token, KV head) row of K and of V once, fp16."""
        return self.attended_tokens() * self.num_kv_heads * self.head_dim * 2 * 2

    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.numel() else 0

    def to(self, device) -> "Workload":
        return dataclasses.replace(
            self, q=self.q.to(device), k_pages=self.k_pages.to(device),
            v_pages=self.v_pages.to(device), page_table=self.page_table.to(device),
            seq_lens=self.seq_lens.to(device))


def _randn_fp16(shape, gen: torch.Generator, device, dtype=torch.float16) -> torch.Tensor:
    """N(0,1) drawn in fp32, rounded to the 16-bit format (fp16 by default);
    drawn in slabs to bound the fp32 temporary for the multi-GiB pools."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    slab = 1 << 26
    for i in range(0, flat.numel(), slab):
        n = min(slab, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=gen, device=device,
                                    dtype=torch.float32).to(dtype)
    return out


def make_custom(name: str, *, batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                page_size: int, seq_lens: Sequence[int] | torch.Tensor, seed: int,
                decoy_pages: int = 0, max_pages: Optional[int] = None, window: int = 0,
                scale: Optional[float] = None, device="cpu",
                dtype=torch.float16) -> Workload:
    """General generator: pages of all sequences drawn without reuse from one
    pool of sum(ceil(L_b/PS)) + decoy_pages pages, by a seeded permutation."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    L = torch.as_tensor(seq_lens, dtype=torch.int64).to("cpu")
    assert L.numel() == batch
    need = [(int(x) + page_size - 1) // page_size for x in L]
    mp = max_pages if max_pages is not None else max(need + [1])
    assert mp >= max(need + [0])
    P = sum(need) + decoy_pages
    q = _randn_fp16((batch, num_q_heads, head_dim), gen, device, dtype)
    k = _randn_fp16((P, page_size, num_kv_heads, head_dim), gen, device, dtype)
    v = _randn_fp16((P, page_size, num_kv_heads, head_dim), gen, device, dtype)
    perm = torch.randperm(P, generator=gen, device=device).to("cpu").to(torch.int32)
    table = torch.full((batch, mp), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    return Workload(name=name, q=q, k_pages=k, v_pages=v, page_table=table.to(device),
                    seq_lens=L.to(torch.int32).to(device),
                    scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
                    window=window, seed=seed)


# name -> (description, builder kwargs)
CONFIGS = {
    # B=1, Hq=4, Hkv=1, D=64, context 256, PS 16, table = permutation of 16 pages
    "tiny": dict(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16,
                 seq_lens=[256], seed=0),
    # Llama-3.1-8B decode shape at 3060 tokens; 64 unused decoy pages in the pool
    "llama": dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                  seq_lens=[3060], seed=1, decoy_pages=64),
    # head_dim sweep at 3060 tokens
    "sweep_d64": dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=64, page_size=16,
                      seq_lens=[3060], seed=2, decoy_pages=64),
    "sweep_d128": dict(batch=1, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                       seq_lens=[3060], seed=2, decoy_pages=64),
    "sweep_d256": dict(batch=1, num_q_heads=16, num_kv_heads=4, head_dim=256, page_size=16,
                       seq_lens=[3060], seed=2, decoy_pages=64),
    # long context: 4 x 131072 tokens, 64/8 heads, PS 64 (1 GiB each for K and V)
    "long": dict(batch=4, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                 seq_lens=[131072] * 4, seed=4),
    # one sequence of the long-context case (512 MiB of K+V, still above L2)
    "long_b1": dict(batch=1, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                    seq_lens=[131072], seed=4),
    "long_w4096": dict(batch=4, num_q_heads=64, num_kv_heads=8, head_dim=128, page_size=64,
                       seq_lens=[131072] * 4, seed=4, window=4096),
    # the head_dim-256 sweep shape (16/4 heads) at one 131072-token sequence:
    # 512 MiB of K+V, above L2, for DRAM-level profiles at D = 256
    "long_d256": dict(batch=1, num_q_heads=16, num_kv_heads=4, head_dim=256, page_size=64,
                      seq_lens=[131072], seed=8),
}

# shapes of the short-context sweep (contexts 1..512, threshold at 256)
SWEEP_SHAPES = {
    "d64": dict(num_q_heads=32, num_kv_heads=8, head_dim=64),
    "d128": dict(num_q_heads=32, num_kv_heads=8, head_dim=128),
    "d256": dict(num_q_heads=16, num_kv_heads=4, head_dim=256),
}


def batched_seq_lens(seed: int = 3, batch: int = 64, max_len: int = 8192) -> torch.Tensor:
    """Batched serving mix: lengths uniform in [1, max_len] from the seed."""
    g = torch.Generator()
    g.manual_seed(seed)
    return torch.randint(1, max_len + 1, (batch,), generator=g, dtype=torch.int64)


def make(name: str, device="cpu", dtype=torch.float16) -> Workload:
    """One of the named workloads, drawn on ``device`` (16-bit format
    ``dtype``: torch.float16 or torch.bfloat16)."""
    if name == "batched":
        L = batched_seq_lens()
        need = int(sum((int(x) + 15) // 16 for x in L))
        return make_custom("batched", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128,
                           page_size=16, seq_lens=L, seed=3, decoy_pages=need // 10,
                           max_pages=512, device=device, dtype=dtype)
    if name == "many_short":  # many short sequences of mixed lengths
        g = torch.Generator()
        g.manual_seed(6)
        L = torch.randint(1, 513, (1000,), generator=g, dtype=torch.int64)
        return make_custom("many_short", batch=1000, num_q_heads=32, num_kv_heads=8,
                           head_dim=128, page_size=16, seq_lens=L, seed=6, device=device,
                           dtype=dtype)
    if name.startswith("seq"):  # e.g. "seq32768" or "seq65536x2": long-case shape, B x L
        L, _, B = name[3:].partition("x")
        return make_custom(name, batch=int(B or 1), num_q_heads=64, num_kv_heads=8,
                           head_dim=128, page_size=64, seq_lens=[int(L)] * int(B or 1), seed=7,
                           device=device, dtype=dtype)
    if name.startswith("ctx"):  # e.g. "ctx300_d128": short-context sweep point
        ctx, shape = name[3:].split("_")
        return make_custom(name, batch=1, page_size=16, seq_lens=[int(ctx)], seed=5,
                           decoy_pages=8, device=device, dtype=dtype, **SWEEP_SHAPES[shape])
    kw = dict(CONFIGS[name])
    return make_custom(name, device=device, dtype=dtype, **kw)
