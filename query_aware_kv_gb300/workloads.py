"""Seeded synthetic inputs for the Quest decode path.

This module only *draws* inputs: a paged fp16 K/V pool, a block table, sequence
lengths, per-step queries and per-step appended tokens.  It contains none of the
method's arithmetic (no bounding boxes, scores, selection or attention), so both the
CUDA path and the CPU oracle can consume what it produces without sharing any
computation.

Layout of what it returns (the layout the library's C-ABI takes):

* ``k_pool``, ``v_pool``: fp16 ``[num_phys][Hkv][P][d]``.  Every slot of every
  physical page is filled with random values, including slots past a sequence's
  length, so that masking of the ragged tail is exercised.
* ``block_table``: int32 ``[B][max_pages]``, logical page -> physical page; pages of
  all sequences are a seeded random permutation of the pool; unused entries are -1.
* ``seq_lens``: int32 ``[B]``, tokens present before the first decode step.
* ``q``: fp16 ``[steps][B][Hq][d]``; ``k_new``/``v_new``: fp16 ``[steps][B][Hkv][d]``.

The workload shapes follow the models the Quest pages evaluate (LongChat-7B-v1.5-32k,
Yarn-Llama-2-7B-128k, a Llama-3.1-8B GQA layout), see "Quest: Query-Aware Sparsity for
Efficient Long-Context LLM Inference" (Tang 2024 summary), Key points, and the GQA note
of "Guide to Quest", Best Practices §2.  No dataset is read: these synthetic tensors
stand in for PG19 / passkey / LongBench activations.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

HEAD_DIM = 128


@dataclass
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    budget: int                 # token budget
    top_k: int                  # pages selected per (sequence, kv head)
    max_pages: int              # row length of the block table
    num_phys: int               # physical pages in the pool
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor      # lengths before the first decode step
    q: torch.Tensor             # [steps][B][Hq][d]
    k_new: torch.Tensor         # [steps][B][Hkv][d]
    v_new: torch.Tensor         # [steps][B][Hkv][d]
    needles: List[Tuple[int, int, int, int]] = field(default_factory=list)  # (b, g, page, slot)
    outlier_channels: Optional[torch.Tensor] = None  # [Hkv][n] int64
    seed: int = 0

    @property
    def steps(self) -> int:
        return int(self.q.shape[0])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def describe(self) -> dict:
        return {
            "workload": self.name, "batch": self.batch, "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads, "head_dim": self.head_dim,
            "page_size": self.page_size, "budget_tokens": self.budget, "top_k_pages": self.top_k,
            "prefill_lens": [int(x) for x in self.seq_lens.tolist()], "decode_steps": self.steps,
            "seed": self.seed,
        }


def pages_for(tokens: int, page_size: int) -> int:
    """Number of pages that hold ``tokens`` tokens (a partial last page counts as one)."""
    return (tokens + page_size - 1) // page_size


def build(name: str, *, batch: int, num_q_heads: int, num_kv_heads: int, page_size: int,
          prefill_lens: Sequence[int], steps: int, budget: int, seed: int = 0,
          device: str | torch.device = "cpu", head_dim: int = HEAD_DIM,
          outliers: int = 0, outlier_scale: float = 8.0,
          needles_per_head: int = 0, needle_mode: str = "none",
          q_noise: float = 0.3, spare_pages: int = 0,
          max_pages: Optional[int] = None) -> Workload:
    """Draw one workload.

    needle_mode:
      * ``"none"``     - queries ~ N(0, I) drawn fresh per step.
      * ``"direction"``- per q head a fixed direction u ~ N(0, I); step t uses
        q_t = u + q_noise * eps_t.  ``needles_per_head`` keys per (sequence, kv head)
        are set to 4*sqrt(d)*u/|u| (u of the group's first q head) at distinct random
        pages and random valid slots.
      * ``"slot0"``    - one needle page per (sequence, kv head) at a random depth whose
        slot-0 key is 4*sqrt(d)*q/|q| for the first step's query (group's first q head).
    """
    if num_q_heads % num_kv_heads:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    if len(prefill_lens) != batch:
        raise ValueError("one prefill length per sequence")
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    d, P, Hkv, Hq = head_dim, page_size, num_kv_heads, num_q_heads
    final_lens = [int(L) + steps for L in prefill_lens]
    pages_needed = [pages_for(L, P) for L in final_lens]
    if max_pages is None:
        max_pages = max(1, max(pages_needed))
    if any(n > max_pages for n in pages_needed):
        raise ValueError("max_pages too small for prefill + steps")
    num_phys = max(1, sum(pages_needed) + spare_pages)

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32)

    # Pool contents: N(0,1) everywhere (slots beyond the sequence hold noise on purpose).
    k_pool = randn(num_phys, Hkv, P, d).to(torch.float16)
    v_pool = randn(num_phys, Hkv, P, d).to(torch.float16)

    # Block table: a seeded random permutation of the physical pages.
    perm = torch.randperm(num_phys, generator=gen, device=dev).to(torch.int32)
    block_table = torch.full((batch, max_pages), -1, dtype=torch.int32, device=dev)
    off = 0
    for b, n in enumerate(pages_needed):
        block_table[b, :n] = perm[off:off + n]
        off += n

    k_new = randn(steps, batch, Hkv, d)
    v_new = randn(steps, batch, Hkv, d).to(torch.float16)

    outlier_channels = None
    if outliers > 0:
        outlier_channels = torch.stack(
            [torch.randperm(d, generator=gen, device=dev)[:outliers] for _ in range(Hkv)])
        for g in range(Hkv):
            ch = outlier_channels[g]
            k_pool[:, g, :, ch] = (k_pool[:, g, :, ch].float() * outlier_scale).to(torch.float16)
            k_new[:, :, g, ch] *= outlier_scale
    k_new = k_new.to(torch.float16)

    G = Hq // Hkv
    needles: List[Tuple[int, int, int, int]] = []
    if needle_mode == "direction":
        u = randn(batch, Hq, d)
        eps = randn(steps, batch, Hq, d)
        q = (u.unsqueeze(0) + q_noise * eps).to(torch.float16)
        for b in range(batch):
            L = int(prefill_lens[b])
            n_pages = pages_for(L, P)
            for g in range(Hkv):
                direction = u[b, g * G]
                key = (4.0 * math.sqrt(d) * direction / direction.norm()).to(torch.float16)
                chosen = torch.randperm(n_pages, generator=gen, device=dev)[:needles_per_head]
                for p in chosen.tolist():
                    valid = min(P, L - p * P)
                    slot = int(torch.randint(valid, (1,), generator=gen, device=dev).item())
                    phys = int(block_table[b, p].item())
                    k_pool[phys, g, slot] = key
                    needles.append((b, g, p, slot))
    elif needle_mode == "slot0":
        q = randn(steps, batch, Hq, d).to(torch.float16)
        for b in range(batch):
            n_pages = pages_for(int(prefill_lens[b]), P)
            for g in range(Hkv):
                qv = q[0, b, g * G].float()
                key = (4.0 * math.sqrt(d) * qv / qv.norm()).to(torch.float16)
                p = int(torch.randint(n_pages, (1,), generator=gen, device=dev).item())
                phys = int(block_table[b, p].item())
                k_pool[phys, g, 0] = key
                needles.append((b, g, p, 0))
    elif needle_mode == "none":
        q = randn(steps, batch, Hq, d).to(torch.float16)
    else:
        raise ValueError(f"unknown needle_mode {needle_mode!r}")

    seq_lens = torch.tensor([int(L) for L in prefill_lens], dtype=torch.int32, device=dev)
    return Workload(name=name, batch=batch, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                    page_size=P, budget=budget, top_k=max(1, budget // P), max_pages=max_pages,
                    num_phys=num_phys, k_pool=k_pool, v_pool=v_pool, block_table=block_table,
                    seq_lens=seq_lens, q=q, k_new=k_new, v_new=v_new, needles=needles,
                    outlier_channels=outlier_channels, seed=seed)


# ---------------------------------------------------------------------------------------
# The five named workloads.  Each decode step appends one token, then attends over the
# cache that includes it, so "context L" is the length seen by the last step.
# ---------------------------------------------------------------------------------------

def tiny(seed: int = 0, device="cpu") -> Workload:
    """1 sequence, 4 MHA heads, d=128, context 1024 (64 pages of 16), budget 256 (16 pages),
    N(0,1) K/V/q, one decode step (1023 prefilled tokens + 1 appended)."""
    return build("tiny_b1_h4_ctx1024_p16_budget256", batch=1, num_q_heads=4, num_kv_heads=4,
                 page_size=16, prefill_lens=[1023], steps=1, budget=256, seed=seed,
                 device=device)


def longchat_32k(seed: int = 0, device="cpu", steps: int = 64, prefill: int = 32768,
                 extra_steps_capacity: int = 0) -> Workload:
    """LongChat-7B-shaped layer: 1 sequence, 32 MHA heads, d=128, 32768 prefilled tokens,
    page 16, budget 2048 (128 pages); K/V ~ N(0,1) with 4 key channels x8 per head;
    8 needle keys per head aligned to a fixed query direction; ``steps`` appended steps."""
    P = 16
    max_pages = pages_for(prefill + steps + extra_steps_capacity, P)
    return build("longchat7b_layer_ctx32k_p16_budget2048", batch=1, num_q_heads=32,
                 num_kv_heads=32, page_size=P, prefill_lens=[prefill], steps=steps,
                 budget=2048, seed=seed, device=device, outliers=4, needles_per_head=8,
                 needle_mode="direction", max_pages=max_pages)


def batched_ragged(seed: int = 0, device="cpu", budget: int = 2048, steps: int = 16,
                   batch: int = 8, lo: int = 8192, hi: int = 32768) -> Workload:
    """8 sequences, 32 MHA heads, contexts ~ U{8192..32768}, page 16, fresh q per step."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (batch,), generator=g).tolist()
    return build(f"batched_ragged_b{batch}_ctx8k-32k_p16_budget{budget}", batch=batch,
                 num_q_heads=32, num_kv_heads=32, page_size=16, prefill_lens=lens,
                 steps=steps, budget=budget, seed=seed, device=device)


def yarn_128k_layer(layer: int, seed: int = 0, device="cpu", budget: int = 2048,
                    context: int = 131072) -> Workload:
    """One layer of the Yarn-Llama-2-7B-128k shape: 1 sequence, 32 MHA heads, context
    131072 (8192 pages of 16), one needle page per head at a random depth whose slot-0 key
    is aligned to that layer's query; layers are independent draws (seed + layer)."""
    return build(f"yarn128k_layer{layer}_ctx128k_p16_budget{budget}", batch=1, num_q_heads=32,
                 num_kv_heads=32, page_size=16, prefill_lens=[context - 1], steps=1,
                 budget=budget, seed=seed * 1000 + layer, device=device, needle_mode="slot0")


def gqa_llama31(seed: int = 0, device="cpu", page_size: int = 16, context: int = 65536,
                batch: int = 4) -> Workload:
    """Llama-3.1-8B GQA shape: 4 sequences, 32 q heads / 8 kv heads, context 65536,
    page 16 or 32, budget 4096, 4 outlier key channels x8 per kv head."""
    return build(f"gqa_llama31_b{batch}_hq32_hkv8_ctx64k_p{page_size}_budget4096",
                 batch=batch, num_q_heads=32, num_kv_heads=8, page_size=page_size,
                 prefill_lens=[context - 1] * batch, steps=1, budget=4096, seed=seed,
                 device=device, outliers=4)
