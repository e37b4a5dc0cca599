"""Seeded synthetic workloads for sparse MLA decode (inputs only).

This module draws the inputs that both the CUDA path and the fp64 oracle
consume: bf16 queries, bf16 latent and rope values of the KV cache (before the
record writer packs them), CSR index streams and per-head sinks.  It holds
none of the method's arithmetic: no packing, quantisation, scoring or softmax.
Each side packs the latent with its own writer.

The five named workloads follow the shapes of the pages' DeepSeek-V3.2 /
Kimi-K3 decode (kv_lora_rank 512, rope 64, top-k 2048, <= 16 heads on the
gfx950 page, 64 heads on the SM100 page); the pages publish no dataset, so
these synthetic draws stand in for real caches.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

LATENT_DIM = 512
ROPE_DIM = 64
QK_DIM = LATENT_DIM + ROPE_DIM
SLAB_ROWS = 1 << 20  # cache rows drawn per generator slab


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    n_q: int
    heads: int
    n_kv_rows: int
    topk: int  # slice length per row (indptr stride)
    latent: str  # "normal" or "student_t3"
    latent_std: float = 1.0
    ragged: bool = False  # causal-prefix ragged rows with -1 entries and padding
    sink: bool = False
    seed: int = 0x5EED

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(QK_DIM)

    @property
    def has_invalid(self) -> bool:
        return self.ragged

    @property
    def max_row_len(self) -> int:
        return self.topk


WORKLOADS = {
    "tiny": Workload("tiny_4x16_k128", 4, 16, 4096, 128, "normal", seed=0x5EED + 1),
    "decode": Workload("decode_64x16_k2048", 64, 16, 131072, 2048, "normal",
                       latent_std=math.sqrt(2.0), seed=0x5EED + 2),
    "ragged": Workload("ragged_256x16_k2048", 256, 16, 262144, 2048, "normal",
                       ragged=True, sink=True, seed=0x5EED + 3),
    "wide": Workload("wide_128x64_k2048", 128, 64, 1048576, 2048, "student_t3",
                     sink=True, seed=0x5EED + 4),
    "long": Workload("long_4x64_k16384", 4, 64, 8388608, 16384, "normal",
                     sink=True, seed=0x5EED + 5),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def latent_slab(w: Workload, slab: int, device="cpu"):
    """bf16 latent [rows, 512] and rope [rows, 64] of cache rows
    [slab * SLAB_ROWS, ...), drawn from a generator seeded by (seed, slab)."""
    start = slab * SLAB_ROWS
    rows = min(SLAB_ROWS, w.n_kv_rows - start)
    g = _gen(device, w.seed * 7919 + 17 * slab + 1)
    if w.latent == "normal":
        lat = torch.randn(rows, LATENT_DIM, generator=g, device=device) * w.latent_std
    elif w.latent == "student_t3":
        # Student-t with 3 degrees of freedom: z / sqrt(chi2_3 / 3), times 2^e with
        # e ~ U{-5..12} per (row, 128-wide block), clipped to |x| <= 57344: the
        # writer's block scales then span 2^-12 .. 2^7, the range the wide
        # workload is specified with (plain t3 blocks alone give 2^-6 .. 2^-3).
        z = torch.randn(rows, LATENT_DIM, generator=g, device=device)
        c = torch.randn(rows, LATENT_DIM, 3, generator=g, device=device).square().sum(-1)
        t = z * torch.sqrt(3.0 / c)
        e = torch.randint(-5, 13, (rows, LATENT_DIM // 128), generator=g, device=device)
        t = t * torch.exp2(e.float()).repeat_interleave(128, dim=1)
        lat = t
    else:
        raise ValueError(w.latent)
    lat = lat.to(torch.bfloat16).clamp_(-57344.0, 57344.0)
    rope = torch.randn(rows, ROPE_DIM, generator=g, device=device).to(torch.bfloat16)
    return lat, rope


def n_slabs(w: Workload) -> int:
    return -(-w.n_kv_rows // SLAB_ROWS)


def latent_all(w: Workload, device="cpu"):
    """The whole cache's bf16 latent and rope (small workloads only)."""
    parts = [latent_slab(w, s, device) for s in range(n_slabs(w))]
    return torch.cat([p[0] for p in parts]), torch.cat([p[1] for p in parts])


def latent_rows(w: Workload, ids: torch.Tensor, device="cpu"):
    """bf16 latent and rope of the given cache rows (redraws the slabs they sit in)."""
    ids = ids.to(torch.int64).cpu()
    lat = torch.empty(len(ids), LATENT_DIM, dtype=torch.bfloat16)
    rope = torch.empty(len(ids), ROPE_DIM, dtype=torch.bfloat16)
    slab_of = ids // SLAB_ROWS
    for s in torch.unique(slab_of).tolist():
        sel = (slab_of == s).nonzero().flatten()
        l_s, r_s = latent_slab(w, s, device)
        local = (ids[sel] - s * SLAB_ROWS).to(l_s.device)
        lat[sel] = l_s[local].cpu()
        rope[sel] = r_s[local].cpu()
    return lat, rope


def queries(w: Workload, device="cpu") -> torch.Tensor:
    g = _gen(device, w.seed * 31 + 2)
    return torch.randn(w.n_q, w.heads, QK_DIM, generator=g, device=device).to(torch.bfloat16)


def sinks(w: Workload, device="cpu") -> Optional[torch.Tensor]:
    if not w.sink:
        return None
    g = _gen(device, w.seed * 31 + 3)
    return torch.randn(w.heads, generator=g, device=device, dtype=torch.float32)


def index_stream(w: Workload, device="cpu"):
    """(indices int32 [n_q * topk], indptr int32 [n_q + 1]).

    Fixed stride: indptr = topk * q.  Plain workloads draw topk unique uniform
    rows of the whole cache per row.  Ragged rows draw L_q ~ U[1, topk] unique
    rows from the causal prefix [0, 1024 + 1000 q) (L_q capped at the prefix
    size), set each to -1 with probability 0.1, and pad the slice with -1.
    """
    g = _gen(device, w.seed * 31 + 4)
    rows = []
    for r in range(w.n_q):
        if not w.ragged:
            rows.append(torch.randperm(w.n_kv_rows, generator=g, device=device)[: w.topk])
            continue
        prefix = min(1024 + 1000 * r, w.n_kv_rows)
        length = int(torch.randint(1, w.topk + 1, (1,), generator=g, device=device).item())
        length = min(length, prefix)
        ids = torch.randperm(prefix, generator=g, device=device)[:length]
        drop = torch.rand(length, generator=g, device=device) < 0.1
        ids = torch.where(drop, torch.full_like(ids, -1), ids)
        pad = torch.full((w.topk - length,), -1, dtype=ids.dtype, device=device)
        rows.append(torch.cat([ids, pad]))
    indices = torch.cat(rows).to(torch.int32)
    indptr = (torch.arange(w.n_q + 1, device=device, dtype=torch.int64) * w.topk).to(torch.int32)
    return indices, indptr


def custom(n_q: int, heads: int, n_kv_rows: int, topk: int, *, ragged=False, sink=False,
           latent="normal", latent_std=1.0, seed=1234) -> Workload:
    """A named-free workload of the given shape (for edge-case tests)."""
    return Workload(f"custom_{n_q}x{heads}_n{n_kv_rows}_k{topk}", n_q, heads, n_kv_rows, topk,
                    latent, latent_std=latent_std, ragged=ragged, sink=sink, seed=seed)
