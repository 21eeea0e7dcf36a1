"""Seeded synthetic inputs for query-aware sparse paged decode.

This module only draws random numbers and lays them out as a paged KV cache.
It holds none of the method's arithmetic (no metadata, no scores, no
selection, no attention), so both the CUDA path and the CPU oracle can take
their inputs from it.

The named workloads stand in for the pages' models (no weights or datasets
are used):

* ``tiny``           -- a correctness case: 2 sequences of 256 tokens, GQA 2,
                        fp32 q/K/V, contiguous page table.
* ``gpt2_345m``      -- GPT2-345M-like decode at 8K context (TinyServe query-
                        aware page selection, section 4.1 table): 8 x 8192
                        tokens, 16 MHA heads, d=64, 30 % of pages selected.
* ``llama3_8b``      -- Llama-3-8B-like GQA decode: 32 sequences of
                        U[4096, 32768] tokens, 32/8 heads, d=128, 128 pages,
                        2 % of pages planted along the group's query.
* ``long_context``   -- 4 sequences of U[65536, 131072] tokens, page 32,
                        keys drawn around 64 centroids, q near one of them.
* ``shared_prefix``  -- 256 sequences sharing 128 aliased prefix pages plus
                        32 private pages each; dense (all pages).  With
                        ``seq_lens`` given, each sequence holds the prefix
                        and ceil(seq_len / P) - prefix_pages private pages.

Slots of a partially filled last page hold NaN in K and V: every consumer
must ignore tokens at or beyond ``seq_len``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

__all__ = ["Spec", "WORKLOADS", "make_inputs", "spec_for", "q_variants"]


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and value recipe of one synthetic paged-KV decode batch."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    seq_lens: Optional[Sequence[int]] = None  # explicit lengths, else drawn
    seq_len_range: Optional[tuple] = None  # inclusive (lo, hi) drawn per sequence
    top_k: Optional[int] = None  # None: all pages (dense)
    q_dtype: torch.dtype = torch.bfloat16
    kv_dtype: torch.dtype = torch.bfloat16
    kind: str = "iid"  # iid | page_offset | planted | centroid | shared_prefix
    contiguous: bool = False  # page id = b * pages_per_seq + j (no shuffle)
    extra_pool_pages: int = 0  # unreferenced pages added to the pool
    prefix_pages: int = 0  # shared_prefix: aliased pages at the head of each table
    suffix_pages: int = 0  # shared_prefix: private pages per sequence
    max_pages: Optional[int] = None  # page-table row capacity (default: longest)
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    "tiny": Spec(
        name="tiny", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
        page_size=16, seq_lens=(256, 256), top_k=4, q_dtype=torch.float32,
        kv_dtype=torch.float32, kind="iid", contiguous=True, seed=0),
    "gpt2_345m": Spec(
        name="gpt2_345m", batch=8, num_q_heads=16, num_kv_heads=16, head_dim=64,
        page_size=16, seq_lens=(8192,) * 8, top_k=154, q_dtype=torch.float32,
        kv_dtype=torch.bfloat16, kind="page_offset", seed=1),
    "llama3_8b": Spec(
        name="llama3_8b", batch=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=16, seq_len_range=(4096, 32768), top_k=128, max_pages=2048,
        kind="planted", seed=2),
    "long_context": Spec(
        name="long_context", batch=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
        page_size=32, seq_len_range=(65536, 131072), top_k=128, max_pages=4096,
        kind="centroid", seed=3),
    "shared_prefix": Spec(
        name="shared_prefix", batch=256, num_q_heads=32, num_kv_heads=8,
        head_dim=128, page_size=16, top_k=None, kind="shared_prefix",
        prefix_pages=128, suffix_pages=32, seed=4),
}


def spec_for(name: str, **overrides) -> Spec:
    """A named workload, optionally with fields replaced (smaller test cases)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


def _draw_seq_lens(spec: Spec, g: torch.Generator) -> torch.Tensor:
    if spec.kind == "shared_prefix":
        n = (spec.prefix_pages + spec.suffix_pages) * spec.page_size
        if spec.seq_lens is not None:
            assert len(spec.seq_lens) == spec.batch
            assert all(spec.prefix_pages * spec.page_size <= x <= n for x in spec.seq_lens)
            return torch.tensor(list(spec.seq_lens), dtype=torch.int32)
        return torch.full((spec.batch,), n, dtype=torch.int32)
    if spec.seq_lens is not None:
        assert len(spec.seq_lens) == spec.batch
        return torch.tensor(list(spec.seq_lens), dtype=torch.int32)
    lo, hi = spec.seq_len_range
    return torch.randint(lo, hi + 1, (spec.batch,), generator=g, dtype=torch.int64).to(torch.int32)


def make_inputs(spec: Spec) -> dict:
    """Draw one decode batch on the CPU.

    Returns a dict of CPU tensors:
      q           [B][Hq][d]              spec.q_dtype
      k_pool      [Npool][Hkv][P][d]      spec.kv_dtype
      v_pool      [Npool][Hkv][P][d]      spec.kv_dtype
      page_table  [B][max_pages] int32    physical page ids, -1 past the sequence
      seq_lens    [B] int32
      n_pages     [B] int32               ceil(seq_len / P)
      top_k       int (or None for dense)
      planted     [B][Hkv][n] int32 logical pages given the planted key
                  offset (-1 padded), or None for other kinds
      aligned     centroid kind: [B][Hkv][n] int32 logical pages whose
                  offset is the centroid the group's query was drawn near
                  (-1 padded), else None
      plus ``spec``.
    """
    g = torch.Generator().manual_seed(1_000_003 * spec.seed + 17)
    B, Hq, Hkv, d, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    G = spec.group
    assert Hq % Hkv == 0
    seq_lens = _draw_seq_lens(spec, g)
    n_pages = (seq_lens + P - 1) // P
    max_pages = spec.max_pages or int(n_pages.max())
    assert int(n_pages.max()) <= max_pages

    # ---- page table (logical page j of sequence b -> physical page id) ----
    if spec.kind == "shared_prefix":
        n_unique = spec.prefix_pages + B * spec.suffix_pages
        n_pool = n_unique + spec.extra_pool_pages
        perm = torch.randperm(n_pool, generator=g).to(torch.int32)
        table = torch.full((B, max_pages), -1, dtype=torch.int32)
        for b in range(B):
            table[b, :spec.prefix_pages] = perm[:spec.prefix_pages]
            s0 = spec.prefix_pages + b * spec.suffix_pages
            own = int(n_pages[b]) - spec.prefix_pages
            table[b, spec.prefix_pages:spec.prefix_pages + own] = perm[s0:s0 + own]
    else:
        total = int(n_pages.sum())
        n_pool = total + spec.extra_pool_pages
        if spec.contiguous:
            ids = torch.arange(n_pool, dtype=torch.int32)
        else:
            ids = torch.randperm(n_pool, generator=g).to(torch.int32)
        table = torch.full((B, max_pages), -1, dtype=torch.int32)
        off = 0
        for b in range(B):
            nb = int(n_pages[b])
            table[b, :nb] = ids[off:off + nb]
            off += nb

    # ---- values -----------------------------------------------------------
    q = torch.randn((B, Hq, d), generator=g, dtype=torch.float32)
    k = torch.randn((n_pool, Hkv, P, d), generator=g, dtype=torch.float32)
    v = torch.randn((n_pool, Hkv, P, d), generator=g, dtype=torch.float32)

    if spec.kind == "page_offset":
        # every (page, KV head) gets its own offset vector, std 0.5, for K and for V
        k += 0.5 * torch.randn((n_pool, Hkv, 1, d), generator=g, dtype=torch.float32)
        v += 0.5 * torch.randn((n_pool, Hkv, 1, d), generator=g, dtype=torch.float32)
    elif spec.kind == "planted":
        # 2 % of each sequence's pages (at least one) get K += 4 u per token,
        # u the unit-norm mean of the query group that reads this KV head
        qg = q.view(B, Hkv, G, d).mean(dim=2)
        u = qg / qg.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        n_plant_max = max(1, int(round(0.02 * int(n_pages.max()))))
        planted = torch.full((B, Hkv, n_plant_max), -1, dtype=torch.int32)
        for b in range(B):
            nb = int(n_pages[b])
            n_plant = max(1, int(round(0.02 * nb)))
            for h in range(Hkv):
                pick = torch.randperm(nb, generator=g)[:n_plant]
                planted[b, h, :n_plant] = pick.sort().values.to(torch.int32)
                phys = table[b, pick].long()
                k[phys, h] += 4.0 * u[b, h]
    elif spec.kind == "centroid":
        n_cent = 64
        cent = torch.randn((Hkv, n_cent, d), generator=g, dtype=torch.float32)
        assign = torch.randint(0, n_cent, (n_pool, Hkv), generator=g)
        off = cent[torch.arange(Hkv)[None, :].expand(n_pool, Hkv), assign]  # [Npool][Hkv][d]
        k += off[:, :, None, :]
        v += off[:, :, None, :]
        star = torch.randint(0, n_cent, (B, Hkv), generator=g)
        for b in range(B):
            for h in range(Hkv):
                q[b, h * G:(h + 1) * G] = cent[h, star[b, h]] + 0.5 * q[b, h * G:(h + 1) * G]
        lists = []
        for b in range(B):
            phys = table[b, :int(n_pages[b])].long()
            lists.append([torch.nonzero(assign[phys, h] == star[b, h]).flatten() for h in range(Hkv)])
        width = max(1, max(len(x) for row in lists for x in row))
        aligned = torch.full((B, Hkv, width), -1, dtype=torch.int32)
        for b in range(B):
            for h in range(Hkv):
                aligned[b, h, :len(lists[b][h])] = lists[b][h].to(torch.int32)

    if spec.kind != "planted":
        planted = None
    if spec.kind != "centroid":
        aligned = None
    q = q.to(spec.q_dtype)
    k = k.to(spec.kv_dtype)
    v = v.to(spec.kv_dtype)

    # slots past the end of each sequence's last page hold garbage (NaN)
    for b in range(B):
        nb = int(n_pages[b])
        valid_last = int(seq_lens[b]) - (nb - 1) * P
        if valid_last < P:
            p = int(table[b, nb - 1])
            k[p, :, valid_last:, :] = float("nan")
            v[p, :, valid_last:, :] = float("nan")

    return dict(spec=spec, q=q, k_pool=k, v_pool=v, page_table=table,
                seq_lens=seq_lens, n_pages=n_pages.to(torch.int32),
                top_k=spec.top_k, max_pages=max_pages, num_pool_pages=n_pool, planted=planted,
                aligned=aligned)


def q_variants(inputs: dict, count: int = 16, noise: float = 0.25, seed: int = 99) -> torch.Tensor:
    """``count`` perturbed copies of q (q + noise * N(0,1)) -> [count][B][Hq][d]."""
    g = torch.Generator().manual_seed(seed)
    q = inputs["q"].float()
    out = q[None] + noise * torch.randn((count,) + tuple(q.shape), generator=g, dtype=torch.float32)
    return out.to(inputs["q"].dtype)


def last_pages(inputs: dict) -> tuple:
    """(physical page id, valid tokens) of every sequence's last page.

    These are the pages a decode step appends to, so their metadata is the
    part refreshed every step.
    """
    P = inputs["spec"].page_size
    sl = inputs["seq_lens"].long()
    nb = inputs["n_pages"].long()
    ids = inputs["page_table"][torch.arange(len(sl)), nb - 1]
    valid = (sl - (nb - 1) * P).to(torch.int32)
    return ids.to(torch.int32), valid


def all_pages(inputs: dict) -> tuple:
    """(physical page id, valid tokens) of every referenced pool page, once each."""
    P = inputs["spec"].page_size
    table = inputs["page_table"]
    sl = inputs["seq_lens"]
    valid = {}
    for b in range(table.shape[0]):
        nb = int(inputs["n_pages"][b])
        for j in range(nb):
            p = int(table[b, j])
            valid[p] = min(P, int(sl[b]) - j * P)
    ids = torch.tensor(sorted(valid), dtype=torch.int32)
    vt = torch.tensor([valid[int(p)] for p in ids], dtype=torch.int32)
    return ids, vt


def dense_bytes(inputs: dict) -> int:
    """K+V bytes a dense decode over every token would read."""
    spec = inputs["spec"]
    es = torch.tensor([], dtype=spec.kv_dtype).element_size()
    return int(inputs["seq_lens"].long().sum()) * spec.num_kv_heads * spec.head_dim * 2 * es


def _check_spec(spec: Spec):
    assert spec.num_q_heads % spec.num_kv_heads == 0
    assert math.log2(spec.group).is_integer()
