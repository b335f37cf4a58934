"""Seeded synthetic inputs shaped like the workloads of the method's pages.

This module only draws inputs: queries, paged K/V caches, block tables and
sequence lengths.  It holds none of the method's arithmetic (no representation
vectors, scores, selection or attention), so that the CUDA path and the oracle
both consume it without sharing any of the computation they are checked on.

Recipe (every draw comes from one seeded ``torch.Generator`` on the target device):
  * q, K, V ~ N(0, 1), rounded once to the storage dtype (bf16 or fp32);
  * one page = ``block_size`` tokens of one request; the cache is laid out
    [page][kv_head][token][head_dim], so one (page, kv head) slab is contiguous;
  * pages shared by a common prefix exist once physically and are referenced by
    every request's block table (prefix sharing with reference counting on the ATB
    reuse page, §2.1 and §3.3);
  * with ``shuffle`` the physical page ids are a seeded random permutation;
  * planted relevance: a seeded ``plant_fraction`` of each request's unshared blocks
    has ``plant_scale * u_h`` added to every key of kv head h, where u_h is the unit
    vector along the sum of the queries of head h's query group;
  * unused block-table entries hold -1.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence

import torch

BF16, F32 = 0, 1


@dataclasses.dataclass
class Case:
    cfg: dict                 # num_q_heads, num_kv_heads, head_dim, block_size, init_tokens,
                              # local_tokens, topk_percent, dense_boundary, dtype
    q: torch.Tensor           # [B][Hq][d]
    k_cache: torch.Tensor     # [P][Hkv][S][d]
    v_cache: torch.Tensor     # [P][Hkv][S][d]
    block_table: torch.Tensor  # [B][max_blocks] int32
    seq_lens: torch.Tensor    # [B] int32
    prompt_lens: torch.Tensor  # [B] int32
    page_ids: torch.Tensor    # [n] int32: every physical page in use, once
    page_valid: torch.Tensor  # [n] int32: tokens present in that page
    name: str = ""

    @property
    def batch(self) -> int:
        return self.block_table.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def num_pages(self) -> int:
        return self.k_cache.shape[0]

    def to(self, device) -> "Case":
        return dataclasses.replace(self, **{f.name: getattr(self, f.name).to(device)
                                            for f in dataclasses.fields(self)
                                            if isinstance(getattr(self, f.name), torch.Tensor)})


def _storage(dtype: int) -> torch.dtype:
    return torch.bfloat16 if dtype == BF16 else torch.float32


def make_case(*, seq_lens: Sequence[int], num_q_heads: int, num_kv_heads: int,
              head_dim: int, dtype: int = BF16, block_size: int = 128,
              init_tokens: int = 1024, local_tokens: int = 7192, topk_percent: float = 0.2,
              dense_boundary: int = 32768, prompt_lens: Sequence[int] | None = None,
              shared_prefix_tokens: int = 0, shuffle: bool = True,
              plant_fraction: float = 0.0, plant_scale: float = 0.5,
              extra_blocks: int = 0, seed: int = 0, device="cpu", name: str = "") -> Case:
    S = block_size
    B = len(seq_lens)
    if shared_prefix_tokens % S:
        raise ValueError("a shared prefix must cover whole pages")
    if any(L < shared_prefix_tokens for L in seq_lens):
        raise ValueError("every request must contain the shared prefix")
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    store = _storage(dtype)

    n_shared = shared_prefix_tokens // S
    nblocks = [(L + S - 1) // S for L in seq_lens]
    max_blocks = max(max(nblocks), 1) + extra_blocks
    P = n_shared + sum(nb - n_shared for nb in nblocks)
    perm = (torch.randperm(P, generator=g, device=device) if shuffle
            else torch.arange(P, device=device)).to(torch.int32).cpu()

    # Logical page numbering: shared prefix first, then each request's own blocks.
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    valid = torch.zeros(P, dtype=torch.int32)
    owner = torch.full((P,), -1, dtype=torch.int64)      # request owning an unshared page
    logical = n_shared
    for b in range(n_shared):
        valid[b] = S
    for r, L in enumerate(seq_lens):
        for b in range(nblocks[r]):
            if b < n_shared:
                table[r, b] = perm[b]
                continue
            table[r, b] = perm[logical]
            valid[logical] = min(S, L - b * S)
            owner[logical] = r
            logical += 1
    phys_valid = torch.zeros(P, dtype=torch.int32)
    phys_valid[perm.long()] = valid
    phys_owner = torch.full((P,), -1, dtype=torch.int64)
    phys_owner[perm.long()] = owner

    q = torch.randn(B, num_q_heads, head_dim, generator=g, device=device).to(store)

    # Planted pages: a seeded fraction of each request's unshared blocks.
    planted = torch.zeros(P, dtype=torch.bool)
    if plant_fraction > 0:
        for r in range(B):
            own = [b for b in range(n_shared, nblocks[r])]
            n_plant = int(round(plant_fraction * len(own)))
            if n_plant:
                pick = torch.randperm(len(own), generator=g, device=device)[:n_plant].cpu()
                for i in pick.tolist():
                    planted[table[r, own[i]].item()] = True
    G = num_q_heads // num_kv_heads
    qsum = q.float().reshape(B, num_kv_heads, G, head_dim).sum(2)
    qdir = qsum / qsum.norm(dim=-1, keepdim=True).clamp_min(1e-30)   # [B][Hkv][d]

    k_cache = torch.empty(P, num_kv_heads, S, head_dim, dtype=store, device=device)
    v_cache = torch.empty_like(k_cache)
    chunk = max(1, (1 << 27) // (num_kv_heads * S * head_dim))
    for p0 in range(0, P, chunk):
        p1 = min(P, p0 + chunk)
        kc = torch.randn(p1 - p0, num_kv_heads, S, head_dim, generator=g, device=device)
        sel = planted[p0:p1].nonzero().flatten()
        if sel.numel():
            rows = phys_owner[p0 + sel]
            kc[sel.to(device)] += plant_scale * qdir[rows.to(device)].unsqueeze(2)
        k_cache[p0:p1] = kc.to(store)
        v_cache[p0:p1] = torch.randn(p1 - p0, num_kv_heads, S, head_dim, generator=g,
                                     device=device).to(store)

    used = torch.nonzero(phys_valid > 0).flatten().to(torch.int32)
    cfg = dict(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
               block_size=S, init_tokens=init_tokens, local_tokens=local_tokens,
               topk_percent=float(topk_percent), dense_boundary=dense_boundary, dtype=dtype)
    Ls = torch.tensor(list(seq_lens), dtype=torch.int32)
    prompts = Ls.clone() if prompt_lens is None else torch.tensor(list(prompt_lens),
                                                                  dtype=torch.int32)
    return Case(cfg=cfg, q=q, k_cache=k_cache, v_cache=v_cache,
                block_table=table.to(device), seq_lens=Ls.to(device),
                prompt_lens=prompts.to(device), page_ids=used.to(device),
                page_valid=phys_valid[used.long()].to(device), name=name)


def _uniform_ints(lo: int, hi: int, n: int, seed: int) -> list[int]:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# ---- the five workloads of the method's evaluation, by shape -----------------------------

def tiny(seed: int = 1, device="cpu", **over) -> Case:
    """1 request, 4 q heads / 1 kv head, d 64, fp32, 4096 tokens, init 256, window 512,
    top-k 20 %, identity block table; DENSE_BOUNDARY 0 so that the sparse path runs."""
    kw = dict(seq_lens=[4096], num_q_heads=4, num_kv_heads=1, head_dim=64, dtype=F32,
              init_tokens=256, local_tokens=512, topk_percent=0.2, dense_boundary=0,
              shuffle=False, seed=seed, device=device, name="tiny-4096-fp32")
    kw.update(over)
    return make_case(**kw)


def llama8b_layer(seq_len: int = 65536, seed: int = 2, device="cpu", **over) -> Case:
    """Llama-3-8B-shaped layer: 32 q / 8 kv heads, d 128, bf16, init 1024, window 7192,
    top-k 0.2, 5 % planted blocks, shuffled pages."""
    kw = dict(seq_lens=[seq_len], num_q_heads=32, num_kv_heads=8, head_dim=128, dtype=BF16,
              plant_fraction=0.05, seed=seed, device=device,
              name=f"llama8b-layer-{seq_len}-bf16")
    kw.update(over)
    return make_case(**kw)


def ragged_batch(n_requests: int = 16, lo: int = 32768, hi: int = 131072, seed: int = 3,
                 device="cpu", **over) -> Case:
    """Ragged paged batch: lengths uniform in [lo, hi], 32/8 heads, d 128, bf16,
    shuffled physical pages."""
    lens = _uniform_ints(lo, hi, n_requests, seed)
    kw = dict(seq_lens=lens, num_q_heads=32, num_kv_heads=8, head_dim=128, dtype=BF16,
              seed=seed, device=device, name=f"ragged-{n_requests}x[{lo},{hi}]-bf16")
    kw.update(over)
    return make_case(**kw)


def dense_vs_sparse(topk_percent: float = 0.2, batch: int = 4, seq_len: int = 131072,
                    seed: int = 4, device="cpu", **over) -> Case:
    """Same seeded cache for every ratio: batch 4 x 131072 tokens, 32/8, d 128, bf16,
    3 % planted blocks; ratio 1.0 is dense paged decode."""
    kw = dict(seq_lens=[seq_len] * batch, num_q_heads=32, num_kv_heads=8, head_dim=128,
              dtype=BF16, topk_percent=topk_percent, plant_fraction=0.03, seed=seed,
              device=device, name=f"dense-vs-sparse-{batch}x{seq_len}-p{topk_percent}")
    kw.update(over)
    return make_case(**kw)


def prefix_shared(n_requests: int = 64, prefix: int = 16384, lo: int = 2048,
                  hi: int = 8192, seed: int = 5, device="cpu", **over) -> Case:
    """70B-shaped prefix sharing: 64/8 heads, d 128, bf16; a shared prefix (one physical
    copy) plus a unique suffix of lo..hi tokens; DENSE_BOUNDARY 0 so the sparse path runs."""
    lens = [prefix + x for x in _uniform_ints(lo, hi, n_requests, seed)]
    kw = dict(seq_lens=lens, num_q_heads=64, num_kv_heads=8, head_dim=128, dtype=BF16,
              shared_prefix_tokens=prefix, dense_boundary=0, seed=seed, device=device,
              name=f"prefix-shared-{n_requests}x({prefix}+[{lo},{hi}])-bf16")
    kw.update(over)
    return make_case(**kw)


def to_oracle_arrays(case: Case) -> dict:
    """Host numpy views for the oracle: bf16 as uint16 bit patterns, fp32 as float32."""
    def host(t: torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view("uint16")
        return t.numpy()
    return dict(q=host(case.q), k_cache=host(case.k_cache), v_cache=host(case.v_cache),
                block_table=host(case.block_table), seq_lens=host(case.seq_lens),
                prompt_lens=host(case.prompt_lens), page_ids=host(case.page_ids),
                page_valid=host(case.page_valid))


def bytes_per_elem(dtype: int) -> int:
    return 2 if dtype == BF16 else 4


def pages_for(seq_len: int, block_size: int = 128) -> int:
    return math.ceil(seq_len / block_size)
