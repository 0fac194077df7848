"""Paged bf16 KV pools, block tables and queries with planted heavy hitters.

Recipe:
  * history lengths L ~ U{hist_min .. hist_max} (or given);
  * every sequence owns ceil(max(L + k, capacity) / 16) pages; the physical
    pages of the pool are a random permutation, so the block table is
    scattered across the pool;
  * K, V ~ N(0, 1) rounded to bf16, pool layout [page][kv_head][16][head_dim];
  * per (sequence, KV head): a random unit direction u and `heavy_per_head`
    distinct heavy tokens drawn from pages [1, P-5) of the history, P =
    ceil(L / 16) (outside the always-kept first page and last four pages);
    a heavy key is z + a*u;
  * every query of the head group (all verify rows and draft steps) is
    (g + c*u) / sqrt(head_dim) with g ~ N(0, I), a = c = sqrt(heavy_score *
    sqrt(head_dim)), so a heavy key scores heavy_score above the N(0, ~1.35)
    background on average.

All randomness comes from one torch.Generator per call, seeded explicitly.
"""

import math
from dataclasses import dataclass

import numpy as np
import torch

PAGE_SIZE = 16


@dataclass
class PagedKV:
    k_pool: torch.Tensor        # [NP][Hkv][16][D] bf16
    v_pool: torch.Tensor        # [NP][Hkv][16][D] bf16
    block_table: torch.Tensor   # [S][max_pages] int32, -1 = unused slot
    hist_lens: torch.Tensor     # [S] int32, L
    u_hat: torch.Tensor         # [S][Hkv][D] float32 heavy direction
    heavy_tokens: torch.Tensor  # [S][Hkv][n_heavy] int64 logical token positions (-1 = none)
    q_heads: int
    k: int
    heavy_score: float

    @property
    def num_seqs(self):
        return self.block_table.shape[0]

    @property
    def kv_heads(self):
        return self.k_pool.shape[1]

    @property
    def head_dim(self):
        return self.k_pool.shape[3]

    @property
    def max_pages(self):
        return self.block_table.shape[1]

    @property
    def num_phys_pages(self):
        return self.k_pool.shape[0]


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns on the host."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _randn_bf16(shape, gen, device, chunk_rows=2048):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def make_paged_kv(num_seqs, q_heads, kv_heads, k, seed, device="cpu", hist_lens=None,
                  hist_min=None, hist_max=None, head_dim=128, capacity_tokens=None,
                  heavy_per_head=8, heavy_score=4.0, spare_pages=0):
    """Build one layer's paged KV cache (see the module docstring)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    S, Hkv, D = int(num_seqs), int(kv_heads), int(head_dim)
    if hist_lens is None:
        hist_lens = torch.randint(int(hist_min), int(hist_max) + 1, (S,), generator=gen, device=device)
    hist_lens = torch.as_tensor(hist_lens, device=device).to(torch.int64)
    need = hist_lens + int(k)
    if capacity_tokens is not None:
        need = torch.clamp(need, min=int(capacity_tokens))
    pages = (need + PAGE_SIZE - 1) // PAGE_SIZE
    total = int(pages.sum().item()) + int(spare_pages)
    max_pages = max(int(pages.max().item()) if S > 0 else 0, 1)

    perm = torch.randperm(max(total, 1), generator=gen, device=device)[:total]
    offs = torch.cumsum(pages, 0) - pages
    slot = torch.arange(max_pages, device=device)[None, :]
    idx = offs[:, None] + slot
    used = slot < pages[:, None]
    block_table = torch.where(used, perm[torch.clamp(idx, max=max(total - 1, 0))],
                              torch.full_like(idx, -1)).to(torch.int32)

    k_pool = _randn_bf16((max(total, 1), Hkv, PAGE_SIZE, D), gen, device)
    v_pool = _randn_bf16((max(total, 1), Hkv, PAGE_SIZE, D), gen, device)

    u_hat = torch.randn((S, Hkv, D), generator=gen, device=device, dtype=torch.float32)
    u_hat = u_hat / u_hat.norm(dim=-1, keepdim=True)

    # Heavy hitters: distinct tokens in pages [1, P-5) of each history.
    hist_pages = (hist_lens + PAGE_SIZE - 1) // PAGE_SIZE
    lo_tok = PAGE_SIZE
    hi_tok = torch.clamp(hist_pages - 5, min=1) * PAGE_SIZE          # exclusive
    span = torch.clamp(hi_tok - lo_tok, min=0)
    nh = int(heavy_per_head)
    heavy = torch.full((S, Hkv, nh), -1, dtype=torch.int64, device=device)
    max_span = int(span.max().item()) if S > 0 else 0
    if nh > 0 and max_span >= nh:
        keys = torch.rand((S, Hkv, max_span), generator=gen, device=device)
        keys = torch.where(torch.arange(max_span, device=device)[None, None, :] < span[:, None, None],
                           keys, torch.full_like(keys, -1.0))
        top = torch.topk(keys, nh, dim=-1).indices
        ok = (span[:, None, None] >= nh).expand(S, Hkv, nh)
        heavy = torch.where(ok, top + lo_tok, heavy)
        a = math.sqrt(float(heavy_score) * math.sqrt(D))
        s_idx, h_idx, j_idx = torch.nonzero(heavy >= 0, as_tuple=True)
        tok = heavy[s_idx, h_idx, j_idx]
        phys = block_table[s_idx, tok // PAGE_SIZE].to(torch.int64)
        rows = k_pool[phys, h_idx, tok % PAGE_SIZE].to(torch.float32)
        k_pool[phys, h_idx, tok % PAGE_SIZE] = (rows + a * u_hat[s_idx, h_idx]).to(torch.bfloat16)

    return PagedKV(k_pool=k_pool, v_pool=v_pool, block_table=block_table,
                   hist_lens=hist_lens.to(torch.int32), u_hat=u_hat, heavy_tokens=heavy,
                   q_heads=int(q_heads), k=int(k), heavy_score=float(heavy_score))


def make_queries(kv: PagedKV, seed, rows=None):
    """Queries aligned with each group's heavy direction.

    rows=None -> [S][Hq][D] (one decode / draft step); rows=T -> [S][T][Hq][D].
    """
    device = kv.k_pool.device
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    S, Hkv, D, Hq = kv.num_seqs, kv.kv_heads, kv.head_dim, kv.q_heads
    G = Hq // Hkv
    c = math.sqrt(kv.heavy_score * math.sqrt(D))
    u = kv.u_hat.repeat_interleave(G, dim=1)          # [S][Hq][D]
    shape = (S, Hq, D) if rows is None else (S, int(rows), Hq, D)
    g = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if rows is not None:
        u = u[:, None]
    return ((g + c * u) / math.sqrt(D)).to(torch.bfloat16)
