"""Shared plumbing for the GPU parity tests: run the CUDA path through the
binding, move the same inputs to the host for the oracle, and compare with
the tolerances the tests state."""

import math

import numpy as np
import torch

import speculative_decode_attention_paged_b300 as s3r
from workloads import bf16_to_bits

# Attention tolerances: max-abs and mean-relative error of the fp32 outputs.
ATTN_MAX_ABS = 1e-2
ATTN_MEAN_REL = 2e-3


def attn_errors(gpu_out, ref_f64):
    g = gpu_out.detach().to(torch.float64).cpu().numpy()
    d = np.abs(g - ref_f64)
    denom = np.abs(ref_f64).mean()
    return float(d.max(initial=0.0)), float(d.mean() / denom) if denom > 0 else float(d.mean())


def assert_attn_close(gpu_out, ref_f64, what=""):
    mx, mr = attn_errors(gpu_out, ref_f64)
    assert mx <= ATTN_MAX_ABS, f"{what}: max-abs {mx:.3e}"
    assert mr <= ATTN_MEAN_REL, f"{what}: mean-rel {mr:.3e}"
    return mx, mr


def kv_desc(kv):
    return s3r.PagedKVDesc(kv.k_pool, kv.v_pool, kv.block_table, kv.q_heads)


def attn_workspace(kv, rows=1):
    return s3r.Workspace(s3r.s3r_attn_workspace_size(kv_desc(kv), rows))


def compact_pool(kv, seqs):
    """The pages of the listed sequences only, as host arrays with a remapped
    block table (plain indexing; keeps full-size oracle checks small)."""
    idx = torch.as_tensor(list(seqs), device=kv.block_table.device, dtype=torch.long)
    bt = kv.block_table[idx].long()
    valid = bt >= 0
    uniq, inv = torch.unique(bt[valid], return_inverse=True)
    new_bt = torch.full_like(bt, -1)
    new_bt[valid] = inv
    return bf16_to_bits(kv.k_pool[uniq]), bf16_to_bits(kv.v_pool[uniq]), new_bt.cpu().numpy()


def host(t):
    return t.detach().cpu().numpy()


def ceil_div(a, b):
    return -(-a // b)


def run_verify_select(kv, q_verify, budget, ws, mass_stride=None, n_sink=1, n_recent=4):
    """verify (with page mass) then select on the GPU; returns everything."""
    S, T = q_verify.shape[0], q_verify.shape[1]
    desc = kv_desc(kv)
    out = torch.empty(q_verify.shape, dtype=torch.float32, device=q_verify.device)
    stride = mass_stride or kv.max_pages
    mass = torch.empty((S, kv.kv_heads, stride), dtype=torch.float32, device=q_verify.device)
    s3r.s3r_verify_attn(desc, kv.hist_lens, q_verify, out, 1.0, ws, page_mass=mass)
    sel_lens = (kv.hist_lens + T).to(torch.int32)
    b_max = budget_b_max(stride, budget, n_sink, n_recent)
    sel = torch.empty((S, kv.kv_heads, b_max), dtype=torch.int32, device=q_verify.device)
    cnt = torch.empty((S, kv.kv_heads), dtype=torch.int32, device=q_verify.device)
    s3r.s3r_select_draft_pages(mass, sel_lens, budget, sel, cnt, ws, n_sink=n_sink, n_recent=n_recent)
    return out, mass, sel, cnt, sel_lens


def budget_b_max(num_pages, budget, n_sink=1, n_recent=4):
    P = int(num_pages)
    mand = min(n_sink, P) + (P - max(max(P - n_recent, 0), min(n_sink, P)))
    return max(min(P, max(math.ceil(budget * P - 1e-9), mand)), 1)


# Selection ties: the GPU selects from its fp32 page mass, the oracle from its
# own fp64 mass.  A page where the two choices differ must lie within
# SELECT_TIE * (rows per KV head) of the cutoff in the oracle's mass (each of
# the G*T rows contributes mass 1, so the window scales with the row count).
SELECT_TIE = 1e-6


def selection_ties_vs_oracle_mass(sel_gpu, cnt_gpu, mass_ref, sel_lens, budget, rows, n_sink=1, n_recent=4):
    """Checks a GPU selection against the oracle's selection from the oracle's
    own mass, and returns the number of tie swaps (pairs of pages, one chosen
    by each side only, both within the window of the cutoff).

    sel_gpu [S][H][b_max], cnt_gpu [S][H] (GPU, from the GPU's mass);
    mass_ref [S][H][>= pages] (oracle fp64); sel_lens [S]; rows = G * T."""
    import oracle
    sel_gpu, cnt_gpu = np.asarray(sel_gpu), np.asarray(cnt_gpu)
    mass_ref = np.asarray(mass_ref, dtype=np.float64)
    S, H = cnt_gpu.shape
    ref_sel, ref_cnt = oracle.select_draft_pages(mass_ref, sel_lens, budget, n_sink, n_recent,
                                                 b_max=sel_gpu.shape[-1])
    assert np.array_equal(cnt_gpu, ref_cnt), "page budgets differ"
    tol = SELECT_TIE * rows
    swaps = 0
    for s in range(S):
        P = ceil_div(int(sel_lens[s]), 16)
        B, mandatory = oracle.selection_budget(P, budget, n_sink, n_recent)
        for h in range(H):
            c = int(cnt_gpu[s, h])
            g = sel_gpu[s, h, :c]
            assert np.all(np.diff(g) > 0), f"({s},{h}): GPU selection not ascending"
            assert np.all(sel_gpu[s, h, c:] == -1)
            gs, rs = set(g.tolist()), set(ref_sel[s, h, :c].tolist())
            if gs == rs:
                continue
            assert mandatory <= gs, f"({s},{h}): a mandatory page is missing"
            rest = sorted(rs - mandatory, key=lambda pg: (-mass_ref[s, h, pg], pg))
            cutoff = mass_ref[s, h, rest[-1]]
            only_g, only_r = gs - rs, rs - gs
            for pg in only_g:
                assert mass_ref[s, h, pg] >= cutoff - tol, \
                    f"({s},{h}) page {pg}: mass {mass_ref[s, h, pg]:.9g} vs cutoff {cutoff:.9g}"
            for pg in only_r:
                assert mass_ref[s, h, pg] <= cutoff + tol, \
                    f"({s},{h}) page {pg}: mass {mass_ref[s, h, pg]:.9g} vs cutoff {cutoff:.9g}"
            swaps += len(only_g)
    return swaps
