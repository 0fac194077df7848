"""GPU parity of the three attention forms against the fp64 oracle.

Tolerances (the bar for attention outputs, fp32 on the GPU side): max-abs
<= 1e-2 and mean-relative (mean |gpu - ref| / mean |ref|) <= 2e-3 over all
output elements.  Page mass:
|gpu - ref| <= 1e-4 * mass + 1e-6 * rows, and every (sequence, KV head) row of
mass sums to its row count.  Selection, end to end: the GPU's pages, chosen
from the GPU's mass, equal the oracle's pages chosen from the oracle's own
fp64 mass, except swaps of pages within 1e-6 * rows of the cutoff, which are
counted and printed."""

import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decode_attention_paged_b300 as s3r
from workloads import (ATTN_QWEN3_1P7B_256SEQ, ATTN_QWEN3_8B_128SEQ, ATTN_TINY, bf16_to_bits, make_paged_kv,
                       make_queries)
from helpers import (assert_attn_close, attn_workspace, budget_b_max, compact_pool, host, kv_desc, run_verify_select,
                     selection_ties_vs_oracle_mass)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _oracle_inputs(kv):
    return bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool), host(kv.block_table)


def _check_mass(mass_gpu, mass_ref, rows):
    g = host(mass_gpu).astype(np.float64)
    w = mass_ref.shape[-1]
    np.testing.assert_array_less(np.abs(g[..., :w] - mass_ref), 1e-4 * np.abs(mass_ref) + 1e-6 * rows)
    assert np.all(g[..., w:] == 0.0)


# ---------------------------------------------------------------- small / ragged shapes

RAGGED = [1, 2, 15, 16, 17, 31, 32, 33, 47, 100, 255, 256, 257, 1000, 1023, 2049, 3001]


@pytest.mark.parametrize("q_heads,kv_heads", [(16, 8), (32, 8), (8, 8), (4, 1), (16, 2), (24, 1), (32, 1)])
def test_dense_decode_ragged(q_heads, kv_heads):
    lens = RAGGED + [5, 600, 64]
    kv = make_paged_kv(len(lens), q_heads, kv_heads, 4, seed=101, device=DEV, hist_lens=lens)
    q = make_queries(kv, 7)
    ws = attn_workspace(kv)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    ctx = kv.hist_lens + 1
    s3r.s3r_dense_decode_attn(kv_desc(kv), ctx, q, out, 1.0, ws)
    ws.check()
    kp, vp, bt = _oracle_inputs(kv)
    ref = oracle.dense_decode_attn(bf16_to_bits(q), kp, vp, bt, host(ctx), 1.0)
    assert_attn_close(out, ref, f"dense {q_heads}/{kv_heads}")


def test_dense_decode_zero_length_gives_zero_rows():
    lens = [0, 40, 0, 17]
    kv = make_paged_kv(4, 16, 8, 4, seed=102, device=DEV, hist_lens=[40, 40, 40, 40])
    q = make_queries(kv, 8)
    ws = attn_workspace(kv)
    out = torch.full(q.shape, 7.0, dtype=torch.float32, device=DEV)
    ctx = torch.tensor(lens, dtype=torch.int32, device=DEV)
    s3r.s3r_dense_decode_attn(kv_desc(kv), ctx, q, out, 1.0, ws)
    ws.check()
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    kp, vp, bt = _oracle_inputs(kv)
    ref = oracle.dense_decode_attn(bf16_to_bits(q), kp, vp, bt, np.array(lens), 1.0)
    assert_attn_close(out, ref, "dense zero-length")


# 17-32 rows per KV head run on the tcgen05 kernel: 32 rows, and 18 / 20 / 24 rows,
# where the second softmax group holds rows past R
@pytest.mark.parametrize("q_heads,kv_heads,T", [(16, 8, 4), (32, 8, 8), (16, 8, 1), (8, 8, 3), (64, 8, 4),
                                                 (4, 1, 8), (16, 8, 9), (32, 8, 5), (24, 8, 8), (64, 8, 3)])
def test_verify_ragged_with_mass(q_heads, kv_heads, T):
    lens = RAGGED
    kv = make_paged_kv(len(lens), q_heads, kv_heads, T, seed=103, device=DEV, hist_lens=lens)
    q = make_queries(kv, 9, rows=T)
    ws = attn_workspace(kv, rows=T)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    mass = torch.empty((len(lens), kv_heads, kv.max_pages + 3), dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, out, 1.0, ws, page_mass=mass)
    ws.check()
    kp, vp, bt = _oracle_inputs(kv)
    ref, mref = oracle.verify_attn(bf16_to_bits(q), kp, vp, bt, host(kv.hist_lens), 1.0)
    assert_attn_close(out, ref, f"verify {q_heads}/{kv_heads} T={T}")
    G = q_heads // kv_heads
    _check_mass(mass, mref, G * T)
    sums = host(mass).astype(np.float64).sum(axis=-1)
    np.testing.assert_allclose(sums, G * T, rtol=1e-4)
    # verify -> mass -> select on the GPU against the oracle's selection from its own mass
    sel_lens = (kv.hist_lens + T).to(torch.int32)
    for budget in (0.1, 0.3):
        b_max = budget_b_max(mass.shape[-1], budget)
        sel = torch.empty((len(lens), kv_heads, b_max), dtype=torch.int32, device=DEV)
        cnt = torch.empty((len(lens), kv_heads), dtype=torch.int32, device=DEV)
        s3r.s3r_select_draft_pages(mass, sel_lens, budget, sel, cnt, ws)
        ws.check()
        swaps = selection_ties_vs_oracle_mass(host(sel), host(cnt), mref, host(sel_lens), budget, G * T)
        assert swaps <= 2, swaps


def test_verify_without_mass_matches_with_mass():
    kv = make_paged_kv(9, 16, 8, 4, seed=104, device=DEV, hist_lens=[50, 3000, 7, 16, 900, 2048, 1, 333, 64])
    q = make_queries(kv, 10, rows=4)
    ws = attn_workspace(kv, rows=4)
    a = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    b = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    mass = torch.empty((9, 8, kv.max_pages), dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, a, 1.0, ws, page_mass=mass)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, b, 1.0, ws)
    ws.check()
    assert torch.equal(a, b)


def test_verify_row_equals_sequential_decodes_on_gpu():
    kv = make_paged_kv(6, 32, 8, 8, seed=105, device=DEV, hist_lens=[17, 500, 1024, 33, 4000, 15])
    q = make_queries(kv, 11, rows=8)
    ws = attn_workspace(kv, rows=8)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, out, 1.0, ws)
    for i in range(8):
        step = torch.empty(q[:, i].shape, dtype=torch.float32, device=DEV)
        s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens + i + 1, q[:, i].contiguous(), step, 1.0, ws)
        diff = (out[:, i].float() - step.float()).abs().max().item()
        assert diff <= 1e-2
    ws.check()


def _random_selection(kv, rng, b_max, count_lo=0):
    S, H = kv.num_seqs, kv.kv_heads
    L = host(kv.hist_lens)
    sel = np.full((S, H, b_max), -1, dtype=np.int32)
    cnt = np.zeros((S, H), dtype=np.int32)
    for s in range(S):
        P = math.ceil(int(L[s]) / 16)
        for h in range(H):
            c = int(rng.integers(min(count_lo, P), min(b_max, P) + 1)) if P > 0 else 0
            pick = rng.choice(P, size=c, replace=False) if c > 0 else np.zeros(0, dtype=np.int64)
            sel[s, h, :c] = pick          # any order
            cnt[s, h] = c
    return sel, cnt


@pytest.mark.parametrize("q_heads,kv_heads", [(16, 8), (32, 8), (4, 1), (32, 1)])
def test_sparse_draft_random_selections(q_heads, kv_heads):
    lens = RAGGED
    kv = make_paged_kv(len(lens), q_heads, kv_heads, 4, seed=106, device=DEV, hist_lens=lens)
    rng = np.random.default_rng(3)
    sel, cnt = _random_selection(kv, rng, b_max=24)
    sel_t = torch.from_numpy(sel).to(DEV)
    cnt_t = torch.from_numpy(cnt).to(DEV)
    ws = attn_workspace(kv)
    kp, vp, bt = _oracle_inputs(kv)
    for j in range(4):
        q = make_queries(kv, 20 + j)
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        s3r.s3r_sparse_draft_attn(kv_desc(kv), kv.hist_lens, j, sel_t, cnt_t, q, out, 1.0, ws)
        ws.check()
        ref = oracle.sparse_draft_attn(bf16_to_bits(q), kp, vp, bt, host(kv.hist_lens), j, sel, cnt, 1.0)
        assert_attn_close(out, ref, f"sparse j={j}")


def test_sparse_all_pages_equals_dense_on_gpu():
    lens = [40, 16, 1000, 3, 257]
    kv = make_paged_kv(len(lens), 16, 8, 4, seed=107, device=DEV, hist_lens=lens)
    P = max(math.ceil(x / 16) for x in lens)
    sel = torch.full((len(lens), 8, P), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros((len(lens), 8), dtype=torch.int32, device=DEV)
    for s, L in enumerate(lens):
        Ps = math.ceil(L / 16)
        sel[s, :, :Ps] = torch.arange(Ps, dtype=torch.int32, device=DEV)
        cnt[s] = Ps
    ws = attn_workspace(kv)
    for j in range(4):
        q = make_queries(kv, 30 + j)
        a = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        b = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        s3r.s3r_sparse_draft_attn(kv_desc(kv), kv.hist_lens, j, sel, cnt, q, a, 1.0, ws)
        s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens + j + 1, q, b, 1.0, ws)
        assert (a.float() - b.float()).abs().max().item() <= 1e-2
    ws.check()


def test_sparse_empty_selection_reads_only_the_tail():
    kv = make_paged_kv(3, 16, 8, 4, seed=108, device=DEV, hist_lens=[35, 64, 100])
    sel = torch.full((3, 8, 4), -1, dtype=torch.int32, device=DEV)
    cnt = torch.zeros((3, 8), dtype=torch.int32, device=DEV)
    ws = attn_workspace(kv)
    kp, vp, bt = _oracle_inputs(kv)
    q = make_queries(kv, 40)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    s3r.s3r_sparse_draft_attn(kv_desc(kv), kv.hist_lens, 2, sel, cnt, q, out, 1.0, ws)
    ws.check()
    ref = oracle.sparse_draft_attn(bf16_to_bits(q), kp, vp, bt, host(kv.hist_lens), 2, host(sel), host(cnt), 1.0)
    assert_attn_close(out, ref, "tail only")


def test_sm_scale_is_applied():
    kv = make_paged_kv(4, 16, 8, 4, seed=109, device=DEV, hist_lens=[300, 20, 77, 1000])
    q = make_queries(kv, 41)
    ws = attn_workspace(kv)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens, q, out, 0.3, ws)
    kp, vp, bt = _oracle_inputs(kv)
    ref = oracle.dense_decode_attn(bf16_to_bits(q), kp, vp, bt, host(kv.hist_lens), 0.3)
    assert_attn_close(out, ref, "sm_scale")


# ---------------------------------------------------------------- the workloads at full size

def _full_round_check(cfg, budget, n_check, seed_q=500):
    # capacity for the verified block and the next round's draft tail
    kv = make_paged_kv(cfg.num_seqs, cfg.q_heads, cfg.kv_heads, 2 * cfg.k, seed=cfg.seed, device=DEV,
                       hist_min=cfg.hist_min, hist_max=cfg.hist_max)
    T = cfg.k
    qv = make_queries(kv, seed_q, rows=T)
    ws = attn_workspace(kv, rows=T)
    out_v, mass, sel, cnt, sel_lens = run_verify_select(kv, qv, budget, ws)
    # next round's drafts read the selection (history grows by the accepted block)
    kv2_hist = sel_lens
    qd = [make_queries(kv, seed_q + 1 + j) for j in range(T)]
    outs_d = []
    for j in range(T):
        o = torch.empty(qd[j].shape, dtype=torch.float32, device=DEV)
        s3r.s3r_sparse_draft_attn(kv_desc(kv), kv2_hist, j, sel, cnt, qd[j], o, 1.0, ws)
        outs_d.append(o)
    qdense = make_queries(kv, seed_q + 99)
    out_dense = torch.empty(qdense.shape, dtype=torch.float32, device=DEV)
    s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens + 1, qdense, out_dense, 1.0, ws)
    torch.cuda.synchronize()
    ws.check()

    # properties at full size, every sequence: mass rows sum to G*T, and verify row j
    # equals a dense decode step over the first L + j + 1 tokens
    G = cfg.q_heads // cfg.kv_heads
    np.testing.assert_allclose(host(mass).astype(np.float64).sum(axis=-1), G * T, rtol=1e-4)
    for j in range(T):
        step = torch.empty(qv[:, j].shape, dtype=torch.float32, device=DEV)
        s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens + j + 1, qv[:, j].contiguous(), step, 1.0, ws)
        assert (out_v[:, j] - step).abs().max().item() <= 1e-2, f"{cfg.name} verify row {j} vs dense"
    ws.check()

    seqs = sorted(np.random.default_rng(cfg.seed).choice(cfg.num_seqs, size=n_check, replace=False).tolist())
    kp, vp, bt = compact_pool(kv, seqs)
    Ls = host(kv.hist_lens)[seqs]
    ref_v, mref = oracle.verify_attn(bf16_to_bits(qv[seqs]), kp, vp, bt, Ls, 1.0)
    assert_attn_close(out_v[seqs], ref_v, f"{cfg.name} verify")
    _check_mass(mass[seqs], mref, G * T)
    # selection from the GPU mass equals the oracle rule applied to the same mass
    sel_ref, cnt_ref = oracle.select_draft_pages(host(mass[seqs]), host(sel_lens)[seqs], budget, 1, 4,
                                                 b_max=sel.shape[-1])
    assert np.array_equal(host(cnt[seqs]), cnt_ref)
    assert np.array_equal(host(sel[seqs]), sel_ref)
    # and, end to end, the oracle's selection from its own fp64 mass, up to counted ties
    swaps = selection_ties_vs_oracle_mass(host(sel[seqs]), host(cnt[seqs]), mref, host(sel_lens)[seqs], budget,
                                          G * T)
    print(f"{cfg.name} budget {budget}: {swaps} selection tie swaps over {n_check * cfg.kv_heads} pairs")
    assert swaps <= max(2, n_check * cfg.kv_heads // 100)
    for j in range(T):
        ref_d = oracle.sparse_draft_attn(bf16_to_bits(qd[j][seqs]), kp, vp, bt, host(kv2_hist)[seqs], j,
                                         host(sel[seqs]), host(cnt[seqs]), 1.0)
        assert_attn_close(outs_d[j][seqs], ref_d, f"{cfg.name} draft j={j}")
    ref_dense = oracle.dense_decode_attn(bf16_to_bits(qdense[seqs]), kp, vp, bt, Ls + 1, 1.0)
    assert_attn_close(out_dense[seqs], ref_dense, f"{cfg.name} dense")


def test_tiny_workload_full():
    _full_round_check(ATTN_TINY, 0.10, n_check=4)


def test_qwen3_1p7b_256seq_sampled():
    _full_round_check(ATTN_QWEN3_1P7B_256SEQ, 0.05, n_check=24)


@pytest.mark.parametrize("budget", [0.05, 0.50])
def test_qwen3_8b_128seq_sampled(budget):
    _full_round_check(ATTN_QWEN3_8B_128SEQ, budget, n_check=16)


def test_long_context_dense_and_verify_with_mass():
    """A 100,003-token history (6,251 pages) next to tiny ones: the page stream
    and the split merges stay exact far beyond the workloads' lengths."""
    lens = [100_003, 3, 17]
    kv = make_paged_kv(len(lens), 16, 8, 4, seed=107, device=DEV, hist_lens=lens, heavy_per_head=4)
    kp, vp, bt = _oracle_inputs(kv)
    ws = attn_workspace(kv, rows=4)
    qd = make_queries(kv, 11)
    out_d = torch.empty(qd.shape, dtype=torch.float32, device=DEV)
    s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens + 1, qd, out_d, 1.0, ws)
    qv = make_queries(kv, 12, rows=4)
    out_v = torch.empty(qv.shape, dtype=torch.float32, device=DEV)
    mass = torch.empty((len(lens), 8, kv.max_pages), dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, qv, out_v, 1.0, ws, page_mass=mass)
    ws.check()
    assert_attn_close(out_d, oracle.dense_decode_attn(bf16_to_bits(qd), kp, vp, bt, host(kv.hist_lens) + 1, 1.0),
                      "long dense")
    ref_v, mref = oracle.verify_attn(bf16_to_bits(qv), kp, vp, bt, host(kv.hist_lens), 1.0)
    assert_attn_close(out_v, ref_v, "long verify")
    _check_mass(mass, mref, 2 * 4)
