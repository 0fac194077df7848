"""Two closed S³R rounds over two layers through the C ABI, checked stage by
stage against the oracle on the inputs each GPU stage consumed:

  draft step j: append the draft row, sparse draft attention over the previous
      round's selection, draft-token sampling from q_j (strided in place);
  verify: append the k + 1 dense block rows, verify them with page mass;
  exact speculative sampling; length commit L' = L + n_acc + 1; selection of
  the next round's pages from the verify mass over L'.

The second round starts from the first round's L' and selection.  Pools are compared bit for
bit, attention with the attention tolerances, page mass with the mass
tolerance, tokens and accepted counts exactly up to the sampler's tie rules,
lengths exactly, and selections exactly when the selection oracle reads the
GPU's fp32 mass and up to counted cutoff ties when it reads its own fp64
mass."""

import math

import numpy as np
import pytest
import torch
from scipy import special

import oracle
import speculative_decode_attention_paged_b300 as s3r
from helpers import assert_attn_close, budget_b_max, host, kv_desc, selection_ties_vs_oracle_mass
from test_gpu_attention import _check_mass
from test_gpu_spec_sample import CDF_TIE, compare
from workloads import bf16_to_bits, make_paged_kv, make_queries, make_spec_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
S, HQ, HKV, K, V, BUDGET, LAYERS, ROUNDS = 6, 16, 8, 4, 2048, 0.25, 2, 2
SEED, OFFSET = 99, 5


def _bf16(shape, gen):
    return torch.randn(shape, generator=gen, device=DEV).to(torch.bfloat16)


def _check_draft_tokens(q_logits_j, got, seed, offset, j):
    ref, det = oracle.sample_draft_tokens(q_logits_j, seed, offset, j)
    for s in np.nonzero(got != ref)[0]:                 # inverse-CDF ties only
        row = special.softmax(q_logits_j[s].astype(np.float64))
        C = np.cumsum(row)
        t = det["u"][s] * C[-1]
        y = int(got[s])
        assert (C[y - 1] if y > 0 else 0.0) <= t + CDF_TIE * C[-1] and C[y] >= t - CDF_TIE * C[-1]
    assert (got != ref).sum() <= 1


def test_two_closed_rounds_two_layers():
    gen = torch.Generator(device=DEV)
    gen.manual_seed(2024)
    L0 = [40, 77, 128, 200, 333, 401]
    kvs = [make_paged_kv(S, HQ, HKV, ROUNDS * (K + 1) + 1, seed=50 + li, device=DEV, hist_lens=L0)
           for li in range(LAYERS)]
    ws = s3r.Workspace(max(s3r.s3r_attn_workspace_size(kv_desc(kv), K + 1) for kv in kvs))
    max_pages = kvs[0].max_pages
    b_max = budget_b_max(max_pages, BUDGET)
    L = kvs[0].hist_lens.clone()
    # the first round's selection: from uniform mass (equal mass -> lowest page ids)
    sel = []
    for kv in kvs:
        pages = torch.full((S, HKV, b_max), -1, dtype=torch.int32, device=DEV)
        cnt = torch.zeros((S, HKV), dtype=torch.int32, device=DEV)
        sel.append((pages, cnt))
    mass0 = torch.ones((S, HKV, max_pages), dtype=torch.float32, device=DEV)
    for kv, (pages, cnt) in zip(kvs, sel):
        s3r.s3r_select_draft_pages(mass0, L, BUDGET, pages, cnt, ws)
    for rnd in range(ROUNDS):
        inp = make_spec_inputs(S, K, V, 3.0, 1.0, seed=300 + rnd, device=DEV)
        p_logits, q_logits = inp.p_logits, inp.q_logits
        Lh = host(L)
        pools0 = [(bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool)) for kv in kvs]
        draft_rows = [[(_bf16((S, 1, HKV, 128), gen), _bf16((S, 1, HKV, 128), gen)) for _ in range(K)]
                      for _ in kvs]
        block_rows = [(_bf16((S, K + 1, HKV, 128), gen), _bf16((S, K + 1, HKV, 128), gen)) for _ in kvs]
        qd = [[make_queries(kv, 1000 * rnd + 10 * li + j) for j in range(K)] for li, kv in enumerate(kvs)]
        qv = [make_queries(kv, 1000 * rnd + 500 + li, rows=K + 1) for li, kv in enumerate(kvs)]
        out_d = [[torch.empty((S, HQ, 128), dtype=torch.float32, device=DEV) for _ in range(K)] for _ in kvs]
        out_v = [torch.empty((S, K + 1, HQ, 128), dtype=torch.float32, device=DEV) for _ in kvs]
        mass = [torch.empty((S, HKV, max_pages), dtype=torch.float32, device=DEV) for _ in kvs]
        drafts = torch.full((S, K), -1, dtype=torch.int32, device=DEV)
        dws = s3r.Workspace(s3r.s3r_sample_draft_workspace_size(S))
        starts = [(L + j).to(torch.int32) for j in range(K)]
        # ---- the round on the GPU
        for j in range(K):
            for li, kv in enumerate(kvs):
                s3r.s3r_kv_append(kv_desc(kv), starts[j], draft_rows[li][j][0], draft_rows[li][j][1], ws)
                s3r.s3r_sparse_draft_attn(kv_desc(kv), L, j, sel[li][0], sel[li][1], qd[li][j], out_d[li][j], 1.0,
                                          ws)
            s3r.s3r_sample_draft_tokens(q_logits[:, j], SEED, OFFSET, j, drafts[:, j], dws)
        pools_before_block = [(bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool)) for kv in kvs]
        for li, kv in enumerate(kvs):
            s3r.s3r_kv_append(kv_desc(kv), L, block_rows[li][0], block_rows[li][1], ws)
            s3r.s3r_verify_attn(kv_desc(kv), L, qv[li], out_v[li], 1.0, ws, page_mass=mass[li])
        sws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(S, K))
        out_t = torch.empty((S, K + 1), dtype=torch.int32, device=DEV)
        nacc = torch.empty((S,), dtype=torch.int32, device=DEV)
        s3r.s3r_spec_sample(p_logits, q_logits, drafts, SEED, OFFSET, out_t, nacc, sws)
        L_new = torch.empty_like(L)
        s3r.s3r_commit_lengths(L, nacc, K, max_pages * 16, L_new, ws)
        new_sel = []
        for li in range(LAYERS):
            pages = torch.empty((S, HKV, b_max), dtype=torch.int32, device=DEV)
            cnt = torch.empty((S, HKV), dtype=torch.int32, device=DEV)
            s3r.s3r_select_draft_pages(mass[li], L_new, BUDGET, pages, cnt, ws)
            new_sel.append((pages, cnt))
        ws.check()
        dws.check()
        sws.check()
        # ---- stage by stage against the oracle
        x = host(drafts)
        ref_masses = []
        for j in range(K):
            _check_draft_tokens(host(q_logits[:, j]), x[:, j], SEED, OFFSET, j)
        for li, kv in enumerate(kvs):
            bt = host(kv.block_table)
            kp, vp = pools0[li]
            for j in range(K):
                kp, vp = oracle.kv_append(kp, vp, bt, Lh + j, bf16_to_bits(draft_rows[li][j][0]),
                                          bf16_to_bits(draft_rows[li][j][1]))
                ref = oracle.sparse_draft_attn(bf16_to_bits(qd[li][j]), kp, vp, bt, Lh, j, host(sel[li][0]),
                                               host(sel[li][1]), 1.0)
                assert_attn_close(out_d[li][j], ref, f"round {rnd} layer {li} draft {j}")
            assert np.array_equal(pools_before_block[li][0], kp) and np.array_equal(pools_before_block[li][1], vp)
            kp, vp = oracle.kv_append(kp, vp, bt, Lh, bf16_to_bits(block_rows[li][0]),
                                      bf16_to_bits(block_rows[li][1]))
            assert np.array_equal(bf16_to_bits(kv.k_pool), kp) and np.array_equal(bf16_to_bits(kv.v_pool), vp)
            ref_o, ref_m = oracle.verify_attn(bf16_to_bits(qv[li]), kp, vp, bt, Lh, 1.0, mass_pages=max_pages)
            assert_attn_close(out_v[li], ref_o, f"round {rnd} layer {li} verify")
            _check_mass(mass[li], ref_m, (HQ // HKV) * (K + 1))
            ref_masses.append(ref_m)
        compare(host(p_logits), host(q_logits), x, SEED, OFFSET, host(out_t), host(nacc))
        assert np.array_equal(host(L_new), oracle.commit_lengths(Lh, host(nacc)))
        for li in range(LAYERS):
            ref_pages, ref_cnt = oracle.select_draft_pages(host(mass[li]).astype(np.float64), host(L_new), BUDGET,
                                                           b_max=b_max)
            assert np.array_equal(host(new_sel[li][1]), ref_cnt)
            assert np.array_equal(host(new_sel[li][0]), ref_pages)
            swaps = selection_ties_vs_oracle_mass(host(new_sel[li][0]), host(new_sel[li][1]), ref_masses[li],
                                                  host(L_new), BUDGET, (HQ // HKV) * (K + 1))
            assert swaps <= 1, swaps
        assert np.all(host(new_sel[0][1]) == np.array([[budget_b_max(math.ceil(x / 16), BUDGET)] * HKV
                                                        for x in host(L_new)]))
        L, sel = L_new, new_sel
