"""Pins for the paged-cache updates of a closed round (kv_append,
commit_lengths) and for the round's chaining: rows read back through a
whole-page rebuild of each history, attention after an append against a
library routine over the history with the row concatenated, the commit closed
form, and a round whose drafter equals the target."""

import math

import numpy as np
import pytest
import torch

from oracle import (PAGE_SIZE, closed_round, commit_lengths, dense_decode_attn, kv_append, select_draft_pages,
                    verify_attn)
from workloads import bf16_to_bits, make_paged_kv, make_queries


def _rebuild(pool, block_table_row, n_pages):
    """[Hkv][n_pages*16][D] history of one sequence: whole pages in block-table
    order, flattened (no per-token index arithmetic)."""
    pages = pool[np.asarray(block_table_row[:n_pages], dtype=np.int64)]        # [P][Hkv][16][D]
    P, Hkv, ps, D = pages.shape
    return pages.transpose(1, 0, 2, 3).reshape(Hkv, P * ps, D)


def _rows(rng, S, T, Hkv, D):
    return rng.integers(0, 1 << 16, size=(S, T, Hkv, D), dtype=np.uint16)


def test_append_reads_back_through_whole_page_rebuild():
    L = [13, 30, 47]
    kv = make_paged_kv(3, 4, 2, 5, seed=3, hist_lens=L, head_dim=8, heavy_per_head=1, spare_pages=2)
    kp, vp, bt = bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool), kv.block_table.numpy()
    rng = np.random.default_rng(0)
    kr, vr = _rows(rng, 3, 5, 2, 8), _rows(rng, 3, 5, 2, 8)
    n_rows = np.array([5, 3, 0])
    k2, v2 = kv_append(kp, vp, bt, L, kr, vr, n_rows)
    touched = np.zeros(kp.shape[:3], dtype=bool)
    for s in range(3):
        P = math.ceil((L[s] + 5) / PAGE_SIZE)
        for pool, after, rows in ((kp, k2, kr), (vp, v2, vr)):
            before_h, after_h = _rebuild(pool, bt[s], P), _rebuild(after, bt[s], P)
            for t in range(5):
                want = rows[s, t] if t < n_rows[s] else before_h[:, L[s] + t]
                assert np.array_equal(after_h[:, L[s] + t], want)
            keep = np.ones(P * PAGE_SIZE, dtype=bool)
            keep[L[s]:L[s] + n_rows[s]] = False
            assert np.array_equal(after_h[:, keep], before_h[:, keep])
        for t in range(n_rows[s]):
            pos = L[s] + t
            touched[bt[s, pos // PAGE_SIZE], :, pos % PAGE_SIZE] = True
    assert np.array_equal(k2[~touched], kp[~touched]) and np.array_equal(v2[~touched], vp[~touched])


def test_decode_after_append_is_attention_over_history_plus_row():
    L = [20, 33]
    kv = make_paged_kv(2, 4, 2, 2, seed=5, hist_lens=L, head_dim=8, heavy_per_head=1, spare_pages=1)
    kp, vp, bt = bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool), kv.block_table.numpy()
    g = torch.Generator().manual_seed(1)
    krow = torch.randn((2, 1, 2, 8), generator=g).to(torch.bfloat16)
    vrow = torch.randn((2, 1, 2, 8), generator=g).to(torch.bfloat16)
    k2, v2 = kv_append(kp, vp, bt, L, bf16_to_bits(krow), bf16_to_bits(vrow))
    q = make_queries(kv, 9)
    got = dense_decode_attn(bf16_to_bits(q), k2, v2, bt, np.array(L) + 1, 0.5)
    K = kv.k_pool.to(torch.float64)
    V = kv.v_pool.to(torch.float64)
    for s in range(2):
        for h in range(2):
            hk = torch.cat([K[int(bt[s, p]), h] for p in range(math.ceil(L[s] / PAGE_SIZE))])[:L[s]]
            hv = torch.cat([V[int(bt[s, p]), h] for p in range(math.ceil(L[s] / PAGE_SIZE))])[:L[s]]
            keys = torch.cat([hk, krow[s, 0, h:h + 1].to(torch.float64)])
            vals = torch.cat([hv, vrow[s, 0, h:h + 1].to(torch.float64)])
            rows = q[s, 2 * h:2 * h + 2].to(torch.float64)
            ref = torch.nn.functional.scaled_dot_product_attention(rows[None, None], keys[None, None],
                                                                   vals[None, None], scale=0.5)[0, 0]
            np.testing.assert_allclose(got[s, 2 * h:2 * h + 2], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_commit_closed_form():
    rng = np.random.default_rng(2)
    L = rng.integers(0, 10_000, size=64)
    n = rng.integers(0, 9, size=64)
    assert np.array_equal(commit_lengths(L, n), L + n + 1)
    assert np.array_equal(commit_lengths(L, np.full(64, 8)), L + 9)        # all 8 drafts accepted
    assert np.array_equal(commit_lengths(L, np.zeros(64, dtype=int)), L + 1)  # only the pending token


def _round_inputs(S, Hq, Hkv, k, D, V, L, seed):
    kv = make_paged_kv(S, Hq, Hkv, k + 2, seed=seed, hist_lens=L, head_dim=D, heavy_per_head=1, spare_pages=1)
    rng = np.random.default_rng(seed)
    bt = kv.block_table.numpy()
    layer = {"k_pool": bf16_to_bits(kv.k_pool), "v_pool": bf16_to_bits(kv.v_pool), "block_table": bt,
             "draft_k": [_rows(rng, S, 1, Hkv, D) & 0xBFFF for _ in range(k)],
             "draft_v": [_rows(rng, S, 1, Hkv, D) & 0xBFFF for _ in range(k)],
             "block_k": _rows(rng, S, k + 1, Hkv, D) & 0xBFFF, "block_v": _rows(rng, S, k + 1, Hkv, D) & 0xBFFF,
             "qd": [bf16_to_bits(make_queries(kv, 100 + j)) for j in range(k)],
             "qv": bf16_to_bits(make_queries(kv, 200, rows=k + 1))}
    return kv, layer


@pytest.mark.parametrize("seed", [0, 1])
def test_round_with_equal_policies_and_full_budget(seed):
    """q = p and budget 1.0: every draft is accepted, so L' = L + k + 1; the
    sparse drafts over all pages are dense decodes of the same cache; every
    page of L' is selected next."""
    S, Hq, Hkv, k, D, V = 3, 4, 2, 3, 8, 50
    L = [17, 40, 63]
    kv, layer = _round_inputs(S, Hq, Hkv, k, D, V, L, seed)
    P = [math.ceil(x / PAGE_SIZE) for x in L]
    b = max(P)
    sel_pages = np.full((S, Hkv, b), -1, dtype=np.int64)
    for s in range(S):
        sel_pages[s, :, :P[s]] = np.arange(P[s])
    sel_count = np.array([[P[s]] * Hkv for s in range(S)])
    rng = np.random.default_rng(seed + 10)
    p_logits = rng.normal(0, 2.0, size=(S, k + 1, V))
    q_logits = p_logits[:, :k].copy()
    r = closed_round([layer], np.array(L), [(sel_pages, sel_count)], p_logits, q_logits, seed=7, offset=1,
                     budget=1.0)
    assert np.all(r["n_accepted"] == k)
    assert np.array_equal(r["out_tokens"][:, :k], r["drafts"])
    assert np.array_equal(r["new_lens"], np.array(L) + k + 1)
    kp, vp = layer["k_pool"], layer["v_pool"]
    for j in range(k):
        kp, vp = kv_append(kp, vp, layer["block_table"], np.array(L) + j, layer["draft_k"][j], layer["draft_v"][j])
        dense = dense_decode_attn(layer["qd"][j], kp, vp, layer["block_table"], np.array(L) + j + 1, 1.0)
        np.testing.assert_allclose(r["draft_out"][0][j], dense, rtol=1e-12, atol=1e-12)
    kp, vp = kv_append(kp, vp, layer["block_table"], np.array(L), layer["block_k"], layer["block_v"])
    assert np.array_equal(r["pools"][0][0], kp) and np.array_equal(r["pools"][0][1], vp)
    _, mass = verify_attn(layer["qv"], kp, vp, layer["block_table"], np.array(L), 1.0,
                          mass_pages=layer["block_table"].shape[1])
    np.testing.assert_allclose(r["mass"][0], mass, rtol=0, atol=0)
    pages, count = r["next_sel"][0]
    want_pages, want_count = select_draft_pages(mass, np.array(L) + k + 1, 1.0)
    assert np.array_equal(count, want_count) and np.array_equal(pages, want_pages)
    assert np.array_equal(count[:, 0], [math.ceil((x + k + 1) / PAGE_SIZE) for x in L])
