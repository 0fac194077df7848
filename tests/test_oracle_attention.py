"""Pins for the attention oracle: it is checked against a library routine
(torch's scaled_dot_product_attention in float64 over a contiguous copy of the
history built page by page), closed forms and the invariants that follow from
the definitions of the three attention forms."""

import math

import numpy as np
import pytest
import torch

from oracle import dense_decode_attn, sparse_draft_attn, verify_attn, PAGE_SIZE
from workloads import make_paged_kv, make_queries, bf16_to_bits


def _tiny(seed, hist_lens, q_heads=4, kv_heads=2, k=3, head_dim=8):
    kv = make_paged_kv(len(hist_lens), q_heads, kv_heads, k, seed, hist_lens=hist_lens,
                       head_dim=head_dim, heavy_per_head=2, spare_pages=3)
    return kv


def _contiguous_history(kv, s, h, n_tokens):
    """K, V of one sequence and KV head as float64 matrices, walking the block
    table page by page (not through the oracle's token gather)."""
    kp = kv.k_pool.to(torch.float64)
    vp = kv.v_pool.to(torch.float64)
    ks, vs = [], []
    for lp in range(math.ceil(n_tokens / PAGE_SIZE)):
        phys = int(kv.block_table[s, lp])
        ks.append(kp[phys, h])
        vs.append(vp[phys, h])
    if not ks:
        return torch.zeros((0, kv.head_dim), dtype=torch.float64), torch.zeros((0, kv.head_dim), dtype=torch.float64)
    return torch.cat(ks)[:n_tokens], torch.cat(vs)[:n_tokens]


def _sdpa(qrows, K, V, mask, scale):
    """Library attention: qrows [R][D], K/V [L][D], mask [R][L] bool."""
    out = torch.nn.functional.scaled_dot_product_attention(
        qrows[None, None], K[None, None], V[None, None], attn_mask=mask[None, None], scale=scale)
    return out[0, 0]


def _np(kv):
    return (bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool), kv.block_table.numpy(), kv.hist_lens.numpy())


@pytest.mark.parametrize("scale", [1.0, 0.37])
def test_dense_matches_library_attention(scale):
    kv = _tiny(11, [37, 64])
    q = make_queries(kv, 5)
    kp, vp, bt, _ = _np(kv)
    ctx = np.array([37, 50])
    got = dense_decode_attn(bf16_to_bits(q), kp, vp, bt, ctx, scale)
    G = kv.q_heads // kv.kv_heads
    for s in range(2):
        for h in range(kv.kv_heads):
            K, V = _contiguous_history(kv, s, h, int(ctx[s]))
            rows = q[s, h * G:(h + 1) * G].to(torch.float64)
            ref = _sdpa(rows, K, V, torch.ones((G, K.shape[0]), dtype=torch.bool), scale)
            np.testing.assert_allclose(got[s, h * G:(h + 1) * G], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_verify_matches_library_causal_attention_and_mass():
    kv = _tiny(12, [29, 48, 5])
    T = kv.k
    q = make_queries(kv, 6, rows=T)
    kp, vp, bt, L = _np(kv)
    got, mass = verify_attn(bf16_to_bits(q), kp, vp, bt, L, 1.0)
    G = kv.q_heads // kv.kv_heads
    for s in range(3):
        n = int(L[s]) + T
        for h in range(kv.kv_heads):
            K, V = _contiguous_history(kv, s, h, n)
            ref_mass = np.zeros(mass.shape[2])
            for i in range(T):
                rows = q[s, i, h * G:(h + 1) * G].to(torch.float64)
                mask = torch.zeros((G, n), dtype=torch.bool)
                mask[:, : int(L[s]) + i + 1] = True
                ref = _sdpa(rows, K, V, mask, 1.0)
                np.testing.assert_allclose(got[s, i, h * G:(h + 1) * G], ref.numpy(), rtol=1e-12, atol=1e-12)
                w = torch.softmax((rows @ K.T).masked_fill(~mask, -math.inf), dim=-1).numpy()
                for t in range(n):
                    ref_mass[t // PAGE_SIZE] += w[:, t].sum()
            np.testing.assert_allclose(mass[s, h], ref_mass, rtol=1e-12, atol=1e-12)
            assert mass[s, h].sum() == pytest.approx(G * T, rel=1e-12)


def test_sparse_matches_library_masked_attention():
    kv = _tiny(13, [70, 41])
    q = make_queries(kv, 7)
    kp, vp, bt, L = _np(kv)
    rng = np.random.default_rng(0)
    b_max = 4
    sel = np.full((2, kv.kv_heads, b_max), -1)
    cnt = np.zeros((2, kv.kv_heads), dtype=np.int64)
    for s in range(2):
        P = math.ceil(int(L[s]) / PAGE_SIZE)
        for h in range(kv.kv_heads):
            pick = np.sort(rng.choice(P, size=min(3, P), replace=False))
            sel[s, h, : len(pick)] = pick
            cnt[s, h] = len(pick)
    G = kv.q_heads // kv.kv_heads
    for j in range(kv.k):
        got = sparse_draft_attn(bf16_to_bits(q), kp, vp, bt, L, j, sel, cnt, 1.0)
        for s in range(2):
            n = int(L[s]) + j + 1
            for h in range(kv.kv_heads):
                K, V = _contiguous_history(kv, s, h, n)
                mask = torch.zeros((G, n), dtype=torch.bool)
                for pg in sel[s, h, : cnt[s, h]]:
                    mask[:, pg * PAGE_SIZE: min((pg + 1) * PAGE_SIZE, int(L[s]))] = True
                mask[:, int(L[s]):] = True
                ref = _sdpa(q[s, h * G:(h + 1) * G].to(torch.float64), K, V, mask, 1.0)
                np.testing.assert_allclose(got[s, h * G:(h + 1) * G], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_closed_forms():
    D = 8
    # One visible token: the output is that token's value row.
    k_pool = np.zeros((1, 1, PAGE_SIZE, D))
    v_pool = np.zeros((1, 1, PAGE_SIZE, D))
    v_pool[0, 0, 0] = np.arange(D) + 0.5
    q = np.ones((1, 1, D))
    out = dense_decode_attn(q, k_pool, v_pool, np.array([[0]]), np.array([1]), 1.0)
    np.testing.assert_array_equal(out[0, 0], v_pool[0, 0, 0])
    # Equal keys: the output is the mean of the values.
    v_pool[0, 0, :5] = np.arange(5 * D).reshape(5, D)
    k_pool[0, 0, :5] = 0.3
    out = dense_decode_attn(q, k_pool, v_pool, np.array([[0]]), np.array([5]), 1.0)
    np.testing.assert_allclose(out[0, 0], v_pool[0, 0, :5].mean(axis=0), rtol=1e-14)
    # Scores 0 and ln 3 give weights 1/4 and 3/4.
    k_pool[:] = 0
    k_pool[0, 0, 1, 0] = 1.0
    v_pool[0, 0, 0] = 4.0
    v_pool[0, 0, 1] = -8.0
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = math.log(3.0)
    out = dense_decode_attn(q, k_pool, v_pool, np.array([[0]]), np.array([2]), 1.0)
    np.testing.assert_allclose(out[0, 0], 0.25 * 4.0 + 0.75 * -8.0, rtol=1e-14)
    # No visible token: zero output.
    out = dense_decode_attn(q, k_pool, v_pool, np.array([[0]]), np.array([0]), 1.0)
    assert not out.any()


def test_budget_one_sparse_equals_dense():
    kv = _tiny(14, [53, 16, 90], k=4)
    q = make_queries(kv, 8)
    kp, vp, bt, L = _np(kv)
    P = max(math.ceil(int(x) / PAGE_SIZE) for x in L)
    sel = np.full((3, kv.kv_heads, P), -1)
    cnt = np.zeros((3, kv.kv_heads), dtype=np.int64)
    for s in range(3):
        Ps = math.ceil(int(L[s]) / PAGE_SIZE)
        sel[s, :, :Ps] = np.arange(Ps)
        cnt[s] = Ps
    for j in range(kv.k):
        sparse = sparse_draft_attn(bf16_to_bits(q), kp, vp, bt, L, j, sel, cnt, 1.0)
        dense = dense_decode_attn(bf16_to_bits(q), kp, vp, bt, L + j + 1, 1.0)
        np.testing.assert_allclose(sparse, dense, rtol=1e-12, atol=1e-13)


def test_verify_rows_equal_sequential_decodes():
    kv = _tiny(15, [31, 64], k=5)
    T = kv.k
    q = make_queries(kv, 9, rows=T)
    kp, vp, bt, L = _np(kv)
    out, _ = verify_attn(bf16_to_bits(q), kp, vp, bt, L, 0.8)
    for i in range(T):
        step = dense_decode_attn(bf16_to_bits(q[:, i]), kp, vp, bt, L + i + 1, 0.8)
        np.testing.assert_allclose(out[:, i], step, rtol=1e-12, atol=1e-13)


def test_gqa_mapping_uses_contiguous_groups():
    # Heads 0..G-1 read KV head 0: make KV head 1 carry huge values and check
    # head 0's output does not see them.
    D = 8
    k_pool = np.zeros((1, 2, PAGE_SIZE, D))
    v_pool = np.zeros((1, 2, PAGE_SIZE, D))
    v_pool[0, 0, :3] = 1.0
    v_pool[0, 1, :3] = 1000.0
    q = np.zeros((1, 4, D))
    out = dense_decode_attn(q, k_pool, v_pool, np.array([[0]]), np.array([3]), 1.0)
    np.testing.assert_allclose(out[0, :2], 1.0)
    np.testing.assert_allclose(out[0, 2:], 1000.0)
