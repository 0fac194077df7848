"""GPU parity of the paged-cache updates against the oracle: appended K/V rows
land bit for bit where the oracle puts them (every other byte of the pools
unchanged), the length commit is exact, bad inputs set their error bits and
write nothing, and draft-token sampling reads strided rows and writes strided
tokens exactly as it does contiguous ones."""

import numpy as np
import pytest
import torch

import oracle
import speculative_decode_attention_paged_b300 as s3r
from helpers import host, kv_desc
from workloads import bf16_to_bits, make_paged_kv

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(S, T, Hkv, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (torch.randn((S, T, Hkv, 128), generator=g, device=DEV).to(torch.bfloat16),
            torch.randn((S, T, Hkv, 128), generator=g, device=DEV).to(torch.bfloat16))


@pytest.mark.parametrize("kv_heads,T,ragged", [(8, 5, False), (8, 5, True), (4, 1, False), (1, 17, True)])
def test_append_matches_oracle_bit_for_bit(kv_heads, T, ragged):
    lens = [0, 13, 15, 16, 30, 47, 255, 1000]
    kv = make_paged_kv(len(lens), 2 * kv_heads, kv_heads, T, seed=7 + T, device=DEV, hist_lens=lens)
    kr, vr = _rows(len(lens), T, kv_heads, seed=T)
    n_rows = None
    if ragged:
        n_rows = torch.tensor([(3 * i) % (T + 1) for i in range(len(lens))], dtype=torch.int32, device=DEV)
    kp0, vp0, bt = bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool), host(kv.block_table)
    ws = s3r.Workspace(256)
    s3r.s3r_kv_append(kv_desc(kv), kv.hist_lens, kr, vr, ws, n_rows=n_rows)
    ws.check()
    kp_ref, vp_ref = oracle.kv_append(kp0, vp0, bt, host(kv.hist_lens), bf16_to_bits(kr), bf16_to_bits(vr),
                                      None if n_rows is None else host(n_rows))
    assert np.array_equal(bf16_to_bits(kv.k_pool), kp_ref)
    assert np.array_equal(bf16_to_bits(kv.v_pool), vp_ref)


def test_append_errors_write_nothing():
    lens = [10, 20, 30, 40]
    kv = make_paged_kv(4, 16, 8, 4, seed=3, device=DEV, hist_lens=lens)
    kp0, vp0 = kv.k_pool.clone(), kv.v_pool.clone()
    kr, vr = _rows(4, 4, 8, seed=1)
    ws = s3r.Workspace(256)
    beyond = torch.tensor([kv.max_pages * 16 - 2] * 4, dtype=torch.int32, device=DEV)   # rows 2, 3 past the table
    s3r.s3r_kv_append(kv_desc(kv), beyond, kr, vr, ws, n_rows=torch.zeros(4, dtype=torch.int32, device=DEV) + 4)
    assert ws.read_error() & s3r.DEVERR_BAD_LENGTH
    kv.k_pool.copy_(kp0)
    kv.v_pool.copy_(vp0)
    s3r.s3r_kv_append(kv_desc(kv), kv.hist_lens, kr, vr, ws,
                      n_rows=torch.tensor([5, 0, 0, 0], dtype=torch.int32, device=DEV))      # count above max_rows
    assert ws.read_error() & s3r.DEVERR_BAD_COUNT
    assert torch.equal(kv.k_pool, kp0) and torch.equal(kv.v_pool, vp0)
    bad_bt = kv.block_table.clone()
    bad_bt[2, 30 // 16] = kv.num_phys_pages + 5                                             # page outside the pool
    desc = s3r.PagedKVDesc(kv.k_pool, kv.v_pool, bad_bt, kv.q_heads)
    s3r.s3r_kv_append(desc, kv.hist_lens, kr, vr, ws,
                      n_rows=torch.tensor([0, 0, 1, 0], dtype=torch.int32, device=DEV))
    assert ws.read_error() & s3r.DEVERR_BAD_PAGE
    assert torch.equal(kv.k_pool, kp0) and torch.equal(kv.v_pool, vp0)


def test_commit_lengths_exact_and_errors():
    L = torch.tensor([0, 5, 100, 4000, 16380, 7], dtype=torch.int32, device=DEV)
    n = torch.tensor([0, 4, 2, 4, 4, 9], dtype=torch.int32, device=DEV)
    out = torch.full_like(L, -7)
    ws = s3r.Workspace(256)
    s3r.s3r_commit_lengths(L, n, 8, 16384, out, ws)
    err = ws.read_error()
    want = oracle.commit_lengths(host(L), host(n))
    got = host(out)
    # 16380 + 4 + 1 exceeds 16384 and 9 exceeds max_accept: those keep their length
    assert np.array_equal(got[:4], want[:4]) and got[4] == 16380 and got[5] == 7
    assert err & s3r.DEVERR_BAD_LENGTH and err & s3r.DEVERR_BAD_COUNT
    s3r.s3r_commit_lengths(L[:4], n[:4], 8, 16384, L[:4], ws)                  # in place
    assert ws.read_error() == 0 and np.array_equal(host(L[:4]), want[:4])


def test_draft_sampling_with_strided_rows_and_tokens():
    n, k, V = 300, 4, 32000
    g = torch.Generator(device=DEV)
    g.manual_seed(4)
    q_logits = torch.randn((n, k, V), generator=g, device=DEV) * 3.0
    drafts = torch.full((n, k), -1, dtype=torch.int32, device=DEV)
    ws = s3r.Workspace(s3r.s3r_sample_draft_workspace_size(n))
    for j in range(k):
        s3r.s3r_sample_draft_tokens(q_logits[:, j], 11, 3, j, drafts[:, j], ws)
    ws.check()
    for j in range(k):
        t = torch.empty((n,), dtype=torch.int32, device=DEV)
        s3r.s3r_sample_draft_tokens(q_logits[:, j].contiguous(), 11, 3, j, t, ws)
        assert torch.equal(t, drafts[:, j])


def _twin_pools(lens, q_heads, kv_heads, k, seed):
    """Two identical caches (same seed): one for the separate calls, one for the fused ones."""
    return [make_paged_kv(len(lens), q_heads, kv_heads, k, seed=seed, device=DEV, hist_lens=lens) for _ in range(2)]


@pytest.mark.parametrize("mode,q_heads,T", [("dense", 16, 1), ("sparse", 16, 1), ("verify", 16, 5),
                                            ("verify", 32, 8)])
def test_fused_append_equals_append_then_attend(mode, q_heads, T):
    """The _append calls leave the same pages and give bit-identical outputs
    (and page mass) as s3r_kv_append followed by the plain call; verify with
    32 rows per KV head runs the tcgen05 kernel."""
    lens = [1, 15, 16, 17, 100, 255, 1000, 2049]
    kv_heads = 8
    sep, fus = _twin_pools(lens, q_heads, kv_heads, 2 * T + 2, seed=61)
    kr, vr = _rows(len(lens), T, kv_heads, seed=62)
    from workloads import make_queries
    outs, masses = [], []
    for kv, fused in ((sep, False), (fus, True)):
        desc = kv_desc(kv)
        ws = s3r.Workspace(s3r.s3r_attn_workspace_size(desc, T))
        L = kv.hist_lens
        if mode == "dense":
            q = make_queries(kv, 70)
            out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
            ctx = (L + 1).to(torch.int32)
            if fused:
                s3r.s3r_dense_decode_attn(desc, ctx, q, out, 1.0, ws, append=(kr, vr))
            else:
                s3r.s3r_kv_append(desc, L, kr, vr, ws)
                s3r.s3r_dense_decode_attn(desc, ctx, q, out, 1.0, ws)
            mass = None
        elif mode == "sparse":
            q = make_queries(kv, 71)
            out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
            j = 2
            sel_cnt = torch.full((len(lens), kv_heads), 2, dtype=torch.int32, device=DEV)
            sel = torch.zeros((len(lens), kv_heads, 2), dtype=torch.int32, device=DEV)
            sel[..., 1] = torch.clamp((L // 16 - 1), min=0)[:, None].to(torch.int32)
            sel_cnt[L < 32] = 1
            start = (L + j).to(torch.int32)
            if fused:
                s3r.s3r_sparse_draft_attn(desc, L, j, sel, sel_cnt, q, out, 1.0, ws, append=(kr, vr))
            else:
                s3r.s3r_kv_append(desc, start, kr, vr, ws)
                s3r.s3r_sparse_draft_attn(desc, L, j, sel, sel_cnt, q, out, 1.0, ws)
            mass = None
        else:
            q = make_queries(kv, 72, rows=T)
            out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
            mass = torch.empty((len(lens), kv_heads, kv.max_pages), dtype=torch.float32, device=DEV)
            if fused:
                s3r.s3r_verify_attn(desc, L, q, out, 1.0, ws, page_mass=mass, append=(kr, vr))
            else:
                s3r.s3r_kv_append(desc, L, kr, vr, ws)
                s3r.s3r_verify_attn(desc, L, q, out, 1.0, ws, page_mass=mass)
        ws.check()
        outs.append(out)
        masses.append(mass)
    assert torch.equal(sep.k_pool, fus.k_pool) and torch.equal(sep.v_pool, fus.v_pool)
    assert torch.equal(outs[0], outs[1])
    if masses[0] is not None:
        assert torch.equal(masses[0], masses[1])
    # and against the oracle: append, then attend
    kp, vp, bt = bf16_to_bits(fus.k_pool), bf16_to_bits(fus.v_pool), host(fus.block_table)
    if mode == "verify":
        ref, mref = oracle.verify_attn(bf16_to_bits(make_queries(fus, 72, rows=T)), kp, vp, bt,
                                       host(fus.hist_lens), 1.0, mass_pages=fus.max_pages)
        from helpers import assert_attn_close
        assert_attn_close(outs[1], ref, f"fused verify {q_heads}/{kv_heads} T={T}")
    elif mode == "dense":
        from helpers import assert_attn_close
        ref = oracle.dense_decode_attn(bf16_to_bits(make_queries(fus, 70)), kp, vp, bt, host(fus.hist_lens) + 1, 1.0)
        assert_attn_close(outs[1], ref, "fused dense")
    else:
        # L = 15 and 17: the selected history page is also the draft tail's
        # first page, so two entries of the stream write and read that page
        from helpers import assert_attn_close
        ref = oracle.sparse_draft_attn(bf16_to_bits(make_queries(fus, 71)), kp, vp, bt, host(fus.hist_lens), j,
                                       host(sel), host(sel_cnt), 1.0)
        assert_attn_close(outs[1], ref, "fused sparse")


def test_fused_append_skips_rows_of_bad_pages():
    lens = [40, 50]
    kv = make_paged_kv(2, 16, 8, 4, seed=63, device=DEV, hist_lens=lens)
    k0, v0 = kv.k_pool.clone(), kv.v_pool.clone()
    bad_bt = kv.block_table.clone()
    bad_bt[1, 50 // 16] = kv.num_phys_pages + 3
    desc = s3r.PagedKVDesc(kv.k_pool, kv.v_pool, bad_bt, 16)
    kr, vr = _rows(2, 1, 8, seed=64)
    from workloads import make_queries
    q = make_queries(kv, 73)
    out = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    ws = s3r.Workspace(s3r.s3r_attn_workspace_size(desc, 1))
    ctx = torch.tensor([41, 51], dtype=torch.int32, device=DEV)
    s3r.s3r_dense_decode_attn(desc, ctx, q, out, 1.0, ws, append=(kr, vr))
    assert ws.read_error() & s3r.DEVERR_BAD_PAGE
    # sequence 0's row landed; sequence 1's page is outside the pool, nothing else changed
    page0 = int(kv.block_table[0, 40 // 16])
    assert torch.equal(kv.k_pool[page0, :, 40 % 16], kr[0, 0])
    changed = (kv.k_pool != k0).any(dim=(1, 2, 3)).nonzero().flatten().tolist()
    assert changed == [page0]
    assert torch.equal(kv.v_pool[page0, :, 40 % 16], vr[0, 0])
