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
