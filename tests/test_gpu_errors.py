"""Data-dependent errors never fault: the kernels skip the bad item, finish,
and set a bit in the workspace's error word (read on the host)."""

import pytest
import torch

import speculative_decode_attention_paged_b300 as s3r
from workloads import make_paged_kv, make_queries, make_spec_inputs
from helpers import attn_workspace, kv_desc

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_out_of_range_page_id_sets_bad_page():
    kv = make_paged_kv(4, 16, 8, 4, seed=201, device=DEV, hist_lens=[100, 200, 300, 400])
    kv.block_table[1, 3] = kv.num_phys_pages + 5
    kv.block_table[2, 0] = -7
    q = make_queries(kv, 1)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    ws = attn_workspace(kv)
    s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens, q, out, 1.0, ws)
    code = ws.read_error()
    assert code & s3r.DEVERR_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    assert ws.read_error() == 0          # cleared by the first read


def test_length_beyond_block_table_sets_bad_length_and_zero_row():
    kv = make_paged_kv(3, 16, 8, 4, seed=202, device=DEV, hist_lens=[64, 64, 64])
    q = make_queries(kv, 2)
    out = torch.full(q.shape, 3.0, dtype=torch.float32, device=DEV)
    ws = attn_workspace(kv)
    ctx = torch.tensor([10, kv.max_pages * 16 + 1, 20], dtype=torch.int32, device=DEV)
    s3r.s3r_dense_decode_attn(kv_desc(kv), ctx, q, out, 1.0, ws)
    assert ws.read_error() & s3r.DEVERR_BAD_LENGTH
    assert torch.all(out[1] == 0)


def test_bad_selection_count_and_page():
    kv = make_paged_kv(2, 16, 8, 4, seed=203, device=DEV, hist_lens=[300, 300])
    sel = torch.zeros((2, 8, 4), dtype=torch.int32, device=DEV)
    sel[0, 0, 1] = 10_000
    cnt = torch.full((2, 8), 2, dtype=torch.int32, device=DEV)
    cnt[1, 3] = 9
    q = make_queries(kv, 3)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    ws = attn_workspace(kv)
    s3r.s3r_sparse_draft_attn(kv_desc(kv), kv.hist_lens, 0, sel, cnt, q, out, 1.0, ws)
    code = ws.read_error()
    assert code & s3r.DEVERR_BAD_PAGE and code & s3r.DEVERR_BAD_COUNT
    assert torch.isfinite(out.float()).all()


def test_draft_token_outside_vocabulary_sets_bad_token():
    inp = make_spec_inputs(8, 3, 100, 3.0, 1.0, seed=5, device=DEV)
    inp.draft_tokens[2, 1] = 100
    inp.draft_tokens[5, 0] = -1
    ws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(8, 3))
    out = torch.empty((8, 4), dtype=torch.int32, device=DEV)
    nacc = torch.empty((8,), dtype=torch.int32, device=DEV)
    s3r.s3r_spec_sample(inp.p_logits, inp.q_logits, inp.draft_tokens, 1, 0, out, nacc, ws)
    assert ws.read_error() & s3r.DEVERR_BAD_TOKEN
    assert int(nacc[5]) == 0 and int(nacc[2]) <= 1
    assert (out[:, 0] >= 0).all() and (out < 100).all()


def test_host_side_rejections():
    kv = make_paged_kv(2, 16, 8, 4, seed=204, device=DEV, hist_lens=[30, 30])
    q = make_queries(kv, 4)
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    small = s3r.Workspace(256)
    with pytest.raises(s3r.S3RError) as e:
        s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens, q, out, 1.0, small)
    assert e.value.status == 4
    ws = attn_workspace(kv, rows=4)
    q5 = make_queries(kv, 5, rows=5)          # 5 rows x G=2 fits; workspace sized for 4 rows
    with pytest.raises(s3r.S3RError):
        s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q5, torch.empty(q5.shape, dtype=torch.float32, device=DEV), 1.0, ws)
    with pytest.raises(s3r.S3RError):
        s3r.s3r_dense_decode_attn(kv_desc(kv), kv.hist_lens, q, out, float("nan"), ws)
