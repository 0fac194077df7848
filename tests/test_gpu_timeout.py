"""The timeout path of the tensor-core verify kernel's bounded waits.

Every wait in the kernel is bounded: when one runs out the kernel sets
S3R_DEVERR_TIMEOUT, every role leaves its loop, the copies still in flight are
waited for (bounded), the tensor memory is freed and the kernel returns.  The
test hook s3r_test_stall_next_verify makes CTA 0 of the next launch skip its
first tile's K copies and that tile's barrier arrival, so the score MMA's wait
runs out after its full spin limit (several seconds) and so does the drain's
wait for that barrier; no fault, trap or unbounded wait is involved.

Checked: the call returns with the TIMEOUT bit in the error word, and after
the workspace is re-zeroed the next call on the same context runs normally
and gives the same outputs, bit for bit, as a call made before the stall (so
the kernel freed its tensor memory and left nothing in flight)."""

import ctypes

import pytest
import torch

import speculative_decode_attention_paged_b300 as s3r
from helpers import attn_workspace, kv_desc
from workloads import make_paged_kv, make_queries

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_stalled_wait_reports_timeout_and_the_context_stays_usable():
    # 32 query rows per KV head (8 rows x 4 heads): the tensor-core verify kernel
    lens = [1000, 2048, 77, 3001, 512, 1500, 16, 2600]
    kv = make_paged_kv(len(lens), 32, 8, 8, seed=211, device=DEV, hist_lens=lens)
    q = make_queries(kv, 212, rows=8)
    ws = attn_workspace(kv, rows=8)
    before = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, before, 1.0, ws)
    ws.check()

    s3r.load_library().s3r_test_stall_next_verify()
    stalled = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, stalled, 1.0, ws)
    code = ws.read_error(clear=True)          # waits for the call (seconds)
    assert code & s3r.DEVERR_TIMEOUT, hex(code)

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert s3r.load_library().s3r_workspace_init(ws.ptr(), ws.nbytes, stream) == 0
    after = torch.full(q.shape, 7.0, dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, after, 1.0, ws)
    ws.check()
    assert torch.equal(after, before)
    # the hook arms one launch only
    again = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    s3r.s3r_verify_attn(kv_desc(kv), kv.hist_lens, q, again, 1.0, ws)
    ws.check()
    assert torch.equal(again, before)
