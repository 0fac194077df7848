"""s3r_spec_sample_noalloc, the sampler for callers that cannot allocate device
memory, against s3r_spec_sample with a caller-allocated workspace.

Such callers (a pre-reserved memory pool, a plugin given only its buffers)
use library-owned scratch instead of a workspace.  The same kernels run on
the same inputs, so tokens and accepted counts must be identical.  Two calls
in a row on different shapes check that scratch left by the first call does
not leak into the second.  This file is collected last on purpose."""

import ctypes

import pytest
import torch

import speculative_decode_attention_paged_b300 as s3r
from workloads import make_spec_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _with_workspace(inp):
    N, k1, _ = inp.p_logits.shape
    ws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(N, k1 - 1))
    out = torch.full((N, k1), 55, dtype=torch.int32, device=DEV)
    nacc = torch.full((N,), 55, dtype=torch.int32, device=DEV)
    s3r.s3r_spec_sample(inp.p_logits, inp.q_logits, inp.draft_tokens, 31, 3, out, nacc, ws)
    ws.check()
    return out, nacc


def _no_alloc_through_c_abi(inp):
    """Direct ctypes call of the C entry point (no workspace argument)."""
    lib = s3r.load_library()
    N, k1, V = inp.p_logits.shape
    out = torch.full((N, k1), 66, dtype=torch.int32, device=DEV)
    nacc = torch.full((N,), 66, dtype=torch.int32, device=DEV)
    err = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = lib.s3r_spec_sample_noalloc(
        ctypes.c_void_p(inp.p_logits.data_ptr()), ctypes.c_void_p(inp.q_logits.data_ptr()),
        ctypes.c_void_p(inp.draft_tokens.data_ptr()), ctypes.c_int32(N), ctypes.c_int32(k1 - 1),
        ctypes.c_int32(V), ctypes.c_uint64(31), ctypes.c_uint64(3), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(nacc.data_ptr()), ctypes.c_void_p(err.data_ptr()), stream)
    assert status == 0, s3r.load_library().s3r_status_string(status)
    torch.cuda.synchronize()
    return out, nacc, int(err.item())


def test_no_alloc_matches_workspace_entry_point_on_two_calls():
    first = make_spec_inputs(512, 8, 151936, 3.0, 1.0, seed=71, device=DEV)
    second = make_spec_inputs(300, 3, 5003, 2.0, 0.5, seed=72, device=DEV)
    bonus_only = make_spec_inputs(700, 0, 32000, 3.0, 1.0, seed=73, device=DEV)   # k = 0: arrival counters
    for inp in (first, second, bonus_only, bonus_only):
        ref_out, ref_nacc = _with_workspace(inp)
        out, nacc, err = _no_alloc_through_c_abi(inp)
        assert err == 0
        assert torch.equal(nacc, ref_nacc)
        assert torch.equal(out, ref_out)


def test_no_alloc_reports_device_errors_and_clears_them():
    bad = make_spec_inputs(16, 2, 100, 3.0, 1.0, seed=73, device=DEV)
    bad.draft_tokens[3, 0] = 100                     # outside the vocabulary
    _, _, err = _no_alloc_through_c_abi(bad)
    assert err & s3r.DEVERR_BAD_TOKEN
    good = make_spec_inputs(16, 2, 100, 3.0, 1.0, seed=74, device=DEV)
    _, _, err = _no_alloc_through_c_abi(good)         # the next call starts clean
    assert err == 0


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    lib = s3r.load_library()
    n, k = 100_000, 8                                # 13.6 MB of row statistics
    need = s3r.s3r_spec_sample_workspace_size(n, k)
    assert need > s3r.NOALLOC_SCRATCH_BYTES
    status = lib.s3r_spec_sample_noalloc(None, None, None, n, k, 151936, 0, 0, None, None, None, None)
    assert status == 2                               # S3R_ERR_UNSUPPORTED, nothing enqueued
