"""The C-ABI library loads, exports every entry point the headers under
include/ declare, and rejects bad arguments on the host before touching a GPU."""

import ctypes
import os
import re

import pytest

import speculative_decode_attention_paged_b300 as s3r
from speculative_decode_attention_paged_b300 import build as s3r_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def _declared():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"S3R_API\s+[^;(]*?\b(s3r_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    s3r_build.build()
    return s3r.load_library()


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ("s3r_dense_decode_attn", "s3r_sparse_draft_attn", "s3r_verify_attn",
                 "s3r_select_draft_pages", "s3r_spec_sample", "s3r_sched_run", "s3r_test_stall_next_verify"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_host_only_queries(lib):
    assert s3r.s3r_version().startswith("s3r-b300")
    assert lib.s3r_status_string(0) == b"S3R_OK"
    assert lib.s3r_status_string(4) == b"S3R_ERR_WORKSPACE"
    assert s3r.s3r_select_workspace_size() == 256
    assert s3r.s3r_spec_sample_workspace_size(2048, 8) >= 256 + 2048 * 17 * 8
    # the no-alloc entry point's documented example fits its fixed scratch
    assert s3r.s3r_spec_sample_workspace_size(2048, 8) == 1_884_672 <= s3r.NOALLOC_SCRATCH_BYTES
    with pytest.raises(s3r.S3RError):
        s3r.s3r_spec_sample_workspace_size(4, 65)


def _kv(**over):
    f = dict(k_pool=None, v_pool=None, num_phys_pages=10, block_table=None, max_pages_per_seq=4,
             num_seqs=0, num_q_heads=16, num_kv_heads=8, head_dim=128, page_size=16)
    f.update(over)
    return s3r._PagedKV(**f)


def test_argument_validation_on_host(lib):
    size = ctypes.c_size_t(0)
    # head_dim / page size the kernels do not implement
    assert lib.s3r_attn_workspace_size(ctypes.byref(_kv(head_dim=64)), 1, ctypes.byref(size)) == 2
    assert lib.s3r_attn_workspace_size(ctypes.byref(_kv(page_size=32)), 1, ctypes.byref(size)) == 2
    # q heads not a multiple of KV heads
    assert lib.s3r_attn_workspace_size(ctypes.byref(_kv(num_q_heads=12)), 1, ctypes.byref(size)) == 1
    # rows per KV head above the limit (G = 16, T = 4)
    assert lib.s3r_attn_workspace_size(ctypes.byref(_kv(num_q_heads=128)), 4, ctypes.byref(size)) == 2
    # attention with a missing workspace
    kv = _kv()
    assert lib.s3r_dense_decode_attn(ctypes.byref(kv), None, None, None, ctypes.c_float(1.0), None, 0, None) == 4
    assert lib.s3r_verify_attn(ctypes.byref(kv), None, 0, None, None, None, 0, ctypes.c_float(1.0), None, 0,
                               None) == 1
    # selection: bad geometry, bad budget, b_max below the budget of mass_stride pages
    assert lib.s3r_select_draft_pages(None, None, 1, 0, 8, ctypes.c_double(0.05), 1, 4, None, None, 8,
                                      None, 0, None) == 1
    assert lib.s3r_select_draft_pages(None, None, 1, 8, 8, ctypes.c_double(1.5), 1, 4, None, None, 8,
                                      None, 0, None) == 1
    # spec sample: k above the limit, empty vocabulary, offset beyond 32 bits
    assert lib.s3r_spec_sample(None, None, None, 1, 65, 10, 0, 0, None, None, None, None, 0, None) == 2
    assert lib.s3r_spec_sample(None, None, None, 1, 4, 0, 0, 0, None, None, None, None, 0, None) == 1
    assert lib.s3r_spec_sample(None, None, None, 1, 4, 10, 0, 1 << 32, None, None, None, None, 0, None) == 1


def test_new_entry_points_validate_on_host(lib):
    kv = _kv()
    # the sequential sampler shares the parallel sampler's checks
    assert lib.s3r_spec_sample_sequential(None, None, None, 1, 65, 10, 0, 0, None, None, None, None, 0, None) == 2
    assert lib.s3r_spec_sample_sequential(None, None, None, -1, 4, 10, 0, 0, None, None, None, None, 0, None) == 1
    # draft sampling: rows closer than the vocabulary, token stride 0, missing workspace
    assert lib.s3r_sample_draft_tokens(None, 4, 100, 99, 0, 0, 0, None, 1, None, 0, None) == 1
    assert lib.s3r_sample_draft_tokens(None, 4, 100, 100, 0, 0, 0, None, 0, None, 0, None) == 1
    assert lib.s3r_sample_draft_tokens(None, 4, 100, 100, 0, 0, 0, None, 1, None, 0, None) == 4
    # KV append: no descriptor, negative rows, unsupported head_dim, missing workspace
    assert lib.s3r_kv_append(None, None, None, 1, None, None, None, 0, None) == 1
    assert lib.s3r_kv_append(ctypes.byref(kv), None, None, -1, None, None, None, 0, None) == 1
    assert lib.s3r_kv_append(ctypes.byref(_kv(head_dim=64)), None, None, 1, None, None, None, 0, None) == 2
    assert lib.s3r_kv_append(ctypes.byref(kv), None, None, 1, None, None, None, 0, None) == 4
    # length commit: negative sizes, missing workspace
    assert lib.s3r_commit_lengths(None, None, -1, 4, 100, None, None, 0, None) == 1
    assert lib.s3r_commit_lengths(None, None, 4, 4, 100, None, None, 0, None) == 4


def test_fused_append_calls_validate_rows_on_host(lib):
    """The *_attn_append calls reject a missing rows struct, a row count other
    than the call's (1 for dense and draft, the verify block's T), missing row
    pointers and rows that are not 16-byte aligned, before any device work.
    The addresses below are never dereferenced: every case fails on the host."""
    kv = _kv(num_seqs=2, k_pool=0x10000, v_pool=0x20000, block_table=0x30000)
    lens, q, out, ws, sel, cnt = 0x40000, 0x50000, 0x60000, 0x100000, 0x70000, 0x80000
    one = 1.0

    def rows(n, k=0x90000, v=0xA0000):
        return ctypes.byref(s3r._KVRows(k_rows=k, v_rows=v, n_rows=n))

    def dense(r, w=ws):
        return lib.s3r_dense_decode_attn_append(ctypes.byref(kv), lens, r, q, out, one, w, 1 << 30, None)

    def draft(r, pos=0):
        return lib.s3r_sparse_draft_attn_append(ctypes.byref(kv), lens, pos, sel, cnt, 4, r, q, out, one, ws,
                                                1 << 30, None)

    def verify(T, r):
        return lib.s3r_verify_attn_append(ctypes.byref(kv), lens, T, r, q, out, None, 0, one, ws, 1 << 30, None)

    assert dense(None) == 1
    assert dense(rows(2)) == 1                   # one row per sequence
    assert dense(rows(1, k=None)) == 1
    assert dense(rows(1, v=0xA0008)) == 1        # not 16-byte aligned
    assert dense(rows(1), w=None) == 4           # the workspace is checked first
    assert draft(None) == 1
    assert draft(rows(3)) == 1
    assert draft(rows(1), pos=-1) == 1
    assert verify(3, None) == 1
    assert verify(3, rows(2)) == 1               # the block's T rows
    assert verify(3, rows(3, k=0x90004)) == 1


def test_no_alloc_checks_arguments_before_touching_its_scratch(lib):
    # Each bad argument is reported as S3R_ERR_INVALID_ARG.  Without a GPU the
    # scratch lookup would fail with S3R_ERR_CUDA, so these statuses also show
    # that the checks run before the shared scratch (and any clear of it).
    assert lib.s3r_spec_sample_noalloc(None, None, None, 4, 2, 0, 0, 0, None, None, None, None) == 1
    assert lib.s3r_spec_sample_noalloc(None, None, None, 4, 2, 10, 0, 1 << 32, None, None, None, None) == 1
    assert lib.s3r_spec_sample_noalloc(None, None, None, 4, 2, 10, 0, 0, None, None, None, None) == 1
    assert lib.s3r_spec_sample_noalloc(None, None, None, -1, 2, 10, 0, 0, None, None, None, None) == 1
