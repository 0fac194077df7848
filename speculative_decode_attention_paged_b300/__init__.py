"""Python binding of the S³R paged decode-attention library (libs3r.so).

Argument marshalling only: every function here takes torch tensors, checks
that they are contiguous CUDA tensors of the right dtype, and passes their
device pointers and sizes to the C entry point of the same name declared in
include/s3r.h.  All computation happens in the CUDA kernels of libs3r.so;
there is no CPU fallback.  If the library has not been built the first call
raises (build it with ``python -m speculative_decode_attention_paged_b300.build``).
"""

import ctypes
import os

import torch

__all__ = [
    "S3RError",
    "S3RDeviceError",
    "PagedKVDesc",
    "Workspace",
    "lib_path",
    "load_library",
    "s3r_version",
    "s3r_attn_workspace_size",
    "s3r_spec_sample_workspace_size",
    "s3r_select_workspace_size",
    "s3r_dense_decode_attn",
    "s3r_sparse_draft_attn",
    "s3r_verify_attn",
    "s3r_select_draft_pages",
    "s3r_spec_sample",
    "s3r_spec_sample_sequential",
    "s3r_spec_sample_noalloc",
    "s3r_sample_draft_workspace_size",
    "s3r_sample_draft_tokens",
    "s3r_kv_append",
    "s3r_commit_lengths",
    "DEVERR_BAD_PAGE",
    "DEVERR_BAD_LENGTH",
    "DEVERR_BAD_TOKEN",
    "DEVERR_TIMEOUT",
    "DEVERR_BAD_COUNT",
]

PAGE_SIZE = 16
HEAD_DIM = 128
MAX_ROWS_PER_KV_HEAD = 32

DEVERR_BAD_PAGE = 0x1
DEVERR_BAD_LENGTH = 0x2
DEVERR_BAD_TOKEN = 0x4
DEVERR_TIMEOUT = 0x8
DEVERR_BAD_COUNT = 0x10

_STATUS = {0: "S3R_OK", 1: "S3R_ERR_INVALID_ARG", 2: "S3R_ERR_UNSUPPORTED", 3: "S3R_ERR_CUDA",
           4: "S3R_ERR_WORKSPACE"}


class S3RError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}")


class S3RDeviceError(RuntimeError):
    def __init__(self, code):
        self.code = code
        super().__init__(f"device error word 0x{code:x}")


class _KVRows(ctypes.Structure):
    _fields_ = [("k_rows", ctypes.c_void_p), ("v_rows", ctypes.c_void_p), ("n_rows", ctypes.c_int32)]


class _PagedKV(ctypes.Structure):
    _fields_ = [
        ("k_pool", ctypes.c_void_p),
        ("v_pool", ctypes.c_void_p),
        ("num_phys_pages", ctypes.c_int64),
        ("block_table", ctypes.c_void_p),
        ("max_pages_per_seq", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SIG = {
    "s3r_version": (ctypes.c_char_p, []),
    "s3r_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "s3r_attn_workspace_size": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _I32, ctypes.POINTER(ctypes.c_size_t)]),
    "s3r_spec_sample_workspace_size": (ctypes.c_int, [_I32, _I32, ctypes.POINTER(ctypes.c_size_t)]),
    "s3r_select_workspace_size": (ctypes.c_int, [ctypes.POINTER(ctypes.c_size_t)]),
    "s3r_workspace_init": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    "s3r_read_device_error": (ctypes.c_int, [_P, _P, ctypes.POINTER(_I32), _I32]),
    "s3r_dense_decode_attn": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, _P, _P, ctypes.c_float, _P,
                                             ctypes.c_size_t, _P]),
    "s3r_sparse_draft_attn": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, _I32, _P, _P, _I32, _P, _P,
                                             ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "s3r_verify_attn": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, _I32, _P, _P, _P, _I32, ctypes.c_float,
                                       _P, ctypes.c_size_t, _P]),
    "s3r_select_draft_pages": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, ctypes.c_double, _I32, _I32, _P, _P,
                                              _I32, _P, ctypes.c_size_t, _P]),
    "s3r_spec_sample": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, ctypes.c_uint64, ctypes.c_uint64, _P, _P,
                                       _P, _P, ctypes.c_size_t, _P]),
    "s3r_spec_sample_sequential": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, ctypes.c_uint64, ctypes.c_uint64,
                                                  _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "s3r_spec_sample_noalloc": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _I32, ctypes.c_uint64, ctypes.c_uint64,
                                               _P, _P, _P, _P]),
    "s3r_sample_draft_workspace_size": (ctypes.c_int, [_I32, ctypes.POINTER(ctypes.c_size_t)]),
    "s3r_sample_draft_tokens": (ctypes.c_int, [_P, _I32, _I32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64,
                                               _I32, _P, ctypes.c_int64, _P, ctypes.c_size_t, _P]),
    "s3r_dense_decode_attn_append": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, ctypes.POINTER(_KVRows), _P, _P,
                                                    ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "s3r_sparse_draft_attn_append": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, _I32, _P, _P, _I32,
                                                    ctypes.POINTER(_KVRows), _P, _P, ctypes.c_float, _P,
                                                    ctypes.c_size_t, _P]),
    "s3r_verify_attn_append": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, _I32, ctypes.POINTER(_KVRows), _P, _P, _P,
                                              _I32, ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "s3r_kv_append": (ctypes.c_int, [ctypes.POINTER(_PagedKV), _P, _P, _I32, _P, _P, _P, ctypes.c_size_t, _P]),
    "s3r_commit_lengths": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, ctypes.c_size_t, _P]),
    "s3r_test_stall_next_verify": (None, []),
}

_lib = None


def lib_path():
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libs3r.so")


def load_library():
    """Load libs3r.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m speculative_decode_attention_paged_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIG.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _call(name, *args):
    status = getattr(load_library(), name)(*args)
    if status != 0:
        raise S3RError(name, status)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on_current_device(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")


def _need(t, dtype, name, shape=None):
    """A contiguous CUDA tensor of `dtype` on the current device; `shape`, when
    given, is the exact shape it must have."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    _on_current_device(t, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def _need_at_least(t, dtype, name, numel):
    _need(t, dtype, name)
    if t.numel() < numel:
        raise ValueError(f"{name} must hold at least {numel} elements")
    return t


def _spec_args(p_logits, q_logits, draft_tokens, out_tokens, n_accepted):
    """Checks every sampler tensor against p_logits' (n, k + 1, vocab)."""
    _need(p_logits, torch.float32, "p_logits")
    if p_logits.dim() != 3 or p_logits.shape[1] < 1:
        raise ValueError("p_logits must be [n][k+1][vocab]")
    n, k1, V = p_logits.shape
    _need(q_logits, torch.float32, "q_logits", (n, k1 - 1, V))
    _need(draft_tokens, torch.int32, "draft_tokens", (n, k1 - 1))
    _need(out_tokens, torch.int32, "out_tokens", (n, k1))
    _need(n_accepted, torch.int32, "n_accepted", (n,))
    return n, k1 - 1, V


class PagedKVDesc:
    """Descriptor of one layer's paged KV cache (device tensors stay owned by
    the caller and must outlive the descriptor's use)."""

    def __init__(self, k_pool, v_pool, block_table, num_q_heads):
        _need(k_pool, torch.bfloat16, "k_pool")
        _need(v_pool, torch.bfloat16, "v_pool")
        _need(block_table, torch.int32, "block_table")
        if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
            raise ValueError("k_pool and v_pool must both be [pages][kv_heads][16][head_dim]")
        self.k_pool, self.v_pool, self.block_table = k_pool, v_pool, block_table
        self.num_q_heads = int(num_q_heads)
        self.c = _PagedKV(
            k_pool=k_pool.data_ptr(), v_pool=v_pool.data_ptr(), num_phys_pages=k_pool.shape[0],
            block_table=block_table.data_ptr(), max_pages_per_seq=block_table.shape[1],
            num_seqs=block_table.shape[0], num_q_heads=self.num_q_heads, num_kv_heads=k_pool.shape[1],
            head_dim=k_pool.shape[3], page_size=k_pool.shape[2])

    @property
    def num_seqs(self):
        return self.c.num_seqs

    @property
    def num_kv_heads(self):
        return self.c.num_kv_heads

    @property
    def max_pages(self):
        return self.c.max_pages_per_seq


class Workspace:
    """Caller-owned device scratch buffer for the library (error word first)."""

    def __init__(self, nbytes, device=None, stream=None):
        nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.view = self.buf[off: off + nbytes]
        self.nbytes = nbytes
        _call("s3r_workspace_init", _ptr(self.view), ctypes.c_size_t(nbytes), _stream(stream))

    def ptr(self):
        return _ptr(self.view)

    def read_error(self, clear=True, stream=None):
        code = _I32(0)
        _call("s3r_read_device_error", self.ptr(), _stream(stream), ctypes.byref(code), _I32(1 if clear else 0))
        return code.value

    def check(self, stream=None):
        code = self.read_error(clear=True, stream=stream)
        if code:
            raise S3RDeviceError(code)


def s3r_version():
    return load_library().s3r_version().decode()


def s3r_attn_workspace_size(kv: PagedKVDesc, max_block_rows=1):
    n = ctypes.c_size_t(0)
    _call("s3r_attn_workspace_size", ctypes.byref(kv.c), _I32(max_block_rows), ctypes.byref(n))
    return n.value


def s3r_spec_sample_workspace_size(n, k):
    out = ctypes.c_size_t(0)
    _call("s3r_spec_sample_workspace_size", _I32(n), _I32(k), ctypes.byref(out))
    return out.value


def s3r_select_workspace_size():
    out = ctypes.c_size_t(0)
    _call("s3r_select_workspace_size", ctypes.byref(out))
    return out.value


def _rows(kv, append, n_rows):
    """s3r_kv_rows for append = (k_rows, v_rows), bf16 [S][n_rows][Hkv][128]."""
    k_rows, v_rows = append
    _need(k_rows, torch.bfloat16, "append k_rows")
    _need(v_rows, torch.bfloat16, "append v_rows")
    if k_rows.shape != v_rows.shape or tuple(k_rows.shape) != (kv.num_seqs, n_rows, kv.num_kv_heads, 128):
        raise ValueError(f"append rows must both be [num_seqs][{n_rows}][num_kv_heads][128]")
    return _KVRows(k_rows.data_ptr(), v_rows.data_ptr(), n_rows)


def s3r_dense_decode_attn(kv: PagedKVDesc, ctx_lens, q, out, sm_scale, ws: Workspace, stream=None, append=None):
    """Dense decode; append=(k_rows, v_rows) [S][1][Hkv][128] first writes the
    row of position ctx_len - 1 into the pages, in the same launch."""
    _need(ctx_lens, torch.int32, "ctx_lens")
    _need(q, torch.bfloat16, "q")
    _need(out, torch.float32, "out")
    if append is None:
        _call("s3r_dense_decode_attn", ctypes.byref(kv.c), _ptr(ctx_lens), _ptr(q), _ptr(out),
              ctypes.c_float(sm_scale), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    else:
        rows = _rows(kv, append, 1)
        _call("s3r_dense_decode_attn_append", ctypes.byref(kv.c), _ptr(ctx_lens), ctypes.byref(rows), _ptr(q),
              _ptr(out), ctypes.c_float(sm_scale), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return out


def s3r_sparse_draft_attn(kv: PagedKVDesc, hist_lens, draft_pos, sel_pages, sel_count, q, out, sm_scale,
                          ws: Workspace, stream=None, append=None):
    """Sparse draft step; append=(k_rows, v_rows) [S][1][Hkv][128] first
    writes the row of position hist_len + draft_pos, in the same launch."""
    _need(hist_lens, torch.int32, "hist_lens")
    _need(sel_pages, torch.int32, "sel_pages")
    _need(sel_count, torch.int32, "sel_count")
    _need(q, torch.bfloat16, "q")
    _need(out, torch.float32, "out")
    if append is None:
        _call("s3r_sparse_draft_attn", ctypes.byref(kv.c), _ptr(hist_lens), _I32(draft_pos), _ptr(sel_pages),
              _ptr(sel_count), _I32(sel_pages.shape[-1]), _ptr(q), _ptr(out), ctypes.c_float(sm_scale),
              ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    else:
        rows = _rows(kv, append, 1)
        _call("s3r_sparse_draft_attn_append", ctypes.byref(kv.c), _ptr(hist_lens), _I32(draft_pos),
              _ptr(sel_pages), _ptr(sel_count), _I32(sel_pages.shape[-1]), ctypes.byref(rows), _ptr(q), _ptr(out),
              ctypes.c_float(sm_scale), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return out


def s3r_verify_attn(kv: PagedKVDesc, hist_lens, q, out, sm_scale, ws: Workspace, page_mass=None, stream=None,
                    append=None):
    """Verify of T = q.shape[1] rows; append=(k_rows, v_rows) [S][T][Hkv][128]
    first writes the block's rows at positions hist_len .. hist_len + T - 1."""
    _need(hist_lens, torch.int32, "hist_lens")
    _need(q, torch.bfloat16, "q")
    _need(out, torch.float32, "out")
    stride = 0
    if page_mass is not None:
        _need(page_mass, torch.float32, "page_mass")
        stride = page_mass.shape[-1]
    if append is None:
        _call("s3r_verify_attn", ctypes.byref(kv.c), _ptr(hist_lens), _I32(q.shape[1]), _ptr(q), _ptr(out),
              _ptr(page_mass), _I32(stride), ctypes.c_float(sm_scale), ws.ptr(), ctypes.c_size_t(ws.nbytes),
              _stream(stream))
    else:
        rows = _rows(kv, append, q.shape[1])
        _call("s3r_verify_attn_append", ctypes.byref(kv.c), _ptr(hist_lens), _I32(q.shape[1]), ctypes.byref(rows),
              _ptr(q), _ptr(out), _ptr(page_mass), _I32(stride), ctypes.c_float(sm_scale), ws.ptr(),
              ctypes.c_size_t(ws.nbytes), _stream(stream))
    return out


def s3r_select_draft_pages(page_mass, sel_lens, budget, sel_pages, sel_count, ws: Workspace, n_sink=1,
                           n_recent=4, stream=None):
    _need(page_mass, torch.float32, "page_mass")
    _need(sel_lens, torch.int32, "sel_lens")
    _need(sel_pages, torch.int32, "sel_pages")
    _need(sel_count, torch.int32, "sel_count")
    S, Hkv, stride = page_mass.shape
    _call("s3r_select_draft_pages", _ptr(page_mass), _ptr(sel_lens), _I32(S), _I32(Hkv), _I32(stride),
          ctypes.c_double(budget), _I32(n_sink), _I32(n_recent), _ptr(sel_pages), _ptr(sel_count),
          _I32(sel_pages.shape[-1]), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return sel_pages, sel_count


def s3r_spec_sample(p_logits, q_logits, draft_tokens, seed, offset, out_tokens, n_accepted, ws: Workspace,
                    stream=None, tie_count=None):
    """Exact speculative sampling.  tie_count: optional int32 CUDA tensor of
    two elements that receives [ratio ties, inverse-CDF ties] (the C side's
    uint32 counters; the counts stay far below 2^31)."""
    n, k, V = _spec_args(p_logits, q_logits, draft_tokens, out_tokens, n_accepted)
    if tie_count is not None:
        _need_at_least(tie_count, torch.int32, "tie_count", 2)
    _call("s3r_spec_sample", _ptr(p_logits), _ptr(q_logits), _ptr(draft_tokens), _I32(n), _I32(k), _I32(V),
          ctypes.c_uint64(seed), ctypes.c_uint64(offset), _ptr(out_tokens), _ptr(n_accepted), _ptr(tie_count),
          ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return out_tokens, n_accepted


def s3r_spec_sample_sequential(p_logits, q_logits, draft_tokens, seed, offset, out_tokens, n_accepted,
                               ws: Workspace, stream=None, tie_count=None):
    """s3r_spec_sample with the ratio tests one position at a time, reading no
    row after a sequence's first rejection; the same results bit for bit."""
    n, k, V = _spec_args(p_logits, q_logits, draft_tokens, out_tokens, n_accepted)
    if tie_count is not None:
        _need_at_least(tie_count, torch.int32, "tie_count", 2)
    _call("s3r_spec_sample_sequential", _ptr(p_logits), _ptr(q_logits), _ptr(draft_tokens), _I32(n), _I32(k),
          _I32(V), ctypes.c_uint64(seed), ctypes.c_uint64(offset), _ptr(out_tokens), _ptr(n_accepted),
          _ptr(tie_count), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return out_tokens, n_accepted


NOALLOC_SCRATCH_BYTES = 2 * 1024 * 1024


def s3r_spec_sample_noalloc(p_logits, q_logits, draft_tokens, seed, offset, out_tokens, n_accepted,
                            device_error=None, stream=None):
    """s3r_spec_sample without a workspace, for callers that cannot allocate
    device memory; the scratch lives in the library (see include/s3r.h).
    device_error: optional int32 CUDA tensor of one element that receives the
    call's device error bits.  Every tensor must be on the current device,
    whose copy of the library's scratch the call uses."""
    n, k, V = _spec_args(p_logits, q_logits, draft_tokens, out_tokens, n_accepted)
    if device_error is not None:
        _need_at_least(device_error, torch.int32, "device_error", 1)
    _call("s3r_spec_sample_noalloc", _ptr(p_logits), _ptr(q_logits), _ptr(draft_tokens), _I32(n), _I32(k),
          _I32(V), ctypes.c_uint64(seed), ctypes.c_uint64(offset), _ptr(out_tokens), _ptr(n_accepted),
          _ptr(device_error), _stream(stream))
    return out_tokens, n_accepted


def s3r_sample_draft_workspace_size(n):
    out = ctypes.c_size_t(0)
    _call("s3r_sample_draft_workspace_size", _I32(n), ctypes.byref(out))
    return out.value


def _need_rows(t, dtype, name, dims):
    """A CUDA tensor of `dims` dimensions whose last dimension is contiguous
    (rows may be strided, e.g. one slice of a larger block)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    _on_current_device(t, name)
    if t.dim() != dims or (dims > 1 and t.stride(-1) != 1):
        raise ValueError(f"{name} must be {dims}-D with a contiguous last dimension")
    return t


def s3r_sample_draft_tokens(logits, seed, offset, draft_pos, tokens, ws: Workspace, stream=None):
    """One draft token per sequence from softmax(logits[s]) (fp32 [n][vocab],
    rows may be strided, e.g. q_logits[:, j]); token s goes to tokens[s]
    (int32 [n], may be strided, e.g. drafts[:, j])."""
    _need_rows(logits, torch.float32, "logits", 2)
    _need_rows(tokens, torch.int32, "tokens", 1)
    n, V = logits.shape
    if tokens.shape[0] != n:
        raise ValueError("tokens must have one entry per logits row")
    _call("s3r_sample_draft_tokens", _ptr(logits), _I32(n), _I32(V), ctypes.c_int64(logits.stride(0) if n > 1 else V),
          ctypes.c_uint64(seed), ctypes.c_uint64(offset), _I32(draft_pos), _ptr(tokens),
          ctypes.c_int64(tokens.stride(0) if n > 1 else 1), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return tokens


def s3r_kv_append(kv: PagedKVDesc, start_lens, k_rows, v_rows, ws: Workspace, n_rows=None, stream=None):
    """Write k_rows / v_rows (bf16 [S][max_rows][Hkv][128]) at positions
    start_lens[s] + t of each sequence's pages; n_rows (int32 [S]) limits the
    rows per sequence (default: all).  The descriptor's pools are written."""
    _need(start_lens, torch.int32, "start_lens")
    _need(k_rows, torch.bfloat16, "k_rows")
    _need(v_rows, torch.bfloat16, "v_rows")
    if k_rows.shape != v_rows.shape or k_rows.dim() != 4 or k_rows.shape[0] != kv.num_seqs:
        raise ValueError("k_rows and v_rows must both be [num_seqs][max_rows][num_kv_heads][head_dim]")
    if n_rows is not None:
        _need(n_rows, torch.int32, "n_rows")
    _call("s3r_kv_append", ctypes.byref(kv.c), _ptr(start_lens), _ptr(n_rows) if n_rows is not None else None,
          _I32(k_rows.shape[1]), _ptr(k_rows), _ptr(v_rows), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))


def s3r_commit_lengths(hist_lens, n_accepted, max_accept, max_len, new_lens, ws: Workspace, stream=None):
    """new_lens = hist_lens + n_accepted + 1 (new_lens may be hist_lens)."""
    _need(hist_lens, torch.int32, "hist_lens")
    _need(n_accepted, torch.int32, "n_accepted")
    _need(new_lens, torch.int32, "new_lens")
    _call("s3r_commit_lengths", _ptr(hist_lens), _ptr(n_accepted), _I32(hist_lens.shape[0]), _I32(max_accept),
          _I32(max_len), _ptr(new_lens), ws.ptr(), ctypes.c_size_t(ws.nbytes), _stream(stream))
    return new_lens
