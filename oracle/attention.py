"""Oracle for the three attention forms of an S³R round over a paged KV cache.

Test infrastructure only (see the package docstring).

What the pages fix
------------------
* Autoregressive decoding reads the whole growing KV cache at every step;
  attention is 72-76% of decode kernel time ([abstract]; [wispaper] "Sparse
  sampling changes the group, not just the speed").  -> ``dense_decode_attn``.
* The drafter is the policy itself running sparse attention over a selected
  part of the history ([wispaper] "S3R drafts sparsely and verifies densely";
  [rebas] "草稿可以稀疏，交卷必须完整"; [ritwork] "Как разреженный черновик
  сохраняет ответы плотной модели").  -> ``sparse_draft_attn``.
* Verification runs full attention over the complete history for the drafted
  block, in parallel ([wispaper] same section and "Dense verification still
  pays the full KV-cache bill").  -> ``verify_attn``.
* The verification attention scores choose the next draft's history
  ([ritwork] "Как разреженный черновик ...", last paragraph).  The page mass
  returned by ``verify_attn`` is that signal.

Readings where the pages are silent
-----------------------------------
* Attention is softmax(sm_scale * q.K^T) V per query head; query head qh uses
  KV head qh // G (contiguous GQA groups).
* KV cache pages hold 16 tokens; pool layout [page][kv_head][16][head_dim].
* ``ctx_lens`` counts the current token (decode query at position ctx_len-1).
* Draft step j sees {t < L : page(t) selected} plus its own tail L..L+j.
* Verify row i (block position L+i) sees tokens 0..L+i (causal inside the
  block).
* Page mass of (s, kv head h, page pg) = sum over the G query heads of the
  group, the T verify rows and the tokens of the page of each row's final
  normalised softmax weight.  Each row contributes total mass 1.
* A row with no visible token yields a zero output (and contributes no mass).

Parity status: pinned (tests/test_oracle_attention.py): brute-force matrix
evaluation on tiny inputs, closed forms (single token, equal keys, two-token
weights), budget 1.0 == dense, k-row verify == k sequential decodes,
sum of page mass == G*T.
"""

import math

import numpy as np

from .bf16 import bf16_bits_to_f64

PAGE_SIZE = 16


def _as_f64(x):
    """bf16 bit arrays are widened exactly; float arrays are cast to float64."""
    x = np.asarray(x)
    if x.dtype in (np.uint16, np.int16):
        return bf16_bits_to_f64(x)
    return x.astype(np.float64)


def _gather_tokens(pool, block_table_row, h, tokens):
    """K (or V) rows of KV head ``h`` for logical token positions ``tokens``.

    Token t lives in logical page t // 16 at slot t % 16; the block table maps
    the logical page to its physical page in the pool.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    phys = np.asarray(block_table_row, dtype=np.int64)[tokens // PAGE_SIZE]
    return _as_f64(pool[phys, h, tokens % PAGE_SIZE, :])


def _attend(qvec, keys, values, sm_scale):
    """softmax(sm_scale * keys @ q) @ values, returning (output, weights)."""
    if keys.shape[0] == 0:
        return np.zeros(values.shape[1]), np.zeros(0)
    scores = sm_scale * (keys @ qvec)
    m = scores.max()
    e = np.exp(scores - m)
    w = e / e.sum()
    return w @ values, w


def _group(q_heads, kv_heads):
    if q_heads % kv_heads != 0:
        raise ValueError("query heads must be a multiple of KV heads")
    return q_heads // kv_heads


def dense_decode_attn(q, k_pool, v_pool, block_table, ctx_lens, sm_scale, seqs=None):
    """Dense autoregressive decode attention (the baseline every speedup is
    measured against: [abstract]; [wispaper] "Sparse sampling changes the
    group, not just the speed").

    q           [S][Hq][D]   bf16 bits or float
    k/v_pool    [NP][Hkv][16][D] bf16 bits
    block_table [S][max_pages] int
    ctx_lens    [S] int, tokens visible to the query (query at ctx_len-1)
    seqs        optional list of sequence indices to evaluate
    returns     [len(seqs)][Hq][D] float64
    """
    S, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    G = _group(Hq, Hkv)
    seqs = list(range(S)) if seqs is None else list(seqs)
    out = np.zeros((len(seqs), Hq, D))
    for oi, s in enumerate(seqs):
        tokens = np.arange(int(ctx_lens[s]))
        for h in range(Hkv):
            keys = _gather_tokens(k_pool, block_table[s], h, tokens)
            vals = _gather_tokens(v_pool, block_table[s], h, tokens)
            for g in range(G):
                qh = h * G + g
                out[oi, qh], _ = _attend(_as_f64(q[s, qh]), keys, vals, sm_scale)
    return out


def draft_visible_tokens(hist_len, draft_pos, selected_pages):
    """Token set of draft step ``draft_pos`` (j): the history tokens t < L whose
    page is selected, then the draft tail L..L+j (reading of [ritwork]
    "Как разреженный черновик ...": sparse proposals read only a selected
    part of the history)."""
    L = int(hist_len)
    hist = np.arange(L, dtype=np.int64)
    hist = hist[np.isin(hist // PAGE_SIZE, np.asarray(selected_pages, dtype=np.int64))]
    tail = np.arange(L, L + int(draft_pos) + 1, dtype=np.int64)
    return np.concatenate([hist, tail])


def sparse_draft_attn(q, k_pool, v_pool, block_table, hist_lens, draft_pos,
                      sel_pages, sel_count, sm_scale, seqs=None):
    """Budgeted sparse draft attention for draft step ``draft_pos`` ([wispaper]
    "S3R drafts sparsely and verifies densely"; [rebas] "草稿可以稀疏，交卷必须完整").

    q          [S][Hq][D]
    hist_lens  [S] int, L = history length before the draft block
    sel_pages  [S][Hkv][b_max] logical page ids (first sel_count entries used)
    sel_count  [S][Hkv]
    returns    [len(seqs)][Hq][D] float64
    """
    S, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    G = _group(Hq, Hkv)
    seqs = list(range(S)) if seqs is None else list(seqs)
    out = np.zeros((len(seqs), Hq, D))
    for oi, s in enumerate(seqs):
        for h in range(Hkv):
            chosen = sel_pages[s][h][: int(sel_count[s][h])]
            tokens = draft_visible_tokens(hist_lens[s], draft_pos, chosen)
            keys = _gather_tokens(k_pool, block_table[s], h, tokens)
            vals = _gather_tokens(v_pool, block_table[s], h, tokens)
            for g in range(G):
                qh = h * G + g
                out[oi, qh], _ = _attend(_as_f64(q[s, qh]), keys, vals, sm_scale)
    return out


def verify_attn(q, k_pool, v_pool, block_table, hist_lens, sm_scale, seqs=None,
                mass_pages=None):
    """Dense causal verification of a T-token block ([wispaper] "S3R drafts
    sparsely and verifies densely", "Dense verification still pays the full
    KV-cache bill") and the page mass of its attention ([ritwork]
    "Как разреженный черновик ...": attention scores choose the next draft's
    history).

    q          [S][T][Hq][D]; row i is the query at position L+i
    hist_lens  [S] int, L
    mass_pages number of page slots in the returned mass (default: the
               largest ceil((L+T)/16) over the evaluated sequences)
    returns    out  [len(seqs)][T][Hq][D] float64
               mass [len(seqs)][Hkv][mass_pages] float64; entries for pages
                    >= ceil((L+T)/16) are zero
    """
    S, T, Hq, D = q.shape
    Hkv = k_pool.shape[1]
    G = _group(Hq, Hkv)
    seqs = list(range(S)) if seqs is None else list(seqs)
    if mass_pages is None:
        mass_pages = max([math.ceil((int(hist_lens[s]) + T) / PAGE_SIZE) for s in seqs] + [0])
    out = np.zeros((len(seqs), T, Hq, D))
    mass = np.zeros((len(seqs), Hkv, mass_pages))
    for oi, s in enumerate(seqs):
        L = int(hist_lens[s])
        for h in range(Hkv):
            tokens = np.arange(L + T)
            keys = _gather_tokens(k_pool, block_table[s], h, tokens)
            vals = _gather_tokens(v_pool, block_table[s], h, tokens)
            for i in range(T):
                visible = L + i + 1
                for g in range(G):
                    qh = h * G + g
                    o, w = _attend(_as_f64(q[s, i, qh]), keys[:visible], vals[:visible], sm_scale)
                    out[oi, i, qh] = o
                    np.add.at(mass[oi, h], tokens[:visible] // PAGE_SIZE, w)
    return out, mass
