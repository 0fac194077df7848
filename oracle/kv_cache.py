"""Oracle for the paged-cache updates of a closed S³R round: appending a block
of K/V rows, and committing the verified block's length.

Test infrastructure only (see the package docstring).

What the pages fix
------------------
* The drafter is the policy itself with sparse attention; it proposes a block
  of tokens, which the dense policy then verifies in parallel ([wispaper]
  "S3R drafts sparsely and verifies densely").  The accepted part of the block
  keeps dense states, recomputed by verification ([wispaper] same section;
  [ritwork] "Как разреженный черновик сохраняет ответы плотной модели").
* At the first rejection the draft is cut: the rejected token and everything
  after it are dropped, and a corrected token takes its place ([rebas]
  "草稿可以稀疏，交卷必须完整"; [ritwork] same section).

Readings where the pages are silent
-----------------------------------
* Block row t of sequence s is the token at position L + t, stored in slot
  (L + t) % 16 of the sequence's logical page (L + t) // 16, i.e. of physical
  page block_table[s][(L + t) // 16] (the cache layout of attention.py).
* Verification runs the pending token and the k drafts (k + 1 rows at
  positions L .. L + k).  With n_acc drafts accepted, positions L .. L + n_acc
  hold the pending token and the accepted drafts, so the new length is
  L + n_acc + 1; the rows after it belong to rejected drafts and are dropped
  by the length alone (the next round's appends overwrite them).

Parity status: pinned by tests/test_oracle_kv_cache.py: appended rows read
back at the right positions through a whole-page rebuild of each sequence's
history and every other row is unchanged; attention after an append equals
library attention over the history with the new row concatenated; the commit
closed form; a round with equal policies and budget 1.0 accepts every draft
and its drafts equal dense decodes.
"""

import numpy as np

from .attention import PAGE_SIZE


def kv_append(k_pool, v_pool, block_table, start_lens, k_rows, v_rows, n_rows=None):
    """Write block rows into copies of the pools and return them.

    k_pool, v_pool  [NP][Hkv][16][D] (bf16 bit patterns or floats)
    block_table     [S][max_pages] physical page ids
    start_lens      [S] position of row 0 of each sequence (its length L)
    k_rows, v_rows  [S][T][Hkv][D], row t to position L + t
    n_rows          [S] rows written per sequence (default T)
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    S, T = k_rows.shape[0], k_rows.shape[1]
    for s in range(S):
        n = T if n_rows is None else int(n_rows[s])
        for t in range(n):
            pos = int(start_lens[s]) + t
            page = int(block_table[s][pos // PAGE_SIZE])
            k_out[page, :, pos % PAGE_SIZE, :] = k_rows[s, t]
            v_out[page, :, pos % PAGE_SIZE, :] = v_rows[s, t]
    return k_out, v_out


def commit_lengths(hist_lens, n_accepted):
    """Length after a verified block: the pending token plus the accepted
    drafts, L + n_acc + 1 ([rebas]; [ritwork]: the block is cut at the first
    rejection)."""
    return np.asarray(hist_lens, dtype=np.int64) + np.asarray(n_accepted, dtype=np.int64) + 1
