"""Oracle for one closed S³R round over a stack of layers: sparse drafting
with draft-token sampling, dense verification with page mass, exact
speculative sampling, the length commit, and the next round's draft pages.

Test infrastructure only (see the package docstring).

The order of the steps is the pages' ([wispaper] "S3R drafts sparsely and
verifies densely": the drafter proposes a block under a budgeted subset of
the history, full attention verifies it in parallel, exact speculative
sampling decides it; [ritwork] "Как разреженный черновик сохраняет ответы
плотной модели": the verification attention scores choose the history of the
next draft).  Each step is the oracle function of its own module; this file
only chains them:

  for draft step j = 0 .. k-1:
      every layer: append the draft row at position L + j, then sparse draft
          attention of step j over the previous round's selection;
      sample draft token x_{j+1} from q_j on the DRAFT stream;
  every layer: append the k + 1 dense rows of [pending token, x_1 .. x_k] at
      positions L .. L + k, then verify those k + 1 rows with page mass;
  exact speculative sampling of (p, q, x) -> n_acc and the emitted tokens;
  commit: L' = L + n_acc + 1 (rows past L' are rolled back);
  every layer: the next round's draft pages from the verify mass over L'.

Parity status: pinned through its parts (each module's own pins) and by
tests/test_oracle_kv_cache.py: with q = p and budget 1.0 every draft is
accepted, L' = L + k + 1, the drafts equal dense decodes and every page is
selected.
"""

import numpy as np

from .attention import sparse_draft_attn, verify_attn
from .draft_sample import sample_draft_tokens
from .kv_cache import commit_lengths, kv_append
from .selection import select_draft_pages
from .spec_sample import spec_sample


def closed_round(layers, hist_lens, sel, p_logits, q_logits, seed, offset, budget, sm_scale=1.0,
                 n_sink=1, n_recent=4):
    """One closed round.

    layers     list of dicts, one per layer: k_pool, v_pool [NP][Hkv][16][D]
               and block_table [S][max_pages] (the cache), draft_k / draft_v
               [k][S][1][Hkv][D] (row of draft step j), block_k / block_v
               [S][k+1][Hkv][D] (dense rows of the verified block), qd
               [k][S][Hq][D] (draft queries), qv [S][k+1][Hq][D] (verify queries)
    hist_lens  [S] L before the round
    sel        list per layer of (sel_pages [S][Hkv][b], sel_count [S][Hkv]),
               the previous round's selection
    p_logits   [S][k+1][V], q_logits [S][k][V]
    returns a dict: pools per layer after the round, draft outputs
    [layer][j] [S][Hq][D], drafts x [S][k], verify outputs and mass per layer,
    out_tokens, n_accepted, new_lens, next selection per layer.
    """
    S = len(hist_lens)
    k = q_logits.shape[1]
    L = np.asarray(hist_lens, dtype=np.int64)
    pools = [(lay["k_pool"], lay["v_pool"]) for lay in layers]
    draft_out = [[None] * k for _ in layers]
    x = np.zeros((S, k), dtype=np.int64)
    for j in range(k):
        for li, lay in enumerate(layers):
            kp, vp = kv_append(pools[li][0], pools[li][1], lay["block_table"], L + j, lay["draft_k"][j],
                               lay["draft_v"][j])
            pools[li] = (kp, vp)
            draft_out[li][j] = sparse_draft_attn(lay["qd"][j], kp, vp, lay["block_table"], L, j, sel[li][0],
                                                 sel[li][1], sm_scale)
        x[:, j], _ = sample_draft_tokens(q_logits[:, j], seed, offset, j)
    verify_out, mass = [], []
    for li, lay in enumerate(layers):
        kp, vp = kv_append(pools[li][0], pools[li][1], lay["block_table"], L, lay["block_k"], lay["block_v"])
        pools[li] = (kp, vp)
        o, m = verify_attn(lay["qv"], kp, vp, lay["block_table"], L, sm_scale,
                           mass_pages=lay["block_table"].shape[1])
        verify_out.append(o)
        mass.append(m)
    out_tokens, n_acc, _ = spec_sample(p_logits, q_logits, x, seed, offset)
    new_lens = commit_lengths(L, n_acc)
    next_sel = [select_draft_pages(m, new_lens, budget, n_sink, n_recent) for m in mass]
    return {"pools": pools, "draft_out": draft_out, "drafts": x, "verify_out": verify_out, "mass": mass,
            "out_tokens": out_tokens, "n_accepted": n_acc, "new_lens": new_lens, "next_sel": next_sel}
