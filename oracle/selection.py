"""Oracle for choosing the next draft's KV pages from verification attention.

Test infrastructure only (see the package docstring).

The pages say only that, after verification, S³R uses the attention scores to
choose the history the next draft reads ([ritwork] "Как разреженный черновик
сохраняет ответы плотной модели", last paragraph), that selection overhead must
stay small ([wispaper] "Where the speedup claim holds") and that the sparse
budget ratio is s = 0.05 ([wispaper] "Throughput gains with comparable task
performance").  The rule itself is not printed, so this library fixes one:

  P  = ceil(sel_len / 16) pages of history
  M  = {0 .. n_sink-1} U {P-n_recent .. P-1}, clipped to [0, P)  (mandatory)
  B  = min(P, max(ceil(budget * P - 1e-9), |M|))                (page budget)
  if B == P: every page
  else: M plus the B-|M| other pages of largest mass, equal mass -> lower
        page index first
  emitted in ascending page order, count B.

Parity status: pinned by tests/test_oracle_select.py against brute force over
all B-subsets on tiny inputs and by its invariants (|sel| = B, M within sel,
ascending, budget 1.0 -> all pages).  The rule is a reading: the pages print
none, so what is pinned is this rule, not a formula of theirs.
"""

import math

import numpy as np

PAGE_SIZE = 16


def selection_budget(num_pages, budget, n_sink, n_recent):
    """(B, mandatory set) for a history of ``num_pages`` pages."""
    P = int(num_pages)
    mandatory = set(range(min(int(n_sink), P))) | set(range(max(P - int(n_recent), 0), P))
    B = min(P, max(math.ceil(float(budget) * P - 1e-9), len(mandatory)))
    return B, mandatory


def select_draft_pages(page_mass, sel_lens, budget, n_sink=1, n_recent=4, b_max=None):
    """Per (sequence, KV head): the selected logical pages and their count.

    page_mass [S][Hkv][mass_stride] float (only the first ceil(sel_len/16)
              entries of each row are read)
    sel_lens  [S] history length the selection covers
    returns   sel_pages [S][Hkv][b_max] int64 (unused slots = -1),
              sel_count [S][Hkv] int64
    """
    mass = np.asarray(page_mass, dtype=np.float64)
    S, Hkv, stride = mass.shape
    counts = np.zeros((S, Hkv), dtype=np.int64)
    chosen_lists = []
    for s in range(S):
        P = math.ceil(int(sel_lens[s]) / PAGE_SIZE)
        if P > stride:
            raise ValueError("mass row shorter than the history's page count")
        B, mandatory = selection_budget(P, budget, n_sink, n_recent)
        for h in range(Hkv):
            if B == P:
                chosen = list(range(P))
            else:
                others = [pg for pg in range(P) if pg not in mandatory]
                others.sort(key=lambda pg: (-mass[s, h, pg], pg))
                chosen = sorted(mandatory | set(others[: B - len(mandatory)]))
            counts[s, h] = len(chosen)
            chosen_lists.append((s, h, chosen))
    width = int(b_max) if b_max is not None else max([len(c) for _, _, c in chosen_lists] + [0])
    sel = np.full((S, Hkv, width), -1, dtype=np.int64)
    for s, h, chosen in chosen_lists:
        if len(chosen) > width:
            raise ValueError("b_max smaller than the page budget")
        sel[s, h, : len(chosen)] = chosen
    return sel, counts
