"""Pins for the page-selection oracle: brute force over every subset on tiny
inputs (with exact ties), the budget arithmetic's special cases and the rule's
invariants on random masses."""

import itertools
import math

import numpy as np
import pytest

from oracle import select_draft_pages, selection_budget


def _brute(mass_row, P, budget, n_sink, n_recent):
    B, M = selection_budget(P, budget, n_sink, n_recent)
    others = [pg for pg in range(P) if pg not in M]
    best = None
    for extra in itertools.combinations(others, B - len(M)):
        chosen = tuple(sorted(M | set(extra)))
        key = (sum(mass_row[list(extra)]) if extra else 0.0, tuple(-c for c in chosen))
        if best is None or key > best[0]:
            best = (key, chosen)
    return list(best[1])


@pytest.mark.parametrize("seed", range(6))
def test_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    S, Hkv = 3, 2
    sel_lens = np.array([16 * 11 + 3, 16 * 9, 16 * 12])
    mass = rng.integers(0, 4, size=(S, Hkv, 12)).astype(np.float64)  # many exact ties
    for budget, n_sink, n_recent in [(0.5, 1, 4), (0.34, 2, 1), (0.7, 0, 0), (0.25, 1, 2)]:
        sel, cnt = select_draft_pages(mass, sel_lens, budget, n_sink, n_recent, b_max=12)
        for s in range(S):
            P = math.ceil(sel_lens[s] / 16)
            for h in range(Hkv):
                ref = _brute(mass[s, h], P, budget, n_sink, n_recent)
                assert list(sel[s, h, : cnt[s, h]]) == ref
                assert (sel[s, h, cnt[s, h]:] == -1).all()


def test_budget_arithmetic():
    assert selection_budget(0, 0.05, 1, 4) == (0, set())
    assert selection_budget(3, 0.05, 1, 4) == (3, {0, 1, 2})
    assert selection_budget(100, 0.05, 1, 4)[0] == 5
    assert selection_budget(101, 0.05, 1, 4)[0] == 6           # ceil(5.05)
    assert selection_budget(1025, 0.05, 1, 4)[0] == 52          # ceil(51.25)
    assert selection_budget(20, 0.05, 1, 4)[0] == 5             # floor at |M|
    assert selection_budget(40, 0.25, 1, 4)[0] == 10            # exact product, no round-up
    assert selection_budget(7, 1.0, 1, 4)[0] == 7
    B, M = selection_budget(10, 0.5, 1, 4)
    assert M == {0, 6, 7, 8, 9} and B == 5


def test_invariants_random():
    rng = np.random.default_rng(7)
    S, Hkv, stride = 5, 3, 80
    sel_lens = rng.integers(1, 16 * stride + 1, size=S)
    mass = rng.random((S, Hkv, stride))
    for budget in (0.0, 0.05, 0.3, 1.0):
        sel, cnt = select_draft_pages(mass, sel_lens, budget, 1, 4, b_max=stride)
        for s in range(S):
            P = math.ceil(sel_lens[s] / 16)
            B, M = selection_budget(P, budget, 1, 4)
            for h in range(Hkv):
                chosen = sel[s, h, : cnt[s, h]]
                assert cnt[s, h] == B
                assert set(M) <= set(chosen)
                assert (np.diff(chosen) > 0).all()
                assert chosen.max(initial=-1) < P
                if budget == 1.0:
                    assert list(chosen) == list(range(P))
                rest = [pg for pg in range(P) if pg not in M]
                picked = [pg for pg in chosen if pg not in M]
                left = [pg for pg in rest if pg not in picked]
                if picked and left:
                    assert min(mass[s, h, picked]) >= max(mass[s, h, left])


def test_selection_tie_judge_accepts_only_cutoff_swaps():
    """The GPU tests judge a selection made from fp32 mass against the oracle's
    selection from fp64 mass; the judge must accept a swap of the two pages
    that straddle the cutoff within the window and reject any other swap."""
    import pytest
    from helpers import SELECT_TIE, selection_ties_vs_oracle_mass
    rows = 8
    P = 40          # 640 tokens; budget 0.25 -> B = 10: pages 0 and 36..39, then 1..5 by mass
    mass = np.linspace(1.0, 0.2, P)[None, None, :].copy()
    mass[0, 0, 20] = mass[0, 0, 5] - 0.5 * SELECT_TIE * rows     # a near-tie with the cutoff page 5
    sel_lens = np.array([P * 16])
    ref_sel, ref_cnt = select_draft_pages(mass, sel_lens, 0.25, 1, 4, b_max=12)
    assert selection_ties_vs_oracle_mass(ref_sel, ref_cnt, mass, sel_lens, 0.25, rows) == 0
    chosen = [int(x) for x in ref_sel[0, 0, : ref_cnt[0, 0]]]
    assert 5 in chosen and 20 not in chosen
    swapped = np.full_like(ref_sel, -1)
    good = sorted(set(chosen) - {5} | {20})
    swapped[0, 0, : len(good)] = good
    assert selection_ties_vs_oracle_mass(swapped, ref_cnt, mass, sel_lens, 0.25, rows) == 1
    bad = sorted(set(chosen) - {5} | {30})      # page 30 lies far below the cutoff
    swapped[0, 0, : len(bad)] = bad
    with pytest.raises(AssertionError):
        selection_ties_vs_oracle_mass(swapped, ref_cnt, mass, sel_lens, 0.25, rows)
