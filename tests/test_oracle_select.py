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
