"""GPU parity of draft-page selection: bit-exact against the oracle rule when
both read the same fp32 page mass (including exact ties), plus edge cases."""


import numpy as np
import pytest
import torch

import oracle
import speculative_decode_attention_paged_b300 as s3r
from helpers import budget_b_max, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(mass, sel_lens, budget, n_sink=1, n_recent=4, b_max=None):
    S, H, stride = mass.shape
    b_max = b_max or budget_b_max(stride, budget, n_sink, n_recent)
    ws = s3r.Workspace(s3r.s3r_select_workspace_size())
    mass_t = torch.from_numpy(mass.astype(np.float32)).to(DEV)
    lens_t = torch.from_numpy(np.asarray(sel_lens, dtype=np.int32)).to(DEV)
    sel = torch.full((S, H, b_max), 123, dtype=torch.int32, device=DEV)
    cnt = torch.full((S, H), 123, dtype=torch.int32, device=DEV)
    s3r.s3r_select_draft_pages(mass_t, lens_t, budget, sel, cnt, ws, n_sink=n_sink, n_recent=n_recent)
    ws.check()
    ref_sel, ref_cnt = oracle.select_draft_pages(mass.astype(np.float32), sel_lens, budget, n_sink, n_recent,
                                                 b_max=b_max)
    return host(sel), host(cnt), ref_sel, ref_cnt


# 37 x 8 pairs run one CTA per pair, 80 x 8 one warp per pair (the two kernels of the call)
@pytest.mark.parametrize("S", [37, 80])
@pytest.mark.parametrize("budget", [0.0, 0.05, 0.1, 0.25, 0.5, 1.0])
def test_random_mass_bit_exact(budget, S):
    rng = np.random.default_rng(int(budget * 1000) + S)
    H, stride = 8, 1100
    sel_lens = rng.integers(0, stride * 16 + 1, size=S)
    sel_lens[:6] = [0, 1, 16, 17, 80, stride * 16]
    mass = rng.gamma(0.5, 1.0, size=(S, H, stride))
    sel, cnt, ref_sel, ref_cnt = _run(mass, sel_lens, budget)
    assert np.array_equal(cnt, ref_cnt)
    assert np.array_equal(sel, ref_sel)


@pytest.mark.parametrize("S", [20, 160])
def test_exact_ties_break_to_lower_page(S):
    rng = np.random.default_rng(5)
    H, stride = 4, 300
    sel_lens = rng.integers(1, stride * 16 + 1, size=S)
    mass = rng.integers(0, 3, size=(S, H, stride)).astype(np.float64)   # heavy ties
    for budget in (0.05, 0.3):
        sel, cnt, ref_sel, ref_cnt = _run(mass, sel_lens, budget)
        assert np.array_equal(sel, ref_sel) and np.array_equal(cnt, ref_cnt)


@pytest.mark.parametrize("n_sink,n_recent", [(0, 0), (1, 4), (3, 0), (0, 7), (2, 2)])
def test_sink_and_recent_variants(n_sink, n_recent):
    rng = np.random.default_rng(n_sink * 10 + n_recent)
    S, H, stride = 16, 2, 200
    sel_lens = rng.integers(1, stride * 16 + 1, size=S)
    mass = rng.random((S, H, stride))
    sel, cnt, ref_sel, ref_cnt = _run(mass, sel_lens, 0.1, n_sink, n_recent)
    assert np.array_equal(sel, ref_sel) and np.array_equal(cnt, ref_cnt)


def test_zero_and_subnormal_masses():
    S, H, stride = 3, 2, 64
    mass = np.zeros((S, H, stride))
    mass[0, 0, 10:20] = 1e-40          # subnormal in fp32
    mass[1, 1, 5] = 3.0
    sel_lens = np.array([stride * 16, 900, 33])
    sel, cnt, ref_sel, ref_cnt = _run(mass, sel_lens, 0.25)
    assert np.array_equal(sel, ref_sel) and np.array_equal(cnt, ref_cnt)
