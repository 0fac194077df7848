"""The speedup model's closed forms and calibration: full acceptance with free
drafts gives k + 1, no acceptance with dense-cost drafts gives 1 / (k + 1);
the accepted-prefix fraction matches a Monte Carlo of sequential acceptance;
the fit recovers a planted correction exactly; held-out errors are those of
the definitions."""

import numpy as np
import pytest

from speculative_decode_attention_paged_b300 import speedup_model as sm


def test_closed_forms():
    for k in (1, 4, 8):
        assert sm.predict(1.0, 0.0, k) == pytest.approx(k + 1)
        assert sm.predict(0.0, 1.0, k) == pytest.approx(1.0 / (k + 1))
        assert sm.predict(0.0, 0.0, k) == pytest.approx(1.0)
        assert sm.predict(0.5, 0.1, k, c=0.3) == pytest.approx((1 + 0.5 * k) / (1.3 + 0.1 * k))


def test_accepted_prefix_fraction_matches_sequential_acceptance():
    rng = np.random.default_rng(0)
    for alpha, k in ((0.8, 4), (0.62, 8), (0.967, 6)):
        ok = rng.random((200_000, k)) < alpha
        n_acc = np.cumprod(ok, axis=1).sum(axis=1)
        assert sm.accepted_prefix_fraction(alpha, k) == pytest.approx(n_acc.mean() / k, abs=3e-3)
    assert sm.accepted_prefix_fraction(1.0, 5) == 1.0 and sm.accepted_prefix_fraction(0.0, 5) == 0.0


def test_fit_recovers_a_planted_correction():
    k, c = 8, 0.437
    rho = np.array([0.02, 0.05, 0.1, 0.25, 0.5, 1.0])
    cost = 1 + k * rho + c
    assert sm.fit_correction(rho, cost, k) == pytest.approx(c, abs=1e-12)
    res = sm.calibrate(rho, cost, k, train=[True, False] * 3)
    assert res["c"] == pytest.approx(c, abs=1e-12)
    assert res["heldout_mape_corrected"] == pytest.approx(0.0, abs=1e-9)
    # without the correction each held-out speedup is off by c / (1 + k rho):
    # |S_model - S| / S = |cost - cost_model| / cost_model
    held = rho[1::2]
    want = 100 * np.mean(c / (1 + k * held))
    assert res["heldout_mape_uncorrected"] == pytest.approx(want, rel=1e-12)


def test_mape_definition():
    assert sm.mape([110, 90], [100, 100]) == pytest.approx(10.0)
    with pytest.raises(ValueError):
        sm.calibrate([0.1], [2.0], 4, train=[True])
