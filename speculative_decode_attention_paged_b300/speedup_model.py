"""Calibrated speedup model of an S³R round over dense autoregressive decoding.

The pages express the speedup as a function of the accepted-prefix fraction
and the effective draft KV-read ratio, with a constant correction fitted on
profiling data, and judge it by its held-out mean absolute percentage error
(wispaper.ai, "Where the speedup claim holds").  They print no formula; this
module takes the plainest one that those two quantities define, for a
memory-bound decode step whose cost is its KV reads:

  a round drafts k tokens, each step reading rho of the dense KV, then
  verifies them with one dense read; it emits 1 + a * k tokens, a the
  accepted-prefix fraction (mean accepted drafts / k).  In units of one dense
  decode step a round costs 1 + k * rho, so

      speedup(a, rho) = (1 + a * k) / (1 + k * rho + c),

  c the constant correction: the round's other costs (verification above one
  dense read, selection, sampling, per-launch latency), in dense-step units.

Calibration works in the cost domain, where c enters linearly: with measured
round times T_round and dense step times T_dense, cost = T_round / T_dense,
and the least-squares c is the mean of cost - 1 - k * rho over the training
points.  The acceptance cancels from the relative error of the speedup, so
MAPE can be taken on costs.
"""

import numpy as np


def accepted_prefix_fraction(alpha, k):
    """Mean accepted drafts / k when each position is accepted with probability
    alpha given the ones before it: sum_{i=1..k} alpha^i / k."""
    alpha = np.asarray(alpha, dtype=np.float64)
    return sum(alpha ** i for i in range(1, k + 1)) / k


def tokens_per_round(a, k):
    return 1.0 + np.asarray(a, dtype=np.float64) * k


def round_cost(rho, k, c=0.0):
    """Cost of a round in dense decode steps."""
    return 1.0 + k * np.asarray(rho, dtype=np.float64) + c


def predict(a, rho, k, c=0.0):
    """Speedup of the round over dense decoding."""
    return tokens_per_round(a, k) / round_cost(rho, k, c)


def fit_correction(rho, cost, k):
    """Least-squares constant c for measured costs (T_round / T_dense)."""
    rho = np.asarray(rho, dtype=np.float64)
    cost = np.asarray(cost, dtype=np.float64)
    if rho.size == 0:
        raise ValueError("no calibration points")
    return float(np.mean(cost - 1.0 - k * rho))


def mape(predicted, measured):
    """Mean absolute percentage error, in percent."""
    p = np.asarray(predicted, dtype=np.float64)
    m = np.asarray(measured, dtype=np.float64)
    return float(100.0 * np.mean(np.abs(p - m) / np.abs(m)))


def calibrate(rho, cost, k, train):
    """Fit c on the points where `train` is true; held-out MAPE of the speedup
    without and with the correction (acceptance cancels, so these are the
    cost errors)."""
    rho = np.asarray(rho, dtype=np.float64)
    cost = np.asarray(cost, dtype=np.float64)
    train = np.asarray(train, dtype=bool)
    c = fit_correction(rho[train], cost[train], k)
    test = ~train
    if not test.any():
        raise ValueError("no held-out points")
    return {"c": c,
            "heldout_mape_uncorrected": mape(1.0 / round_cost(rho[test], k), 1.0 / cost[test]),
            "heldout_mape_corrected": mape(1.0 / round_cost(rho[test], k, c), 1.0 / cost[test]),
            "train_mape_corrected": mape(1.0 / round_cost(rho[train], k, c), 1.0 / cost[train])}
