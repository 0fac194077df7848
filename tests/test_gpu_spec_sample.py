"""GPU parity of exact speculative sampling against the oracle.

Given identical fp32 logits and identical Philox uniforms, accept/reject
decisions and sampled tokens must match bit for bit, except floating-point
ties, which are counted and bounded:
  * a ratio tie: |u - p_i(x_i)/q_i(x_i)| <= 1e-6;
  * a resample tie: the GPU token is still a valid inverse-CDF answer for the
    oracle's fp64 CDF C of the row within 1e-6 * Z:
    C[y-1] <= u*Z + 1e-6*Z and C[y] >= u*Z - 1e-6*Z.
Every disagreement must also be one the GPU counted itself (the sampler's
tie counters flag the decisions that lie within those windows on its side).
The exactness theorem itself is checked on the GPU too (chi-square of the
first emitted token against p_1 over 10^6 sequences)."""

import numpy as np
import pytest
import torch
from scipy import special, stats

import oracle
import speculative_decode_attention_paged_b300 as s3r
from workloads import SAMPLER_ROLLOUT_2048SEQ, SAMPLER_TINY, make_spec_inputs
from helpers import host

pytestmark = pytest.mark.gpu
DEV = "cuda"
RATIO_TIE = 1e-6
CDF_TIE = 1e-6


def _gpu(inp, seed, offset=0, with_ties=False):
    N, k1, V = inp.p_logits.shape
    k = k1 - 1
    ws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(N, k))
    out = torch.full((N, k + 1), 77, dtype=torch.int32, device=DEV)
    nacc = torch.full((N,), 77, dtype=torch.int32, device=DEV)
    ties = torch.full((2,), 99, dtype=torch.int32, device=DEV)
    s3r.s3r_spec_sample(inp.p_logits, inp.q_logits, inp.draft_tokens, seed, offset, out, nacc, ws, tie_count=ties)
    ws.check()
    if with_ties:
        return host(out), host(nacc), host(ties)
    return host(out), host(nacc)


def compare(p_logits, q_logits, drafts, seed, offset, out_g, nacc_g, max_tie_frac=0.01, seq_ids=None,
            gpu_ties=None):
    """Oracle on the same host arrays; returns (ratio_ties, cdf_ties), the
    disagreements that the tie windows allow.  gpu_ties: the GPU's own
    [ratio, inverse-CDF] tie counts over the same sequences, which must cover
    every disagreement."""
    out_o, nacc_o, det = oracle.spec_sample(p_logits, q_logits, drafts, seed, offset, seq_ids=seq_ids)
    N, k = drafts.shape
    ratio_ties = cdf_ties = 0
    for n in range(N):
        if nacc_g[n] != nacc_o[n]:
            i = min(nacc_g[n], nacc_o[n])     # first position where the decisions differ
            gap = abs(det["u_accept"][n, i] - det["ratio"][n, i])
            assert gap <= RATIO_TIE, f"seq {n}: accept decision differs at {i}, |u - ratio| = {gap:.3e}"
            ratio_ties += 1
            continue
        assert np.array_equal(out_g[n, : nacc_g[n]], out_o[n, : nacc_o[n]])
        assert np.all(out_g[n, nacc_g[n] + 1:] == -1)
        yg, yo = int(out_g[n, nacc_g[n]]), int(out_o[n, nacc_o[n]])
        if yg != yo:
            a = int(nacc_o[n])
            if a < k:
                row = oracle.residual_row(p_logits[n, a], q_logits[n, a])
            else:
                row = np.exp(p_logits[n, k].astype(np.float64) - p_logits[n, k].max())
                row /= row.sum()
            C = np.cumsum(row)
            Z = C[-1]
            t = det["u_resample"][n] * Z
            lo = C[yg - 1] if yg > 0 else 0.0
            assert 0 <= yg < len(row) and row[yg] > 0, f"seq {n}: token {yg} has zero probability"
            assert lo <= t + CDF_TIE * Z and C[yg] >= t - CDF_TIE * Z, f"seq {n}: token {yg} vs {yo}"
            cdf_ties += 1
    assert ratio_ties + cdf_ties <= max(2, max_tie_frac * N), (ratio_ties, cdf_ties)
    if gpu_ties is not None:
        assert ratio_ties <= gpu_ties[0] and cdf_ties <= gpu_ties[1], ((ratio_ties, cdf_ties), tuple(gpu_ties))
    return ratio_ties, cdf_ties


def test_tiny_sampler_full():
    cfg = SAMPLER_TINY
    inp = make_spec_inputs(cfg.num_seqs, cfg.k, cfg.vocab, cfg.p_sigma, cfg.q_sigmas[0], cfg.seed, device=DEV)
    out, nacc, ties = _gpu(inp, cfg.philox_seed, with_ties=True)
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), cfg.philox_seed, 0, out, nacc,
            gpu_ties=ties)


@pytest.mark.parametrize("sigma", [0.3, 1.0, 3.0])
def test_qwen_vocab_many_sequences(sigma):
    inp = make_spec_inputs(256, 8, 151936, 3.0, sigma, seed=int(sigma * 10), device=DEV)
    out, nacc, ties = _gpu(inp, seed=12345, offset=7, with_ties=True)
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 12345, 7, out, nacc, gpu_ties=ties)


@pytest.mark.parametrize("V", [1, 2, 3, 5, 127, 1000, 4099, 300000])
def test_odd_vocab_sizes(V):
    inp = make_spec_inputs(64 if V < 100_000 else 8, 4, V, 2.0, 1.0, seed=V, device=DEV)
    out, nacc, ties = _gpu(inp, seed=99, with_ties=True)
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 99, 0, out, nacc, gpu_ties=ties)


def test_q_equals_p_accepts_everything():
    inp = make_spec_inputs(128, 6, 5000, 3.0, 0.0, seed=3, device=DEV)
    out, nacc = _gpu(inp, seed=5)
    assert np.all(nacc == 6)
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 5, 0, out, nacc)


def test_k_zero_samples_bonus_only():
    inp = make_spec_inputs(32, 0, 1000, 3.0, 1.0, seed=4, device=DEV)
    out, nacc = _gpu(inp, seed=6)
    assert np.all(nacc == 0)
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 6, 0, out, nacc)


def test_rollout_2048seq_sampled():
    cfg = SAMPLER_ROLLOUT_2048SEQ
    for sigma in cfg.q_sigmas:
        inp = make_spec_inputs(cfg.num_seqs, cfg.k, cfg.vocab, cfg.p_sigma, sigma, cfg.seed, device=DEV)
        out, nacc = _gpu(inp, cfg.philox_seed)
        # acceptance is what the noise level implies (~95% / ~80% per position)
        rate = (nacc[:, None] > np.arange(cfg.k)[None, :]).sum() / max(1, (np.minimum(nacc + 1, cfg.k)).sum())
        assert 0.5 < rate < 1.0
        rng = np.random.default_rng(int(sigma * 100))
        seqs = np.sort(rng.choice(cfg.num_seqs, size=128, replace=False))
        compare(host(inp.p_logits[seqs]), host(inp.q_logits[seqs]), host(inp.draft_tokens[seqs]),
                cfg.philox_seed, 0, out[seqs], nacc[seqs], seq_ids=seqs)


def test_exactness_theorem_on_gpu():
    """First emitted token ~ p_1 over 10^6 sequences (chi-square)."""
    N, k, V = 1_000_000, 3, 12
    rng = np.random.default_rng(9)
    p_row = rng.normal(0, 1.5, size=(k + 1, V)).astype(np.float32)
    q_row = (p_row[:k] + rng.normal(0, 1.0, size=(k, V))).astype(np.float32)
    p = torch.from_numpy(p_row).to(DEV).expand(N, k + 1, V).contiguous()
    q = torch.from_numpy(q_row).to(DEV).expand(N, k, V).contiguous()
    qprob = special.softmax(q_row.astype(np.float64), axis=-1)
    x = np.stack([rng.choice(V, size=N, p=qprob[i]) for i in range(k)], axis=1).astype(np.int32)
    inp = type("I", (), {})()
    inp.p_logits, inp.q_logits, inp.draft_tokens = p, q, torch.from_numpy(x).to(DEV)
    out, nacc = _gpu(inp, seed=2024)
    pprob = special.softmax(p_row.astype(np.float64), axis=-1)
    for j in range(k + 1):
        have = nacc >= j
        counts = np.bincount(out[have, j], minlength=V)
        assert stats.chisquare(counts, pprob[j] * have.sum()).pvalue > 1e-3



def _nearest_boundary_gap(row, target):
    """Distance from target to the nearer end of the interval (C[y-1], C[y]]
    that holds it, relative to Z = C[-1] (fp64)."""
    C = np.cumsum(row)
    Z = C[-1]
    y = min(int(np.argmax(C > target)), len(C) - 1)
    lo = C[y - 1] if y > 0 else 0.0
    return min(target - lo, C[y] - target) / Z


def test_tie_counters_count_planted_near_ties():
    """The GPU's tie counters flag the decisions within the windows.  Half the
    sequences get a draft whose ratio p/q is planted within +-2e-6 of its
    acceptance uniform; the other half accept every draft (q = p) and get a
    bonus row whose first CDF boundary is planted within +-2e-6 of the
    resampling uniform.  The oracle's fp64 gaps then bound the counts: every
    gap within 0.7 of the window must be counted, none beyond 1.3 of it (the
    GPU decides on fp32 row statistics)."""
    from oracle import philox_uniform
    N, k, V, seed = 2048, 3, 64, 4242
    rng = np.random.default_rng(32)
    p_logits = rng.normal(0, 1.0, size=(N, k + 1, V))
    q_logits = p_logits[:, :k] + rng.normal(0, 0.5, size=(N, k, V))
    drafts = rng.integers(0, V, size=(N, k))
    half = N // 2
    delta = rng.uniform(-2e-6, 2e-6, size=N)
    # ratio ties at position 0: q_0 uniform, p_0 = e^a at the draft, 1 elsewhere
    n1 = np.arange(half)
    t = np.clip(philox_uniform(seed, 0, n1, 0, 0) + delta[n1], 1e-3, None)
    q_logits[n1, 0] = 0.0
    p_logits[n1, 0] = 0.0
    p_logits[n1, 0, drafts[n1, 0]] = np.log(t * (V - 1) / (V - t))
    # inverse-CDF ties in the bonus row: q = p accepts everything; token 0 of
    # p_k holds mass t next to the uniform of (n, k, RESAMPLE)
    n2 = np.arange(half, N)
    q_logits[n2] = p_logits[n2, :k]
    t2 = np.clip(philox_uniform(seed, 0, n2, k, 1) + delta[n2], 1e-3, 1.0 - 1e-3)
    p_logits[n2, k] = 0.0
    p_logits[n2, k, 0] = np.log(t2 * (V - 1) / (1.0 - t2))
    p32, q32, d32 = p_logits.astype(np.float32), q_logits.astype(np.float32), drafts.astype(np.int32)
    inp = type("I", (), {})()
    inp.p_logits, inp.q_logits, inp.draft_tokens = (torch.from_numpy(x).to(DEV) for x in (p32, q32, d32))
    out, nacc, ties = _gpu(inp, seed=seed, with_ties=True)
    compare(p32, q32, d32, seed, 0, out, nacc, gpu_ties=ties, max_tie_frac=1.0)

    _, nacc_o, det = oracle.spec_sample(p32, q32, d32, seed, 0)
    gap = np.abs(det["u_accept"] - det["ratio"]) / RATIO_TIE
    tested = np.arange(k)[None, :] <= np.minimum(nacc_o, k - 1)[:, None]
    r_sure, r_maybe = int(((gap <= 0.7) & tested).sum()), int(((gap <= 1.3) & tested).sum())
    cgap = np.empty(N)
    for n in range(N):
        a = int(nacc_o[n])
        if a < k:
            row = oracle.residual_row(p32[n, a], q32[n, a])
        else:
            row = special.softmax(p32[n, k].astype(np.float64))
        cgap[n] = _nearest_boundary_gap(row, det["u_resample"][n] * row.sum()) / CDF_TIE
    c_sure, c_maybe = int((cgap <= 0.7).sum()), int((cgap <= 1.3).sum())
    assert r_sure > 200 and c_sure > 200          # the planted ties are there
    assert r_sure <= ties[0] <= r_maybe, (r_sure, int(ties[0]), r_maybe)
    assert c_sure <= ties[1] <= c_maybe, (c_sure, int(ties[1]), c_maybe)
