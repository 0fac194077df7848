"""GPU checks of the sequential (early-exit) speculative sampler.

It computes the same function as the parallel sampler with the ratio tests
taken one position at a time, so on the same inputs its accepted counts and
tokens must equal the parallel sampler's bit for bit, and so must its tie
counts; against the oracle the same tie rules apply (ratio ties within 1e-6,
inverse-CDF ties within 1e-6 * Z).  Its per-sequence arrival counters must be left at zero, so a
workspace serves any number of calls."""

import numpy as np
import pytest
import torch

import speculative_decode_attention_paged_b300 as s3r
from helpers import host
from test_gpu_spec_sample import compare
from workloads import make_spec_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(fn, p, q, x, seed, offset=0, ws=None, ties=None):
    N, k1, V = p.shape
    if ws is None:
        ws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(N, k1 - 1))
    out = torch.full((N, k1), 77, dtype=torch.int32, device=DEV)
    nacc = torch.full((N,), 77, dtype=torch.int32, device=DEV)
    fn(p, q, x, seed, offset, out, nacc, ws, tie_count=ties)
    return host(out), host(nacc), ws


def _both(inp, seed, offset=0):
    ties_p = torch.full((2,), 55, dtype=torch.int32, device=DEV)
    ties_s = torch.full((2,), 66, dtype=torch.int32, device=DEV)
    out_p, nacc_p, ws = _run(s3r.s3r_spec_sample, inp.p_logits, inp.q_logits, inp.draft_tokens, seed, offset,
                             ties=ties_p)
    ws.check()
    out_s, nacc_s, ws = _run(s3r.s3r_spec_sample_sequential, inp.p_logits, inp.q_logits, inp.draft_tokens, seed,
                             offset, ties=ties_s)
    ws.check()
    assert torch.equal(ties_p, ties_s)
    return (out_p, nacc_p), (out_s, nacc_s)


@pytest.mark.parametrize("N,k,V,sigma", [
    (4, 4, 4096, 0.5), (64, 4, 1, 1.0), (64, 4, 7, 1.0), (64, 3, 4099, 1.0), (200, 8, 1000, 3.0),
    (256, 8, 151936, 0.3), (256, 8, 151936, 1.0), (128, 4, 151936, 3.0), (96, 1, 32000, 1.0)])
def test_equals_parallel_sampler_bit_for_bit(N, k, V, sigma):
    inp = make_spec_inputs(N, k, V, 3.0, sigma, seed=N + k + V, device=DEV)
    (out_p, nacc_p), (out_s, nacc_s) = _both(inp, seed=4242, offset=3)
    assert np.array_equal(nacc_p, nacc_s)
    assert np.array_equal(out_p, out_s)


def test_matches_oracle_qwen_vocab():
    inp = make_spec_inputs(128, 8, 151936, 3.0, 1.0, seed=17, device=DEV)
    out, nacc, ws = _run(s3r.s3r_spec_sample_sequential, inp.p_logits, inp.q_logits, inp.draft_tokens, 99, 5)
    ws.check()
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 99, 5, out, nacc)


def test_all_accepted_and_bonus_only():
    inp = make_spec_inputs(128, 6, 5000, 3.0, 0.0, seed=3, device=DEV)      # q = p: every draft accepted
    (out_p, nacc_p), (out_s, nacc_s) = _both(inp, seed=5)
    assert np.all(nacc_s == 6) and np.array_equal(out_p, out_s)
    inp0 = make_spec_inputs(32, 0, 1000, 3.0, 1.0, seed=4, device=DEV)     # k = 0
    (out_p, nacc_p), (out_s, nacc_s) = _both(inp0, seed=6)
    assert np.all(nacc_s == 0) and np.array_equal(out_p, out_s)


def test_scalar_path_for_unaligned_logits():
    """Logits 4 bytes past a 16-byte boundary take the scalar-load kernels."""
    inp = make_spec_inputs(64, 4, 4096, 3.0, 1.0, seed=8, device=DEV)
    N, k1, V = inp.p_logits.shape
    pbuf = torch.empty(inp.p_logits.numel() + 1, dtype=torch.float32, device=DEV)
    qbuf = torch.empty(inp.q_logits.numel() + 1, dtype=torch.float32, device=DEV)
    p = pbuf[1:].view(N, k1, V)
    q = qbuf[1:].view(N, k1 - 1, V)
    p.copy_(inp.p_logits)
    q.copy_(inp.q_logits)
    assert p.data_ptr() % 16 != 0
    out, nacc, ws = _run(s3r.s3r_spec_sample_sequential, p, q, inp.draft_tokens, 11)
    ws.check()
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 11, 0, out, nacc)


def test_counters_reset_between_calls_and_after_bad_tokens():
    inp = make_spec_inputs(96, 4, 3000, 3.0, 1.0, seed=21, device=DEV)
    first_out, first_nacc, ws = _run(s3r.s3r_spec_sample_sequential, inp.p_logits, inp.q_logits,
                                     inp.draft_tokens, 7)
    for _ in range(3):
        out, nacc, _ = _run(s3r.s3r_spec_sample_sequential, inp.p_logits, inp.q_logits, inp.draft_tokens, 7, ws=ws)
        assert np.array_equal(out, first_out) and np.array_equal(nacc, first_nacc)
    ws.check()
    bad = inp.draft_tokens.clone()
    bad[5, 0] = 3000                                  # outside the vocabulary: rejected at position 0, reported
    out, nacc, _ = _run(s3r.s3r_spec_sample_sequential, inp.p_logits, inp.q_logits, bad, 7, ws=ws)
    assert ws.read_error() & s3r.DEVERR_BAD_TOKEN
    assert nacc[5] == 0
    out, nacc, _ = _run(s3r.s3r_spec_sample_sequential, inp.p_logits, inp.q_logits, inp.draft_tokens, 7, ws=ws)
    assert ws.read_error() == 0
    assert np.array_equal(out, first_out) and np.array_equal(nacc, first_nacc)


def test_draft_sampling_reuses_its_workspace():
    """The k = 0 kernel's counters are left at zero: repeated draft-token calls
    on one workspace agree."""
    n, V = 300, 151936
    g = torch.Generator(device=DEV)
    g.manual_seed(12)
    logits = torch.randn((n, V), generator=g, device=DEV) * 3.0
    ws = s3r.Workspace(s3r.s3r_sample_draft_workspace_size(n))
    toks = []
    for _ in range(3):
        t = torch.full((n,), -5, dtype=torch.int32, device=DEV)
        s3r.s3r_sample_draft_tokens(logits, 9, 2, 1, t, ws)
        toks.append(host(t))
    ws.check()
    assert all(np.array_equal(toks[0], t) for t in toks[1:])
    assert np.all((toks[0] >= 0) & (toks[0] < V))


def test_long_blocks_beyond_one_warp_of_drafts():
    """k = 40: the parallel ratio tests take two 32-lane passes and the
    sequential sampler 41 steps; both agree with each other and the oracle."""
    inp = make_spec_inputs(24, 40, 1000, 3.0, 0.05, seed=40, device=DEV)
    (out_p, nacc_p), (out_s, nacc_s) = _both(inp, seed=8, offset=2)
    assert np.array_equal(nacc_p, nacc_s) and np.array_equal(out_p, out_s)
    assert nacc_s.max() > 32                     # some block got past the first warp of tests
    compare(host(inp.p_logits), host(inp.q_logits), host(inp.draft_tokens), 8, 2, out_s, nacc_s)
