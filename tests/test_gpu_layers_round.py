"""GPU parity of the closed 28-layer S³R round at its own shapes: 28 layers of
the Qwen3-1.7B attention geometry, 32 sequences with histories U{4096..16384}
in a pool sized for 16K tokens per sequence (60.1 GB), budget 0.05, k = 4,
V = 151936.  The round is the one the benchmark times (bench.LayersRound),
replayed from its CUDA graph, and it is checked against the oracle stage by
stage:

  * layers 0 and 27, three sampled sequences (the shortest, the longest and
    one between): every draft step's output (sparse attention over the
    previous round's pages plus the draft tail, after that step's row was
    appended), the verify output and page mass of the k + 1 block rows, and
    the sequences' pages of K and V after the round, bit for bit against the
    oracle's appends;
  * all 32 sequences: the sampled draft tokens, the accepted counts and
    emitted tokens (tie rules of the sampler tests), the committed lengths
    L' = L + n_acc + 1;
  * layers 0 and 27: the next round's pages of the sampled sequences, bit for
    bit against the selection rule applied to the GPU's mass, and against the
    oracle's selection from its own fp64 mass up to counted cutoff ties.

Each replay restarts from the same L and rewrites the same slots, so the
pages read back before the replay serve as the oracle's starting cache: every
position the round reads at or after L is written by the round before it is
read."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_attn_close, compact_pool, host, selection_ties_vs_oracle_mass
from test_gpu_attention import _check_mass
from test_gpu_closed_round import _check_draft_tokens
from test_gpu_spec_sample import compare
from workloads import bf16_to_bits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_28_layer_round_in_its_cuda_graph():
    import bench
    lr = bench.LayersRound(torch.device(DEV, torch.cuda.current_device()))
    try:
        _check_round(lr)
    finally:
        del lr
        torch.cuda.empty_cache()


def _check_round(lr):
    assert lr.n_layers == 28 and lr.S == 32 and lr.pool_gb > 60.0
    lr.s3r_round()                       # warm-up, as the benchmark does
    torch.cuda.synchronize()
    lr.check()
    g_round, _ = lr.capture(dense=False)
    k, S, G = lr.k, lr.S, lr.Hq // lr.Hkv
    L = lr.L_host.numpy().astype(np.int64)
    order = np.argsort(L, kind="stable")
    seqs = sorted({int(order[0]), int(order[S // 2]), int(order[-1])})
    check_layers = (0, lr.n_layers - 1)
    before = {}
    for li in check_layers:
        l = lr.layers[li]
        kp, vp, bt = compact_pool(l["kv"], seqs)
        before[li] = (kp, vp, bt, host(l["sel"][seqs]), host(l["cnt"][seqs]))
    g_round.replay()
    torch.cuda.synchronize()
    lr.check()

    sc = lr.scfg
    q_logits = host(lr.spec.q_logits)
    p_logits = host(lr.spec.p_logits)
    x = host(lr.drafts)
    for j in range(k):
        _check_draft_tokens(q_logits[:, j], x[:, j], sc.philox_seed, 0, j)
    out_t, nacc = host(lr.out_tokens), host(lr.n_acc)
    compare(p_logits, q_logits, x, sc.philox_seed, 0, out_t, nacc)
    L_next = host(lr.L_next)
    assert np.array_equal(L_next, oracle.commit_lengths(L, nacc))

    Ls = L[seqs]
    for li in check_layers:
        l = lr.layers[li]
        kp, vp, bt, sel, cnt = before[li]
        for j in range(k):
            kp, vp = oracle.kv_append(kp, vp, bt, Ls + j, bf16_to_bits(l["draft_kv"][j][0][seqs]),
                                      bf16_to_bits(l["draft_kv"][j][1][seqs]))
            ref = oracle.sparse_draft_attn(bf16_to_bits(l["qd"][j][seqs]), kp, vp, bt, Ls, j, sel, cnt, 1.0)
            assert_attn_close(l["out_d"][j][seqs], ref, f"layer {li} draft {j}")
        kp, vp = oracle.kv_append(kp, vp, bt, Ls, bf16_to_bits(l["block_kv"][0][seqs]),
                                  bf16_to_bits(l["block_kv"][1][seqs]))
        kp_gpu, vp_gpu, _ = compact_pool(l["kv"], seqs)
        assert np.array_equal(kp_gpu, kp) and np.array_equal(vp_gpu, vp), f"layer {li}: pages after the round"
        ref_o, ref_m = oracle.verify_attn(bf16_to_bits(l["qv"][seqs]), kp, vp, bt, Ls, 1.0,
                                          mass_pages=l["kv"].max_pages)
        assert_attn_close(l["out_v"][seqs], ref_o, f"layer {li} verify")
        _check_mass(l["mass"][seqs], ref_m, G * (k + 1))
        # the next round's pages over L'
        mass_gpu = host(l["mass"][seqs]).astype(np.float64)
        b_max = l["sel_next"].shape[-1]
        ref_pages, ref_cnt = oracle.select_draft_pages(mass_gpu, L_next[seqs], lr.budget, b_max=b_max)
        assert np.array_equal(host(l["cnt_next"][seqs]), ref_cnt)
        assert np.array_equal(host(l["sel_next"][seqs]), ref_pages)
        swaps = selection_ties_vs_oracle_mass(host(l["sel_next"][seqs]), host(l["cnt_next"][seqs]), ref_m,
                                              L_next[seqs], lr.budget, G * (k + 1))
        print(f"layer {li}: {swaps} selection tie swaps over {len(seqs) * lr.Hkv} pairs")
        assert swaps <= 1
