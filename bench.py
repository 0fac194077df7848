"""Benchmark of the S³R paged decode-attention hot path on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl s3r|reference]

One step is one pass of the whole hot path over one batch of synthetic input
shaped like the Qwen3-1.7B rollout workload (one attention layer, 256
sequences, histories U{4096..16384}, 16 query / 8 KV heads, head_dim 128,
16-token bf16 pages in a randomly permuted pool, k = 4, budget 0.05, Qwen3
vocabulary 151936 for the sampler):

  1. k dense decode steps (the autoregressive baseline, positions L .. L+k-1);
  2. verification of the k-token block with page mass;
  3. draft-page selection from that mass (history L + k);
  4. k sparse draft steps of the next round over the selected pages;
  5. exact speculative sampling of the 256 drafted blocks.

`value` is the algorithmic HBM throughput of the whole step in GB/s (KV bytes
of every attention call + queries/outputs + page mass + selection + logits:
the bytes the step must move at least once) divided by the device time of the
step; the per-phase split, the draft+verify attention tokens/s, the dense
tokens/s and the effective tokens/s at the measured acceptance are extra keys.
`e2e` repeats the step through the same calls with host inputs and results:
each step's inputs are copied from pinned host memory and its results copied
back inside the timed region, two buffer sets letting one step's upload
overlap the previous step's kernels.  The reference arm (--impl reference)
times the fp64 CPU oracle on a bounded sample of the same workload.

Other workloads (--workload, one JSON line each): `sweep` (Qwen3-8B geometry,
budgets 0.05 .. 0.50), `sampler` (2048 sequences x k = 8, parallel and
sequential samplers, draft-token sampling), `layers` (the closed 28-layer
round against 4 dense steps), `scheduler` (the AIMD KV scheduler simulation,
host only) and `speedup` (the speedup-model calibration).
"""

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from workloads import (ATTN_QWEN3_1P7B_256SEQ, ATTN_QWEN3_1P7B_28LAYER, ATTN_QWEN3_8B_128SEQ,  # noqa: E402
                       ATTN_TINY, ROLLOUT_ACCEPTANCE_MATCHED_SIGMAS, SAMPLER_ROLLOUT_2048SEQ, SAMPLER_ROUND_256SEQ,
                       SAMPLER_TINY, make_paged_kv, make_queries, make_rollout_requests, make_spec_inputs)

METRIC = "KV GB/s (% of 8 TB/s) and draft+verify attention tokens/s at 1 B300"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
KV_TOKEN_BYTES_PER_HEAD = 2 * 128 * 2          # K + V rows of one token of one KV head, bf16
SMI_FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def ceil_div(a, b):
    return -(-a // b)


def selection_budget_pages(P, budget, n_sink=1, n_recent=4):
    mand = min(n_sink, P) + (P - max(max(P - n_recent, 0), min(n_sink, P)))
    return min(P, max(math.ceil(budget * P - 1e-9), mand))


# ---------------------------------------------------------------- workload

class Workload:
    """Device-resident inputs of one step (built once, reused every step)."""

    def __init__(self, device, attn_cfg=ATTN_QWEN3_1P7B_256SEQ, sampler_cfg=SAMPLER_ROUND_256SEQ, num_seqs=None):
        self.cfg = attn_cfg
        self.scfg = sampler_cfg
        if num_seqs is not None:
            import dataclasses
            self.cfg = dataclasses.replace(self.cfg, num_seqs=int(num_seqs))
            self.scfg = dataclasses.replace(self.scfg, num_seqs=int(num_seqs))
        c = self.cfg
        self.k = c.k
        self.budget = c.budgets[0]
        # capacity for the verified block and the next round's draft tail
        self.kv = make_paged_kv(c.num_seqs, c.q_heads, c.kv_heads, 2 * c.k, seed=c.seed, device=device,
                                hist_min=c.hist_min, hist_max=c.hist_max,
                                heavy_per_head=c.heavy_per_head, heavy_score=c.heavy_score)
        kv = self.kv
        S, Hq, Hkv, k = kv.num_seqs, kv.q_heads, kv.kv_heads, self.k
        self.S, self.Hq, self.Hkv = S, Hq, Hkv
        self.q_verify = make_queries(kv, 1000, rows=k)
        self.q_dense = [make_queries(kv, 1100 + j) for j in range(k)]
        self.q_draft = [make_queries(kv, 1200 + j) for j in range(k)]
        self.ctx_dense = [(kv.hist_lens + j + 1).to(torch.int32) for j in range(k)]
        self.sel_lens = (kv.hist_lens + k).to(torch.int32)
        self.mass_stride = kv.max_pages
        self.b_max = selection_budget_pages(self.mass_stride, self.budget)
        sc = self.scfg
        self.spec = make_spec_inputs(sc.num_seqs, sc.k, sc.vocab, sc.p_sigma, sc.q_sigmas[0], sc.seed,
                                     device=device)
        self.N, self.V = sc.num_seqs, sc.vocab
        # outputs
        f32 = dict(dtype=torch.float32, device=device)
        self.out_dense = [torch.empty(q.shape, **f32) for q in self.q_dense]
        self.out_verify = torch.empty(self.q_verify.shape, **f32)
        self.out_draft = [torch.empty(q.shape, **f32) for q in self.q_draft]
        self.mass = torch.empty((S, Hkv, self.mass_stride), **f32)
        self.sel = torch.empty((S, Hkv, self.b_max), dtype=torch.int32, device=device)
        self.cnt = torch.empty((S, Hkv), dtype=torch.int32, device=device)
        self.out_tokens = torch.empty((self.N, sc.k + 1), dtype=torch.int32, device=device)
        self.n_acc = torch.empty((self.N,), dtype=torch.int32, device=device)

    # ---- algorithmic bytes (per call), used for value and the roofline
    def dense_bytes(self, j):
        L = self.kv.hist_lens.double()
        kv_bytes = float((L + j + 1).sum()) * self.Hkv * KV_TOKEN_BYTES_PER_HEAD
        return kv_bytes + self.S * self.Hq * 128 * (2 + 4)

    def verify_bytes(self):
        L = self.kv.hist_lens.double()
        kv_bytes = float((L + self.k).sum()) * self.Hkv * KV_TOKEN_BYTES_PER_HEAD
        return kv_bytes + self.S * self.k * self.Hq * 128 * (2 + 4) + self.S * self.Hkv * self.mass_stride * 4

    def select_bytes(self):
        return self.S * self.Hkv * (self.mass_stride + self.b_max + 1) * 4

    def draft_tokens_visible(self, j):
        """Tokens each (sequence, KV head) of draft step j reads (host count
        from the selection, which is the same every step)."""
        sel = self.sel.cpu().numpy()
        cnt = self.cnt.cpu().numpy()
        Lsel = self.sel_lens.cpu().numpy().astype(np.int64)
        total = 0
        for s in range(self.S):
            L = int(Lsel[s])
            for h in range(self.Hkv):
                pages = sel[s, h, : cnt[s, h]].astype(np.int64)
                total += int(np.minimum(pages * 16 + 16, L).sum() - np.minimum(pages * 16, L).sum())
            total += self.Hkv * (j + 1)
        return total

    def draft_bytes(self, j):
        return (self._draft_tok[j] * KV_TOKEN_BYTES_PER_HEAD + self.S * self.Hq * 128 * (2 + 4)
                + self.S * self.Hkv * (self.b_max + 1) * 4)

    def sample_bytes(self):
        k = self.scfg.k
        return self.N * (2 * k + 1) * self.V * 4 + self.N * (k + (k + 1) + 1) * 4

    def finalize_bytes(self):
        self._draft_tok = [self.draft_tokens_visible(j) for j in range(self.k)]
        self.bytes = {
            "dense": [self.dense_bytes(j) for j in range(self.k)],
            "verify": self.verify_bytes(),
            "select": self.select_bytes(),
            "draft": [self.draft_bytes(j) for j in range(self.k)],
            "sample": self.sample_bytes(),
        }
        b = self.bytes
        self.step_bytes = sum(b["dense"]) + b["verify"] + b["select"] + sum(b["draft"]) + b["sample"]


class Runner:
    """Issues one step through the C-ABI binding, with events between phases."""

    PHASES = ("dense", "verify", "select", "draft", "sample")

    def __init__(self, w: Workload):
        import speculative_decode_attention_paged_b300 as s3r
        self.s3r = s3r
        self.w = w
        self.desc = s3r.PagedKVDesc(w.kv.k_pool, w.kv.v_pool, w.kv.block_table, w.kv.q_heads)
        dev = w.kv.k_pool.device
        self.ws = s3r.Workspace(s3r.s3r_attn_workspace_size(self.desc, w.k), device=dev)
        self.sws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(w.N, w.scfg.k), device=dev)
        # dense x k, verify, select, drafts x k, sampler (one kernel per call)
        self.launches_per_step = w.k + 1 + 1 + w.k + 1

    def step(self, ev=None):
        """ev: list of 2k+4 events recorded at the phase boundaries, or None."""
        s3r, w = self.s3r, self.w
        i = 0

        def mark():
            nonlocal i
            if ev is not None:
                ev[i].record()
            i += 1

        mark()
        for j in range(w.k):
            s3r.s3r_dense_decode_attn(self.desc, w.ctx_dense[j], w.q_dense[j], w.out_dense[j], 1.0, self.ws)
            mark()
        s3r.s3r_verify_attn(self.desc, w.kv.hist_lens, w.q_verify, w.out_verify, 1.0, self.ws, page_mass=w.mass)
        mark()
        s3r.s3r_select_draft_pages(w.mass, w.sel_lens, w.budget, w.sel, w.cnt, self.ws)
        mark()
        for j in range(w.k):
            s3r.s3r_sparse_draft_attn(self.desc, w.sel_lens, j, w.sel, w.cnt, w.q_draft[j], w.out_draft[j], 1.0,
                                      self.ws)
            mark()
        s3r.s3r_spec_sample(w.spec.p_logits, w.spec.q_logits, w.spec.draft_tokens, w.scfg.philox_seed, 0,
                            w.out_tokens, w.n_acc, self.sws)
        mark()

    def n_events(self):
        return 2 * self.w.k + 4


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) taken while the timed region runs."""

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        import tempfile
        self.path = os.path.join(tempfile.gettempdir(), f"s3r_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                if self.uuid and parts[0] != self.uuid:
                    continue
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": num(rows[0][2]),
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------- distributed plumbing

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def aggregate_gbs(step_bytes, ms_per_step, world):
    """Whole-job throughput of `world` replicas each moving step_bytes per
    step, timed by the slowest rank (ms_per_step = max over ranks)."""
    return world * step_bytes / (ms_per_step * 1e-3) / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU baseline (the oracle)

def _oracle_inputs(seed, n_seqs):
    """Host inputs of `n_seqs` sequences of the 256-sequence round, regenerated
    on the CPU with the same recipe (shapes, distributions) and their own seed."""
    from workloads import bf16_to_bits
    c = ATTN_QWEN3_1P7B_256SEQ
    sc = SAMPLER_ROUND_256SEQ
    kv = make_paged_kv(n_seqs, c.q_heads, c.kv_heads, 2 * c.k, seed=c.seed + 100 + seed, device="cpu",
                       hist_min=c.hist_min, hist_max=c.hist_max)
    spec = make_spec_inputs(n_seqs, sc.k, sc.vocab, sc.p_sigma, sc.q_sigmas[0], sc.seed + 100 + seed)
    return (bf16_to_bits(kv.k_pool), bf16_to_bits(kv.v_pool), kv.block_table.numpy(),
            kv.hist_lens.numpy().astype(np.int64), bf16_to_bits(make_queries(kv, 1000, rows=c.k)),
            bf16_to_bits(make_queries(kv, 1100)), spec.p_logits.numpy(), spec.q_logits.numpy(),
            spec.draft_tokens.numpy())


def _oracle_pass(inputs, s):
    """The fp64 oracle over one whole sequence s of `inputs`: k dense decode
    steps, verify with page mass, selection, k sparse drafts and exact
    speculative sampling; returns the algorithmic bytes of that work."""
    import oracle
    c = ATTN_QWEN3_1P7B_256SEQ
    sc = SAMPLER_ROUND_256SEQ
    kp, vp, bt, L, qv, qd, p_l, q_l, x_l = inputs
    n_seqs = len(L)
    k, Hkv, Hq = c.k, c.kv_heads, c.q_heads
    one = [s]
    done = 0.0
    for j in range(k):
        oracle.dense_decode_attn(qd, kp, vp, bt, L + j + 1, 1.0, seqs=one)
        done += (L[s] + j + 1) * Hkv * KV_TOKEN_BYTES_PER_HEAD + Hq * 128 * 6
    _, mass = oracle.verify_attn(qv, kp, vp, bt, L, 1.0, seqs=one, mass_pages=bt.shape[1])
    done += (L[s] + k) * Hkv * KV_TOKEN_BYTES_PER_HEAD + k * Hq * 128 * 6 + Hkv * bt.shape[1] * 4
    sel, cnt = oracle.select_draft_pages(mass, L[one] + k, c.budgets[0], 1, 4)
    done += Hkv * (bt.shape[1] + sel.shape[-1]) * 4
    sel_full = np.full((n_seqs, Hkv, sel.shape[-1]), -1, dtype=np.int64)
    cnt_full = np.zeros((n_seqs, Hkv), dtype=np.int64)
    sel_full[s], cnt_full[s] = sel[0], cnt[0]
    for j in range(k):
        oracle.sparse_draft_attn(qd, kp, vp, bt, L + k, j, sel_full, cnt_full, 1.0, seqs=one)
        vis = 0
        for h in range(Hkv):
            pg = sel[0, h, : cnt[0, h]]
            vis += int(np.minimum(pg * 16 + 16, L[s] + k).sum() - np.minimum(pg * 16, L[s] + k).sum()) + j + 1
        done += vis * KV_TOKEN_BYTES_PER_HEAD + Hq * 128 * 6
    oracle.spec_sample(p_l[one], q_l[one], x_l[one], sc.philox_seed, 0, seq_ids=one)
    done += (2 * sc.k + 1) * sc.vocab * 4
    return done


def _oracle_loop(inputs, seconds):
    """Whole-sequence oracle passes over `inputs` until `seconds` of CPU time
    are spent (at least one pass); returns (bytes, seconds, passes)."""
    n = len(inputs[3])
    done, passes = 0.0, 0
    t0 = time.perf_counter()
    while True:
        done += _oracle_pass(inputs, passes % n)
        passes += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return done, time.perf_counter() - t0, passes


def _oracle_worker(wid, n_seqs, cmd_q, res_q, barrier):
    """One oracle process of OracleFarm: builds its own sequences, then runs a
    timed loop for each command until it receives None."""
    inputs = _oracle_inputs(1000 + wid, n_seqs)
    res_q.put(("ready", wid))
    while True:
        seconds = cmd_q.get()
        if seconds is None:
            return
        barrier.wait()
        res_q.put(_oracle_loop(inputs, seconds))


_SINGLE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS")


class OracleFarm:
    """The fp64 oracle on the host's cores: one single-threaded process per
    core (started with spawn, so no CUDA state is inherited), each over its
    own sequences of the same recipe.  run(seconds) times all of them
    together and returns (bytes, wall seconds, passes): the oracle's whole-job
    throughput on `workers` cores."""

    def __init__(self, workers=None, seqs_per_worker=2):
        import multiprocessing as mp
        self.cpu_count = os.cpu_count() or 1
        # one per core, at most 128 (about 0.3 GB of host memory each)
        self.workers = max(1, int(workers or min(self.cpu_count, 128)))
        ctx = mp.get_context("spawn")
        self.cmd = [ctx.Queue() for _ in range(self.workers)]
        self.res = ctx.Queue()
        self.barrier = ctx.Barrier(self.workers)
        saved = {k: os.environ.get(k) for k in _SINGLE_THREAD_ENV}
        for k in _SINGLE_THREAD_ENV:
            os.environ[k] = "1"
        try:
            self.procs = [ctx.Process(target=_oracle_worker, args=(i, seqs_per_worker, self.cmd[i], self.res,
                                                                   self.barrier), daemon=True)
                          for i in range(self.workers)]
            for pr in self.procs:
                pr.start()
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        for _ in range(self.workers):
            self.res.get(timeout=600)
        self.seqs = self.workers * seqs_per_worker

    def run(self, seconds):
        for q in self.cmd:
            q.put(float(seconds))
        out = [self.res.get(timeout=600 + 10 * seconds) for _ in range(self.workers)]
        return sum(o[0] for o in out), max(o[1] for o in out), sum(o[2] for o in out)

    def close(self):
        for q in self.cmd:
            q.put(None)
        for pr in self.procs:
            pr.join(timeout=30)

    def describe(self, passes, seconds):
        return (f"{passes} whole-sequence passes in {seconds:.1f} s by {self.workers} single-threaded oracle "
                f"processes ({self.cpu_count} host cores), {self.seqs} distinct sequences of the 256-sequence "
                f"round's recipe (histories U{{4096..16384}}): 4 dense decode steps, verify+mass, select, "
                f"4 sparse drafts, spec sample over V=151936; fp64 NumPy oracle")


# ---------------------------------------------------------------- arms

def run_reference(args, world, rank):
    if rank != 0:
        return 0
    farm = OracleFarm(args.cpu_workers)
    try:
        per_step = max(1.0, 60.0 / max(args.steps + args.warmup, 1))
        for _ in range(args.warmup):
            farm.run(per_step / 4)
        total_b, total_t, passes = 0.0, 0.0, 0
        for _ in range(args.steps):
            b, t, n = farm.run(per_step)
            total_b += b
            total_t += t
            passes += n
    finally:
        farm.close()
    value = total_b / total_t / 1e9
    desc = farm.describe(passes, total_t)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "qwen3-1.7b-geom 1 layer, 256 seqs x U{4096..16384}, 16/8 heads, d=128, k=4, "
                               "budget 0.05, vocab 151936 (bounded sample per step)",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": farm.workers, "cpu_count": farm.cpu_count,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def selection_tie_sample(w, n=8):
    """The round's selection (from the GPU's fp32 mass) against the oracle's
    selection from its own fp64 verify mass, on n sequences spread over the
    batch: pages chosen by one side only are cutoff ties when the oracle's
    mass of the page lies within 1e-6 * (G * T) of the cutoff, mismatches
    otherwise."""
    import oracle
    from workloads import bf16_to_bits
    seqs = sorted({int(x) for x in np.linspace(0, w.S - 1, n)})
    idx = torch.as_tensor(seqs, device=w.kv.block_table.device, dtype=torch.long)
    bt = w.kv.block_table[idx].long()
    uniq, inv = torch.unique(bt[bt >= 0], return_inverse=True)
    bt_c = torch.full_like(bt, -1)
    bt_c[bt >= 0] = inv
    kp, vp = bf16_to_bits(w.kv.k_pool[uniq]), bf16_to_bits(w.kv.v_pool[uniq])
    L = w.kv.hist_lens.cpu().numpy().astype(np.int64)[seqs]
    _, mref = oracle.verify_attn(bf16_to_bits(w.q_verify[idx]), kp, vp, bt_c.cpu().numpy(), L, 1.0,
                                 mass_pages=w.mass_stride)
    sel_lens = w.sel_lens.cpu().numpy()[seqs]
    ref_sel, ref_cnt = oracle.select_draft_pages(mref, sel_lens, w.budget, 1, 4, b_max=w.b_max)
    sel, cnt = w.sel[idx].cpu().numpy(), w.cnt[idx].cpu().numpy()
    tol = 1e-6 * (w.Hq // w.Hkv) * w.k
    ties = mismatched = 0
    for i in range(len(seqs)):
        P = ceil_div(int(sel_lens[i]), 16)
        mand = set(range(min(1, P))) | set(range(max(P - 4, 0), P))
        for h in range(w.Hkv):
            g = set(sel[i, h, : cnt[i, h]].tolist())
            r = set(ref_sel[i, h, : ref_cnt[i, h]].tolist())
            if g == r:
                continue
            rest = sorted(r - mand, key=lambda pg: (-mref[i, h, pg], pg))
            cut = mref[i, h, rest[-1]] if rest else 0.0
            for pg in g - r:
                ties, mismatched = (ties + 1, mismatched) if mref[i, h, pg] >= cut - tol else (ties, mismatched + 1)
            for pg in r - g:
                if mref[i, h, pg] > cut + tol:
                    mismatched += 1
    return {"pairs": len(seqs) * w.Hkv, "tie_swaps": ties, "mismatched_pages": mismatched,
            "window": "1e-6 x G x T of the oracle's fp64 mass"}


def sampler_vs_oracle(p, q, x, out, nacc, seed, n=64):
    """The GPU sampler's decisions against the oracle's on n sequences spread
    over the batch (the same fp32 logits and Philox uniforms): a differing
    accepted count is a ratio tie when |u - p/q| <= 1e-6 at the first position
    where the two differ; a differing token is an inverse-CDF tie when it is
    still a valid answer for the oracle's fp64 CDF within 1e-6 * Z; anything
    else is a mismatch."""
    import oracle
    N, k1, _ = p.shape
    k = k1 - 1
    seqs = np.unique(np.linspace(0, N - 1, n).astype(np.int64))
    idx = torch.as_tensor(seqs, device=p.device)
    P, Q, X = p[idx].cpu().numpy(), q[idx].cpu().numpy(), x[idx].cpu().numpy()
    og, ng = out[idx].cpu().numpy(), nacc[idx].cpu().numpy()
    out_o, nacc_o, det = oracle.spec_sample(P, Q, X, seed, 0, seq_ids=seqs)
    ratio = cdf = bad = 0
    for i in range(len(seqs)):
        if ng[i] != nacc_o[i]:
            j = int(min(ng[i], nacc_o[i]))
            if abs(det["u_accept"][i, j] - det["ratio"][i, j]) <= 1e-6:
                ratio += 1
            else:
                bad += 1
            continue
        if np.array_equal(og[i], out_o[i]):
            continue
        a = int(nacc_o[i])
        y = int(og[i, a])
        if a < k:
            row = oracle.residual_row(P[i, a], Q[i, a])
        else:
            e = np.exp(P[i, k].astype(np.float64) - P[i, k].max())
            row = e / e.sum()
        C = np.cumsum(row)
        Z, t = C[-1], det["u_resample"][i] * C[-1]
        ok = 0 <= y < len(row) and row[y] > 0 and (C[y - 1] if y > 0 else 0.0) <= t + 1e-6 * Z \
            and C[y] >= t - 1e-6 * Z and np.array_equal(og[i, :a], out_o[i, :a])
        cdf, bad = (cdf + 1, bad) if ok else (cdf, bad + 1)
    return {"sequences": int(len(seqs)), "ratio_ties": ratio, "cdf_ties": cdf, "mismatches": bad}


def run_tiny(args):
    """The 4-sequence x 2048-token case (one layer, 16 q / 8 KV heads, k = 4,
    budget 0.10; sampler 4 x k = 4 x V = 4096): latency per call of every
    step, through the same binding calls as the round (L2-resident: a latency
    case, not a bandwidth one)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    w = Workload(dev, attn_cfg=ATTN_TINY, sampler_cfg=SAMPLER_TINY)
    r = Runner(w)
    for _ in range(max(3, args.warmup)):
        r.step()
    torch.cuda.synchronize()
    n = 50
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(r.n_events())] for _ in range(n)]
    for i in range(n):
        r.step(evs[i])
    torch.cuda.synchronize()
    r.ws.check()
    r.sws.check()
    k = w.k
    d = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(r.n_events() - 1)] for e in evs]) * 1e3
    return {"workload": "4 seqs x 2048 tokens, 16 q / 8 kv heads, k=4, budget 0.10; sampler 4 x k=4 x V=4096",
            "dense_decode_us": float(d[:, 0:k].mean()), "verify_mass_us": float(d[:, k].mean()),
            "select_us": float(d[:, k + 1].mean()), "sparse_draft_us": float(d[:, k + 2: 2 * k + 2].mean()),
            "spec_sample_us": float(d[:, 2 * k + 2].mean()), "calls_timed": n}


def run_extras(args):
    """Compact results of the other workloads for the default bench line (each
    leg at up to 10 timed steps; a leg that fails reports its error instead)."""
    sub = argparse.Namespace(**vars(args))
    sub.steps, sub.warmup, sub.seqs, sub.layers, sub.all_16k = min(args.steps, 10), 3, None, None, False
    out = {}

    def sweep_c(r):
        return {"dense_gbs": r["dense"]["gbs"], "verify_T8_G4_ms": r["verify_T8_G4"]["ms"],
                "verify_T8_G4_gbs": r["verify_T8_G4"]["gbs"],
                "budgets": {b: {"draft_kv_gb_per_step": v["draft_kv_gb_per_step"], "draft_gbs": v["draft_gbs"],
                                "draft_ms_per_step": v["draft_ms_per_step"],
                                "draft_verify_tokens_per_s": v["draft_verify_tokens_per_s"]}
                            for b, v in r["budgets"].items()}}

    def sampler_c(r):
        return {sg: {"gbs": v["gbs"], "ms": v["ms"], "recipe": v["recipe"], "mean_accepted": v["mean_accepted"],
                     "per_position_acceptance": float(np.mean(v["per_position_acceptance"])),
                     "sampled_tokens_per_s": v["sampled_tokens_per_s"],
                     "gpu_ratio_within_1e-6": v["gpu_ratio_within_1e-6"],
                     "gpu_cdf_target_within_1e-6_Z": v["gpu_cdf_target_within_1e-6_Z"],
                     "vs_oracle": v["vs_oracle"], "sequential_ms": v["sequential"]["ms"]}
                for sg, v in r["sigma"].items()}

    def layers_c(r):
        return {k_: r[k_] for k_ in ("value", "round_ms", "dense_4_steps_ms", "round_vs_4_dense_time",
                                     "emitted_tokens_speedup", "s3r_emitted_tokens_per_s",
                                     "dense_emitted_tokens_per_s", "mean_accepted", "round_gb")}

    legs = (("tiny_4seq_2048_latency", run_tiny, lambda r: {k_: v for k_, v in r.items() if k_ != "workload"}),
            ("qwen3_8b_128seq_sweep", run_sweep, sweep_c),
            ("sampler_2048seq_k8", run_sampler, sampler_c),
            ("layers_28_closed_round", run_layers, layers_c))
    for name, fn, compact in legs:
        try:
            out[name] = compact(fn(sub))
        except Exception as e:  # one leg's failure must not cost the contract line
            out[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def run_s3r(args, world, rank, local):
    import speculative_decode_attention_paged_b300 as s3r
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    # the oracle's processes start before the first GPU call (spawned: no CUDA state is inherited)
    farm = OracleFarm(args.cpu_workers) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None
    s3r.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = Workload(dev, num_seqs=args.seqs)
    r = Runner(w)
    r.step()
    torch.cuda.synchronize()
    w.finalize_bytes()
    r.ws.check()
    r.sws.check()

    for _ in range(args.warmup):
        r.step()
    torch.cuda.synchronize()

    K = args.steps
    nev = r.n_events()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(K)]
    props = torch.cuda.get_device_properties(dev)
    uuid = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) is not None else None
    clocks = ClockSampler(uuid) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.5)
    barrier(world)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for i in range(K):
        r.step(evs[i])
    t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clock_info = clocks.stop() if clocks else None
    total_ms = t_start.elapsed_time(t_end)
    total_ms_max = allreduce_max(total_ms, world)
    r.ws.check()
    r.sws.check()

    # per-phase durations (ms), averaged over the K steps
    k = w.k
    ph = {"dense": [], "verify": [], "select": [], "draft": [], "sample": []}
    dense_launch_ms = []
    for e in evs:
        d = [e[j].elapsed_time(e[j + 1]) for j in range(nev - 1)]
        ph["dense"].append(sum(d[0:k]))
        dense_launch_ms.extend(d[0:k])
        ph["verify"].append(d[k])
        ph["select"].append(d[k + 1])
        ph["draft"].append(sum(d[k + 2: 2 * k + 2]))
        ph["sample"].append(d[2 * k + 2])
    pm = {key: statistics.mean(v) for key, v in ph.items()}

    ms_per_step = total_ms_max / K
    value = aggregate_gbs(w.step_bytes, ms_per_step, world)
    b = w.bytes
    dense_avg_bytes = sum(b["dense"]) / k
    dense_launch = statistics.mean(dense_launch_ms)
    achieved = dense_avg_bytes / (dense_launch * 1e-3) / 1e9
    peaks = measured_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    nacc = w.n_acc.cpu().numpy()
    mean_emitted = float((nacc + 1).mean())
    t_round = (pm["verify"] + pm["select"] + pm["draft"]) * 1e-3
    dv_tokens = w.S * k / t_round
    dense_tokens = w.S * k / (pm["dense"] * 1e-3)
    eff_tokens = w.S * mean_emitted / (t_round + pm["sample"] * 1e-3)

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    phases = {
        "dense_x%d" % k: {"ms": pm["dense"], "gb": sum(b["dense"]) / 1e9, "gbs": gbs(sum(b["dense"]), pm["dense"])},
        "verify": {"ms": pm["verify"], "gb": b["verify"] / 1e9, "gbs": gbs(b["verify"], pm["verify"])},
        "select": {"ms": pm["select"], "gb": b["select"] / 1e9, "gbs": gbs(b["select"], pm["select"])},
        "draft_x%d" % k: {"ms": pm["draft"], "gb": sum(b["draft"]) / 1e9, "gbs": gbs(sum(b["draft"]), pm["draft"])},
        "spec_sample": {"ms": pm["sample"], "gb": b["sample"] / 1e9, "gbs": gbs(b["sample"], pm["sample"])},
    }

    # ---- end to end: host (pinned) inputs -> device -> C-ABI calls -> host results
    e2e = run_e2e(w, r, max(4, min(K, 10)), world)

    # ---- tie accounting of the round (untimed): the sampler's own counters and
    # the selection against the oracle's fp64 mass on sampled sequences
    ties = torch.zeros((2,), dtype=torch.int32, device=dev)
    s3r.s3r_spec_sample(w.spec.p_logits, w.spec.q_logits, w.spec.draft_tokens, w.scfg.philox_seed, 0,
                        w.out_tokens, w.n_acc, r.sws, tie_count=ties)
    r.sws.check()
    tie_report = {
        # decisions inside the tie windows, counted by the sampler itself over all
        # sequences: an upper bound on what rounding could flip (a pick of a token
        # whose mass is below 2e-6 of the row always counts)
        "sampler_gpu_counters": {"ratio_within_1e-6": int(ties[0]), "cdf_target_within_1e-6_Z": int(ties[1]),
                                 "sequences": w.N},
        "sampler_vs_oracle": sampler_vs_oracle(w.spec.p_logits, w.spec.q_logits, w.spec.draft_tokens, w.out_tokens,
                                               w.n_acc, w.scfg.philox_seed) if rank == 0 else None,
        "selection": selection_tie_sample(w) if rank == 0 else None}
    round_ms = pm["verify"] + pm["select"] + pm["draft"] + pm["sample"]
    round_bytes = b["verify"] + b["select"] + sum(b["draft"]) + b["sample"]
    extras = run_extras(args) if (rank == 0 and world == 1 and not args.no_extra) else None

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"qwen3-1.7b-geom 1 layer: {w.S} seqs x U{{4096..16384}}, 16 q / 8 kv heads, d=128, "
                               "16-token bf16 pages (permuted pool), k=4, budget 0.05; sampler 256 x k=4 x "
                               "V=151936 fp32, sigma=1.0",
                   "step": "4 dense decode + verify(page mass) + select + 4 sparse drafts + spec sample",
                   "l2": "inputs larger than L2 (step reads %.1f GB vs 126 MB L2)" % (w.step_bytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "1 gpu"},
        "kv_pct_of_8tbs": 100.0 * value / NOMINAL_HBM_GBS,
        "pct_of_measured_hbm": 100.0 * value / peak,
        "draft_verify_attn_tokens_per_s": dv_tokens * world,
        "dense_decode_tokens_per_s": dense_tokens * world,
        "effective_tokens_per_s": eff_tokens * world,
        "mean_accepted_plus_one": mean_emitted,
        "round_vs_dense_speedup": pm["dense"] / round_ms,
        "s3r_round_gbs": gbs(round_bytes, round_ms),
        "s3r_round_pct_of_8tbs": 100.0 * gbs(round_bytes, round_ms) / NOMINAL_HBM_GBS,
        "emitted_tokens_speedup": (w.S * mean_emitted / round_ms) / (w.S * k / pm["dense"]),
        "ties": tie_report,
        "phases": phases,
        "roofline": {"kernel": "attn_partial_kernel (dense decode)",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "bytes_per_launch": dense_avg_bytes, "launch_ms": dense_launch,
                     "traffic": (DENSE_TRAFFIC_RATIO * dense_avg_bytes) if DENSE_TRAFFIC_RATIO else None},
        "gpu_launches": r.launches_per_step * K,
        "e2e": e2e,
        "clocks": clock_info,
    }
    if extras is not None:
        line["other_workloads"] = extras
    if farm is not None:
        try:
            cb, ct, passes = farm.run(args.cpu_seconds)
        finally:
            farm.close()
        line["cpu_baseline"] = {"value": cb / ct / 1e9, "unit": UNIT, "cores": farm.workers,
                                "cpu_count": farm.cpu_count, "kind": "oracle", "sample": farm.describe(passes, ct)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# Roofline denominators when MEASURED_PEAKS.json is absent: one earlier
# measurement of a B300 (copy bandwidth; dense bf16 GEMM held for seconds).
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1400.0


def measured_peaks(root=None):
    """The measured peaks file at the repo root as a dict ({} if absent)."""
    try:
        with open(os.path.join(root or ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


# (dram__bytes_read.sum + dram__bytes_write.sum) / algorithmic bytes of one
# dense-decode launch of attn_partial_kernel, from an ncu capture of the
# 32-sequence case of this workload; traffic grows with the KV streamed, so the
# full launch's traffic is this ratio times its algorithmic bytes.  None when
# the kernel has changed since the capture.
DENSE_TRAFFIC_RATIO = (1348030976 + 2870784) / 1346994176


def _mirror(w):
    """A second set of the step's per-step buffers (inputs and outputs) over
    the same KV pool, so one step's inputs can be uploaded while another step
    runs."""
    import copy
    from workloads import SpecInputs
    m = copy.copy(w)
    m.q_verify = torch.empty_like(w.q_verify)
    m.q_dense = [torch.empty_like(t) for t in w.q_dense]
    m.q_draft = [torch.empty_like(t) for t in w.q_draft]
    m.spec = SpecInputs(torch.empty_like(w.spec.p_logits), torch.empty_like(w.spec.q_logits),
                        torch.empty_like(w.spec.draft_tokens))
    m.out_dense = [torch.empty_like(t) for t in w.out_dense]
    m.out_verify = torch.empty_like(w.out_verify)
    m.out_draft = [torch.empty_like(t) for t in w.out_draft]
    m.mass = torch.empty_like(w.mass)
    m.sel = torch.empty_like(w.sel)
    m.cnt = torch.empty_like(w.cnt)
    m.out_tokens = torch.empty_like(w.out_tokens)
    m.n_acc = torch.empty_like(w.n_acc)
    return m


def _step_io(w):
    ins = [w.q_verify] + w.q_dense + w.q_draft + [w.spec.p_logits, w.spec.q_logits, w.spec.draft_tokens]
    outs = w.out_dense + [w.out_verify, w.mass, w.sel, w.cnt] + w.out_draft + [w.out_tokens, w.n_acc]
    return ins, outs


def run_e2e(w, r, steps, world):
    """Same step through the public API with host buffers: every step's inputs
    are copied from pinned host memory and every result copied back inside the
    timed region.  Two buffer sets alternate: while step i runs on one, the
    inputs of step i + 1 upload into the other (a copy stream per direction),
    and a set is refilled only after its step ran and its results were read."""
    ins0, outs0 = _step_io(w)
    h_in = [t.cpu().pin_memory() for t in ins0]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs0]
    h2d = sum(t.numel() * t.element_size() for t in ins0)
    d2h = sum(t.numel() * t.element_size() for t in outs0)
    wb = _mirror(w)
    rb = Runner(wb)
    sets = [(r, _step_io(w)), (rb, _step_io(wb))]
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()

    def pipeline(n):
        computed = [None, None]      # per set: event after its step ran
        read = [None, None]          # per set: event after its results were copied back
        ready = [None, None]         # per set: event after its inputs arrived

        def upload(i):
            b = i % 2
            with torch.cuda.stream(up):
                for e in (computed[b], read[b]):
                    if e is not None:
                        up.wait_event(e)
                for d, h in zip(sets[b][1][0], h_in):
                    d.copy_(h, non_blocking=True)
                ready[b] = torch.cuda.Event()
                ready[b].record(up)

        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            comp.wait_event(ready[b])
            if read[b] is not None:
                comp.wait_event(read[b])
            sets[b][0].step()
            computed[b] = torch.cuda.Event()
            computed[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                for h, d in zip(h_out, sets[b][1][1]):
                    h.copy_(d, non_blocking=True)
                read[b] = torch.cuda.Event()
                read[b].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)

    pipeline(2)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b_ev = torch.cuda.Event(enable_timing=True)
    a.record()
    up.wait_stream(comp)
    down.wait_stream(comp)
    pipeline(steps)
    b_ev.record()
    torch.cuda.synchronize()
    ms = allreduce_max(a.elapsed_time(b_ev), world) / steps
    for o0, o1 in zip(outs0, _step_io(wb)[1]):
        if not torch.equal(o0, o1):
            raise RuntimeError("the two buffer sets computed different results")
    return {"value": world * w.step_bytes / (ms * 1e-3) / 1e9, "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "buffer_sets": 2}


# ---------------------------------------------------------------- extra workloads (one JSON line each)

def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _visible_draft_tokens(sel, cnt, sel_lens, j):
    """Tokens all (sequence, KV head) pairs of draft step j read."""
    sel = sel.cpu().numpy().astype(np.int64)
    cnt = cnt.cpu().numpy()
    L = sel_lens.cpu().numpy().astype(np.int64)
    total = 0
    S, H, _ = sel.shape
    for s in range(S):
        for h in range(H):
            pg = sel[s, h, : cnt[s, h]]
            total += int(np.minimum(pg * 16 + 16, L[s]).sum() - np.minimum(pg * 16, L[s]).sum())
    return total + S * H * (j + 1)


def _timed(fn, steps, warmup):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = _events(2)
    a.record()
    for _ in range(steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _clock_sampler():
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    uuid = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) is not None else None
    c = ClockSampler(uuid)
    c.start()
    time.sleep(0.3)
    return c


def run_sweep(args):
    """Qwen3-8B attention geometry, one layer: 128 sequences x U{8192..24576},
    32 q / 8 KV heads, k = T = 8 (32 query rows per KV head in verify); a dense
    decode step, verify with page mass, then per budget in {0.05, 0.10, 0.25,
    0.50}: select + 8 sparse draft steps."""
    import speculative_decode_attention_paged_b300 as s3r
    dev = torch.device("cuda", torch.cuda.current_device())
    c = ATTN_QWEN3_8B_128SEQ
    S = args.seqs or c.num_seqs
    kv = make_paged_kv(S, c.q_heads, c.kv_heads, 2 * c.k, seed=c.seed, device=dev,
                       hist_min=c.hist_min, hist_max=c.hist_max)
    k, Hq, Hkv = c.k, c.q_heads, c.kv_heads
    desc = s3r.PagedKVDesc(kv.k_pool, kv.v_pool, kv.block_table, Hq)
    ws = s3r.Workspace(s3r.s3r_attn_workspace_size(desc, k), device=dev)
    L = kv.hist_lens
    qv = make_queries(kv, 3000, rows=k)
    qd = [make_queries(kv, 3100 + j) for j in range(k)]
    out_v = torch.empty(qv.shape, dtype=torch.float32, device=dev)
    out_d = torch.empty(qd[0].shape, dtype=torch.float32, device=dev)
    mass = torch.empty((S, Hkv, kv.max_pages), dtype=torch.float32, device=dev)
    sel_lens = (L + k).to(torch.int32)
    clocks = _clock_sampler()
    Lsum = float(L.double().sum())
    dense_bytes = (Lsum + S) * Hkv * KV_TOKEN_BYTES_PER_HEAD + S * Hq * 128 * 6
    ctx = (L + 1).to(torch.int32)
    t_dense = _timed(lambda: s3r.s3r_dense_decode_attn(desc, ctx, qd[0], out_d, 1.0, ws), args.steps, args.warmup)
    verify_bytes = (Lsum + S * k) * Hkv * KV_TOKEN_BYTES_PER_HEAD + S * k * Hq * 128 * 6 + S * Hkv * kv.max_pages * 4
    t_verify = _timed(lambda: s3r.s3r_verify_attn(desc, L, qv, out_v, 1.0, ws, page_mass=mass), args.steps,
                      args.warmup)
    budgets = {}
    total_b, total_t = dense_bytes + verify_bytes, t_dense + t_verify
    for budget in c.budgets:
        b_max = selection_budget_pages(kv.max_pages, budget)
        sel = torch.empty((S, Hkv, b_max), dtype=torch.int32, device=dev)
        cnt = torch.empty((S, Hkv), dtype=torch.int32, device=dev)
        t_sel = _timed(lambda: s3r.s3r_select_draft_pages(mass, sel_lens, budget, sel, cnt, ws), args.steps,
                       args.warmup)
        ws.check()
        tok = [_visible_draft_tokens(sel, cnt, sel_lens, j) for j in range(k)]
        dbytes = [t * KV_TOKEN_BYTES_PER_HEAD + S * Hq * 128 * 6 + S * Hkv * (b_max + 1) * 4 for t in tok]

        def drafts():
            for j in range(k):
                s3r.s3r_sparse_draft_attn(desc, sel_lens, j, sel, cnt, qd[j], out_d, 1.0, ws)

        t_d = _timed(drafts, max(1, args.steps // 2), args.warmup)
        budgets[str(budget)] = {"draft_kv_gb_per_step": tok[0] * KV_TOKEN_BYTES_PER_HEAD / 1e9,
                                "draft_ms_per_step": t_d / k, "draft_gbs": sum(dbytes) / (t_d * 1e-3) / 1e9,
                                "select_ms": t_sel,
                                "round_ms": t_d + t_verify + t_sel,
                                "draft_verify_tokens_per_s": S * k / ((t_d + t_verify + t_sel) * 1e-3)}
        total_b += sum(dbytes)
        total_t += t_d
    ws.check()
    clock_info = clocks.stop()
    return {"workload": f"qwen3-8b-geom 1 layer: {S} seqs x U{{8192..24576}}, 32 q / 8 kv heads, d=128, k=T=8",
            "metric": METRIC, "value": total_b / (total_t * 1e-3) / 1e9, "unit": UNIT,
            "dense": {"ms": t_dense, "gb": dense_bytes / 1e9, "gbs": dense_bytes / (t_dense * 1e-3) / 1e9},
            "verify_T8_G4": {"ms": t_verify, "gb": verify_bytes / 1e9, "gbs": verify_bytes / (t_verify * 1e-3) / 1e9},
            "budgets": budgets, "clocks": clock_info}


def run_sampler(args):
    """Exact speculative sampling at rollout scale: 2048 sequences (256 prompts
    x 8 responses) x k = 8 over V = 151936, sigma in {0.3, 1.0} (the recipe)
    and {0.12, 0.5} (the levels that give the ~95% and ~80% per-position
    acceptance the workload aims for).  Per sigma: the parallel and the
    sequential sampler, the acceptance and the sampler's tie counts."""
    import speculative_decode_attention_paged_b300 as s3r
    dev = torch.device("cuda", torch.cuda.current_device())
    sc = SAMPLER_ROLLOUT_2048SEQ
    N = args.seqs or sc.num_seqs
    res = {}
    for sigma in tuple(sc.q_sigmas) + tuple(ROLLOUT_ACCEPTANCE_MATCHED_SIGMAS):
        inp = make_spec_inputs(N, sc.k, sc.vocab, sc.p_sigma, sigma, sc.seed, device=dev)
        ws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(N, sc.k), device=dev)
        out = torch.empty((N, sc.k + 1), dtype=torch.int32, device=dev)
        nacc = torch.empty((N,), dtype=torch.int32, device=dev)
        ties = torch.zeros((2,), dtype=torch.int32, device=dev)
        clocks = _clock_sampler()
        t = _timed(lambda: s3r.s3r_spec_sample(inp.p_logits, inp.q_logits, inp.draft_tokens, sc.philox_seed, 0,
                                               out, nacc, ws), args.steps, args.warmup)
        clock_info = clocks.stop()
        s3r.s3r_spec_sample(inp.p_logits, inp.q_logits, inp.draft_tokens, sc.philox_seed, 0, out, nacc, ws,
                            tie_count=ties)
        ws.check()
        a = nacc.cpu().numpy()
        nbytes = N * (2 * sc.k + 1) * sc.vocab * 4 + N * (2 * sc.k + 2) * 4
        reached = np.array([(a >= i).sum() for i in range(sc.k)])
        accepted = np.array([(a > i).sum() for i in range(sc.k)])
        # the sequential sampler on the same inputs: rows up to each first rejection only
        out_s = torch.empty_like(out)
        nacc_s = torch.empty_like(nacc)
        t_seq = _timed(lambda: s3r.s3r_spec_sample_sequential(inp.p_logits, inp.q_logits, inp.draft_tokens,
                                                              sc.philox_seed, 0, out_s, nacc_s, ws),
                       args.steps, args.warmup)
        ws.check()
        if not (torch.equal(out_s, out) and torch.equal(nacc_s, nacc)):
            raise RuntimeError("sequential sampler differs from the parallel sampler")
        rows_read = int(np.where(a < sc.k, 2 * (a + 1), 2 * sc.k + 1).sum())
        seq_bytes = rows_read * sc.vocab * 4
        sequential = {"ms": t_seq, "rows_read": rows_read, "rows_total": N * (2 * sc.k + 1),
                      "gb": seq_bytes / 1e9, "gbs": seq_bytes / (t_seq * 1e-3) / 1e9,
                      "speedup_vs_parallel": t / t_seq}
        res[str(sigma)] = {"ms": t, "gb": nbytes / 1e9, "gbs": nbytes / (t * 1e-3) / 1e9,
                           "recipe": "matched acceptance" if sigma in ROLLOUT_ACCEPTANCE_MATCHED_SIGMAS else "as written",
                           "gpu_ratio_within_1e-6": int(ties[0]), "gpu_cdf_target_within_1e-6_Z": int(ties[1]),
                           "vs_oracle": sampler_vs_oracle(inp.p_logits, inp.q_logits, inp.draft_tokens, out, nacc,
                                                          sc.philox_seed, n=32),
                           "sequential": sequential,
                           "mean_accepted": float(a.mean()), "mean_emitted": float((a + 1).mean()),
                           "per_position_acceptance": [float(x) for x in accepted / np.maximum(reached, 1)],
                           "accepted_histogram": np.bincount(a, minlength=sc.k + 1).tolist(),
                           "sampled_tokens_per_s": float((a + 1).sum() / (t * 1e-3)), "clocks": clock_info}
        del inp
        torch.cuda.empty_cache()
    vals = [r["gbs"] for r in res.values()]
    # draft-token sampling: one token per sequence from softmax(q) of one draft step
    g = torch.Generator(device=dev)
    g.manual_seed(sc.seed + 7)
    logits = torch.randn((N, sc.vocab), generator=g, device=dev) * sc.p_sigma
    dws = s3r.Workspace(s3r.s3r_sample_draft_workspace_size(N), device=dev)
    dtok = torch.empty((N,), dtype=torch.int32, device=dev)
    t = _timed(lambda: s3r.s3r_sample_draft_tokens(logits, sc.philox_seed, 0, 0, dtok, dws), args.steps, args.warmup)
    dws.check()
    dbytes = N * sc.vocab * 4 + N * 4
    draft = {"ms": t, "gb": dbytes / 1e9, "gbs": dbytes / (t * 1e-3) / 1e9, "tokens_per_s": N / (t * 1e-3)}
    return {"workload": f"spec sample: {N} seqs x k={sc.k} x V={sc.vocab} fp32, p~N(0,3^2), q=p+N(0,s^2)",
            "metric": METRIC, "value": float(np.mean(vals)), "unit": UNIT, "sigma": res,
            "draft_token_sampling": draft}


class LayersRound:
    """Closed multi-layer S³R round: all 28 layers of the Qwen3-1.7B attention
    geometry, 32 sequences with histories U{4096..16384} in a pool sized for
    16K tokens per sequence (~60 GB), per-layer random queries and K/V rows,
    budget 0.05, k = 4, synthetic logits over V = 151936 (p ~ N(0, 3^2),
    q = p + N(0, 1)).  One round (s3r_round), captured in one CUDA graph:
      4 draft steps: every layer writes its draft row at L + j and runs sparse
        draft attention over the previous round's pages, in one launch; the
        draft token is sampled from q_j in place;
      verify: every layer writes the k + 1 dense rows of [pending token,
        drafts] at L .. L + k (s3r_kv_append) and verifies them with page
        mass;
      exact speculative sampling of the 32 blocks, the length commit
        L' = L + n_acc + 1, and every layer's pages for the next round over L'.
    Compared with 4 dense decode steps (dense_steps, a second graph): every
    layer writes the step's row and runs dense attention in one launch, then a
    token is sampled from p_j.
    Both restart from the same L at every replay (the appends rewrite the same
    slots), so every replay is the same round.  The GPU parity test of this
    workload replays the same graph and checks it against the oracle."""

    def __init__(self, dev, n_layers=None, num_seqs=None, all_16k=False):
        import speculative_decode_attention_paged_b300 as s3r
        self.s3r = s3r
        c = ATTN_QWEN3_1P7B_28LAYER
        sc = SAMPLER_ROUND_256SEQ
        self.cfg, self.scfg = c, sc
        S, k, Hq, Hkv = (num_seqs or c.num_seqs), c.k, c.q_heads, c.kv_heads
        self.n_layers = n_layers or c.layers
        self.S, self.k, self.Hq, self.Hkv = S, k, Hq, Hkv
        self.budget, self.V = c.budgets[0], sc.vocab
        self.all_16k = all_16k
        gen = torch.Generator(device="cpu")
        gen.manual_seed(c.seed)
        L = torch.randint(c.hist_min, c.hist_max + 1, (S,), generator=gen).to(torch.int32)
        if all_16k:
            L = torch.full((S,), c.capacity_tokens - 2 * k, dtype=torch.int32)
        self.L_host = L
        rows_gen = torch.Generator(device=dev)
        rows_gen.manual_seed(c.seed + 1)

        def bf16_rows(*shape):
            return (torch.randn(shape, generator=rows_gen, device=dev)).to(torch.bfloat16)

        self.layers = []
        for li in range(self.n_layers):
            kv = make_paged_kv(S, Hq, Hkv, 2 * k, seed=c.seed * 1000 + li, device=dev, hist_lens=L.to(dev),
                               capacity_tokens=c.capacity_tokens)
            desc = s3r.PagedKVDesc(kv.k_pool, kv.v_pool, kv.block_table, Hq)
            b_max = selection_budget_pages(kv.max_pages, self.budget)
            self.layers.append(dict(
                kv=kv, desc=desc,
                qv=make_queries(kv, 5000 + li, rows=k + 1),
                qd=[make_queries(kv, 5100 + 16 * li + j) for j in range(k)],
                draft_kv=[(bf16_rows(S, 1, Hkv, 128), bf16_rows(S, 1, Hkv, 128)) for _ in range(k)],
                block_kv=(bf16_rows(S, k + 1, Hkv, 128), bf16_rows(S, k + 1, Hkv, 128)),
                out_v=torch.empty((S, k + 1, Hq, 128), dtype=torch.float32, device=dev),
                out_d=[torch.empty((S, Hq, 128), dtype=torch.float32, device=dev) for _ in range(k)],
                mass=torch.empty((S, Hkv, kv.max_pages), dtype=torch.float32, device=dev),
                sel=torch.empty((S, Hkv, b_max), dtype=torch.int32, device=dev),
                cnt=torch.empty((S, Hkv), dtype=torch.int32, device=dev),
                sel_next=torch.empty((S, Hkv, b_max), dtype=torch.int32, device=dev),
                cnt_next=torch.empty((S, Hkv), dtype=torch.int32, device=dev)))
        self.max_len = self.layers[0]["kv"].max_pages * 16
        self.spec = make_spec_inputs(S, k, self.V, sc.p_sigma, sc.q_sigmas[0], sc.seed, device=dev)
        self.drafts = torch.empty((S, k), dtype=torch.int32, device=dev)
        self.out_tokens = torch.empty((S, k + 1), dtype=torch.int32, device=dev)
        self.n_acc = torch.empty((S,), dtype=torch.int32, device=dev)
        self.dense_tokens = torch.empty((S, k), dtype=torch.int32, device=dev)
        self.Ld = L.to(dev)
        self.L_next = torch.empty_like(self.Ld)
        self.ctx = [(self.Ld + j + 1).to(torch.int32) for j in range(k)]
        self.ws = s3r.Workspace(s3r.s3r_attn_workspace_size(self.layers[0]["desc"], k + 1), device=dev)
        self.sws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(S, k), device=dev)
        self.dws = s3r.Workspace(s3r.s3r_sample_draft_workspace_size(S), device=dev)
        self.pool_gb = sum(2 * l["kv"].k_pool.numel() * 2 for l in self.layers) / 1e9
        # the first round's pages: a verify of the block at L, selected over L + k (a previous round)
        for l in self.layers:
            s3r.s3r_kv_append(l["desc"], self.Ld, l["block_kv"][0], l["block_kv"][1], self.ws)
            s3r.s3r_verify_attn(l["desc"], self.Ld, l["qv"], l["out_v"], 1.0, self.ws, page_mass=l["mass"])
            s3r.s3r_select_draft_pages(l["mass"], (self.Ld + k).to(torch.int32), self.budget, l["sel"], l["cnt"],
                                       self.ws)

    def s3r_round(self):
        s3r, sc, k = self.s3r, self.scfg, self.k
        for j in range(k):
            for l in self.layers:
                s3r.s3r_sparse_draft_attn(l["desc"], self.Ld, j, l["sel"], l["cnt"], l["qd"][j], l["out_d"][j], 1.0,
                                          self.ws, append=l["draft_kv"][j])
            s3r.s3r_sample_draft_tokens(self.spec.q_logits[:, j], sc.philox_seed, 0, j, self.drafts[:, j], self.dws)
        for l in self.layers:
            # the block's k + 1 rows by their own launch: timed in the round, this
            # beat the fused verify call (12.26 vs 12.34 ms at 28 layers)
            s3r.s3r_kv_append(l["desc"], self.Ld, l["block_kv"][0], l["block_kv"][1], self.ws)
            s3r.s3r_verify_attn(l["desc"], self.Ld, l["qv"], l["out_v"], 1.0, self.ws, page_mass=l["mass"])
        s3r.s3r_spec_sample(self.spec.p_logits, self.spec.q_logits, self.drafts, sc.philox_seed, 0, self.out_tokens,
                            self.n_acc, self.sws)
        s3r.s3r_commit_lengths(self.Ld, self.n_acc, k, self.max_len, self.L_next, self.ws)
        for l in self.layers:
            s3r.s3r_select_draft_pages(l["mass"], self.L_next, self.budget, l["sel_next"], l["cnt_next"], self.ws)

    def dense_steps(self):
        s3r, sc = self.s3r, self.scfg
        for j in range(self.k):
            for l in self.layers:
                s3r.s3r_dense_decode_attn(l["desc"], self.ctx[j], l["qd"][j], l["out_d"][j], 1.0, self.ws,
                                          append=l["draft_kv"][j])
            s3r.s3r_sample_draft_tokens(self.spec.p_logits[:, j], sc.philox_seed, 0, j, self.dense_tokens[:, j],
                                        self.dws)

    def check(self):
        for w in (self.ws, self.sws, self.dws):
            w.check()

    def capture(self, dense=True):
        """CUDA graphs of the round (and of the 4 dense steps); the calls
        enqueue on torch's current stream, here a side stream under capture."""
        g_round = torch.cuda.CUDAGraph()
        g_dense = torch.cuda.CUDAGraph() if dense else None
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g_round, stream=side, capture_error_mode="thread_local"):
                self.s3r_round()
            if dense:
                with torch.cuda.graph(g_dense, stream=side, capture_error_mode="thread_local"):
                    self.dense_steps()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        return g_round, g_dense

    def launches_per_round(self):
        # per layer: k drafts, block append, verify, selection; then k draft-token samplings,
        # the sampler and the length commit
        return self.n_layers * (self.k + 3) + self.k + 1 + 1


def run_layers(args):
    """The closed 28-layer round (LayersRound) against 4 dense decode steps,
    both as CUDA graphs."""
    dev = torch.device("cuda", torch.cuda.current_device())
    lr = LayersRound(dev, n_layers=args.layers, num_seqs=args.seqs, all_16k=args.all_16k)
    S, k, Hq, Hkv, n_layers, V = lr.S, lr.k, lr.Hq, lr.Hkv, lr.n_layers, lr.V
    L, Ld, layers = lr.L_host, lr.Ld, lr.layers
    lr.s3r_round()
    lr.dense_steps()
    torch.cuda.synchronize()
    lr.check()
    g_round, g_dense = lr.capture()
    clocks = _clock_sampler()
    t_round = _timed(g_round.replay, args.steps, args.warmup)
    t_dense = _timed(g_dense.replay, args.steps, args.warmup)
    t_round_eager = _timed(lr.s3r_round, max(2, args.steps // 4), 1)
    clock_info = clocks.stop()
    lr.check()
    a = lr.n_acc.cpu().numpy().astype(np.int64)
    if not np.array_equal(lr.L_next.cpu().numpy(), L.numpy() + a + 1):
        raise RuntimeError("length commit differs from L + n_acc + 1")
    Lsum = float(L.double().sum())
    tok = [sum(_visible_draft_tokens(l["sel"], l["cnt"], Ld, j) for l in layers) for j in range(k)]
    row_bytes = Hkv * KV_TOKEN_BYTES_PER_HEAD                       # K + V of one token, all KV heads
    draft_bytes = sum(t * KV_TOKEN_BYTES_PER_HEAD for t in tok) + k * n_layers * S * Hq * 128 * 6
    verify_bytes = n_layers * ((Lsum + S * (k + 1)) * row_bytes + S * (k + 1) * Hq * 128 * 6
                               + 2 * S * Hkv * layers[0]["kv"].max_pages * 4)
    append_bytes = n_layers * 2 * S * (2 * k + 1) * row_bytes       # rows read and written
    sample_bytes = S * k * V * 4 + S * (2 * k + 1) * V * 4
    dense_bytes = n_layers * sum((Lsum + S * (j + 1)) * row_bytes + S * Hq * 128 * 6 for j in range(k)) \
        + n_layers * 2 * S * k * row_bytes + S * k * V * 4
    round_bytes = draft_bytes + verify_bytes + append_bytes + sample_bytes
    emitted = float((a + 1).sum())
    return {"workload": f"qwen3-1.7b-geom {n_layers} layers: {S} seqs x "
                        + ("all 16K" if args.all_16k else "U{4096..16384}") + f" in a {lr.pool_gb:.1f} GB pool, "
                        f"budget {lr.budget}, k={k}, verify k+1 rows, V={V} (sigma {lr.scfg.q_sigmas[0]}); "
                        "closed round in one CUDA graph",
            "metric": METRIC, "value": round_bytes / (t_round * 1e-3) / 1e9, "unit": UNIT,
            "round_ms": t_round, "round_ms_eager": t_round_eager, "round_gb": round_bytes / 1e9,
            "dense_4_steps_ms": t_dense, "dense_gb": dense_bytes / 1e9,
            "dense_gbs": dense_bytes / (t_dense * 1e-3) / 1e9,
            "round_vs_4_dense_time": t_dense / t_round,
            "mean_accepted": float(a.mean()), "mean_emitted_per_round": emitted / S,
            "s3r_emitted_tokens_per_s": emitted / (t_round * 1e-3),
            "dense_emitted_tokens_per_s": S * k / (t_dense * 1e-3),
            "emitted_tokens_speedup": (emitted / t_round) / (S * k / t_dense),
            "launches_per_round": lr.launches_per_round(),
            "launches_per_dense_4_steps": k * (n_layers + 1), "clocks": clock_info}


def run_speedup(args):
    """Speedup-model calibration on measured kernel times: Qwen3-8B attention
    geometry, one layer, 128 sequences x U{8192..24576}, k = 8, V = 151936.
    A dense step is dense decode attention plus sampling one token from p; an
    S3R round at budget b is k x (sparse draft attention + draft-token
    sampling) + verify with page mass + exact speculative sampling + page
    selection.  Each is timed as a whole (gigabytes per iteration, above L2).
    rho(b) = draft KV bytes per step / dense KV bytes per step (algorithmic);
    cost(b) = T_round(b) / T_dense.  The constant correction is fitted on
    alternate budgets and judged on the others."""
    import speculative_decode_attention_paged_b300 as s3r
    from speculative_decode_attention_paged_b300 import speedup_model as sm
    dev = torch.device("cuda", torch.cuda.current_device())
    c = ATTN_QWEN3_8B_128SEQ
    sc = SAMPLER_ROUND_256SEQ
    S = args.seqs or c.num_seqs
    k, Hq, Hkv = c.k, c.q_heads, c.kv_heads
    kv = make_paged_kv(S, Hq, Hkv, 2 * k, seed=c.seed, device=dev, hist_min=c.hist_min, hist_max=c.hist_max)
    desc = s3r.PagedKVDesc(kv.k_pool, kv.v_pool, kv.block_table, Hq)
    ws = s3r.Workspace(s3r.s3r_attn_workspace_size(desc, k), device=dev)
    L = kv.hist_lens
    qv = make_queries(kv, 3000, rows=k)
    qd = [make_queries(kv, 3100 + j) for j in range(k)]
    out_v = torch.empty(qv.shape, dtype=torch.float32, device=dev)
    out_d = torch.empty(qd[0].shape, dtype=torch.float32, device=dev)
    mass = torch.empty((S, Hkv, kv.max_pages), dtype=torch.float32, device=dev)
    sel_lens = (L + k).to(torch.int32)
    ctx = (L + 1).to(torch.int32)
    spec = make_spec_inputs(S, k, sc.vocab, sc.p_sigma, sc.q_sigmas[0], sc.seed, device=dev)
    drafts = torch.empty((S, k), dtype=torch.int32, device=dev)
    out_t = torch.empty((S, k + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((S,), dtype=torch.int32, device=dev)
    tok1 = torch.empty((S,), dtype=torch.int32, device=dev)
    sws = s3r.Workspace(s3r.s3r_spec_sample_workspace_size(S, k), device=dev)
    dws = s3r.Workspace(s3r.s3r_sample_draft_workspace_size(S), device=dev)
    s3r.s3r_verify_attn(desc, L, qv, out_v, 1.0, ws, page_mass=mass)
    clocks = _clock_sampler()

    def dense_step():
        s3r.s3r_dense_decode_attn(desc, ctx, qd[0], out_d, 1.0, ws)
        s3r.s3r_sample_draft_tokens(spec.p_logits[:, 0], sc.philox_seed, 0, 0, tok1, dws)

    t_dense = _timed(dense_step, args.steps, args.warmup)
    dense_kv = float((L.double() + 1).sum()) * Hkv * KV_TOKEN_BYTES_PER_HEAD
    budgets = (0.02, 0.05, 0.10, 0.15, 0.20, 0.25, 0.35, 0.50, 0.75, 1.00)
    rows = []
    for b in budgets:
        b_max = selection_budget_pages(kv.max_pages, b)
        sel = torch.empty((S, Hkv, b_max), dtype=torch.int32, device=dev)
        cnt = torch.empty((S, Hkv), dtype=torch.int32, device=dev)
        s3r.s3r_select_draft_pages(mass, sel_lens, b, sel, cnt, ws)
        draft_kv = sum(_visible_draft_tokens(sel, cnt, sel_lens, j) for j in range(k)) * KV_TOKEN_BYTES_PER_HEAD / k

        def s3r_round():
            for j in range(k):
                s3r.s3r_sparse_draft_attn(desc, sel_lens, j, sel, cnt, qd[j], out_d, 1.0, ws)
                s3r.s3r_sample_draft_tokens(spec.q_logits[:, j], sc.philox_seed, 0, j, drafts[:, j], dws)
            s3r.s3r_verify_attn(desc, L, qv, out_v, 1.0, ws, page_mass=mass)
            s3r.s3r_spec_sample(spec.p_logits, spec.q_logits, drafts, sc.philox_seed, 0, out_t, nacc, sws)
            s3r.s3r_select_draft_pages(mass, sel_lens, b, sel, cnt, ws)

        t_round = _timed(s3r_round, max(3, args.steps // 2), args.warmup)
        rows.append({"budget": b, "rho": draft_kv / dense_kv, "round_ms": t_round, "cost": t_round / t_dense})
    for w in (ws, sws, dws):
        w.check()
    clock_info = clocks.stop()
    rho = np.array([r["rho"] for r in rows])
    cost = np.array([r["cost"] for r in rows])
    train = np.arange(len(rows)) % 2 == 0
    cal = sm.calibrate(rho, cost, k, train)
    for r in rows:
        r["model_cost_uncorrected"] = float(sm.round_cost(r["rho"], k))
        r["model_cost_corrected"] = float(sm.round_cost(r["rho"], k, cal["c"]))
    a_meas = float(nacc.double().mean().item()) / k
    # the pages' two budget points (per-position acceptance 80.4% at 0.05 and 96.7%
    # at 0.50, draft length 6 on their system): what the measured costs predict
    context = {}
    for b, alpha in ((0.05, 0.804), (0.50, 0.967)):
        i = budgets.index(b)
        a = float(sm.accepted_prefix_fraction(alpha, k))
        context[str(b)] = {"alpha": alpha, "accepted_prefix_fraction": a,
                           "predicted_speedup": float(sm.predict(a, rho[i], k, cal["c"])),
                           "measured_cost_speedup": float(sm.tokens_per_round(a, k) / cost[i])}
    return {"workload": f"speedup-model calibration, qwen3-8b-geom 1 layer: {S} seqs x U{{8192..24576}}, k={k}, "
                        f"V={sc.vocab}, budgets {list(budgets)}",
            "metric": "held-out MAPE of the calibrated speedup model", "value": cal["heldout_mape_corrected"],
            "unit": "%", "higher_is_better": False, "dense_step_ms": t_dense, "points": rows, "calibration": cal,
            "train_budgets": [budgets[i] for i in range(len(budgets)) if train[i]],
            "synthetic_accepted_prefix_fraction": a_meas,
            "speedup_at_synthetic_acceptance": {str(r["budget"]): float(sm.tokens_per_round(a_meas, k) / r["cost"])
                                                for r in rows},
            "context_pages_budget_points": context, "clocks": clock_info}


def _host_link_gbs():
    """Host-to-device copy rate of pinned memory (1 GiB, median of 5), or None
    without a GPU."""
    if not torch.cuda.is_available():
        return None
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    times = []
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return n / (float(np.median(times[1:])) * 1e-3) / 1e9


def run_scheduler(args):
    """KV-aware AIMD scheduler against offload with a fixed limit of 256 and
    recompute, simulated by the library's host scheduler over a KV page pool:
    256 prompts x 8 responses, prompts U{512..2048}, responses log-uniform on
    [512, 16384], k = 4 with per-position acceptance 0.8; Qwen3-8B KV geometry
    (36 layers x 8 KV heads x 128, bf16: 2.36 MB per 16-token page) in 100 GB
    of HBM.  Reported per policy: pages moved per 1000 generated tokens,
    cumulative moved and recomputed pages, rounds, mean concurrency; and a
    modelled generation rate: per round k + 1 passes over the 16.4 GB of bf16
    weights and attention reads of (1 + k * budget) x the running contexts,
    both at the measured HBM copy rate; moved pages at the measured host-link
    rate; recomputed pages at a prefill cost of 2 x 8e9 x 16 FLOP each at the
    measured sustained bf16 rate.  The AIMD constants (not printed by the
    pages) are those that maximised this modelled rate over a small grid."""
    from speculative_decode_attention_paged_b300 import scheduler as sched
    w = make_rollout_requests(256, 8, seed=17, prompt_lo=512, prompt_hi=2048, response_lo=512,
                              response_hi=16384, k=4, alpha=0.8)
    page_tokens, k, budget = 16, 4, 0.05
    kv_token_bytes = 36 * 8 * 128 * 2 * 2
    weight_bytes = 16.4e9
    page_bytes = kv_token_bytes * page_tokens
    pool = int(100e9 // page_bytes)
    peaks = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS)) * 1e9
    tflops = float(peaks.get("bf16_tflops_sustained", FALLBACK_BF16_TFLOPS_SUSTAINED)) * 1e12
    link = _host_link_gbs()
    link_src = "measured" if link is not None else "assumed"
    link = (link or 55.0) * 1e9
    t_page_move = page_bytes / link
    t_page_recompute = 2 * 8e9 * page_tokens / tflops
    common = dict(pool_pages=pool, page_size=page_tokens, block_tokens=k + 1)
    policies = {
        "aimd": dict(policy=sched.AIMD, limit_init=64, limit_min=16, limit_max=1024, add_step=4, mult=0.5,
                     util_low=0.8, util_high=0.98, backlog_max=64),
        "offload_fixed_256": dict(policy=sched.FIXED_OFFLOAD, limit_init=256, limit_min=256, limit_max=256,
                                  add_step=0, mult=1.0, util_low=0.0, util_high=1.0, backlog_max=0),
        "recompute_fixed_256": dict(policy=sched.RECOMPUTE, limit_init=256, limit_min=256, limit_max=256,
                                    add_step=0, mult=1.0, util_low=0.0, util_high=1.0, backlog_max=0),
    }
    res = {}
    for name, pol in policies.items():
        cfg = dict(common, **pol)
        t0 = time.perf_counter()
        tot, trace = sched.run(cfg, w.prompt_lens, w.response_lens, w.emits, max_steps=200_000)
        sim_s = time.perf_counter() - t0
        attn_s = sum(t["ctx_tokens"] for t in trace) * kv_token_bytes * (1 + k * budget) / hbm
        weights_s = tot["steps"] * (k + 1) * weight_bytes / hbm
        move_s = (tot["offloaded"] + tot["restored"]) * t_page_move
        recompute_s = tot["recomputed"] * t_page_recompute
        model_s = attn_s + weights_s + move_s + recompute_s
        res[name] = {"rounds": tot["steps"], "tokens": tot["tokens"], "stalled": tot["stalled"],
                     "pages_moved": tot["offloaded"] + tot["restored"],
                     "pages_moved_per_1000_tokens": 1000.0 * (tot["offloaded"] + tot["restored"]) / tot["tokens"],
                     "pages_recomputed": tot["recomputed"],
                     "moved_plus_recomputed_pages": tot["offloaded"] + tot["restored"] + tot["recomputed"],
                     "preemptions": tot["preemptions"], "mean_concurrency": tot["running_sum"] / tot["steps"],
                     "peak_pages": tot["peak_used"], "final_limit": tot["limit_final"],
                     "model_s": model_s, "model_attention_s": attn_s, "model_weights_s": weights_s,
                     "model_transfer_s": move_s,
                     "model_recompute_s": recompute_s, "model_tokens_per_s": tot["tokens"] / model_s,
                     "simulation_s": sim_s}
    return {"workload": "AIMD KV scheduler simulation: 2048 rollout requests, Qwen3-8B KV geometry, "
                        f"{pool} pages of 16 tokens (100 GB)",
            "metric": "KV cache pages moved per 1000 generated tokens", "value":
                res["aimd"]["pages_moved_per_1000_tokens"], "unit": "pages/1000 tokens",
            "higher_is_better": False, "policies": res,
            "model": {"hbm_gbs": hbm / 1e9, "host_link_gbs": link / 1e9, "host_link": link_src,
                      "bf16_tflops": tflops / 1e12, "page_bytes": page_bytes, "weight_bytes": weight_bytes,
                      "draft_budget": budget, "k": k}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("s3r", "reference"), default="s3r")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-workers", type=int, default=None,
                    help="oracle processes for the CPU baseline (default: one per host core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="leave the other workloads' compact results out of the default line")
    ap.add_argument("--workload", choices=("round", "tiny", "sweep", "sampler", "layers", "scheduler", "speedup"),
                    default="round",
                    help="round (default): the 256-sequence S3R round + dense baseline, with compact results of "
                         "tiny, sweep, sampler and layers; tiny: 4 x 2048 latency per call; sweep: Qwen3-8B "
                         "geometry budget sweep; sampler: 2048 x k=8 sampler; layers: the 28-layer closed round; "
                         "scheduler: the AIMD KV scheduler simulation (host); speedup: the speedup-model "
                         "calibration on measured round and dense-step times")
    ap.add_argument("--layers", type=int, default=None, help="fewer layers for --workload layers")
    ap.add_argument("--all-16k", action="store_true", help="--workload layers with every history at 16K")
    ap.add_argument("--seqs", type=int, default=None,
                    help="fewer sequences than the 256 of the workload (small profiling case only)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "s3r":
        print("note: fewer than 3 warm-up steps; timing rules want >= 3", file=sys.stderr)
    world, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, world, rank)
        if args.workload != "round":
            import speculative_decode_attention_paged_b300 as s3r
            s3r.load_library()
            leg = {"tiny": run_tiny, "sweep": run_sweep, "sampler": run_sampler, "layers": run_layers,
                   "scheduler": run_scheduler, "speedup": run_speedup}[args.workload]
            line = leg(args)
            line.update({"n_gpus": world, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
                         "data": "synthetic", "l2": "inputs larger than L2"})
            if rank == 0:
                print(json.dumps(line), flush=True)
            return 0
        return run_s3r(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
