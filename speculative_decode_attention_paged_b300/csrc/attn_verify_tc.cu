// Dense causal verification of a drafted block on the 5th-generation tensor
// cores (tcgen05 + TMEM), with the page-mass epilogue.
//
// What is computed is the verify form of the paged attention (wispaper.ai,
// "S3R drafts sparsely and verifies densely"; "Dense verification still pays
// the full KV-cache bill"): the T x G query rows of a (sequence, KV head) pair
// attend causally to its whole history, and the attention mass per page feeds
// the next draft's page selection (rit.work, "Как разреженный черновик
// сохраняет ответы плотной модели").
//
// How:
//   * The page stream of all pairs is split into one contiguous share per CTA
//     (persistent grid, one CTA per SM).  A share is walked in tiles of up to
//     8 pages (128 tokens) of one pair.
//   * Scores are computed transposed, S^T = K Q^T (M = 128 tokens, N = 32
//     query rows, K = head_dim), so no MMA row is padding: K tiles land from
//     TMA in the K-major 128-byte-swizzled layout the MMA reads, and so does
//     the query block (one 4-D TMA box per 64-column half).
//   * O^T += V^T P^T (M = 128 = head_dim, K = 16 tokens per MMA): V is read
//     in place as an MN-major operand; P^T is written by the softmax threads
//     as a bf16 high part and a bf16 remainder stacked along N (N = 64: the
//     32 rows twice), so one MMA per page carries ~16 bits of P and the two
//     32-column halves of O^T are added at the end.  (An MMA costs at least
//     ~61 cycles whatever its N up to 128, so fewer, wider MMAs pay.)
//   * Warp roles: warps 0, 10, 11 = TMA producers (3 stages of 8 pages of K
//     and V; a tile's page boxes are spread over the three warps),
//     warp 1 = MMA issuer (one thread) and TMEM owner, warps 2-9 = softmax in
//     two warpgroups of 16 query rows each: a thread owns one token of the
//     tile (one TMEM lane) and its group's 16 rows; row maxima and sums are
//     reduced with butterfly reduce-scatters.  The running
//     max is refreshed only when a tile's max exceeds it by more than 2^8
//     (then O^T is rescaled in TMEM); otherwise p <= 256 and the stale max is
//     exact to use.  Accumulators: S^T double-buffered and O^T in TMEM.
//   * Pairs cut by share boundaries leave (m, l, O) partials; the last CTA to
//     finish a pair merges them.  Page mass is formed as in the CUDA-core
//     kernel: per-(page, row) log-sum-exps, normalised by each row's LSE.
//   * Every wait is bounded; a timeout sets S3R_DEVERR_TIMEOUT and a shared
//     abort flag, every role then leaves its loop, the MMA issuer drains its
//     MMAs and the TMEM is freed.

#include "attn_common.cuh"
#include "attn_paged.cuh"
#include "s3r_device.cuh"

namespace s3r {

namespace {

using namespace attn;

constexpr int kTcTilePages = 8;                        // 128 tokens: the MMA's M
constexpr int kTcStages = 3;
// Tile metadata ring, twice the stage ring: a stage's K half is reloaded as
// soon as the score MMA has read it, while the output MMA and the softmax warps
// of that tile still read its metadata; slot t % 6 is rewritten only for tile
// t + 6, whose K waits for S(t + 3), which the issuer starts only after PV(t).
constexpr int kMetaSlots = 2 * kTcStages;
constexpr int kTcRegion = kTcTilePages * kHalfBytes;   // 16 KiB: one 64-column half of 8 pages
constexpr int kTcStageBytes = 4 * kTcRegion;           // K lo, K hi, V lo, V hi halves
constexpr int kTcRows = 32;                            // MMA N: query rows per KV head
constexpr int kTcQHalf = kTcRows * 128;                // 4 KiB: 32 rows x 64 columns
constexpr int kTcPBytes = 128 * 2 * kTcRows * 2;       // 16 KiB of bf16 P^T: high part | remainder
constexpr int kTcProducers = 3;                        // warps issuing TMA: 0, 10, 11
constexpr int kTcThreads = 384;                        // producers, MMA, 2 x 4 softmax warps
constexpr int kSoftmaxThreads = 256;
constexpr int kWgThreads = 128;
constexpr int kRowsWg = 16;                            // query rows per softmax warpgroup
constexpr int kWgBar0 = 1;                             // named barriers 1, 2: one per warpgroup
constexpr int kAllBar = 3;                             // named barrier 3: both warpgroups
constexpr uint32_t kTmemCols = 128;                    // S^T x 2 (32 columns each), O^T (64)
constexpr uint32_t kColS = 0, kColO = 64;              // O^T: 32 columns from P high, 32 from P low
constexpr float kRescaleSlack = 8.f;

enum : int { kTileFirst = 1, kTileLast = 2, kTileWhole = 4, kTileEnd = 8 };

struct TileMeta {
  int pair, e0, n, np, L, flags;
  long long start;                 // global stream index of the pair's first page
  int lo[kTcTilePages];            // visible token range [lo, hi) of each page;
  int hi[kTcTilePages];            // lo == hi when the page is not loaded
};

struct TcSmem {
  size_t stages, q, p, meta, bars, red_max, red_sum, rowbuf, misc, scratch, prefix, total;
};

__host__ __device__ inline TcSmem tc_smem_layout(int n_chunks) {
  TcSmem s{};
  size_t off = 0;
  s.stages = off;  off += static_cast<size_t>(kTcStages) * kTcStageBytes;
  s.q = off;       off += 2 * kTcQHalf;
  s.p = off;       off += kTcPBytes;
  s.meta = off;    off += kMetaSlots * sizeof(TileMeta);
  s.bars = off;    off += 32 * sizeof(uint64_t);
  s.red_max = off; off += 2 * 2 * 4 * 16 * sizeof(float);   // [group][buffer][quarter][row]
  s.red_sum = off; off += 2 * 4 * 16 * sizeof(float);       // [group][quarter][row]
  s.rowbuf = off;  off += 3 * 32 * sizeof(float);   // row LSE, row max, row 1/sum
  s.misc = off;    off += 4 * sizeof(int);          // TMEM base, abort flag, last-arrival flag
  s.scratch = off; off += 32 * sizeof(int);
  s.prefix = off;  off += static_cast<size_t>(n_chunks + 1) * sizeof(int);
  s.total = off + 1024;                             // alignment slack
  return s;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int* err) {
  for (uint32_t i = 0; i < kMaxSpin; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  report_error(err, S3R_DEVERR_TIMEOUT);
  return false;
}

// Butterfly reduce-scatter of v[VALS] over groups of WIDTH lanes (VALS <=
// WIDTH, both powers of two): afterwards v[0] holds the group's reduction of
// row (lane % WIDTH) / (WIDTH / VALS).  Fixed order: deterministic.
template <int WIDTH, int VALS, bool MAX>
__device__ __forceinline__ void reduce_scatter(float (&v)[VALS], int lane) {
#pragma unroll
  for (int step = 0; (VALS >> (step + 1)) >= 1; ++step) {
    const int off = WIDTH >> (step + 1);
    const int n = VALS >> (step + 1);
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < n; ++j) {
      const float send = up ? v[j] : v[j + n];
      const float keep = up ? v[j + n] : v[j];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[j] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
#pragma unroll
  for (int off = WIDTH / VALS / 2; off >= 1; off >>= 1) {
    const float recv = __shfl_xor_sync(0xffffffffu, v[0], off);
    v[0] = MAX ? fmaxf(v[0], recv) : v[0] + recv;
  }
}

__device__ __forceinline__ int64_t q_row_off(const AttnArgs& a, int s, int h, int r) {
  const int i = r / a.G, g = r - (r / a.G) * a.G;
  return ((static_cast<int64_t>(s) * a.T + i) * a.Hq + h * a.G + g) * kHeadDim;
}

template <bool MASS>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_verify_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap,
                          const __grid_constant__ CUtensorMap qmap, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const TcSmem L = tc_smem_layout(a.n_chunks);
  uint8_t* stages = smem + L.stages;
  uint8_t* qbuf = smem + L.q;
  uint8_t* pbuf = smem + L.p;
  TileMeta* meta = reinterpret_cast<TileMeta*>(smem + L.meta);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  // K and V halves of a stage have their own full / empty barriers: K is free
  // again as soon as the score MMA has read it, V once the output MMA has.
  uint64_t* k_full = bars;                  // [3]
  uint64_t* k_empty = bars + 3;             // [3]
  uint64_t* v_full = bars + 6;              // [3]
  uint64_t* v_empty = bars + 9;             // [3]
  uint64_t* q_full = bars + 12;
  uint64_t* q_empty = bars + 13;
  uint64_t* s_full = bars + 14;             // [2]
  uint64_t* s_free = bars + 16;             // [2]
  uint64_t* p_full = bars + 18;
  uint64_t* o_done = bars + 19;
  uint64_t* drain = bars + 20;
  // Softmax warps learn of tile t's metadata from meta_full[t % 6], not from
  // k_full: K of a stage may be reloaded (k_full moving on) before they look.
  uint64_t* meta_full = bars + 21;          // [kMetaSlots]
  float* red_max = reinterpret_cast<float*>(smem + L.red_max);
  float* red_sum = reinterpret_cast<float*>(smem + L.red_sum);
  float* row_lse = reinterpret_cast<float*>(smem + L.rowbuf);    // [32]
  float* row_max = row_lse + 32;
  float* row_inv = row_lse + 64;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc) + 1;
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + L.misc) + 2;
  int* scratch = reinterpret_cast<int*>(smem + L.scratch);
  int* prefix = reinterpret_cast<int*>(smem + L.prefix);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], 8);
    }
    mbar_init(p_full, 8);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    for (int s = 0; s < kMetaSlots; ++s) mbar_init(&meta_full[s], 1);
    *abort_flag = 0;
    *last_flag = 0;
  }
  // Operand buffers start as zeros, so rows no TMA writes stay finite.
  {
    int4* z = reinterpret_cast<int4*>(smem);
    const int n16 = static_cast<int>((L.meta) / 16);
    for (int i = tid; i < n16; i += kTcThreads) z[i] = make_int4(0, 0, 0, 0);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  // ---- plan: pages per chunk of 32 pairs, then an exclusive scan
  plan_chunk_pages(a, prefix, warp, kTcThreads / 32, lane);
  fence_barrier_init();
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  block_exclusive_scan<kTcThreads>(prefix, a.n_chunks, scratch);

  const uint32_t tmem = *tmem_slot;
  const int64_t N = prefix[a.n_chunks];
  const int tw = gridDim.x;
  const int cta = blockIdx.x;
  const int64_t x0 = share_start(N, cta, tw);
  const int64_t x1 = share_start(N, cta + 1, tw);

  if (warp == 0 || warp >= 10) {
    // =========================== TMA producers: every producer warp walks the same tiles;
    // warp 0 (pid 0) also writes the tile metadata, the expected byte count and the query
    // block; the page boxes of a tile are spread over the producers (a warp pays ~86 cycles
    // per box it issues, so one warp alone cannot keep a 64 KiB stage in flight).
    const int pid = warp == 0 ? 0 : warp - 9;
    int t = 0;
    bool ok = true;
    const uint64_t policy = l2_policy_evict_first();
    if (x0 < x1) {
      // the pair holding x0: chunk by binary search, then a warp scan
      int pair;
      int64_t pstart;
      {
        int lo = 0, hi = a.n_chunks - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (prefix[mid] <= x0) lo = mid; else hi = mid - 1;
        }
        const int c = lo;
        const int pp = c * kPairChunk + lane;
        const int np = pp < a.n_pairs ? pair_geom(a, pp, false).np : 0;
        int incl = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const unsigned ball = __ballot_sync(0xffffffffu, incl > x0 - prefix[c]);
        const int l = __ffs(ball) - 1;
        pair = c * kPairChunk + l;
        pstart = prefix[c] + __shfl_sync(0xffffffffu, incl - np, l);
      }
      PairGeom g = pair_geom(a, pair, false);
      int e = static_cast<int>(x0 - pstart);
      int64_t x = x0;
      int q_uses = 0;
      bool first_of_pair = true;
      int cpair = -1, cbase = 0;           // lane l caches entry cbase + l of pair cpair
      Entry cache{-1, 0, 0, -1};
      while (x < x1) {
        if (e >= g.np) {
          do {
            ++pair;
            g = pair_geom(a, pair, false);
          } while (g.np == 0);
          pstart = x;
          e = 0;
          first_of_pair = true;
        }
        const int64_t rest = x1 - x;
        const int n = min(kTcTilePages, min(g.np - e, rest < kTcTilePages ? static_cast<int>(rest) : kTcTilePages));
        const bool last = (e + n == g.np) || (x + n == x1);
        const bool whole = (pstart >= x0) && (pstart + g.np <= x1);
        if (pair != cpair || e + n > cbase + 32) {   // refill before waiting: the loads overlap the wait
          cpair = pair;
          cbase = e;
          cache = cbase + lane < g.np ? pair_entry(a, pair, g, cbase + lane) : Entry{-1, 0, 0, -1};
        }
        const int st = t % kTcStages;
        const uint32_t ph = static_cast<uint32_t>((t / kTcStages) & 1);
        int okw = 1;
        if (lane == 0) okw = wait_or_abort(&k_empty[st], ph ^ 1u, abort_flag, a.err);
        if (!__shfl_sync(0xffffffffu, okw, 0)) { ok = false; break; }
        const int s = pair / a.Hkv, h = pair - (pair / a.Hkv) * a.Hkv;
        if (first_of_pair && pid == 0) {
          if (lane == 0) okw = wait_or_abort(q_empty, static_cast<uint32_t>(q_uses & 1) ^ 1u, abort_flag, a.err);
          if (!__shfl_sync(0xffffffffu, okw, 0)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2u * 128u * static_cast<uint32_t>(a.R));
            tma_load_4d(qbuf, &qmap, 0, h * a.G, 0, s, q_full);
            tma_load_4d(qbuf + kTcQHalf, &qmap, 64, h * a.G, 0, s, q_full);
          }
        }
        if (first_of_pair) ++q_uses;
        const int src_lane = e - cbase + (lane & (kTcTilePages - 1));
        Entry en;
        en.lp = -1;
        en.lo = __shfl_sync(0xffffffffu, cache.lo, src_lane);
        en.hi = __shfl_sync(0xffffffffu, cache.hi, src_lane);
        en.phys = __shfl_sync(0xffffffffu, cache.phys, src_lane);
        const bool load = lane < n && en.phys >= 0;
        TileMeta& m = meta[t % kMetaSlots];
        if (pid == 0 && lane < kTcTilePages) {
          m.lo[lane] = load ? en.lo : 0;
          m.hi[lane] = load ? en.hi : 0;
        }
        const unsigned loadmask = __ballot_sync(0xffffffffu, load);
        if (pid == 0 && lane == 0) {
          m.pair = pair;
          m.e0 = e;
          m.n = n;
          m.np = g.np;
          m.L = g.L;
          m.flags = (first_of_pair ? kTileFirst : 0) | (last ? kTileLast : 0) | (whole ? kTileWhole : 0);
          m.start = pstart;
        }
        __syncwarp();
        // test of the bounded waits: CTA 0's first tile gets no K and no arrival
        const bool stall_k = a.test_stall != 0 && blockIdx.x == 0 && t == 0;
        if (pid == 0 && lane == 0) {
          mbar_arrive(&meta_full[t % kMetaSlots]);
          if (!stall_k) mbar_arrive_expect_tx(&k_full[st], __popc(loadmask) * 2u * kHalfBytes);
        }
        __syncwarp();
        // appended block rows of this tile's pages, each written by the producer
        // warp that issues the page's boxes, before it issues them
        if (a.app_rows > 0 && (g.L + a.app_rows - 1) / kPage >= e && g.L / kPage < e + n) {
          for (int p = pid; p < n; p += kTcProducers)
            append_rows_in_page<8>(a, s, h, g.L, e + p, __shfl_sync(0xffffffffu, en.phys, p), lane);
        }
        const bool mine = load && (lane % kTcProducers) == pid;
        uint8_t* dst = stages + static_cast<size_t>(st) * kTcStageBytes + lane * kHalfBytes;
        const int y = h * kPage;
        if (mine && !stall_k) {
          tma_load_3d(dst, &kmap, 0, y, en.phys, &k_full[st], policy);
          tma_load_3d(dst + kTcRegion, &kmap, 64, y, en.phys, &k_full[st], policy);
        }
        // V of this tile once the output MMA of the stage's previous tile is done
        if (lane == 0) okw = wait_or_abort(&v_empty[st], ph ^ 1u, abort_flag, a.err);
        if (!__shfl_sync(0xffffffffu, okw, 0)) { ok = false; break; }
        if (pid == 0 && lane == 0) mbar_arrive_expect_tx(&v_full[st], __popc(loadmask) * 2u * kHalfBytes);
        __syncwarp();
        if (mine) {
          tma_load_3d(dst + 2 * kTcRegion, &vmap, 0, y, en.phys, &v_full[st], policy);
          tma_load_3d(dst + 3 * kTcRegion, &vmap, 64, y, en.phys, &v_full[st], policy);
        }
        x += n;
        e += n;
        ++t;
        first_of_pair = false;
      }
    }
    if (ok && pid == 0) {
      // end marker for the MMA and softmax roles
      const int st = t % kTcStages;
      int okw = 1;
      if (lane == 0) okw = wait_or_abort(&k_empty[st], static_cast<uint32_t>((t / kTcStages) & 1) ^ 1u,
                                         abort_flag, a.err);
      if (__shfl_sync(0xffffffffu, okw, 0) && lane == 0) {
        meta[t % kMetaSlots].flags = kTileEnd;
        mbar_arrive(&meta_full[t % kMetaSlots]);
        mbar_arrive(&k_full[st]);
      }
    }
    // Copies this warp may still have in flight (only after an abort).
    if (pid == 0 && lane == 0 && *abort_flag) {
      for (int k = max(0, t - kTcStages); k < t; ++k) {
        mbar_wait_bounded(&k_full[k % kTcStages], static_cast<uint32_t>((k / kTcStages) & 1));
        mbar_wait_bounded(&v_full[k % kTcStages], static_cast<uint32_t>((k / kTcStages) & 1));
      }
    }
  } else if (warp == 1) {
    // =========================== MMA issuer (one thread)
    if (lane == 0) {
      const uint32_t idesc_s = umma_idesc_bf16(128, kTcRows, false, false);
      const uint32_t idesc_o = umma_idesc_bf16(128, 2 * kTcRows, true, true);
      uint32_t q_ph = 0;
      bool ok = true;
      auto issue_s = [&](int t, int flags) -> bool {
        const int st = t % kTcStages, b = t & 1;
        if (flags & kTileFirst) {
          if (!wait_or_abort(q_full, q_ph, abort_flag, a.err)) return false;
          q_ph ^= 1u;
        }
        if (!wait_or_abort(&s_free[b], static_cast<uint32_t>((t >> 1) & 1) ^ 1u, abort_flag, a.err)) return false;
        tc_fence_after_sync();
        const uint64_t ad0 = umma_smem_desc(smem_u32(stages + static_cast<size_t>(st) * kTcStageBytes), 16, 1024,
                                            kUmmaLayoutSw128);
        const uint64_t bd0 = umma_smem_desc(smem_u32(qbuf), 16, 1024, kUmmaLayoutSw128);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          // start addresses advance in 16-byte units inside the low descriptor field
          const uint64_t ad = ad0 + static_cast<uint64_t>(((ks >> 2) * kTcRegion + (ks & 3) * 32) >> 4);
          const uint64_t bd = bd0 + static_cast<uint64_t>(((ks >> 2) * kTcQHalf + (ks & 3) * 32) >> 4);
          umma_bf16(tmem + kColS + 32u * b, ad, bd, idesc_s, ks > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        umma_commit(&k_empty[st]);            // K of this stage may be reloaded
        if (flags & kTileLast) umma_commit(q_empty);
        return true;
      };
      auto ph_of = [](int x) { return static_cast<uint32_t>((x / kTcStages) & 1); };
      // S(t) is issued as soon as tile t's K lands; PV(t) as soon as its P is
      // written: the issuer polls both, so a late K never holds back a PV.
      int t = 0, s_next = 0;
      bool end_seen = false;
      if (wait_or_abort(&k_full[0], 0, abort_flag, a.err)) {
        const int f = meta[0].flags;
        if (f & kTileEnd) end_seen = true;
        else if ((ok = issue_s(0, f))) s_next = 1;
      } else {
        ok = false;
      }
      while (ok && s_next > t) {
        for (uint32_t spin = 0;; ++spin) {
          if (!end_seen && s_next == t + 1 && mbar_test_wait(&k_full[s_next % kTcStages], ph_of(s_next))) {
            const int f = meta[s_next % kMetaSlots].flags;
            if (f & kTileEnd) {
              end_seen = true;
            } else {
              if (!issue_s(s_next, f)) { ok = false; break; }
              ++s_next;
            }
          }
          if (mbar_test_wait(p_full, static_cast<uint32_t>(t & 1))) break;
          if (*abort_flag) { ok = false; break; }
          if (spin >= 16u * kMaxSpin) {
            *abort_flag = 1;
            report_error(a.err, S3R_DEVERR_TIMEOUT);
            ok = false;
            break;
          }
        }
        if (!ok) break;
        // O^T += V^T P^T for tile t
        const int st = t % kTcStages;
        if (!wait_or_abort(&v_full[st], ph_of(t), abort_flag, a.err)) { ok = false; break; }
        tc_fence_after_sync();
        const int n = meta[t % kMetaSlots].n;
        const bool first = (meta[t % kMetaSlots].flags & kTileFirst) != 0;
        const uint64_t vd0 = umma_smem_desc(smem_u32(stages + static_cast<size_t>(st) * kTcStageBytes) +
                                                2 * kTcRegion,
                                            kTcRegion, 1024, kUmmaLayoutSw128);
        // P^T: MN-major, no swizzle; 8-row core blocks 128 B apart along N, 8-token blocks 1 KiB apart
        const uint64_t pd0 = umma_smem_desc(smem_u32(pbuf), 1024, 128, kUmmaLayoutNone);
        for (int p = 0; p < n; ++p) {
          umma_bf16(tmem + kColO, vd0 + static_cast<uint64_t>((p * kHalfBytes) >> 4),
                    pd0 + static_cast<uint64_t>((p * 2048) >> 4), idesc_o, (first && p == 0) ? 0u : 1u);
        }
        umma_commit(o_done);
        umma_commit(&v_empty[st]);
        ++t;
        if (s_next == t && !end_seen) {      // S(t) still waits for its K
          if (!wait_or_abort(&k_full[t % kTcStages], ph_of(t), abort_flag, a.err)) { ok = false; break; }
          const int f = meta[t % kMetaSlots].flags;
          if (f & kTileEnd) end_seen = true;
          else if ((ok = issue_s(t, f))) ++s_next;
        }
      }
      if (!ok) *abort_flag = 1;
      // no MMA may be in flight when the TMEM is freed
      umma_commit(drain);
      mbar_wait_bounded(drain, 0);
    }
    __syncwarp();
  } else {
    // =========================== softmax: two warpgroups of 4 warps, 16 rows each
    const int wg = (warp - 2) >> 2;                // warpgroup: rows wg*16 .. wg*16+15
    const int r0 = wg * kRowsWg;
    const int q4 = warp & 3;                       // TMEM lane quarter this warp may access
    const int i = q4 * 32 + lane;                  // token slot of the tile = TMEM lane
    const int sm_tid = tid - 64;                   // 0..255 over both warpgroups
    const int wg_bar = kWgBar0 + wg;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    float* rmax = red_max + wg * 128;              // [2 buffers][4 quarters][16 rows]
    float* rsum = red_sum + wg * 64;               // [4 quarters][16 rows]
    float m_run[kRowsWg], l_part[kRowsWg];
#pragma unroll
    for (int j = 0; j < kRowsWg; ++j) {
      m_run[j] = kNegInf;
      l_part[j] = 0.f;
    }
    int seg_index = 0;
    for (int t = 0;; ++t) {
      const int b = t & 1;
      bool ok = wait_or_abort(&meta_full[t % kMetaSlots], static_cast<uint32_t>((t / kMetaSlots) & 1),
                              abort_flag, a.err);
      const TileMeta& m = meta[t % kMetaSlots];
      const int flags = ok ? m.flags : kTileEnd;
      if (ok && !(flags & kTileEnd))
        ok = wait_or_abort(&s_full[b], static_cast<uint32_t>((t >> 1) & 1), abort_flag, a.err);
      if (!named_bar_and(kAllBar, kSoftmaxThreads, ok)) break;
      if (flags & kTileEnd) break;
      const int pair = m.pair, e0 = m.e0, n = m.n, np = m.np, Lh = m.L;
      const int page = i >> 4;
      const int lo = page < n ? m.lo[page] : 0;
      const int hi = page < n ? m.hi[page] : 0;
      const long long pstart = m.start;
      if (flags & kTileFirst) {
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j) {
          m_run[j] = kNegInf;
          l_part[j] = 0.f;
        }
      }
      tc_fence_after_sync();
      float x[kRowsWg];
      tmem_ld16(lane_addr + kColS + 32u * b + r0, x);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);

      // scale and mask: token pos is visible to rows r >= r_min (causal), r < R
      const int pos = (e0 + page) * kPage + (i & 15);
      const bool tok = pos >= lo && pos < hi;
      const int r_min = pos <= Lh ? 0 : (pos - Lh) * a.G;
      // x stays unscaled: the scale enters the vote and the exponent by fma
      if (!(tok && r_min == 0 && r0 + kRowsWg <= a.R)) {   // some row may not see the token
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j) {
          const int r = r0 + j;
          if (!(tok && r >= r_min && r < a.R)) x[j] = kNegInf;
        }
      }

      // The running max only moves when some score exceeds it by more than
      // the slack: one vote decides whether this tile needs the exact max.
      float v[kRowsWg];
      bool exceed = false;
#pragma unroll
      for (int j = 0; j < kRowsWg; ++j) exceed |= fmaf(x[j], a.scale_log2, -m_run[j]) > kRescaleSlack;
      bool ok_acc = true;
      bool waited_prev = false;
      if (named_bar_or(wg_bar, kWgThreads, exceed)) {
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j) v[j] = x[j] * a.scale_log2;
        reduce_scatter<32, kRowsWg, true>(v, lane);   // lanes 2j, 2j+1: row j of this warp
        float* rm = rmax + (t & 1) * 64;
        if ((lane & 1) == 0) rm[q4 * 16 + (lane >> 1)] = v[0];
        named_bar_sync(wg_bar, kWgThreads);
        const int jr = lane >> 1;
        const float tmax_l = fmaxf(fmaxf(rm[jr], rm[16 + jr]), fmaxf(rm[32 + jr], rm[48 + jr]));
        float alpha[kRowsWg];
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j) {
          const float tm = __shfl_sync(0xffffffffu, tmax_l, 2 * j);
          const float mn = fmaxf(m_run[j], tm);
          alpha[j] = mn == kNegInf ? 1.f : (m_run[j] == kNegInf ? 0.f : fast_exp2(m_run[j] - mn));
          m_run[j] = mn;
          l_part[j] *= alpha[j];
        }
        if (!(flags & kTileFirst)) {
          // O^T holds this pair's earlier tiles: rescale this group's columns once PV(t-1) is done
          const bool okw = wait_or_abort(o_done, static_cast<uint32_t>((t - 1) & 1), abort_flag, a.err);
          if (named_bar_and(wg_bar, kWgThreads, okw)) {
            tc_fence_after_sync();
            float o[kRowsWg];
            tmem_ld16(lane_addr + kColO + r0, o);
#pragma unroll
            for (int j = 0; j < kRowsWg; ++j) o[j] *= alpha[j];
            tmem_st16(lane_addr + kColO + r0, o);
            tmem_ld16(lane_addr + kColO + 32 + r0, o);
#pragma unroll
            for (int j = 0; j < kRowsWg; ++j) o[j] *= alpha[j];
            tmem_st16(lane_addr + kColO + 32 + r0, o);
            tc_fence_before_sync();
          } else {
            ok_acc = false;
          }
          waited_prev = true;
        }
      }
      float mu[kRowsWg];
      float m_lane = 0.f;   // m_use of row (lane & 15) of this group
#pragma unroll
      for (int j = 0; j < kRowsWg; ++j) {
        mu[j] = m_run[j] == kNegInf ? 0.f : m_run[j];
        if (j == (lane & 15)) m_lane = mu[j];
      }
#pragma unroll
      for (int j = 0; j < kRowsWg; ++j) {
        x[j] = fast_exp2(fmaf(x[j], a.scale_log2, -mu[j]));
        l_part[j] += x[j];
      }
      // P^T (bf16 high part and remainder); the buffer is free once PV(t-1) is done
      if (t > 0 && !waited_prev)
        ok_acc = ok_acc && wait_or_abort(o_done, static_cast<uint32_t>((t - 1) & 1), abort_flag, a.err);
      if (!named_bar_and(kAllBar, kSoftmaxThreads, ok_acc)) break;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t h4[4], l4[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) split_bf16x2(x[c * 8 + 2 * jj], x[c * 8 + 2 * jj + 1], h4[jj], l4[jj]);
        const int off = (i >> 3) * 1024 + (2 * wg + c) * 128 + (i & 7) * 16;
        *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(h4[0], h4[1], h4[2], h4[3]);
        *reinterpret_cast<uint4*>(pbuf + off + 4 * 128) = make_uint4(l4[0], l4[1], l4[2], l4[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      if (MASS) {
        // per (page, row) log-sum-exp, after P^T is handed to the output MMA (it
        // runs meanwhile): the sum over the 16 tokens of the page
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j) v[j] = x[j];
        reduce_scatter<16, kRowsWg, false>(v, lane);   // lane holds row (lane & 15)
        const int r = r0 + (lane & 15);
        if (page < n && r < a.R) {
          a.page_lse[(static_cast<int64_t>(pair) * a.max_pages + e0 + page) * a.R + r] =
              v[0] > 0.f ? m_lane + fast_log2(v[0]) : kNegInf;
        }
      }

      if (!(flags & kTileLast)) continue;
      // =========================== end of this pair's segment
      ok = wait_or_abort(o_done, static_cast<uint32_t>(t & 1), abort_flag, a.err);
      if (!named_bar_and(kAllBar, kSoftmaxThreads, ok)) break;
      tc_fence_after_sync();
      float o[kRowsWg];
      tmem_ld16(lane_addr + kColO + r0, o);       // thread i holds column d = i of the group's rows
      tmem_ld16(lane_addr + kColO + 32 + r0, v);  // the P-remainder half
#pragma unroll
      for (int j = 0; j < kRowsWg; ++j) o[j] += v[j];
      tc_fence_before_sync();
#pragma unroll
      for (int j = 0; j < kRowsWg; ++j) v[j] = l_part[j];
      reduce_scatter<32, kRowsWg, false>(v, lane);
      if ((lane & 1) == 0) rsum[q4 * 16 + (lane >> 1)] = v[0];
      named_bar_sync(wg_bar, kWgThreads);
      const int jr = lane >> 1;                    // lanes 2j, 2j+1: row r0 + j
      const float L_l = (rsum[jr] + rsum[16 + jr]) + (rsum[32 + jr] + rsum[48 + jr]);
      float m_jr = 0.f;
#pragma unroll
      for (int j = 0; j < kRowsWg; ++j)
        if (j == jr) m_jr = mu[j];
      const int s = pair / a.Hkv, h = pair - (pair / a.Hkv) * a.Hkv;
      int last = 0;
      if (flags & kTileWhole) {
        const float inv_l = L_l > 0.f ? 1.f / L_l : 0.f;
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j) {
          const float ir = __shfl_sync(0xffffffffu, inv_l, 2 * j);
          if (r0 + j < a.R) a.out[q_row_off(a, s, h, r0 + j) + i] = o[j] * ir;
        }
        if (MASS && q4 == 0 && (lane & 1) == 0) row_lse[r0 + jr] = L_l > 0.f ? m_jr + fast_log2(L_l) : kNegInf;
      } else {
        const int slot = cta * 2 + (seg_index == 0 ? 0 : 1);
#pragma unroll
        for (int j = 0; j < kRowsWg; ++j)
          if (r0 + j < a.R) a.part_o[(static_cast<int64_t>(slot) * a.R + r0 + j) * kHeadDim + i] = o[j];
        if (q4 == 0 && (lane & 1) == 0 && r0 + jr < a.R)
          *reinterpret_cast<float2*>(a.part_ml + (static_cast<int64_t>(slot) * a.R + r0 + jr) * 2) =
              make_float2(m_jr, L_l);
        __threadfence();
        named_bar_sync(kAllBar, kSoftmaxThreads);
        const int gwa = share_of(N, pstart, tw);
        const int nseg = N >= tw ? share_of(N, pstart + np - 1, tw) - gwa + 1 : np;
        if (sm_tid == 0) *last_flag = atomicAdd(a.arrivals + pair, 1) == nseg - 1;
        named_bar_sync(kAllBar, kSoftmaxThreads);
        last = *last_flag;
        if (last) {
          __threadfence();
          auto slot_of = [&](int j) -> int {
            if (N >= tw) return (gwa + j) * 2 + ((j == 0 && share_start(N, gwa, tw) < pstart) ? 1 : 0);
            return share_of(N, pstart + j, tw) * 2;
          };
          if (q4 == 0 && lane < kRowsWg) {
            float M = kNegInf, Ls = 0.f;
            if (r0 + lane < a.R) {
              for (int j = 0; j < nseg; ++j) {
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(
                    a.part_ml + (static_cast<int64_t>(slot_of(j)) * a.R + r0 + lane) * 2));
                if (ml.y > 0.f) {
                  const float mn = fmaxf(M, ml.x);
                  Ls = Ls * fast_exp2(M - mn) + ml.y * fast_exp2(ml.x - mn);
                  M = mn;
                }
              }
            }
            row_max[r0 + lane] = M;
            row_inv[r0 + lane] = Ls > 0.f ? 1.f / Ls : 0.f;
            row_lse[r0 + lane] = Ls > 0.f ? M + fast_log2(Ls) : kNegInf;
          }
          named_bar_sync(wg_bar, kWgThreads);
          for (int j = 0; j < kRowsWg && r0 + j < a.R; ++j) {
            const int r = r0 + j;
            const float Mr = row_max[r], ir = row_inv[r];
            float acc = 0.f;
            for (int sg = 0; sg < nseg; ++sg) {
              const int64_t row = static_cast<int64_t>(slot_of(sg)) * a.R + r;
              const float mr = __ldcg(a.part_ml + row * 2);
              const float w = mr == kNegInf ? 0.f : fast_exp2(mr - Mr) * ir;
              acc += w * __ldcg(a.part_o + row * kHeadDim + i);
            }
            a.out[q_row_off(a, s, h, r) + i] = acc;
          }
          if (sm_tid == 0) a.arrivals[pair] = 0;
        }
      }
      if (MASS && ((flags & kTileWhole) || last)) {
        named_bar_sync(kAllBar, kSoftmaxThreads);
        float* dst = a.page_mass + static_cast<int64_t>(pair) * a.mass_stride;
        const float* plse = a.page_lse + static_cast<int64_t>(pair) * a.max_pages * a.R;
        if ((a.R & 3) == 0 && a.R <= kTcRows) {
          // Pages lp and lp + 256 at once: 16 loads of 16 bytes in flight per
          // thread.  One page at a time left the pipeline stalled for about six
          // dependent load round trips per pair; three or four pages at once
          // were slower again (their loads compete with the stage ring's).
          constexpr int kU = 2;
          for (int lp0 = sm_tid; lp0 < a.mass_stride; lp0 += kU * kSoftmaxThreads) {
            float4 v[kU][kTcRows / 4];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              const int lp = lp0 + u * kSoftmaxThreads;
#pragma unroll
              for (int q = 0; q < kTcRows / 4; ++q)
                v[u][q] = (lp < np && 4 * q < a.R)
                              ? __ldcg(reinterpret_cast<const float4*>(plse + static_cast<int64_t>(lp) * a.R) + q)
                              : make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
              float m = 0.f;
#pragma unroll
              for (int q = 0; q < kTcRows / 4; ++q) {
                const float e[4] = {v[u][q].x, v[u][q].y, v[u][q].z, v[u][q].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float L = 4 * q + k < a.R ? row_lse[4 * q + k] : kNegInf;
                  if (e[k] != kNegInf && L != kNegInf) m += fast_exp2(e[k] - L);
                }
              }
              const int lp = lp0 + u * kSoftmaxThreads;
              if (lp < a.mass_stride) dst[lp] = m;
            }
          }
        } else {
          for (int lp = sm_tid; lp < a.mass_stride; lp += kSoftmaxThreads)
            dst[lp] = lp < np ? page_mass_of(plse + static_cast<int64_t>(lp) * a.R, row_lse, a.R) : 0.f;
        }
      }
      ++seg_index;
      named_bar_sync(kAllBar, kSoftmaxThreads);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t verify_tc_smem_bytes(int n_chunks) { return tc_smem_layout(n_chunks).total; }

cudaError_t launch_verify_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                             const AttnArgs& a, int grid, cudaStream_t stream) {
  const size_t smem = verify_tc_smem_bytes(a.n_chunks);
  const bool mass = a.page_mass != nullptr;
  auto kern = mass ? attn_verify_tc_kernel<true> : attn_verify_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, smem, stream>>>(kmap, vmap, qmap, a);
  return cudaGetLastError();
}

}  // namespace s3r
