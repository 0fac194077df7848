// Paged split-KV attention for the three attention forms of an S³R round.
//
// What is computed (per the S³R pages):
//   * dense decode: every step reads the whole history (arXiv abstract;
//     wispaper.ai "Sparse sampling changes the group, not just the speed");
//   * sparse draft: the policy reads only its selected pages plus its own
//     draft tail (wispaper.ai "S3R drafts sparsely and verifies densely");
//   * verify: T drafted positions attend causally to the complete history
//     (same section; "Dense verification still pays the full KV-cache bill"),
//     and the verify attention mass per page feeds the next draft's selection
//     (rit.work "Как разреженный черновик сохраняет ответы плотной модели").
//
// How (B300 design):
//   * Work unit = one 16-token page of one (sequence, KV head) pair: a 4 KiB K
//     tile + a 4 KiB V tile, contiguous in the pool.  All pages of all pairs
//     form one global stream; each warp of a persistent grid (one 8-warp CTA
//     per SM) takes an equal contiguous share of it, so load balance is exact
//     whatever the mix of context lengths.  A pair cut by share boundaries
//     leaves a partial (m, l, O) per segment (at most two per warp); each
//     writer publishes its segment with a fence and an arrival counter, and
//     the last segment to arrive merges them (log-sum-exp merge) in place, so
//     one launch does the whole call.
//   * Each warp runs its own 2-stage TMA pipeline (cp.async.bulk.tensor, one
//     mbarrier per stage, 128-byte swizzle so ldmatrix reads are
//     bank-conflict free).  Page ids are fetched 32 at a time, one per lane.
//   * The G (decode / draft) or T*G (verify) query rows of a pair share every
//     K/V tile: S = Q K^T and O += P V run on bf16 mma.sync m16n8k16 with the
//     16 tokens of a page as one n16 / k16 block, fp32 accumulation and an
//     online softmax in registers (exp2 domain).
//   * Verify with page mass also stores, per (page, row), the base-2
//     log-sum-exp of the row's scores over the page; the warp that completes
//     a pair turns it into the normalised mass sum_r 2^(lse_page,r - LSE_r).
//   * Data-dependent errors (bad page id, bad length) skip the page and set a
//     bit in the device error word; every wait is bounded.

#include "attn_common.cuh"
#include "attn_paged.cuh"
#include "s3r_device.cuh"

namespace s3r {

namespace {

using namespace attn;

constexpr int kStageBytes = 2 * kTileBytes;   // K tile + V tile
constexpr int kThreads = kAttnWarps * 32;

// Smem address of the 16-byte chunk holding (token, d0..d0+7) of a swizzled
// K or V tile: two 64-column halves of 16 rows x 128 B, 128B-swizzled.
__device__ __forceinline__ uint32_t tile_addr(uint32_t tile, int token, int d0) {
  const int half = d0 >> 6;
  const int chunk = (d0 & 63) >> 3;
  return tile + half * kHalfBytes + token * 128 + ((chunk ^ (token & 7)) << 4);
}

template <int MT, bool MASS>
__global__ void __launch_bounds__(kThreads, 1)
    attn_partial_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stage_mem = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kAttnWarps * kAttnStages * kStageBytes);
  int4* meta = reinterpret_cast<int4*>(bars + kAttnWarps * kAttnStages);   // 2 int4 per stage
  int* scratch = reinterpret_cast<int*>(meta + 2 * kAttnWarps * kAttnStages);   // 32 ints
  float* lse_all = reinterpret_cast<float*>(scratch + 32);               // [warps][32] row LSEs
  int* prefix = reinterpret_cast<int*>(lse_all + kAttnWarps * 32);       // n_chunks + 1

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid < kAttnWarps * kAttnStages) mbar_init(&bars[tid], 1);

  // ---- plan: pages per chunk of 32 pairs, then an exclusive scan
  plan_chunk_pages(a, prefix, warp, kAttnWarps, lane);
  fence_barrier_init();
  __syncthreads();
  block_exclusive_scan<kThreads>(prefix, a.n_chunks, scratch);

  const int64_t N = prefix[a.n_chunks];
  const int tw = a.total_warps;
  const int gw = blockIdx.x * kAttnWarps + warp;
  const int64_t x0 = share_start(N, gw, tw);
  const int64_t x1 = share_start(N, gw + 1, tw);
  if (x0 >= x1) return;

  uint8_t* my_stages = stage_mem + warp * kAttnStages * kStageBytes;
  uint64_t* my_bars = bars + warp * kAttnStages;
  int4* my_meta = meta + 2 * warp * kAttnStages;
  const uint64_t policy = l2_policy_evict_first();

  // ---- locate the pair holding x0: chunk by binary search, then a warp scan
  int pr_pair;
  int64_t pr_pair_start;
  {
    int lo = 0, hi = a.n_chunks - 1;   // largest c with prefix[c] <= x0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= x0) lo = mid; else hi = mid - 1;
    }
    const int c = lo;
    const int pair = c * kPairChunk + lane;
    const int np = pair < a.n_pairs ? pair_geom(a, pair, false).np : 0;
    int incl = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int64_t rel = x0 - prefix[c];
    const unsigned ball = __ballot_sync(0xffffffffu, incl > rel);
    const int l = __ffs(ball) - 1;
    pr_pair = c * kPairChunk + l;
    pr_pair_start = prefix[c] + __shfl_sync(0xffffffffu, incl - np, l);
  }

  // ---- producer state (warp-uniform except the per-lane entry cache)
  PairGeom pr_g = pair_geom(a, pr_pair, false);
  int pr_e = static_cast<int>(x0 - pr_pair_start);
  int pr_base = pr_e;
  Entry cache = pr_base + lane < pr_g.np ? pair_entry(a, pr_pair, pr_g, pr_base + lane)
                                         : Entry{-1, 0, 0, -1};
  int64_t pr_x = x0;
  int64_t pr_k = 0;
  const bool app_one = a.app_rows == 1;
  uint4 pr_row = app_one ? load_single_row(a, pr_pair / a.Hkv, pr_pair % a.Hkv, lane) : uint4{};

  auto produce = [&]() {
    if (pr_x >= x1) return;
    if (pr_e >= pr_g.np) {
      do {
        ++pr_pair;
        pr_g = pair_geom(a, pr_pair, false);
      } while (pr_g.np == 0);
      pr_e = 0;
      pr_base = 0;
      cache = lane < pr_g.np ? pair_entry(a, pr_pair, pr_g, lane) : Entry{-1, 0, 0, -1};
      if (app_one) pr_row = load_single_row(a, pr_pair / a.Hkv, pr_pair % a.Hkv, lane);
    } else if (pr_e - pr_base >= 32) {
      pr_base = pr_e;
      cache = pr_base + lane < pr_g.np ? pair_entry(a, pr_pair, pr_g, pr_base + lane)
                                       : Entry{-1, 0, 0, -1};
    }
    const int li = pr_e - pr_base;
    const int lp = __shfl_sync(0xffffffffu, cache.lp, li);
    const int elo = __shfl_sync(0xffffffffu, cache.lo, li);
    const int ehi = __shfl_sync(0xffffffffu, cache.hi, li);
    const int phys = __shfl_sync(0xffffffffu, cache.phys, li);
    const int st = static_cast<int>(pr_k % kAttnStages);
    if (app_one)
      store_single_row(a, pr_pair % a.Hkv, pr_g.L, lp, phys, lane, pr_row);
    else
      append_rows_in_page<1>(a, pr_pair / a.Hkv, pr_pair % a.Hkv, pr_g.L, lp, phys, lane);
    if (lane == 0) {
      my_meta[2 * st] = make_int4(lp, elo, ehi, phys);
      my_meta[2 * st + 1] = make_int4(pr_pair, pr_e, pr_g.np, pr_g.L);
      uint64_t* bar = &my_bars[st];
      if (phys >= 0) {
        mbar_arrive_expect_tx(bar, kStageBytes);
        uint8_t* dst = my_stages + st * kStageBytes;
        const int y = (pr_pair % a.Hkv) * kPage;
        fence_proxy_async_smem();
        tma_load_3d(dst, &kmap, 0, y, phys, bar, policy);
        tma_load_3d(dst + kHalfBytes, &kmap, 64, y, phys, bar, policy);
        tma_load_3d(dst + kTileBytes, &vmap, 0, y, phys, bar, policy);
        tma_load_3d(dst + kTileBytes + kHalfBytes, &vmap, 64, y, phys, bar, policy);
      } else {
        mbar_arrive_expect_tx(bar, 0);
      }
    }
    ++pr_e;
    ++pr_x;
    ++pr_k;
  };

  for (int i = 0; i < kAttnStages; ++i) produce();

  // ---- consumer state
  const int qg = lane >> 2;      // row within an m16 tile (and +8)
  const int qt = lane & 3;       // column pair selector
  uint32_t qf[MT][8][4];
  float o[MT][16][4];
  float m_r[MT][2], l_r[MT][2];
  int cur_pair = -1, cur_s = 0, cur_h = 0, cur_L = 0, cur_np = 0, seg_first = 0, seg_last = 0;
  int seg_index = 0;
  int64_t cur_start = 0;           // global stream index of the current pair's first page
  float* my_lse = lse_all + warp * 32;

  // Per-lane constant parts of the ldmatrix row addresses.
  const int k_tok = ((lane >> 4) << 3) + (lane & 7);
  const int k_dsel = (lane >> 3) & 1;
  const int v_tok = (((lane >> 3) & 1) << 3) + (lane & 7);
  const int v_dsel = lane >> 4;

  auto q_row_offset = [&](int r) -> int64_t {
    const int i = r / a.G;
    const int g = r - i * a.G;
    return ((static_cast<int64_t>(cur_s) * a.T + i) * a.Hq + cur_h * a.G + g) * kHeadDim;
  };

  auto begin_pair = [&](int pair, int e_first, int np, int L) {
    cur_pair = pair;
    cur_s = pair / a.Hkv;
    cur_h = pair - cur_s * a.Hkv;
    cur_L = L;
    cur_np = np;
    seg_first = e_first;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      m_r[mt][0] = m_r[mt][1] = kNegInf;
      l_r[mt][0] = l_r[mt][1] = 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n) o[mt][n][0] = o[mt][n][1] = o[mt][n][2] = o[mt][n][3] = 0.f;
      const int r0 = mt * 16 + qg, r1 = r0 + 8;
      const bool v0 = r0 < a.R, v1 = r1 < a.R;
      const uint32_t* q0 = v0 ? reinterpret_cast<const uint32_t*>(a.q + q_row_offset(r0)) : nullptr;
      const uint32_t* q1 = v1 ? reinterpret_cast<const uint32_t*>(a.q + q_row_offset(r1)) : nullptr;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int c0 = (ks * 16 + qt * 2) >> 1, c1 = c0 + 4;   // 32-bit word index
        qf[mt][ks][0] = v0 ? __ldg(q0 + c0) : 0u;
        qf[mt][ks][1] = v1 ? __ldg(q1 + c0) : 0u;
        qf[mt][ks][2] = v0 ? __ldg(q0 + c1) : 0u;
        qf[mt][ks][3] = v1 ? __ldg(q1 + c1) : 0u;
      }
    }
  };

  // Page mass of the current pair from the per-(page, row) log-sum-exps and
  // the rows' final LSEs in my_lse; zero beyond its np pages.
  auto write_mass = [&]() {
    __syncwarp();
    float* dst = a.page_mass + static_cast<int64_t>(cur_pair) * a.mass_stride;
    const float* pl = a.page_lse + static_cast<int64_t>(cur_pair) * a.max_pages * a.R;
    write_pair_mass<16>(dst, pl, my_lse, a.R, cur_np, a.mass_stride, lane, 32);
  };

  // Slot of segment j of a pair cut by warp shares: the pair's pages start at
  // global index X and span shares gwa..; with N >= tw every share holds a
  // page, otherwise every non-empty share holds exactly one page.  a_off: the
  // first share started before the pair (its partial is that warp's second).
  auto segment_slot = [&](int64_t X, int gwa, bool a_off, int j) -> int {
    if (N >= tw) return (gwa + j) * 2 + ((j == 0 && a_off) ? 1 : 0);
    return share_of(N, X + j, tw) * 2;
  };

  // Merge the partials of the current (cut) pair.  Pass 1: lane r < R folds
  // row r's (m, l) over the segments, eight loads in flight at a time.  Pass 2:
  // every lane merges 4 of the 128 columns of each row, again with the loads
  // of eight segments issued together.
  auto merge_pair = [&](int nseg, int gwa) {
    constexpr int kBatch = 8;
    const bool a_off = N >= tw && share_start(N, gwa, tw) < cur_start;
    float M = kNegInf, Ls = 0.f;
    if (lane < a.R) {
      for (int j0 = 0; j0 < nseg; j0 += kBatch) {
        float2 ml[kBatch];
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
          const int j = j0 + jj;
          ml[jj] = j < nseg ? __ldcg(reinterpret_cast<const float2*>(
                                  a.part_ml + (static_cast<int64_t>(segment_slot(cur_start, gwa, a_off, j)) * a.R +
                                               lane) * 2))
                            : make_float2(kNegInf, 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
          if (ml[jj].y > 0.f) {
            const float mn = fmaxf(M, ml[jj].x);
            Ls = Ls * fast_exp2(M - mn) + ml[jj].y * fast_exp2(ml[jj].x - mn);
            M = mn;
          }
        }
      }
      if (MASS) my_lse[lane] = Ls > 0.f ? M + fast_log2(Ls) : kNegInf;
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    for (int r = 0; r < a.R; ++r) {
      const float Mr = __shfl_sync(0xffffffffu, M, r);
      const float ir = __shfl_sync(0xffffffffu, inv, r);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = 0; j0 < nseg; j0 += kBatch) {
        float mr[kBatch];
        float4 o[kBatch];
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
          const int j = j0 + jj;
          if (j < nseg) {
            const int64_t row = static_cast<int64_t>(segment_slot(cur_start, gwa, a_off, j)) * a.R + r;
            mr[jj] = __ldcg(a.part_ml + row * 2);
            o[jj] = __ldcg(reinterpret_cast<const float4*>(a.part_o + row * kHeadDim) + lane);
          } else {
            mr[jj] = kNegInf;
            o[jj] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
          const float w = mr[jj] == kNegInf ? 0.f : fast_exp2(mr[jj] - Mr) * ir;
          acc.x += w * o[jj].x;
          acc.y += w * o[jj].y;
          acc.z += w * o[jj].z;
          acc.w += w * o[jj].w;
        }
      }
      reinterpret_cast<float4*>(a.out + q_row_offset(r))[lane] = acc;
    }
  };

  auto finish_pair = [&]() {
    const bool whole = (seg_first == 0) && (seg_last == cur_np - 1);
    const int slot = gw * 2 + (seg_index == 0 ? 0 : 1);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int r = mt * 16 + qg + hb * 8;
        const float l = quad_sum(l_r[mt][hb]);
        const float m = m_r[mt][hb];
        if (r >= a.R) continue;
        if (whole) {
          const float inv = l > 0.f ? 1.f / l : 0.f;
          float* dst = a.out + q_row_offset(r);
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            *reinterpret_cast<float2*>(dst + n * 8 + qt * 2) =
                make_float2(o[mt][n][2 * hb] * inv, o[mt][n][2 * hb + 1] * inv);
          }
          if (MASS && qt == 0) my_lse[r] = l > 0.f ? m + fast_log2(l) : kNegInf;
        } else {
          float* po = a.part_o + (static_cast<int64_t>(slot) * a.R + r) * kHeadDim;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            *reinterpret_cast<float2*>(po + n * 8 + qt * 2) =
                make_float2(o[mt][n][2 * hb], o[mt][n][2 * hb + 1]);
          }
          if (qt == 0) {
            *reinterpret_cast<float2*>(a.part_ml + (static_cast<int64_t>(slot) * a.R + r) * 2) =
                make_float2(m, l);
          }
        }
      }
    }
    if (whole) {
      if (MASS && a.page_mass != nullptr) write_mass();
    } else {
      // Publish this segment; the last of the pair's segments to arrive merges.
      const int gwa = share_of(N, cur_start, tw);
      const int nseg = N >= tw ? share_of(N, cur_start + cur_np - 1, tw) - gwa + 1 : cur_np;
      fence_acq_rel_gpu();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(a.arrivals + cur_pair, 1) == nseg - 1;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        fence_acq_rel_gpu();
        merge_pair(nseg, gwa);
        if (MASS && a.page_mass != nullptr) write_mass();
        if (lane == 0) a.arrivals[cur_pair] = 0;   // ready for the next call
      }
    }
    ++seg_index;
  };

  bool ok = true;
  int64_t k_fail = 0;
  const int64_t n_total = x1 - x0;
  for (int64_t k = 0; k < n_total; ++k) {
    const int st = static_cast<int>(k % kAttnStages);
    const uint32_t parity = static_cast<uint32_t>((k / kAttnStages) & 1);
    if (!mbar_wait_bounded(&my_bars[st], parity)) {
      if (lane == 0) report_error(a.err, S3R_DEVERR_TIMEOUT);
      ok = false;
      k_fail = k;
      break;
    }
    const int4 m0 = my_meta[2 * st];
    const int4 m1 = my_meta[2 * st + 1];
    const int lp = m0.x, elo = m0.y, ehi = m0.z, phys = m0.w;
    if (m1.x != cur_pair) {
      if (cur_pair >= 0) finish_pair();
      begin_pair(m1.x, m1.y, m1.z, m1.w);
      cur_start = x0 + k - m1.y;
    }
    seg_last = m1.y;

    if (phys >= 0) {
      const uint32_t kt = smem_u32(my_stages + st * kStageBytes);
      const uint32_t vt = kt + kTileBytes;
      const int page0 = lp * kPage;

      // S = Q K^T for the page's 16 tokens.
      float sacc[MT][2][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          sacc[mt][nt][0] = sacc[mt][nt][1] = sacc[mt][nt][2] = sacc[mt][nt][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(tile_addr(kt, k_tok, ks * 16 + k_dsel * 8), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(sacc[mt][0], qf[mt][ks], b0, b1);
          mma_bf16_16816(sacc[mt][1], qf[mt][ks], b2, b3);
        }
      }

      // Mask: page token range, and for verify the causal limit of each row.
      const bool need_mask = (elo > page0) || (ehi < page0 + kPage) ||
                             (a.mode == kModeVerify && page0 + kPage - 1 > cur_L);
      uint32_t pa[MT][4], pl[MT][4];
      float ps_h[MT][2], mu_h[MT][2];   // page mass: this lane's row sums and the max they use
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int j = 0; j < 4; ++j) x[nt][j] = sacc[mt][nt][j] * a.scale_log2;
        if (need_mask) {
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const int r = mt * 16 + qg + hb * 8;
            const int lim = a.mode == kModeVerify ? cur_L + r / a.G : 0x7fffffff;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int t = page0 + nt * 8 + qt * 2 + e;
                if (t < elo || t >= ehi || t > lim) x[nt][hb * 2 + e] = kNegInf;
              }
          }
        }
        float alpha[2];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          float mx = fmaxf(fmaxf(x[0][2 * hb], x[0][2 * hb + 1]), fmaxf(x[1][2 * hb], x[1][2 * hb + 1]));
          mx = quad_max(mx);
          const float m_new = fmaxf(m_r[mt][hb], mx);
          const float m_use = m_new == kNegInf ? 0.f : m_new;
          alpha[hb] = fast_exp2(m_r[mt][hb] - m_use);
          float psum = 0.f;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float p = fast_exp2(x[nt][2 * hb + e] - m_use);
              x[nt][2 * hb + e] = p;
              psum += p;
            }
          l_r[mt][hb] = l_r[mt][hb] * alpha[hb] + psum;
          m_r[mt][hb] = m_new;
          ps_h[mt][hb] = psum;
          mu_h[mt][hb] = m_use;
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
          o[mt][n][0] *= alpha[0];
          o[mt][n][1] *= alpha[0];
          o[mt][n][2] *= alpha[1];
          o[mt][n][3] *= alpha[1];
        }
        // P as bf16 hi + lo parts: P V is then exact to ~2^-16 relative.
        split_bf16x2(x[0][0], x[0][1], pa[mt][0], pl[mt][0]);
        split_bf16x2(x[0][2], x[0][3], pa[mt][1], pl[mt][1]);
        split_bf16x2(x[1][0], x[1][1], pa[mt][2], pl[mt][2]);
        split_bf16x2(x[1][2], x[1][3], pa[mt][3], pl[mt][3]);
      }

      // O += P V.
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(tile_addr(vt, v_tok, c * 16 + v_dsel * 8), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16_16816(o[mt][2 * c], pa[mt], b0, b1);
          mma_bf16_16816(o[mt][2 * c + 1], pa[mt], b2, b3);
          mma_bf16_16816(o[mt][2 * c], pl[mt], b0, b1);
          mma_bf16_16816(o[mt][2 * c + 1], pl[mt], b2, b3);
        }
      }
      if (MASS) {
        // the page's log-sum-exp per row, after the output MMAs are issued
        float* pg = a.page_lse + (static_cast<int64_t>(cur_pair) * a.max_pages + lp) * a.R;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            const float ps = quad_sum(ps_h[mt][hb]);
            const int r = mt * 16 + qg + hb * 8;
            if (qt == 0 && r < a.R) pg[r] = ps > 0.f ? mu_h[mt][hb] + fast_log2(ps) : kNegInf;
          }
      }
    } else if (MASS && lp >= 0) {
      // Nothing visible on this page: it holds no mass.
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const int r = mt * 16 + qg + hb * 8;
          if (qt == 0 && r < a.R)
            a.page_lse[(static_cast<int64_t>(cur_pair) * a.max_pages + lp) * a.R + r] = kNegInf;
        }
    }
    __syncwarp();
    produce();
  }

  if (ok) {
    finish_pair();
  } else {
    // Drain whatever copies this warp still has in flight (bounded).
    for (int64_t k = k_fail; k < pr_k; ++k) {
      const int st = static_cast<int>(k % kAttnStages);
      mbar_wait_bounded(&my_bars[st], static_cast<uint32_t>((k / kAttnStages) & 1));
    }
  }
}

template <int MT, bool MASS>
cudaError_t launch_variant(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a,
                           int grid, cudaStream_t stream) {
  const size_t smem = attn_smem_bytes(a.n_chunks);
  cudaError_t e = cudaFuncSetAttribute(attn_partial_kernel<MT, MASS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  attn_partial_kernel<MT, MASS><<<grid, kThreads, smem, stream>>>(kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace

size_t attn_smem_bytes(int n_chunks) {
  return 1024 + static_cast<size_t>(kAttnWarps) * kAttnStages * kStageBytes +
         static_cast<size_t>(kAttnWarps) * kAttnStages * (8 + 32) + 32 * 4 + kAttnWarps * 32 * 4 +
         static_cast<size_t>(n_chunks + 1) * 4;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

AttnWorkspaceLayout attn_workspace_layout(int n_pairs, int rows, int max_pages, int total_warps,
                                          bool with_mass) {
  AttnWorkspaceLayout L{};
  size_t off = 0;
  L.err_off = off;
  off += 256;
  L.arrivals_off = off;
  off = align256(off + static_cast<size_t>(n_pairs) * 4);
  L.part_o_off = off;
  off = align256(off + static_cast<size_t>(2) * total_warps * rows * kHeadDim * 4);
  L.part_ml_off = off;
  off = align256(off + static_cast<size_t>(2) * total_warps * rows * 2 * 4);
  L.page_lse_off = off;
  if (with_mass) off = align256(off + static_cast<size_t>(n_pairs) * max_pages * rows * 4);
  L.total = off;
  return L;
}

cudaError_t launch_attention(const CUtensorMap& kmap, const CUtensorMap& vmap, const AttnArgs& a,
                             int grid, cudaStream_t stream) {
  const bool mass = a.mode == kModeVerify && a.page_mass != nullptr;
  if (a.R <= 16) {
    return mass ? launch_variant<1, true>(kmap, vmap, a, grid, stream)
                : launch_variant<1, false>(kmap, vmap, a, grid, stream);
  }
  return mass ? launch_variant<2, true>(kmap, vmap, a, grid, stream)
              : launch_variant<2, false>(kmap, vmap, a, grid, stream);
}

}  // namespace s3r
