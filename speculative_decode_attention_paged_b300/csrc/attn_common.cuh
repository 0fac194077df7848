// Paged page-stream helpers shared by the S³R attention kernels: the pages of
// every (sequence, KV head) pair of a call form one global stream, split into
// equal contiguous shares across the workers of a persistent grid.
#pragma once

#include "attn_paged.cuh"
#include "s3r_device.cuh"

namespace s3r {
namespace attn {
namespace {   // internal linkage: every kernel file gets its own copy

constexpr float kNegInf = -__builtin_huge_valf();

struct PairGeom {
  int np;     // pages in the pair's stream
  int L;      // ctx_len (dense) or hist_len (sparse / verify)
  int cnt;    // selected pages (sparse)
};

// The inputs of a pair's geometry: its sequence's length and (sparse) its
// selection count.  Loaded apart from their use so that callers can have the
// loads of many pairs in flight together.
struct GeomIn {
  int len;
  int cnt;
};

__device__ __forceinline__ GeomIn pair_geom_load(const AttnArgs& a, int pair) {
  GeomIn in;
  in.len = __ldg(a.lens + pair / a.Hkv);
  in.cnt = a.mode == kModeSparse ? __ldg(a.sel_count + pair) : 0;
  return in;
}

// Pages of a pair in the global stream, with its length and selection count,
// from its loaded inputs.
__device__ PairGeom pair_geom_of(const AttnArgs& a, GeomIn in, bool report) {
  PairGeom g{0, 0, 0};
  const int len = in.len;
  const int cap = a.max_pages * kPage;
  if (a.mode == kModeDense) {
    if (len < 0 || len > cap) {
      if (report) report_error(a.err, S3R_DEVERR_BAD_LENGTH);
      return g;
    }
    g.L = len;
    g.np = (len + kPage - 1) / kPage;
  } else if (a.mode == kModeVerify) {
    if (len < 0 || len + a.T > cap) {
      if (report) report_error(a.err, S3R_DEVERR_BAD_LENGTH);
      return g;
    }
    g.L = len;
    g.np = (len + a.T + kPage - 1) / kPage;
  } else {
    const int last = len + a.draft_pos;
    if (len < 0 || last >= cap) {
      if (report) report_error(a.err, S3R_DEVERR_BAD_LENGTH);
      return g;
    }
    int cnt = in.cnt;
    if (cnt < 0 || cnt > a.b_max) {
      if (report) report_error(a.err, S3R_DEVERR_BAD_COUNT);
      cnt = 0;
    }
    g.L = len;
    g.cnt = cnt;
    g.np = cnt + (last / kPage - len / kPage + 1);
  }
  return g;
}

// Pages of pair `pair` in the global stream, with its length and selection count.
__device__ PairGeom pair_geom(const AttnArgs& a, int pair, bool report) {
  return pair_geom_of(a, pair_geom_load(a, pair), report);
}

struct Entry {
  int lp;     // logical page
  int lo;     // first visible token (absolute)
  int hi;     // one past the last visible token
  int phys;   // physical page, -1 = nothing to load
};

// Entry e of pair `pair`'s page stream.
__device__ Entry pair_entry(const AttnArgs& a, int pair, const PairGeom& g, int e) {
  Entry r{-1, 0, 0, -1};
  const int s = pair / a.Hkv;
  if (a.mode == kModeDense) {
    r.lp = e;
    r.lo = e * kPage;
    r.hi = min(r.lo + kPage, g.L);
  } else if (a.mode == kModeVerify) {
    r.lp = e;
    r.lo = e * kPage;
    r.hi = min(r.lo + kPage, g.L + a.T);
  } else if (e < g.cnt) {
    const int lp = __ldg(a.sel_pages + static_cast<int64_t>(pair) * a.b_max + e);
    if (lp < 0 || lp >= a.max_pages) {
      report_error(a.err, S3R_DEVERR_BAD_PAGE);
      return r;
    }
    r.lp = lp;
    r.lo = lp * kPage;
    r.hi = min(r.lo + kPage, g.L);
  } else {
    r.lp = g.L / kPage + (e - g.cnt);
    r.lo = max(r.lp * kPage, g.L);
    r.hi = min(r.lp * kPage + kPage, g.L + a.draft_pos + 1);
  }
  if (r.lo < r.hi) {
    const int phys = __ldg(a.block_table + static_cast<int64_t>(s) * a.max_pages + r.lp);
    if (phys < 0 || static_cast<int64_t>(phys) >= a.num_phys_pages) {
      report_error(a.err, S3R_DEVERR_BAD_PAGE);
    } else {
      r.phys = phys;
    }
  }
  return r;
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}

__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Global page index where warp share `gw` starts (shares split N pages evenly).
__device__ __forceinline__ int64_t share_start(int64_t N, int gw, int tw) {
  return N * gw / tw;
}

// The warp share holding global page x (the last share whose start is <= x).
__device__ __forceinline__ int share_of(int64_t N, int64_t x, int tw) {
  return static_cast<int>(((x + 1) * tw - 1) / N);
}

// In-CTA exclusive scan of vals[0..n) in place; vals[n] receives the total.
// THREADS = the CTA's thread count (a multiple of 32, at most 1024).
template <int THREADS>
__device__ void block_exclusive_scan(int* vals, int n, int* scratch) {
  constexpr int kWarpsB = THREADS / 32;
  const int tid = threadIdx.x;
  const int per = (n + THREADS - 1) / THREADS;
  const int b = min(tid * per, n), e = min(b + per, n);
  int local = 0;
  for (int i = b; i < e; ++i) local += vals[i];
  // warp inclusive scan of the thread sums
  const int lane = tid & 31, warp = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarpsB ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    if (lane < kWarpsB) scratch[lane] = w;   // inclusive warp totals
  }
  __syncthreads();
  int run = incl - local + (warp > 0 ? scratch[warp - 1] : 0);
  for (int i = b; i < e; ++i) {
    const int v = vals[i];
    vals[i] = run;
    run += v;
  }
  if (tid == THREADS - 1) vals[n] = run;
  __syncthreads();
}

// Normalised page mass of one pair: dst[lp] = sum over rows r < R of
// 2^(lse[lp][r] - LSE[r]) for pages lp < np, zero for np <= lp < stride.
// Thread t of nthreads takes pages t, t + nthreads, ...; it keeps the loads of
// kU pages x 4 rows in flight (a page at a time left one dependent load chain
// per page, which ran at the end of the kernel), and sums each page's rows in
// the order r = 0, 1, ....
template <int kU>
__device__ __forceinline__ void write_pair_mass(float* dst, const float* lse, const float* row_lse, int R, int np,
                                                int stride, int t, int nthreads) {
  for (int lp0 = t; lp0 < stride; lp0 += nthreads * kU) {
    float acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = 0.f;
    if (lp0 < np) {
      for (int r0 = 0; r0 < R; r0 += 4) {
        float v[kU][4];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int lp = lp0 + u * nthreads;
#pragma unroll
          for (int k = 0; k < 4; ++k)
            v[u][k] = (lp < np && r0 + k < R) ? __ldcg(lse + static_cast<int64_t>(lp) * R + r0 + k) : kNegInf;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (r0 + k < R) {
            const float L = row_lse[r0 + k];
#pragma unroll
            for (int u = 0; u < kU; ++u)
              if (v[u][k] != kNegInf && L != kNegInf) acc[u] += fast_exp2(v[u][k] - L);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int lp = lp0 + u * nthreads;
      if (lp < stride) dst[lp] = lp < np ? acc[u] : 0.f;
    }
  }
}

// Normalised mass of one page: sum over rows r < R of 2^(lse_page[r] - LSE[r]).
// lse_page is 16-byte aligned when R is a multiple of 4.
__device__ __forceinline__ float page_mass_of(const float* lse_page, const float* row_lse, int R) {
  float mass = 0.f;
  if ((R & 3) == 0) {
#pragma unroll 8
    for (int r = 0; r < R; r += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(lse_page + r));
      const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float L = row_lse[r + k];
        if (e[k] != kNegInf && L != kNegInf) mass += fast_exp2(e[k] - L);
      }
    }
  } else {
    for (int r = 0; r < R; ++r) {
      const float v = __ldcg(lse_page + r);
      const float L = row_lse[r];
      if (v != kNegInf && L != kNegInf) mass += fast_exp2(v - L);
    }
  }
  return mass;
}

// Zero output rows (and zero page mass) of a pair with no page to read.
__device__ void zero_pair(const AttnArgs& a, int pair) {
  const int s = pair / a.Hkv, h = pair - (pair / a.Hkv) * a.Hkv;
  for (int r = 0; r < a.R; ++r) {
    const int i = r / a.G, g = r - (r / a.G) * a.G;
    float4* dst = reinterpret_cast<float4*>(
        a.out + ((static_cast<int64_t>(s) * a.T + i) * a.Hq + h * a.G + g) * kHeadDim);
    for (int c = 0; c < kHeadDim / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (a.page_mass != nullptr) {
    float* m = a.page_mass + static_cast<int64_t>(pair) * a.mass_stride;
    for (int lp = 0; lp < a.mass_stride; ++lp) m[lp] = 0.f;
  }
}

// The call's appended rows that fall in logical page lp of pair (s, h), whose
// physical page is phys: written into the pool by the whole warp (lanes 0-15
// the K row, lanes 16-31 the V row, 16 bytes each), then ordered before the
// TMA load of that page that this warp issues next.  Each entry of a pair's
// page stream is read by one warp only, so no reader sees the page before the
// rows land.  (A draft page that is both selected and the draft tail is two
// entries: both writers store the same bytes.)  The loads of up to kBatch rows
// are in flight before any of their stores.
template <int kBatch>
__device__ __forceinline__ void append_rows_in_page(const AttnArgs& a, int s, int h, int L, int lp, int phys,
                                                    int lane) {
  if (a.app_rows == 0 || phys < 0) return;
  const int p0 = a.mode == kModeDense ? L - 1 : (a.mode == kModeSparse ? L + a.draft_pos : L);
  const int lo = max(p0, lp * kPage), hi = min(p0 + a.app_rows, (lp + 1) * kPage);
  if (lo >= hi) return;
  const int piece = lane & 15;
  const uint4* src = lane < 16 ? a.app_k : a.app_v;
  uint4* dst = lane < 16 ? a.k_pool_w : a.v_pool_w;
  for (int base = lo; base < hi; base += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const int pos = base + r;
      if (pos < hi) v[r] = __ldg(src + ((static_cast<int64_t>(s) * a.app_rows + (pos - p0)) * a.Hkv + h) * 16 + piece);
    }
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const int pos = base + r;
      if (pos < hi) dst[((static_cast<int64_t>(phys) * a.Hkv + h) * kPage + (pos % kPage)) * 16 + piece] = v[r];
    }
  }
  fence_proxy_async_global();
  __syncwarp();
}

// The one appended row of pair (s, h) (calls with app_rows == 1), this lane's
// 16-byte piece of it: K for lanes 0-15, V for 16-31.  Loaded when a warp
// starts on the pair, so the load overlaps the pair's earlier pages.
__device__ __forceinline__ uint4 load_single_row(const AttnArgs& a, int s, int h, int lane) {
  const uint4* src = lane < 16 ? a.app_k : a.app_v;
  return __ldg(src + (static_cast<int64_t>(s) * a.Hkv + h) * 16 + (lane & 15));
}

// Store of that row if it falls in logical page lp (physical page phys), then
// the same ordering before the page's TMA load as append_rows_in_page.
__device__ __forceinline__ void store_single_row(const AttnArgs& a, int h, int L, int lp, int phys, int lane,
                                                 uint4 v) {
  if (phys < 0) return;
  const int pos = a.mode == kModeDense ? L - 1 : (a.mode == kModeSparse ? L + a.draft_pos : L);
  if (pos / kPage != lp) return;
  uint4* dst = lane < 16 ? a.k_pool_w : a.v_pool_w;
  dst[((static_cast<int64_t>(phys) * a.Hkv + h) * kPage + (pos % kPage)) * 16 + (lane & 15)] = v;
  fence_proxy_async_global();
  __syncwarp();
}

// Plan of a call: pages of every chunk of kPairChunk pairs into prefix[c],
// before the exclusive scan.  Warp w of nwarps takes chunks w, w + nwarps,
// ...; the geometry loads of kPlanBatch chunks are issued before any of them is
// used, so their latencies overlap (a chain of one load round trip per chunk
// was most of a call's start-up).  Pairs with nothing to read get zero
// outputs here, each from one CTA.
constexpr int kPlanBatch = 8;

__device__ __forceinline__ void plan_chunk_pages(const AttnArgs& a, int* prefix, int warp, int nwarps, int lane) {
  for (int c0 = warp; c0 < a.n_chunks; c0 += kPlanBatch * nwarps) {
    GeomIn in[kPlanBatch];
#pragma unroll
    for (int u = 0; u < kPlanBatch; ++u) {
      const int c = c0 + u * nwarps;
      const int pair = c * kPairChunk + lane;
      in[u] = (c < a.n_chunks && pair < a.n_pairs) ? pair_geom_load(a, pair) : GeomIn{0, 0};
    }
#pragma unroll
    for (int u = 0; u < kPlanBatch; ++u) {
      const int c = c0 + u * nwarps;
      const int pair = c * kPairChunk + lane;
      int np = 0;
      if (c < a.n_chunks && pair < a.n_pairs) {
        np = pair_geom_of(a, in[u], blockIdx.x == 0).np;
        if (np == 0 && (c % static_cast<int>(gridDim.x)) == static_cast<int>(blockIdx.x)) zero_pair(a, pair);
      }
      np = warp_sum(np);
      if (lane == 0 && c < a.n_chunks) prefix[c] = np;
    }
  }
}

}  // namespace
}  // namespace attn
}  // namespace s3r
