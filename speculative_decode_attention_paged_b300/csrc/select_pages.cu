// Draft-page selection from verify attention mass.
//
// The S³R pages say the verification attention scores choose the history the
// next draft reads (rit.work, "Как разреженный черновик сохраняет ответы
// плотной модели") and that selection must stay cheap (wispaper.ai, "Where the
// speedup claim holds").  The rule is this library's: per (sequence, KV head)
// keep the first n_sink and last n_recent pages, then the pages of largest
// mass up to B = min(P, max(ceil(budget * P - 1e-9), |mandatory|)) pages,
// equal mass -> lower page id; emit ascending.
//
// One warp per (sequence, KV head) (one CTA per pair when there are few
// pairs; see select_pages_cta_kernel).  The warp first stages its mass row in
// shared memory (coalesced loads, several in flight per lane); a 4-pass
// MSB-first radix select (8 bits a pass, warp-private 256-bin histogram in
// shared memory) then finds the K-th largest mass; ties at the threshold are
// ranked by page id with ballots; the chosen pages are compacted in ascending
// order with ballots.  Every pass after the load reads shared memory only.

#include <algorithm>

#include "s3r_device.cuh"

namespace s3r {

namespace {

constexpr int kSelWarps = 8;

__device__ __forceinline__ uint32_t mass_key(float m) {
  // Non-negative finite masses order like their bit patterns; anything else
  // (negative, -0, NaN) ranks lowest.
  return (m > 0.f && m < __builtin_huge_valf()) ? __float_as_uint(m) : 0u;
}

__global__ void __launch_bounds__(kSelWarps * 32)
    select_pages_kernel(const float* __restrict__ mass, const int32_t* __restrict__ sel_lens,
                        int n_pairs, int Hkv, int stride, double budget, int n_sink, int n_recent,
                        int32_t* __restrict__ sel_pages, int32_t* __restrict__ sel_count, int b_max,
                        int* err) {
  extern __shared__ int sel_smem[];
  const int warps = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x * warps + warp;
  if (pair >= n_pairs) return;
  int* hist = sel_smem + warp * 256;
  float* row = reinterpret_cast<float*>(sel_smem + warps * 256) + static_cast<int64_t>(warp) * stride;
  const int s = pair / Hkv;
  const float* grow = mass + static_cast<int64_t>(pair) * stride;
  int32_t* out = sel_pages + static_cast<int64_t>(pair) * b_max;

  const int len = __ldg(sel_lens + s);
  const int P = len >= 0 ? (len + kPage - 1) / kPage : -1;
  if (P < 0 || P > stride) {
    if (lane == 0) {
      report_error(err, S3R_DEVERR_BAD_LENGTH);
      sel_count[pair] = 0;
    }
    for (int i = lane; i < b_max; i += 32) out[i] = -1;
    return;
  }
  {
    int pg = lane;
    for (; pg + 15 * 32 < P; pg += 16 * 32) {   // 16 loads in flight per lane
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __ldg(grow + pg + j * 32);
#pragma unroll
      for (int j = 0; j < 16; ++j) row[pg + j * 32] = v[j];
    }
    for (; pg < P; pg += 32) row[pg] = __ldg(grow + pg);
    __syncwarp();
  }
  const int sink_end = min(n_sink, P);
  const int rec_start = max(P - n_recent, 0);
  const int n_mand = sink_end + (P - max(rec_start, sink_end));
  // fp64 with explicit rounding steps (no contraction), as the rule states.
  const double want = ceil(__dsub_rn(__dmul_rn(budget, static_cast<double>(P)), 1e-9));
  int B = static_cast<int>(fmin(static_cast<double>(P), fmax(want, static_cast<double>(n_mand))));
  if (B > b_max) {
    if (lane == 0) report_error(err, S3R_DEVERR_BAD_COUNT);
    B = b_max;
  }
  const int K = B - n_mand;   // extra pages to pick by mass
  auto mandatory = [&](int pg) { return pg < sink_end || pg >= rec_start; };

  uint32_t thresh = 0;
  int take_eq = 0;             // how many keys equal to thresh to take (lowest ids)
  const bool take_all = (B == P);
  if (!take_all && K > 0) {
    uint32_t prefix = 0, pmask = 0;
    int k_rem = K;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = lane; i < 256; i += 32) hist[i] = 0;
      __syncwarp();
      for (int pg = lane; pg < P; pg += 32) {
        if (mandatory(pg)) continue;
        const uint32_t key = mass_key(row[pg]);
        if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
      __syncwarp();
      // Lane l owns digits 255-8l .. 248-8l (descending); find the digit where
      // the count of larger-or-equal keys first reaches k_rem.
      int cnt[8];
      int local = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[255 - 8 * lane - j];
        local += cnt[j];
      }
      int incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int excl = incl - local;
      const unsigned ball = __ballot_sync(0xffffffffu, incl >= k_rem);
      const int owner = __ffs(ball) - 1;
      int digit = 0, above = 0;
      if (lane == owner) {
        int run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + cnt[j] >= k_rem) {
            digit = 255 - 8 * lane - j;
            above = run;
            break;
          }
          run += cnt[j];
        }
      }
      digit = __shfl_sync(0xffffffffu, digit, owner);
      above = __shfl_sync(0xffffffffu, above, owner);
      k_rem -= above;
      prefix |= static_cast<uint32_t>(digit) << shift;
      pmask |= 255u << shift;
      __syncwarp();
    }
    thresh = prefix;
    take_eq = k_rem;
  }

  // Compact the chosen pages in ascending order.
  int written = 0, eq_seen = 0;
  for (int base = 0; base < P; base += 32) {
    const int pg = base + lane;
    const bool in = pg < P;
    const bool cand = in && !take_all && K > 0 && !mandatory(pg);
    const uint32_t key = cand ? mass_key(row[pg]) : 0u;
    bool chosen = in && (take_all || mandatory(pg) || (cand && key > thresh));
    // Keys equal to the threshold: the lowest page ids first.
    const bool is_eq = cand && key == thresh;
    const unsigned eqb = __ballot_sync(0xffffffffu, is_eq);
    if (is_eq) chosen = eq_seen + __popc(eqb & ((1u << lane) - 1u)) < take_eq;
    eq_seen += __popc(eqb);
    const unsigned chb = __ballot_sync(0xffffffffu, chosen);
    const int slot = written + __popc(chb & ((1u << lane) - 1u));
    if (chosen && slot < b_max) out[slot] = pg;
    written += __popc(chb);
  }
  written = min(written, b_max);
  for (int i = written + lane; i < b_max; i += 32) out[i] = -1;
  if (lane == 0) sel_count[pair] = written;
}

// The same selection with one CTA of kSelCtaThreads threads per (sequence, KV
// head): the row is staged by the whole CTA, each radix pass histograms the
// candidates into one shared 256-bin histogram, warp 0 finds the digit, and
// the pages are compacted 256 at a time in page order (ballots within warps,
// counts across warps), so ties at the threshold go to the lowest page ids as
// in the warp version.  Results are identical; a pair's work is spread over 8
// warps instead of 1.
constexpr int kSelCtaThreads = 256;
// Pair counts below this take one CTA per pair (four per SM of the B300's 148).
constexpr int kSelCtaMaxPairs = 4 * 148;

__global__ void __launch_bounds__(kSelCtaThreads)
    select_pages_cta_kernel(const float* __restrict__ mass, const int32_t* __restrict__ sel_lens,
                            int n_pairs, int Hkv, int stride, double budget, int n_sink, int n_recent,
                            int32_t* __restrict__ sel_pages, int32_t* __restrict__ sel_count, int b_max,
                            int* err) {
  extern __shared__ int sel_smem[];
  __shared__ int s_hist[256];
  __shared__ int s_digit, s_above;
  __shared__ int s_weq[kSelCtaThreads / 32], s_wcnt[kSelCtaThreads / 32];
  constexpr int kW = kSelCtaThreads / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = blockIdx.x;
  if (pair >= n_pairs) return;
  float* row = reinterpret_cast<float*>(sel_smem);
  const int s = pair / Hkv;
  const float* grow = mass + static_cast<int64_t>(pair) * stride;
  int32_t* out = sel_pages + static_cast<int64_t>(pair) * b_max;

  const int len = __ldg(sel_lens + s);
  const int P = len >= 0 ? (len + kPage - 1) / kPage : -1;
  if (P < 0 || P > stride) {
    if (tid == 0) {
      report_error(err, S3R_DEVERR_BAD_LENGTH);
      sel_count[pair] = 0;
    }
    for (int i = tid; i < b_max; i += kSelCtaThreads) out[i] = -1;
    return;
  }
  for (int pg = tid; pg < P; pg += kSelCtaThreads) row[pg] = __ldg(grow + pg);
  __syncthreads();
  const int sink_end = min(n_sink, P);
  const int rec_start = max(P - n_recent, 0);
  const int n_mand = sink_end + (P - max(rec_start, sink_end));
  // fp64 with explicit rounding steps (no contraction), as the rule states.
  const double want = ceil(__dsub_rn(__dmul_rn(budget, static_cast<double>(P)), 1e-9));
  int B = static_cast<int>(fmin(static_cast<double>(P), fmax(want, static_cast<double>(n_mand))));
  if (B > b_max) {
    if (tid == 0) report_error(err, S3R_DEVERR_BAD_COUNT);
    B = b_max;
  }
  const int K = B - n_mand;   // extra pages to pick by mass
  auto mandatory = [&](int pg) { return pg < sink_end || pg >= rec_start; };

  uint32_t thresh = 0;
  int take_eq = 0;             // how many keys equal to thresh to take (lowest ids)
  const bool take_all = (B == P);
  if (!take_all && K > 0) {
    uint32_t prefix = 0, pmask = 0;
    int k_rem = K;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      s_hist[tid] = 0;
      __syncthreads();
      for (int pg = tid; pg < P; pg += kSelCtaThreads) {
        if (mandatory(pg)) continue;
        const uint32_t key = mass_key(row[pg]);
        if ((key & pmask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (warp == 0) {
        // Lane l owns digits 255-8l .. 248-8l (descending); the digit where the
        // count of larger-or-equal keys first reaches k_rem.
        int cnt[8];
        int local = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          cnt[j] = s_hist[255 - 8 * lane - j];
          local += cnt[j];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const int excl = incl - local;
        const unsigned ball = __ballot_sync(0xffffffffu, incl >= k_rem);
        const int owner = __ffs(ball) - 1;
        if (lane == owner) {
          int run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run + cnt[j] >= k_rem) {
              s_digit = 255 - 8 * lane - j;
              s_above = run;
              break;
            }
            run += cnt[j];
          }
        }
      }
      __syncthreads();
      const int digit = s_digit;
      k_rem -= s_above;
      prefix |= static_cast<uint32_t>(digit) << shift;
      pmask |= 255u << shift;
    }
    thresh = prefix;
    take_eq = k_rem;
  }

  // Compact the chosen pages in ascending order, 256 pages at a time.
  const unsigned lower = (1u << lane) - 1u;
  int written = 0, eq_seen = 0;
  for (int base = 0; base < P; base += kSelCtaThreads) {
    const int pg = base + tid;
    const bool in = pg < P;
    const bool cand = in && !take_all && K > 0 && !mandatory(pg);
    const uint32_t key = cand ? mass_key(row[pg]) : 0u;
    bool chosen = in && (take_all || mandatory(pg) || (cand && key > thresh));
    const bool is_eq = cand && key == thresh;
    const unsigned eqb = __ballot_sync(0xffffffffu, is_eq);
    if (lane == 0) s_weq[warp] = __popc(eqb);
    __syncthreads();
    int eq_before = 0, eq_total = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int c = s_weq[w];
      eq_before += w < warp ? c : 0;
      eq_total += c;
    }
    // Keys equal to the threshold: the lowest page ids first.
    if (is_eq) chosen = eq_seen + eq_before + __popc(eqb & lower) < take_eq;
    eq_seen += eq_total;
    const unsigned chb = __ballot_sync(0xffffffffu, chosen);
    if (lane == 0) s_wcnt[warp] = __popc(chb);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kW; ++w) {
      const int c = s_wcnt[w];
      before += w < warp ? c : 0;
      total += c;
    }
    const int slot = written + before + __popc(chb & lower);
    if (chosen && slot < b_max) out[slot] = pg;
    written += total;
    __syncthreads();
  }
  written = min(written, b_max);
  for (int i = written + tid; i < b_max; i += kSelCtaThreads) out[i] = -1;
  if (tid == 0) sel_count[pair] = written;
}

}  // namespace

cudaError_t launch_select_pages(const float* mass, const int32_t* sel_lens, int S, int Hkv,
                                int stride, double budget, int n_sink, int n_recent,
                                int32_t* sel_pages, int32_t* sel_count, int b_max, int* err,
                                cudaStream_t stream) {
  const int n_pairs = S * Hkv;
  if (n_pairs == 0) return cudaSuccess;
  // Few pairs leave most of the GPU idle with one warp per pair: give each
  // pair a CTA instead (256 pairs: 14.6 against 21.7 us; at 2048 pairs the
  // warp per pair is faster, 24.1 against 26.7 us).
  if (n_pairs < kSelCtaMaxPairs) {
    const size_t smem_cta = static_cast<size_t>(stride) * sizeof(float);
    if (smem_cta > (200u << 10)) return cudaErrorInvalidValue;
    if (smem_cta > (40u << 10)) {
      const cudaError_t e = cudaFuncSetAttribute(select_pages_cta_kernel,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem_cta));
      if (e != cudaSuccess) return e;
    }
    select_pages_cta_kernel<<<n_pairs, kSelCtaThreads, smem_cta, stream>>>(mass, sel_lens, n_pairs, Hkv, stride,
                                                                           budget, n_sink, n_recent, sel_pages,
                                                                           sel_count, b_max, err);
    return cudaGetLastError();
  }
  // Warps per CTA: as many as keep (histogram + staged row) per warp within
  // 96 KB of shared memory, so two CTAs fit on an SM.
  const size_t per_warp = 256 * sizeof(int) + static_cast<size_t>(stride) * sizeof(float);
  int warps = static_cast<int>(std::min<size_t>(kSelWarps, std::max<size_t>(1, (96u << 10) / per_warp)));
  const size_t smem = per_warp * warps;
  if (smem > (200u << 10)) return cudaErrorInvalidValue;
  if (smem > (48u << 10)) {
    const cudaError_t e = cudaFuncSetAttribute(select_pages_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int grid = (n_pairs + warps - 1) / warps;
  select_pages_kernel<<<grid, warps * 32, smem, stream>>>(mass, sel_lens, n_pairs, Hkv, stride, budget,
                                                          n_sink, n_recent, sel_pages, sel_count, b_max,
                                                          err);
  return cudaGetLastError();
}

}  // namespace s3r
