// Exact speculative sampling over the full vocabulary.
//
// The S³R pages: full-attention verification accepts or rejects the drafted
// tokens through exact speculative sampling, which keeps the output
// distributed as the dense policy (wispaper.ai, "S3R drafts sparsely and
// verifies densely"); after the first rejection the correcting token comes
// from the residual distribution (rit.work, "Как разреженный черновик
// сохраняет ответы плотной модели"; rebasdaily.com, "草稿可以稀疏，交卷必须完整").
//
// The steps, each parallel over rows or chunks of rows.  Each row is cut into
// 32 contiguous chunks.
//   row stats   one CTA per logit row (k+1 target rows and k draft rows per
//               sequence): the row max m and z = sum_v 2^((x_v - m) log2 e)
//               in one streaming pass with 16-byte loads; the bonus row p_k
//               also keeps its 32 chunk (max, sum) pairs, which are its chunk
//               masses;
//   ratio tests one warp per sequence: the k tests p_i(x_i)/q_i(x_i) against
//               Philox uniforms (fp64 ratio from fp32 row stats); a = the
//               first rejected position (k if none);
//   chunk sums  one CTA per (sequence, 8 chunks) of a sequence that rejected:
//               fp64 sums over each chunk of the residual max(0, p_a - q_a)
//               and of p_a (the fallback when the residual vanishes);
//   pick        one CTA per sequence: the chunk masses locate the chunk
//               holding u * Z; that chunk alone is scanned in token-id order
//               (fp32 sums over contiguous per-thread runs, fp64 prefix across
//               runs) to find the token.
// The parallel sampler runs them all in one launch (spec_fused_kernel): CTAs
// take tasks in ticket order, first every row of sequence 0, 1, ..., then the
// chunk sums of each sequence; the last row of a sequence to finish runs its
// ratio tests (and, if every draft was accepted, its bonus pick), and the last
// of its chunk-sum tasks its pick.  A sequence's chunk sums so re-read p_a and
// q_a while later sequences' rows still stream.
// With k = 0 there is nothing to test and the row is its own bonus row:
// bonus_sample streams each row with 4 CTAs, the last of which merges the
// chunk statistics and picks the token.
// The sequential variant replaces the row tasks and ratio tests by k + 1
// launches of seq_step, one per position, which read a sequence's rows only up
// to its first rejection; chunk_sum and pick then do the chunk sums and the
// pick as separate launches.

#include <cfloat>

#include "philox.cuh"
#include "s3r_device.cuh"
#include "spec_sample.cuh"

namespace s3r {

namespace {

constexpr int kStatThreads = 256;
constexpr double kLog2eD = 1.4426950408889634074;
// Tie windows of the optional tie counters: a ratio test with |u - p/q| at
// most kRatioTie, and an inverse-CDF pick whose target u * Z lies within
// kCdfTie * Z of an end of the chosen token's CDF interval.
constexpr double kRatioTie = 1e-6;
constexpr double kCdfTie = 1e-6;

// 2^((x - m) log2 e) with m pre-scaled: mlog2 = m * log2 e.
__device__ __forceinline__ float scaled_exp(float x, float mlog2) {
  return fast_exp2(fmaf(x, kLog2e, -mlog2));
}

__device__ __forceinline__ void merge_stats(float& m, float& z, float m2, float z2) {
  const float mn = fmaxf(m, m2);
  if (mn == -FLT_MAX * 2.f) return;   // both empty (-inf)
  const float a = m == mn ? 1.f : fast_exp2((m - mn) * kLog2e);
  const float b = m2 == mn ? 1.f : fast_exp2((m2 - mn) * kLog2e);
  z = z * a + z2 * b;
  m = mn;
}

// A row is also split over kRowParts CTAs of 8 warps, one warp per chunk.
constexpr int kRowParts = 4;
static_assert(kSampleChunks == kRowParts * (kStatThreads / 32), "one warp per chunk");

// Contiguous chunk `c` of a row of V tokens: [lo, hi).  The chunk length is a
// multiple of 4 so float4 loads stay aligned when V is.
__device__ __forceinline__ int chunk_len(int V) {
  return ((V + kSampleChunks - 1) / kSampleChunks + 3) & ~3;
}

// One warp streams x[lo, hi) once: the online maximum m and
// z = sum 2^((x - m) log2 e), merged across the warp (lane 0 holds the result).
template <bool VEC>
__device__ __forceinline__ float2 warp_chunk_stats(const float* __restrict__ x, int lo, int hi, int lane) {
  const float neg_inf = -__builtin_huge_valf();
  float m = neg_inf, z = 0.f;
  if (VEC) {
    const float4* x4 = reinterpret_cast<const float4*>(x + lo);
    const int n4 = (hi - lo) >> 2;
    for (int base = 0; base < n4; base += 4 * 32) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = base + j * 32 + lane;
        v[j] = idx < n4 ? __ldcs(x4 + idx) : make_float4(neg_inf, neg_inf, neg_inf, neg_inf);
      }
      float bm = neg_inf;
#pragma unroll
      for (int j = 0; j < 4; ++j) bm = fmaxf(bm, fmaxf(fmaxf(v[j].x, v[j].y), fmaxf(v[j].z, v[j].w)));
      if (bm > m) {
        z = m == neg_inf ? 0.f : z * fast_exp2((m - bm) * kLog2e);
        m = bm;
      }
      if (m == neg_inf) continue;
      const float ml = m * kLog2e;
      float bs = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        bs += (scaled_exp(v[j].x, ml) + scaled_exp(v[j].y, ml)) +
              (scaled_exp(v[j].z, ml) + scaled_exp(v[j].w, ml));
      z += bs;
    }
  } else {
    for (int base = lo; base < hi; base += 4 * 32) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = base + j * 32 + lane;
        v[j] = idx < hi ? __ldcs(x + idx) : neg_inf;
      }
      const float bm = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      if (bm > m) {
        z = m == neg_inf ? 0.f : z * fast_exp2((m - bm) * kLog2e);
        m = bm;
      }
      if (m == neg_inf) continue;
      const float ml = m * kLog2e;
      z += (scaled_exp(v[0], ml) + scaled_exp(v[1], ml)) + (scaled_exp(v[2], ml) + scaled_exp(v[3], ml));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    merge_stats(m, z, m2, z2);
  }
  return make_float2(m, z);
}

// The whole CTA streams row x once; warp w takes chunks w, w + 8, ...; the
// per-chunk (max, sum) land in s_c[kSampleChunks].  Ends with a barrier.
template <bool VEC>
__device__ __forceinline__ void block_chunk_stats(const float* __restrict__ x, int V, float2* s_c) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CL = chunk_len(V);
  for (int c = warp; c < kSampleChunks; c += kStatThreads / 32) {
    const int lo = min(c * CL, V), hi = min(lo + CL, V);
    const float2 s = warp_chunk_stats<VEC>(x, lo, hi, lane);
    if (lane == 0) s_c[c] = s;
  }
  __syncthreads();
}

// Warp-wide: lane c holds chunk c's (max, sum); the row's (max, sum) in lane 0.
__device__ __forceinline__ float2 merge_chunk_stats(float2 s) {
  float m = s.x, z = s.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    merge_stats(m, z, m2, z2);
  }
  return make_float2(m, z);
}

// Probability mass of a chunk from its statistics and the row's:
// z_c 2^((m_c - m) log2 e) / z, in fp64; 0 for an empty chunk (and for the
// undefined all -inf row).
__device__ __forceinline__ double chunk_mass(float2 c, float2 row) {
  const double v = static_cast<double>(c.y) *
                   exp2((static_cast<double>(c.x) - static_cast<double>(row.x)) * kLog2eD) /
                   static_cast<double>(row.y);
  return v > 0.0 ? v : 0.0;
}

// The row a sequence samples from, in probability space: the residual
// max(0, p(v) - q(v)) after a rejection, or p(v) itself for the bonus token
// (q == null).  One inline definition, so every kernel computes the same values.
struct SampleRow {
  const float* p;
  const float* q;
  float mp, izp, mq, izq;   // row max * log2 e and 1 / sum, target and draft
  __device__ __forceinline__ float prob(float lp) const { return scaled_exp(lp, mp) * izp; }
  __device__ __forceinline__ float resid(float pv, float lq) const {
    return q == nullptr ? pv : fmaxf(pv - scaled_exp(lq, mq) * izq, 0.f);
  }
  __device__ __forceinline__ float value(float lp, float lq) const { return resid(prob(lp), lq); }
  __device__ __forceinline__ float at(int v) const {
    return value(__ldg(p + v), q != nullptr ? __ldg(q + v) : 0.f);
  }
};

__device__ __forceinline__ SampleRow sample_row(const float* p, const float* q, const float2* stats,
                                                int N, int k, int V, int n, int a, bool use_p) {
  SampleRow row;
  const float2 sp = __ldcg(stats + static_cast<int64_t>(n) * (k + 1) + a);
  row.p = p + (static_cast<int64_t>(n) * (k + 1) + a) * V;
  row.mp = sp.x * kLog2e;
  row.izp = 1.f / sp.y;
  row.q = nullptr;
  row.mq = 0.f;
  row.izq = 0.f;
  if (a < k && !use_p) {
    const float2 sq = __ldcg(stats + static_cast<int64_t>(N) * (k + 1) + static_cast<int64_t>(n) * k + a);
    row.q = q + (static_cast<int64_t>(n) * k + a) * V;
    row.mq = sq.x * kLog2e;
    row.izq = 1.f / sq.y;
  }
  return row;
}

// p(x) / q(x) of one drafted token x, formed in fp64 from the fp32 logits
// p(x), q(x) and the rows' (max, sum).
__device__ __forceinline__ double draft_ratio(float lp, float lq, float2 sp, float2 sq) {
  const double e = (static_cast<double>(lp) - sp.x) - (static_cast<double>(lq) - sq.x);
  return exp2(e * kLog2eD) * static_cast<double>(sq.y) / static_cast<double>(sp.y);
}

// The ratio test: x is rejected unless u < p(x) / q(x).
__device__ __forceinline__ bool ratio_rejects(double ratio, float u) { return !(static_cast<double>(u) < ratio); }

// A ratio test whose uniform lies within kRatioTie of the ratio: a decision
// that rounding in the row statistics could flip.
__device__ __forceinline__ bool ratio_tie(double ratio, float u) {
  return fabs(static_cast<double>(u) - ratio) <= kRatioTie;
}

// One warp per sequence: the k ratio tests.  Draft x_i is accepted iff
// u(n, i-1, ACCEPT) < p_i(x_i) / q_i(x_i); the ratio is formed in fp64 from the
// fp32 logits and row statistics.  Writes a = index of the first rejection
// (k if none), the accepted drafts and the -1 padding after position a.  With
// ties != null, ties[0] gains the number of tests up to and including the
// first rejection whose uniform lies within kRatioTie of the ratio.
__device__ __forceinline__ int accept_sequence(const float* __restrict__ p, const float* __restrict__ q,
                                               const int32_t* __restrict__ drafts, int N, int k, int V,
                                               uint64_t seed, uint32_t offset, const float2* __restrict__ stats,
                                               int32_t* __restrict__ accept, int32_t* __restrict__ out_tokens,
                                               int32_t* __restrict__ n_accepted, int* err,
                                               uint32_t* __restrict__ ties, int n, int lane) {
  const int np_rows = N * (k + 1);
  int first = k;
  uint64_t tie_bits = 0;   // bit i: test i is a tie (k <= 64)
  for (int base = 0; base < k; base += 32) {
    const int i = base + lane;
    bool rej = false, tie = false;
    if (i < k) {
      const int x = __ldg(drafts + static_cast<int64_t>(n) * k + i);
      if (x < 0 || x >= V) {
        report_error(err, S3R_DEVERR_BAD_TOKEN);
        rej = true;
      } else {
        const double ratio = draft_ratio(__ldg(p + (static_cast<int64_t>(n) * (k + 1) + i) * V + x),
                                         __ldg(q + (static_cast<int64_t>(n) * k + i) * V + x),
                                         __ldcg(stats + static_cast<int64_t>(n) * (k + 1) + i),
                                         __ldcg(stats + np_rows + static_cast<int64_t>(n) * k + i));
        const float u = philox_uniform(seed, offset, n, i, kStreamAccept);
        rej = ratio_rejects(ratio, u);
        tie = ratio_tie(ratio, u);
      }
    }
    const unsigned b = __ballot_sync(0xffffffffu, rej);
    tie_bits |= static_cast<uint64_t>(__ballot_sync(0xffffffffu, tie)) << base;
    if (b != 0u && first == k) first = base + __ffs(b) - 1;
  }
  if (ties != nullptr && lane == 0) {
    const uint64_t upto = first >= 63 ? ~uint64_t{0} : ((uint64_t{1} << (first + 1)) - 1);
    const int c = __popcll(tie_bits & upto);
    if (c > 0) atomicAdd(ties, static_cast<uint32_t>(c));
  }
  int32_t* out = out_tokens + static_cast<int64_t>(n) * (k + 1);
  for (int i = lane; i <= k; i += 32) {
    if (i < first) out[i] = __ldg(drafts + static_cast<int64_t>(n) * k + i);
    else if (i > first) out[i] = -1;
  }
  if (lane == 0) {
    accept[n] = first;
    n_accepted[n] = first;
  }
  return first;
}

// s += x with Kahan compensation c (the sum is s - c).
__device__ __forceinline__ void kahan_add(float& s, float& c, float x) {
  const float y = x - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// One warp per chunk of a sequence that rejected a draft (kRowParts CTAs of 8
// warps per sequence): the sums over the chunk of the residual
// max(0, p_a - q_a) and of p_a itself (the fallback when the residual
// vanishes), fp32 over each 16-value batch, compensated across batches, fp64
// across lanes.  Sequences that accepted every draft sample the bonus row
// p_k, whose chunk masses the row statistics already hold: their CTAs return
// at once.  Coalesced 16-byte loads.
template <bool VEC>
__device__ __forceinline__ void residual_chunk_sums(const float* __restrict__ p, const float* __restrict__ q,
                                                   int N, int k, int V, const float2* __restrict__ stats,
                                                   double2* __restrict__ chunk_sums, int n, int part, int a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const SampleRow row = sample_row(p, q, stats, N, k, V, n, a, false);
  const int CL = chunk_len(V);
  const int c = part * (kStatThreads / 32) + warp;
  const int lo = min(c * CL, V), hi = min(lo + CL, V);
  float sr = 0.f, cr = 0.f, sp = 0.f, cp = 0.f;
  if (VEC) {
    const float4* p4 = reinterpret_cast<const float4*>(row.p + lo);
    const float4* q4 = reinterpret_cast<const float4*>(row.q + lo);
    const int n4 = (hi - lo) >> 2;
    const float neg_inf = -__builtin_huge_valf();
    for (int base = 0; base < n4; base += 4 * 32) {
      float4 lp[4], lq[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = base + j * 32 + lane;
        lp[j] = i < n4 ? __ldcs(p4 + i) : make_float4(neg_inf, neg_inf, neg_inf, neg_inf);
        lq[j] = i < n4 ? __ldcs(q4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float br = 0.f, bp = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float px = row.prob(lp[j].x), py = row.prob(lp[j].y);
        const float pz = row.prob(lp[j].z), pw = row.prob(lp[j].w);
        br += (row.resid(px, lq[j].x) + row.resid(py, lq[j].y)) +
              (row.resid(pz, lq[j].z) + row.resid(pw, lq[j].w));
        bp += (px + py) + (pz + pw);
      }
      kahan_add(sr, cr, br);
      kahan_add(sp, cp, bp);
    }
  } else {
    for (int base = lo; base < hi; base += 4 * 32) {
      float br = 0.f, bp = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = base + j * 32 + lane;
        if (v < hi) {
          const float pv = row.prob(__ldcs(row.p + v));
          br += row.resid(pv, __ldcs(row.q + v));
          bp += pv;
        }
      }
      kahan_add(sr, cr, br);
      kahan_add(sp, cp, bp);
    }
  }
  double dr = static_cast<double>(sr) - static_cast<double>(cr);
  double dp = static_cast<double>(sp) - static_cast<double>(cp);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dr += __shfl_xor_sync(0xffffffffu, dr, o);
    dp += __shfl_xor_sync(0xffffffffu, dp, o);
  }
  if (lane == 0) chunk_sums[static_cast<int64_t>(n) * kSampleChunks + c] = make_double2(dr, dp);
}

template <bool VEC>
__global__ void __launch_bounds__(kStatThreads)
    chunk_sum_kernel(const float* __restrict__ p, const float* __restrict__ q, int N, int k, int V,
                     const float2* __restrict__ stats, const int32_t* __restrict__ accept,
                     double2* __restrict__ chunk_sums) {
  const int n = blockIdx.x / kRowParts;
  const int part = blockIdx.x - n * kRowParts;
  const int a = __ldg(accept + n);
  if (a == k) return;
  residual_chunk_sums<VEC>(p, q, N, k, V, stats, chunk_sums, n, part, a);
}

// Warp-wide, lane c holding chunk c's mass v >= 0 (fp64): the chunk where the
// inverse CDF of u lands -- the first whose inclusive prefix (token order)
// exceeds u * Z, Z the last prefix; the last chunk with mass if rounding puts
// none past it; chunk 0 if every mass is 0 -- the target's offset into it, and Z.
__device__ __forceinline__ void choose_chunk(double v, double u, int lane, int& chunk, double& tgt, double& total) {
  double incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  total = __shfl_sync(0xffffffffu, incl, 31);
  const double target = u * total;
  const unsigned over = __ballot_sync(0xffffffffu, incl > target);
  const unsigned pos = __ballot_sync(0xffffffffu, v > 0.0);
  chunk = over != 0u ? __ffs(over) - 1 : (pos != 0u ? 31 - __clz(pos) : 0);
  const double prev = __shfl_sync(0xffffffffu, incl, chunk > 0 ? chunk - 1 : 0);
  tgt = target - (chunk > 0 ? prev : 0.0);
}

constexpr int kPickThreads = 256;
static_assert(kPickThreads == kStatThreads, "the bonus sampler runs both phases in one CTA");

struct PickSmem {
  double warp_tot[kPickThreads / 32];
  int owner, last, pick, tie;
};

// Block-wide inverse CDF inside chunk [lo, hi) of `row`: the first token whose
// running mass exceeds tgt, where the chunk is cut into contiguous per-thread
// runs summed in fp32 and prefix-summed across runs in fp64 (token order).
// The run holding the target is the last non-empty run whose exclusive prefix
// is <= tgt (thread 0's is 0, so one always is); its thread walks it again
// (the same values, now from L1).  When rounding leaves the target past that
// run, the run's last token with mass is taken, else the chunk's.  Nothing is
// staged in shared memory, so kernels that stream rows before picking keep
// their L1 for loads in flight.  Every thread returns the token.  sm.tie is
// set when the target lies within eps of either end of the picked token's
// interval of the running sum (or a rounding fallback picked it).
__device__ __forceinline__ int block_pick_in_chunk(const SampleRow& row, int lo, int hi, double tgt,
                                                   double eps, PickSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int len = hi - lo;
  if (tid == 0) {
    sm.owner = -1;
    sm.last = -1;
    sm.pick = -1;
    sm.tie = 0;
  }
  const int E = (len + kPickThreads - 1) / kPickThreads;
  const int r0 = min(lo + tid * E, hi), r1 = min(r0 + E, hi);
  float part = 0.f;
  int my_last = -1;
  for (int v0 = r0; v0 < r1; v0 += 8) {
    float lp[8], lq[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const bool in = v0 + j < r1;
      lp[j] = in ? __ldg(row.p + v0 + j) : -__builtin_huge_valf();
      lq[j] = (in && row.q != nullptr) ? __ldg(row.q + v0 + j) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float r = row.value(lp[j], lq[j]);
      part += r;
      if (r > 0.f) my_last = v0 + j;
    }
  }
  // Exclusive fp64 prefix of the run sums in thread order.
  double incl = static_cast<double>(part);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  double excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.0;
  if (lane == 31) sm.warp_tot[warp] = incl;
  __syncthreads();
  if (my_last >= 0) atomicMax(&sm.last, my_last);
  for (int w = 0; w < warp; ++w) excl += sm.warp_tot[w];
  if (r0 < r1 && excl <= tgt) atomicMax(&sm.owner, tid);
  __syncthreads();
  if (tid == sm.owner) {
    const double rem = tgt - excl;
    float run = 0.f;
    int pick = -1;
    bool tie = true;   // a rounding fallback is a boundary case
    for (int v = r0; v < r1; ++v) {
      const float r = row.at(v);
      const float before = run;
      run += r;
      if (r > 0.f && static_cast<double>(run) > rem) {
        pick = v;
        tie = static_cast<double>(run) - rem <= eps || rem - static_cast<double>(before) <= eps;
        break;
      }
    }
    sm.pick = pick >= 0 ? pick : my_last;
    sm.tie = tie ? 1 : 0;
  }
  __syncthreads();
  const int tok = sm.pick >= 0 ? sm.pick : (sm.last >= 0 ? sm.last : lo);
  return tok < hi ? tok : hi - 1;
}

// One CTA per sequence after the ratio tests: the 32 chunk masses (the
// residual's, or p_a's when the residual vanishes, or the bonus row's from its
// chunk statistics) locate the chunk holding u * Z; that chunk is scanned in
// token-id order.
// Block-wide (every thread of the CTA): sequence n's token at position a.
__device__ __forceinline__ void pick_sequence(const float* __restrict__ p, const float* __restrict__ q, int N,
                                              int k, int V, uint64_t seed, uint32_t offset,
                                              const float2* __restrict__ stats,
                                              const float2* __restrict__ bonus_chunks, int a,
                                              const double2* __restrict__ chunk_sums,
                                              int32_t* __restrict__ out_tokens, uint32_t* __restrict__ ties,
                                              int n) {
  __shared__ PickSmem sm;
  __shared__ int s_chunk, s_use_p;
  __shared__ double s_tgt, s_eps;
  const int tid = threadIdx.x;
  if (tid < 32) {
    double2 cs;
    if (a == k) {
      const double v = chunk_mass(__ldcg(bonus_chunks + static_cast<int64_t>(n) * kSampleChunks + tid),
                                  __ldcg(stats + static_cast<int64_t>(n) * (k + 1) + k));
      cs = make_double2(v, v);
    } else {
      cs = __ldcg(chunk_sums + static_cast<int64_t>(n) * kSampleChunks + tid);
    }
    double zr = cs.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) zr += __shfl_xor_sync(0xffffffffu, zr, o);
    const bool use_p = (a == k) || !(zr > 0.0);
    double v = use_p ? cs.y : cs.x;
    v = v > 0.0 ? v : 0.0;
    // the uniform of counter (n, a, RESAMPLE, offset)
    const double u = static_cast<double>(philox_uniform(seed, offset, n, a, kStreamResample));
    int chunk;
    double tgt, total;
    choose_chunk(v, u, tid, chunk, tgt, total);
    if (tid == 0) {
      s_chunk = chunk;
      s_use_p = use_p ? 1 : 0;
      s_tgt = tgt;
      s_eps = kCdfTie * total;
    }
  }
  __syncthreads();
  const SampleRow row = sample_row(p, q, stats, N, k, V, n, a, s_use_p != 0);
  const int CL = chunk_len(V);
  const int lo = min(s_chunk * CL, V), hi = min(lo + CL, V);
  const int tok = block_pick_in_chunk(row, lo, hi, s_tgt, s_eps, sm);
  if (tid == 0) {
    out_tokens[static_cast<int64_t>(n) * (k + 1) + a] = tok;
    if (ties != nullptr && sm.tie) atomicAdd(ties + 1, 1u);
  }
}

__global__ void __launch_bounds__(kPickThreads)
    pick_kernel(const float* __restrict__ p, const float* __restrict__ q, int N, int k, int V,
                uint64_t seed, uint32_t offset, const float2* __restrict__ stats,
                const float2* __restrict__ bonus_chunks, const int32_t* __restrict__ accept,
                const double2* __restrict__ chunk_sums, int32_t* __restrict__ out_tokens,
                uint32_t* __restrict__ ties) {
  const int n = blockIdx.x;
  pick_sequence(p, q, N, k, V, seed, offset, stats, bonus_chunks, __ldg(accept + n), chunk_sums, out_tokens, ties,
                n);
}

// Rows split over CTAs: each of kRowParts CTAs streams 8 chunks of a row (one
// warp per chunk) and stores their (max, sum) pairs; the CTA that arrives
// last on the sequence's counter (the stores published by a fence before the
// arrival) merges the pairs, acts for the sequence and resets the counter.
// The chunk pairs and their merge are those of the one-launch sampler's row
// tasks (block_chunk_stats, merge_chunk_stats), so the row statistics are
// bitwise the same on every path.

// This CTA's 8 chunks of row x into dst[kSampleChunks]; true in every thread
// of the CTA that arrived last among `arrivals_expected` on *counter.
template <bool VEC>
__device__ __forceinline__ bool split_chunks_arrive(const float* __restrict__ x, int V, int part,
                                                    float2* __restrict__ dst, int* counter,
                                                    int arrivals_expected) {
  __shared__ int s_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int CL = chunk_len(V);
  const int c = part * (kStatThreads / 32) + warp;
  const int lo = min(c * CL, V), hi = min(lo + CL, V);
  const float2 s = warp_chunk_stats<VEC>(x, lo, hi, lane);
  if (lane == 0) dst[c] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    fence_acq_rel_gpu();
    s_last = atomicAdd(counter, 1) == arrivals_expected - 1;
  }
  __syncthreads();
  const bool last = s_last != 0;
  if (last) fence_acq_rel_gpu();
  return last;
}

// k = 0: one token per sequence from softmax(p_n) (row n at p + n * row_stride,
// token n at out_tokens[n * token_stride]), kRowParts CTAs per row;
// the last to arrive takes the chunk holding u * Z from the merged chunk
// statistics and scans it.  The uniform is the one of counter
// (n, u_pos, u_stream, offset).  Writes n_accepted[n] = 0.
template <bool VEC>
__global__ void __launch_bounds__(kStatThreads)
    bonus_sample_kernel(const float* __restrict__ p, int V, int64_t row_stride, uint64_t seed, uint32_t offset,
                        uint32_t u_stream, int u_pos, float2* __restrict__ chunks, int* __restrict__ arrivals,
                        int32_t* __restrict__ out_tokens, int64_t token_stride,
                        int32_t* __restrict__ n_accepted, uint32_t* __restrict__ ties) {
  __shared__ PickSmem sm;
  __shared__ float2 s_row;
  __shared__ int s_chunk;
  __shared__ double s_tgt, s_eps;
  const int n = blockIdx.x / kRowParts;
  const int part = blockIdx.x - n * kRowParts;
  const int tid = threadIdx.x;
  const float* x = p + static_cast<int64_t>(n) * row_stride;
  float2* cs_n = chunks + static_cast<int64_t>(n) * kSampleChunks;
  if (!split_chunks_arrive<VEC>(x, V, part, cs_n, arrivals + n, kRowParts)) return;
  if (tid < 32) {
    const float2 cs = __ldcg(cs_n + tid);
    float2 r = merge_chunk_stats(cs);
    r.x = __shfl_sync(0xffffffffu, r.x, 0);
    r.y = __shfl_sync(0xffffffffu, r.y, 0);
    const double u = static_cast<double>(philox_uniform(seed, offset, n, u_pos, u_stream));
    int chunk;
    double tgt, total;
    choose_chunk(chunk_mass(cs, r), u, tid, chunk, tgt, total);
    if (tid == 0) {
      s_chunk = chunk;
      s_tgt = tgt;
      s_eps = kCdfTie * total;
      s_row = r;
      arrivals[n] = 0;
      n_accepted[n] = 0;
    }
  }
  __syncthreads();
  SampleRow row;
  row.p = x;
  row.q = nullptr;
  row.mp = s_row.x * kLog2e;
  row.izp = 1.f / s_row.y;
  row.mq = 0.f;
  row.izq = 0.f;
  const int CL = chunk_len(V);
  const int lo = min(s_chunk * CL, V), hi = min(lo + CL, V);
  const int tok = block_pick_in_chunk(row, lo, hi, s_tgt, s_eps, sm);
  if (tid == 0) {
    out_tokens[static_cast<int64_t>(n) * token_stride] = tok;
    if (ties != nullptr && sm.tie) atomicAdd(ties + 1, 1u);
  }
}

// Step i of the sequential (early-exit) ratio tests.  For i < k the rows p_i
// and q_i of every sequence that has not rejected yet (accept[n] == k) are
// streamed, kRowParts CTAs each; the last CTA merges both rows' statistics,
// stores them where the one-launch sampler's row tasks do, and tests draft i.  For i == k the bonus
// row p_k of every sequence that accepted all k drafts is streamed and its
// chunk statistics kept for the pick.  A sequence is finished at its
// rejection (or at i == k): accepted drafts, -1 padding and n_accepted are
// written then.  Sequences that rejected earlier return at once, so no row
// after a sequence's first rejection is read.
template <bool VEC>
__global__ void __launch_bounds__(kStatThreads)
    seq_step_kernel(const float* __restrict__ p, const float* __restrict__ q,
                    const int32_t* __restrict__ drafts, int N, int k, int V, int i, uint64_t seed,
                    uint32_t offset, float2* __restrict__ stats, float2* __restrict__ pchunks,
                    float2* __restrict__ qchunks, int32_t* accept, int* __restrict__ arrivals,
                    int32_t* __restrict__ out_tokens, int32_t* __restrict__ n_accepted, int* err,
                    uint32_t* __restrict__ ties) {
  const int rows = i < k ? 2 : 1;
  const int per_seq = rows * kRowParts;
  const int n = blockIdx.x / per_seq;
  const int rem = blockIdx.x - n * per_seq;
  const int which = rem / kRowParts;      // 0: p_i, 1: q_i
  const int part = rem - which * kRowParts;
  if (i > 0 && accept[n] != k) return;    // rejected at an earlier position
  const float* x = which == 0 ? p + (static_cast<int64_t>(n) * (k + 1) + i) * V
                              : q + (static_cast<int64_t>(n) * k + i) * V;
  float2* pc = pchunks + static_cast<int64_t>(n) * kSampleChunks;
  float2* qc = qchunks + static_cast<int64_t>(n) * kSampleChunks;
  if (!split_chunks_arrive<VEC>(x, V, part, which == 0 ? pc : qc, arrivals + n, per_seq)) return;
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  const float2 rp = merge_chunk_stats(__ldcg(pc + lane));
  float2 rq = make_float2(0.f, 0.f);
  if (i < k) rq = merge_chunk_stats(__ldcg(qc + lane));
  int first = k;
  if (lane == 0) {
    arrivals[n] = 0;
    stats[static_cast<int64_t>(n) * (k + 1) + i] = rp;
    if (i < k) {
      stats[static_cast<int64_t>(N) * (k + 1) + static_cast<int64_t>(n) * k + i] = rq;
      const int x_i = __ldg(drafts + static_cast<int64_t>(n) * k + i);
      bool rej = true;
      if (x_i < 0 || x_i >= V) {
        report_error(err, S3R_DEVERR_BAD_TOKEN);
      } else {
        const double ratio = draft_ratio(__ldg(p + (static_cast<int64_t>(n) * (k + 1) + i) * V + x_i),
                                         __ldg(q + (static_cast<int64_t>(n) * k + i) * V + x_i), rp, rq);
        const float u = philox_uniform(seed, offset, n, i, kStreamAccept);
        rej = ratio_rejects(ratio, u);
        if (ties != nullptr && ratio_tie(ratio, u)) atomicAdd(ties, 1u);
      }
      first = rej ? i : k;
      accept[n] = first;
    }
  }
  first = __shfl_sync(0xffffffffu, first, 0);
  if (i == k || first == i) {
    int32_t* out = out_tokens + static_cast<int64_t>(n) * (k + 1);
    for (int j = lane; j <= k; j += 32) {
      if (j < first) out[j] = __ldg(drafts + static_cast<int64_t>(n) * k + j);
      else if (j > first) out[j] = -1;
    }
    if (lane == 0) n_accepted[n] = first;
  }
}

__device__ __forceinline__ int ld_acquire_gpu(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(int* ptr, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// The parallel sampler in one launch.  Each CTA takes a ticket; tickets
// [0, N(2k+1)) are the rows, sequence-major (p_0..p_k, then q_0..q_{k-1} of
// sequence 0, then of sequence 1, ...), and the next N * kRowParts tickets the
// chunk-sum tasks of sequence 0, 1, ....  Row task: the row's statistics (and
// the bonus row's chunk statistics); the last of a sequence's 2k+1 rows to
// finish runs the ratio tests, picks the bonus token if every draft was
// accepted, and marks the sequence ready.  Chunk-sum task: waits until its
// sequence is ready -- every row task holds a lower ticket, so it has started
// and waits on nothing, and the wait ends -- then sums its 8 chunks of the
// residual row a (nothing if a == k); the last of the sequence's tasks picks
// the token and clears the sequence's counters.  The last CTA to finish clears
// the ticket.  The arithmetic of every step is that of the separate kernels.
template <bool VEC>
__global__ void __launch_bounds__(kStatThreads)
    spec_fused_kernel(const float* __restrict__ p, const float* __restrict__ q, const int32_t* __restrict__ drafts,
                      int N, int k, int V, uint64_t seed, uint32_t offset, float2* __restrict__ stats,
                      float2* __restrict__ bonus, int32_t* __restrict__ accept, double2* __restrict__ chunk_sums,
                      int32_t* __restrict__ out_tokens, int32_t* __restrict__ n_accepted, int* err,
                      uint32_t* __restrict__ ties, int* __restrict__ row_arrive, int* __restrict__ res_arrive,
                      int* __restrict__ ready, int* __restrict__ ticket) {
  __shared__ int s_task, s_flag, s_first;
  __shared__ float2 s_c[kSampleChunks];
  const int tid = threadIdx.x;
  if (tid == 0) s_task = atomicAdd(ticket, 1);
  __syncthreads();
  const int task = s_task;
  const int R = 2 * k + 1;
  const int row_tasks = N * R;
  if (task < row_tasks) {
    const int n = task / R, r = task - (task / R) * R;
    const bool is_p = r <= k;
    const int64_t row = is_p ? static_cast<int64_t>(n) * (k + 1) + r
                             : static_cast<int64_t>(N) * (k + 1) + static_cast<int64_t>(n) * k + (r - k - 1);
    const float* x = is_p ? p + (static_cast<int64_t>(n) * (k + 1) + r) * V
                          : q + (static_cast<int64_t>(n) * k + (r - k - 1)) * V;
    block_chunk_stats<VEC>(x, V, s_c);
    if (tid < 32) {
      const float2 cs = s_c[tid];
      const float2 rr = merge_chunk_stats(cs);
      if (tid == 0) stats[row] = rr;
      if (r == k) bonus[static_cast<int64_t>(n) * kSampleChunks + tid] = cs;
    }
    __syncthreads();
    if (tid == 0) {
      fence_acq_rel_gpu();
      s_flag = atomicAdd(row_arrive + n, 1) == R - 1;
    }
    __syncthreads();
    if (s_flag) {
      fence_acq_rel_gpu();
      if (tid < 32) {
        const int first = accept_sequence(p, q, drafts, N, k, V, seed, offset, stats, accept, out_tokens,
                                          n_accepted, err, ties, n, tid);
        if (tid == 0) s_first = first;
      }
      __syncthreads();
      if (s_first == k) pick_sequence(p, q, N, k, V, seed, offset, stats, bonus, k, chunk_sums, out_tokens, ties, n);
      if (tid == 0) {
        row_arrive[n] = 0;
        fence_acq_rel_gpu();
        st_release_gpu(ready + n, 1);
      }
    }
  } else {
    const int rt = task - row_tasks;
    const int n = rt / kRowParts, part = rt - (rt / kRowParts) * kRowParts;
    if (tid == 0) {
      int ok = 0;
      for (uint32_t i = 0; i < kMaxSpin; ++i) {
        if (ld_acquire_gpu(ready + n) != 0) {
          ok = 1;
          break;
        }
        __nanosleep(256);
      }
      if (!ok) report_error(err, S3R_DEVERR_TIMEOUT);
      s_flag = ok;
    }
    __syncthreads();
    const int ok = s_flag;
    fence_acq_rel_gpu();
    const int a = ok ? __ldcg(accept + n) : k;
    if (a < k) residual_chunk_sums<VEC>(p, q, N, k, V, stats, chunk_sums, n, part, a);
    __syncthreads();
    if (tid == 0) {
      fence_acq_rel_gpu();
      s_flag = atomicAdd(res_arrive + n, 1) == kRowParts - 1;
    }
    __syncthreads();
    if (s_flag) {
      fence_acq_rel_gpu();
      if (a < k) pick_sequence(p, q, N, k, V, seed, offset, stats, bonus, a, chunk_sums, out_tokens, ties, n);
      if (tid == 0) {
        res_arrive[n] = 0;
        ready[n] = 0;
      }
    }
  }
  if (tid == 0 && atomicAdd(ticket + 1, 1) == static_cast<int>(gridDim.x) - 1) {
    ticket[0] = 0;
    ticket[1] = 0;
  }
}

// chunk_sum then pick, after the ratio tests have set accept[] and the stats.
cudaError_t launch_residual_pick(const float* p, const float* q, int N, int k, int V, uint64_t seed,
                                 uint32_t offset, const float2* stats, const float2* bonus,
                                 const int32_t* accept, double2* chunks, int32_t* out_tokens, bool vec,
                                 uint32_t* ties, cudaStream_t stream) {
  const unsigned chunk_blocks = static_cast<unsigned>(static_cast<int64_t>(N) * kRowParts);
  if (vec) {
    chunk_sum_kernel<true><<<chunk_blocks, kStatThreads, 0, stream>>>(p, q, N, k, V, stats, accept, chunks);
  } else {
    chunk_sum_kernel<false><<<chunk_blocks, kStatThreads, 0, stream>>>(p, q, N, k, V, stats, accept, chunks);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pick_kernel<<<N, kPickThreads, 0, stream>>>(p, q, N, k, V, seed, offset, stats, bonus, accept, chunks,
                                              out_tokens, ties);
  return cudaGetLastError();
}

}  // namespace

SpecWorkspaceLayout spec_workspace_layout(int64_t N, int k) {
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SpecWorkspaceLayout L{};
  L.err_off = 0;
  L.stats_off = 256;
  L.accept_off = L.stats_off + al(static_cast<size_t>(N) * (2 * k + 1) * sizeof(float2));
  L.chunk_off = L.accept_off + al(static_cast<size_t>(N) * sizeof(int32_t));
  L.bonus_off = L.chunk_off + al(static_cast<size_t>(N) * kSampleChunks * sizeof(double2));
  L.arrive_off = L.bonus_off + al(static_cast<size_t>(N) * kSampleChunks * sizeof(float2));
  L.res_arrive_off = L.arrive_off + static_cast<size_t>(N) * sizeof(int);
  L.ready_off = L.res_arrive_off + static_cast<size_t>(N) * sizeof(int);
  L.ticket_off = L.ready_off + static_cast<size_t>(N) * sizeof(int);
  L.total = al(L.ticket_off + 2 * sizeof(int));
  return L;
}

cudaError_t launch_spec_sample(const float* p, const float* q, const int32_t* drafts, int N, int k,
                               int V, uint64_t seed, uint32_t offset, void* ws,
                               int32_t* out_tokens, int32_t* n_accepted, cudaStream_t stream,
                               uint32_t u_stream, int u_pos, int64_t row_stride, int64_t token_stride,
                               uint32_t* ties) {
  if (N == 0) return cudaSuccess;
  const SpecWorkspaceLayout L = spec_workspace_layout(N, k);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w + L.err_off);
  float2* stats = reinterpret_cast<float2*>(w + L.stats_off);
  int32_t* accept = reinterpret_cast<int32_t*>(w + L.accept_off);
  double2* chunks = reinterpret_cast<double2*>(w + L.chunk_off);
  float2* bonus = reinterpret_cast<float2*>(w + L.bonus_off);
  int* arrivals = reinterpret_cast<int*>(w + L.arrive_off);
  const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                   (k == 0 || reinterpret_cast<uintptr_t>(q) % 16 == 0);
  if (k == 0) {
    const int pos = u_pos >= 0 ? u_pos : 0;
    const int64_t stride = row_stride > 0 ? row_stride : V;
    const bool vec0 = vec && stride % 4 == 0;
    const unsigned blocks = static_cast<unsigned>(static_cast<int64_t>(N) * kRowParts);
    if (vec0) {
      bonus_sample_kernel<true><<<blocks, kStatThreads, 0, stream>>>(p, V, stride, seed, offset, u_stream, pos,
                                                                     bonus, arrivals, out_tokens, token_stride,
                                                                     n_accepted, ties);
    } else {
      bonus_sample_kernel<false><<<blocks, kStatThreads, 0, stream>>>(p, V, stride, seed, offset, u_stream, pos,
                                                                      bonus, arrivals, out_tokens, token_stride,
                                                                      n_accepted, ties);
    }
    return cudaGetLastError();
  }
  int* res_arrive = reinterpret_cast<int*>(w + L.res_arrive_off);
  int* ready = reinterpret_cast<int*>(w + L.ready_off);
  int* ticket = reinterpret_cast<int*>(w + L.ticket_off);
  const unsigned blocks = static_cast<unsigned>(static_cast<int64_t>(N) * (2 * k + 1 + kRowParts));
  if (vec) {
    spec_fused_kernel<true><<<blocks, kStatThreads, 0, stream>>>(p, q, drafts, N, k, V, seed, offset, stats, bonus,
                                                                 accept, chunks, out_tokens, n_accepted, err, ties,
                                                                 arrivals, res_arrive, ready, ticket);
  } else {
    spec_fused_kernel<false><<<blocks, kStatThreads, 0, stream>>>(p, q, drafts, N, k, V, seed, offset, stats,
                                                                  bonus, accept, chunks, out_tokens, n_accepted, err,
                                                                  ties, arrivals, res_arrive, ready, ticket);
  }
  return cudaGetLastError();
}

cudaError_t launch_spec_sample_sequential(const float* p, const float* q, const int32_t* drafts, int N, int k,
                                          int V, uint64_t seed, uint32_t offset, void* ws,
                                          int32_t* out_tokens, int32_t* n_accepted, cudaStream_t stream,
                                          uint32_t* ties) {
  if (N == 0) return cudaSuccess;
  if (k == 0)
    return launch_spec_sample(p, q, drafts, N, k, V, seed, offset, ws, out_tokens, n_accepted, stream, 1, -1, 0, 1,
                              ties);
  const SpecWorkspaceLayout L = spec_workspace_layout(N, k);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w + L.err_off);
  float2* stats = reinterpret_cast<float2*>(w + L.stats_off);
  int32_t* accept = reinterpret_cast<int32_t*>(w + L.accept_off);
  double2* chunks = reinterpret_cast<double2*>(w + L.chunk_off);
  // the draft rows' chunk statistics live in the chunk-sum area until the
  // residual chunk sums overwrite it after the last step
  float2* qchunks = reinterpret_cast<float2*>(chunks);
  float2* bonus = reinterpret_cast<float2*>(w + L.bonus_off);
  int* arrivals = reinterpret_cast<int*>(w + L.arrive_off);
  const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(q) % 16 == 0);
  for (int i = 0; i <= k; ++i) {
    const unsigned blocks = static_cast<unsigned>(static_cast<int64_t>(N) * (i < k ? 2 : 1) * kRowParts);
    if (vec) {
      seq_step_kernel<true><<<blocks, kStatThreads, 0, stream>>>(p, q, drafts, N, k, V, i, seed, offset, stats,
                                                                 bonus, qchunks, accept, arrivals, out_tokens,
                                                                 n_accepted, err, ties);
    } else {
      seq_step_kernel<false><<<blocks, kStatThreads, 0, stream>>>(p, q, drafts, N, k, V, i, seed, offset, stats,
                                                                  bonus, qchunks, accept, arrivals, out_tokens,
                                                                  n_accepted, err, ties);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_residual_pick(p, q, N, k, V, seed, offset, stats, bonus, accept, chunks, out_tokens, vec, ties,
                              stream);
}

}  // namespace s3r
