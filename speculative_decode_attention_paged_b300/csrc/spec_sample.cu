// Exact speculative sampling over the full vocabulary.
//
// The S³R pages: full-attention verification accepts or rejects the drafted
// tokens through exact speculative sampling, which keeps the output
// distributed as the dense policy (wispaper.ai, "S3R drafts sparsely and
// verifies densely"); after the first rejection the correcting token comes
// from the residual distribution (rit.work, "Как разреженный черновик
// сохраняет ответы плотной модели"; rebasdaily.com, "草稿可以稀疏，交卷必须完整").
//
// Four kernels, all parallel over rows or chunks of rows:
//   row_stats   one CTA per logit row (k+1 target rows and k draft rows per
//               sequence): the row max m and z = sum_v 2^((x_v - m) log2 e),
//               one streaming pass with 16-byte loads;
//   accept      one warp per sequence: the k ratio tests p_i(x_i)/q_i(x_i)
//               against Philox uniforms (fp64 ratio from fp32 row stats);
//               a = the first rejected position (k if none);
//   chunk_sum   one CTA per (sequence, chunk of the row): fp64 sums over the
//               chunk of the residual max(0, p_a - q_a) (or of p_k for the
//               bonus token) and of p_a (the fallback when the residual
//               vanishes);
//   pick        one CTA per sequence: the chunk sums locate the chunk holding
//               u * Z; that chunk alone is scanned in token-id order (fp64
//               prefix over contiguous per-thread runs) to find the token.

#include <cfloat>

#include "philox.cuh"
#include "s3r_device.cuh"
#include "spec_sample.cuh"

namespace s3r {

namespace {

constexpr int kStatThreads = 256;
constexpr double kLog2eD = 1.4426950408889634074;

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

template <bool VEC>
__global__ void __launch_bounds__(kStatThreads)
    row_stats_kernel(const float* __restrict__ p, const float* __restrict__ q, int N, int k, int V,
                     float2* __restrict__ stats) {
  const int row = blockIdx.x;
  const int np = N * (k + 1);
  const float* x = row < np ? p + static_cast<int64_t>(row) * V
                            : q + static_cast<int64_t>(row - np) * V;
  const int tid = threadIdx.x;
  const float neg_inf = -__builtin_huge_valf();
  float m = neg_inf, z = 0.f;
  if (VEC) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int n4 = V >> 2;
    for (int base = 0; base < n4; base += 4 * kStatThreads) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = base + j * kStatThreads + tid;
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
    for (int base = 0; base < V; base += 4 * kStatThreads) {
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = base + j * kStatThreads + tid;
        v[j] = idx < V ? __ldcs(x + idx) : neg_inf;
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
  // Block reduction of (m, z).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
    merge_stats(m, z, m2, z2);
  }
  __shared__ float sm[kStatThreads / 32], sz[kStatThreads / 32];
  if ((tid & 31) == 0) {
    sm[tid >> 5] = m;
    sz[tid >> 5] = z;
  }
  __syncthreads();
  if (tid == 0) {
    float M = sm[0], Z = sz[0];
    for (int w = 1; w < kStatThreads / 32; ++w) merge_stats(M, Z, sm[w], sz[w]);
    stats[row] = make_float2(M, Z);
  }
}

// The row a sequence samples from, in probability space: the residual
// max(0, p(v) - q(v)) after a rejection, or p(v) itself for the bonus token
// (q == null).  One inline function, so every kernel computes the same values.
struct SampleRow {
  const float* p;
  const float* q;
  float mp, izp, mq, izq;   // row max * log2 e and 1 / sum, target and draft
  __device__ __forceinline__ float value(float lp, float lq) const {
    const float pv = scaled_exp(lp, mp) * izp;
    if (q == nullptr) return pv;
    return fmaxf(pv - scaled_exp(lq, mq) * izq, 0.f);
  }
  __device__ __forceinline__ float at(int v) const {
    return value(__ldg(p + v), q != nullptr ? __ldg(q + v) : 0.f);
  }
};

__device__ __forceinline__ SampleRow sample_row(const float* p, const float* q, const float2* stats,
                                                int N, int k, int V, int n, int a, bool use_p) {
  SampleRow row;
  const float2 sp = stats[static_cast<int64_t>(n) * (k + 1) + a];
  row.p = p + (static_cast<int64_t>(n) * (k + 1) + a) * V;
  row.mp = sp.x * kLog2e;
  row.izp = 1.f / sp.y;
  row.q = nullptr;
  row.mq = 0.f;
  row.izq = 0.f;
  if (a < k && !use_p) {
    const float2 sq = stats[static_cast<int64_t>(N) * (k + 1) + static_cast<int64_t>(n) * k + a];
    row.q = q + (static_cast<int64_t>(n) * k + a) * V;
    row.mq = sq.x * kLog2e;
    row.izq = 1.f / sq.y;
  }
  return row;
}

// Contiguous chunk `c` of a row of V tokens: [lo, hi).  The chunk length is a
// multiple of 4 so float4 loads stay aligned when V is.
__device__ __forceinline__ int chunk_len(int V) {
  return ((V + kSampleChunks - 1) / kSampleChunks + 3) & ~3;
}

// One warp per sequence: the k ratio tests.  Draft x_i is accepted iff
// u(n, i-1, ACCEPT) < p_i(x_i) / q_i(x_i); the ratio is formed in fp64 from the
// fp32 logits and row statistics.  Writes a = index of the first rejection
// (k if none), the accepted drafts and the -1 padding after position a.
__global__ void __launch_bounds__(256)
    accept_kernel(const float* __restrict__ p, const float* __restrict__ q,
                  const int32_t* __restrict__ drafts, int N, int k, int V, uint64_t seed,
                  uint32_t offset, const float2* __restrict__ stats, int32_t* __restrict__ accept,
                  int32_t* __restrict__ out_tokens, int32_t* __restrict__ n_accepted, int* err) {
  const int lane = threadIdx.x & 31;
  const int n = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (n >= N) return;
  const int np_rows = N * (k + 1);
  int first = k;
  for (int base = 0; base < k; base += 32) {
    const int i = base + lane;
    bool rej = false;
    if (i < k) {
      const int x = __ldg(drafts + static_cast<int64_t>(n) * k + i);
      if (x < 0 || x >= V) {
        report_error(err, S3R_DEVERR_BAD_TOKEN);
        rej = true;
      } else {
        const float lp = __ldg(p + (static_cast<int64_t>(n) * (k + 1) + i) * V + x);
        const float lq = __ldg(q + (static_cast<int64_t>(n) * k + i) * V + x);
        const float2 sp = stats[static_cast<int64_t>(n) * (k + 1) + i];
        const float2 sq = stats[np_rows + static_cast<int64_t>(n) * k + i];
        const double e = (static_cast<double>(lp) - sp.x) - (static_cast<double>(lq) - sq.x);
        const double ratio = exp2(e * kLog2eD) * static_cast<double>(sq.y) / static_cast<double>(sp.y);
        const float u = philox_uniform(seed, offset, n, i, kStreamAccept);
        rej = !(static_cast<double>(u) < ratio);
      }
    }
    const unsigned b = __ballot_sync(0xffffffffu, rej);
    if (b != 0u && first == k) first = base + __ffs(b) - 1;
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
}

// Block-wide sum of two doubles (fixed reduction order); result in thread 0.
template <int THREADS>
__device__ __forceinline__ double2 block_sum2(double x, double y) {
  __shared__ double2 s_w[THREADS / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    x += __shfl_xor_sync(0xffffffffu, x, o);
    y += __shfl_xor_sync(0xffffffffu, y, o);
  }
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = make_double2(x, y);
  __syncthreads();
  double2 t = make_double2(0.0, 0.0);
  if (threadIdx.x == 0) {
    for (int w = 0; w < THREADS / 32; ++w) {
      t.x += s_w[w].x;
      t.y += s_w[w].y;
    }
  }
  return t;
}

// One CTA per (sequence, chunk): the sums over the chunk of the residual row
// max(0, p_a - q_a) and of p_a itself (the fallback when the residual
// vanishes), or of p_k twice for the bonus row.  Coalesced 16-byte loads.
template <bool VEC>
__global__ void __launch_bounds__(256)
    chunk_sum_kernel(const float* __restrict__ p, const float* __restrict__ q, int N, int k, int V,
                     const float2* __restrict__ stats, const int32_t* __restrict__ accept,
                     double2* __restrict__ chunk_sums) {
  const int n = blockIdx.x / kSampleChunks;
  const int c = blockIdx.x - n * kSampleChunks;
  const int tid = threadIdx.x;
  const int a = __ldg(accept + n);
  const SampleRow row = sample_row(p, q, stats, N, k, V, n, a, false);
  const SampleRow prow = sample_row(p, q, stats, N, k, V, n, a, true);
  const int CL = chunk_len(V);
  const int lo = min(c * CL, V), hi = min(lo + CL, V);
  float sr = 0.f, sp = 0.f;
  if (VEC) {
    const float4* p4 = reinterpret_cast<const float4*>(row.p + lo);
    const float4* q4 = row.q != nullptr ? reinterpret_cast<const float4*>(row.q + lo) : nullptr;
    const int n4 = (hi - lo) >> 2;
    for (int b = tid; b < n4; b += 4 * 256) {
      float4 lp[4], lq[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = b + j * 256;
        lp[j] = i < n4 ? p4[i] : make_float4(-__builtin_huge_valf(), -__builtin_huge_valf(),
                                              -__builtin_huge_valf(), -__builtin_huge_valf());
        lq[j] = (q4 != nullptr && i < n4) ? q4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sr += ((row.value(lp[j].x, lq[j].x) + row.value(lp[j].y, lq[j].y)) +
               (row.value(lp[j].z, lq[j].z) + row.value(lp[j].w, lq[j].w)));
        sp += ((prow.value(lp[j].x, 0.f) + prow.value(lp[j].y, 0.f)) +
               (prow.value(lp[j].z, 0.f) + prow.value(lp[j].w, 0.f)));
      }
    }
  } else {
    for (int v = lo + tid; v < hi; v += 256) {
      const float lp = __ldg(row.p + v);
      sr += row.value(lp, row.q != nullptr ? __ldg(row.q + v) : 0.f);
      sp += prow.value(lp, 0.f);
    }
  }
  const double2 t = block_sum2<256>(static_cast<double>(sr), static_cast<double>(sp));
  if (tid == 0) chunk_sums[blockIdx.x] = t;
}

// One CTA per sequence: inverse CDF in token-id order.  The 32 chunk sums
// (loaded in parallel) give the chunk holding u * Z; that chunk's residual
// values are computed once into shared memory with coalesced loads, cut into
// contiguous runs, one per thread, whose fp64 sums are prefix-summed in thread
// order; the thread whose run spans the target walks it to the token.
constexpr int kPickThreads = 256;
constexpr int kPickMaxChunk = 8192;    // chunk values staged in shared memory (V <= 262,144)

__global__ void __launch_bounds__(kPickThreads)
    pick_kernel(const float* __restrict__ p, const float* __restrict__ q, int N, int k, int V,
                uint64_t seed, uint32_t offset, uint32_t u_stream, int u_pos,
                const float2* __restrict__ stats,
                const int32_t* __restrict__ accept, const double2* __restrict__ chunk_sums,
                int32_t* __restrict__ out_tokens) {
  __shared__ double2 s_cs[kSampleChunks];
  __shared__ double s_excl[kPickThreads + 1];
  __shared__ float s_r[kPickMaxChunk];
  __shared__ int s_chunk, s_use_p, s_pick, s_last;
  __shared__ double s_tgt;
  const int n = blockIdx.x;
  const int tid = threadIdx.x;
  const int a = __ldg(accept + n);
  if (tid < kSampleChunks) s_cs[tid] = chunk_sums[static_cast<int64_t>(n) * kSampleChunks + tid];
  __syncthreads();
  if (tid == 0) {
    double zr = 0.0;
    for (int c = 0; c < kSampleChunks; ++c) zr += s_cs[c].x;
    const bool use_p = (a == k) || !(zr > 0.0);
    double Z = 0.0;
    for (int c = 0; c < kSampleChunks; ++c) Z += use_p ? s_cs[c].y : s_cs[c].x;
    // the uniform of counter (n, position, stream, offset): position a on the
    // RESAMPLE stream for verification, the draft step on the DRAFT stream
    const double target =
        static_cast<double>(philox_uniform(seed, offset, n, u_pos >= 0 ? u_pos : a, u_stream)) * Z;
    // First chunk whose inclusive prefix exceeds the target, else the last
    // chunk with positive mass.
    double run = 0.0, base = 0.0, last_base = 0.0;
    int pick = -1, last = 0;
    for (int c = 0; c < kSampleChunks; ++c) {
      const double v = use_p ? s_cs[c].y : s_cs[c].x;
      if (v > 0.0) {
        last = c;
        last_base = run;
      }
      if (pick < 0 && run + v > target) {
        pick = c;
        base = run;
      }
      run += v;
    }
    if (pick < 0) {
      pick = last;
      base = last_base;
    }
    s_chunk = pick;
    s_use_p = use_p ? 1 : 0;
    s_tgt = target - base;
    s_pick = 0x7fffffff;
    s_last = -1;
  }
  __syncthreads();
  const SampleRow row = sample_row(p, q, stats, N, k, V, n, a, s_use_p != 0);
  const int CL = chunk_len(V);
  const int lo = min(s_chunk * CL, V), hi = min(lo + CL, V);
  const int len = hi - lo;
  const bool staged = len <= kPickMaxChunk;
  if (staged) {
    for (int v = tid; v < len; v += kPickThreads) s_r[v] = row.at(lo + v);
    __syncthreads();
  }
  auto value = [&](int v) -> float { return staged ? s_r[v - lo] : row.at(v); };
  const int E = (len + kPickThreads - 1) / kPickThreads;
  const int r0 = min(lo + tid * E, hi), r1 = min(r0 + E, hi);
  double part = 0.0;
  int my_last = -1;
  for (int v = r0; v < r1; ++v) {
    const float r = value(v);
    part += static_cast<double>(r);
    if (r > 0.f) my_last = v;
  }
  s_excl[tid] = part;
  if (my_last >= 0) atomicMax(&s_last, my_last);
  __syncthreads();
  if (tid == 0) {
    // Exclusive prefix in thread order, sequential so it is monotone.
    double run = 0.0;
    for (int t = 0; t < kPickThreads; ++t) {
      const double v = s_excl[t];
      s_excl[t] = run;
      run += v;
    }
    s_excl[kPickThreads] = __longlong_as_double(0x7ff0000000000000LL);   // +inf
  }
  __syncthreads();
  const double tgt = s_tgt;
  if (s_excl[tid] <= tgt && tgt < s_excl[tid + 1]) {
    double run = s_excl[tid];
    int pick = -1;
    for (int v = r0; v < r1; ++v) {
      const float r = value(v);
      run += static_cast<double>(r);
      if (r > 0.f && run > tgt) {
        pick = v;
        break;
      }
    }
    if (pick < 0) pick = my_last;
    if (pick >= 0) atomicMin(&s_pick, pick);
  }
  __syncthreads();
  if (tid == 0) {
    int tok = s_pick != 0x7fffffff ? s_pick : s_last;
    if (tok < 0) tok = lo < V ? lo : V - 1;
    out_tokens[static_cast<int64_t>(n) * (k + 1) + a] = tok;
  }
}

}  // namespace

SpecWorkspaceLayout spec_workspace_layout(int64_t N, int k) {
  auto al = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SpecWorkspaceLayout L{};
  L.err_off = 0;
  L.stats_off = 256;
  L.accept_off = L.stats_off + al(static_cast<size_t>(N) * (2 * k + 1) * sizeof(float2));
  L.chunk_off = L.accept_off + al(static_cast<size_t>(N) * sizeof(int32_t));
  L.total = L.chunk_off + al(static_cast<size_t>(N) * kSampleChunks * sizeof(double2));
  return L;
}

cudaError_t launch_spec_sample(const float* p, const float* q, const int32_t* drafts, int N, int k,
                               int V, uint64_t seed, uint32_t offset, void* ws,
                               int32_t* out_tokens, int32_t* n_accepted, cudaStream_t stream,
                               uint32_t u_stream, int u_pos) {
  if (N == 0) return cudaSuccess;
  const SpecWorkspaceLayout L = spec_workspace_layout(N, k);
  uint8_t* w = static_cast<uint8_t*>(ws);
  int* err = reinterpret_cast<int*>(w + L.err_off);
  float2* stats = reinterpret_cast<float2*>(w + L.stats_off);
  int32_t* accept = reinterpret_cast<int32_t*>(w + L.accept_off);
  double2* chunks = reinterpret_cast<double2*>(w + L.chunk_off);
  const int rows = N * (2 * k + 1);
  const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                   (k == 0 || reinterpret_cast<uintptr_t>(q) % 16 == 0);
  if (vec) {
    row_stats_kernel<true><<<rows, kStatThreads, 0, stream>>>(p, q, N, k, V, stats);
  } else {
    row_stats_kernel<false><<<rows, kStatThreads, 0, stream>>>(p, q, N, k, V, stats);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  accept_kernel<<<(N + 7) / 8, 256, 0, stream>>>(p, q, drafts, N, k, V, seed, offset, stats, accept,
                                                  out_tokens, n_accepted, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t chunk_blocks = static_cast<int64_t>(N) * kSampleChunks;
  if (vec) {
    chunk_sum_kernel<true><<<static_cast<unsigned>(chunk_blocks), 256, 0, stream>>>(p, q, N, k, V, stats,
                                                                                   accept, chunks);
  } else {
    chunk_sum_kernel<false><<<static_cast<unsigned>(chunk_blocks), 256, 0, stream>>>(p, q, N, k, V, stats,
                                                                                    accept, chunks);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pick_kernel<<<N, kPickThreads, 0, stream>>>(p, q, N, k, V, seed, offset, u_stream, u_pos, stats, accept,
                                              chunks, out_tokens);
  return cudaGetLastError();
}

}  // namespace s3r
