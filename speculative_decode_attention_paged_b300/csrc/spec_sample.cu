// Exact speculative sampling over the full vocabulary.
//
// The S³R pages: full-attention verification accepts or rejects the drafted
// tokens through exact speculative sampling, which keeps the output
// distributed as the dense policy (wispaper.ai, "S3R drafts sparsely and
// verifies densely"); after the first rejection the correcting token comes
// from the residual distribution (rit.work, "Как разреженный черновик
// сохраняет ответы плотной модели"; rebasdaily.com, "草稿可以稀疏，交卷必须完整").
//
// Two kernels:
//   row_stats     one CTA per logit row (k+1 target rows and k draft rows per
//                 sequence): the row max m and z = sum_v 2^((x_v - m) log2 e),
//                 one streaming pass with 16-byte loads;
//   decide        one CTA per sequence: the k ratio tests p_i(x_i)/q_i(x_i)
//                 against Philox uniforms (fp64 ratio from fp32 row stats),
//                 then an inverse CDF in token-id order over the residual
//                 max(0, p - q) (or p_{k+1} for the bonus): each warp owns a
//                 contiguous segment of the row; warp-scan step sums are
//                 accumulated in fp64; the warp whose segment holds u * Z
//                 rescans it with the same arithmetic to find the token.

#include <cfloat>

#include "philox.cuh"
#include "s3r_device.cuh"

namespace s3r {

namespace {

constexpr int kStatThreads = 256;
constexpr int kDecideWarps = 8;
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

struct ResidualRow {
  const float* p;
  const float* q;   // null -> sample from p itself
  float mp, izp, mq, izq;
  int V;
  __device__ __forceinline__ float at(int v) const {
    const float pv = scaled_exp(__ldg(p + v), mp) * izp;
    if (q == nullptr) return pv;
    return fmaxf(pv - scaled_exp(__ldg(q + v), mq) * izq, 0.f);
  }
  // The four values a lane owns in one 128-element step (0 beyond V).
  __device__ __forceinline__ void four(int e0, float (&r)[4]) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) r[i] = e0 + i < V ? at(e0 + i) : 0.f;
  }
};

__global__ void __launch_bounds__(kDecideWarps * 32)
    decide_kernel(const float* __restrict__ p, const float* __restrict__ q,
                  const int32_t* __restrict__ drafts, int N, int k, int V, uint64_t seed,
                  uint32_t offset, const float2* __restrict__ stats, int32_t* __restrict__ out_tokens,
                  int32_t* __restrict__ n_accepted, int* err) {
  __shared__ int s_acc[64];
  __shared__ double s_wtot[kDecideWarps];
  __shared__ int s_token;
  const int n = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int np_rows = N * (k + 1);

  if (tid < k) {
    const int x = __ldg(drafts + static_cast<int64_t>(n) * k + tid);
    bool acc = false;
    if (x < 0 || x >= V) {
      report_error(err, S3R_DEVERR_BAD_TOKEN);
    } else {
      const float lp = __ldg(p + (static_cast<int64_t>(n) * (k + 1) + tid) * V + x);
      const float lq = __ldg(q + (static_cast<int64_t>(n) * k + tid) * V + x);
      const float2 sp = stats[static_cast<int64_t>(n) * (k + 1) + tid];
      const float2 sq = stats[np_rows + static_cast<int64_t>(n) * k + tid];
      const double e = (static_cast<double>(lp) - sp.x) - (static_cast<double>(lq) - sq.x);
      const double ratio = exp2(e * kLog2eD) * static_cast<double>(sq.y) / static_cast<double>(sp.y);
      const float u = philox_uniform(seed, offset, n, tid, kStreamAccept);
      acc = static_cast<double>(u) < ratio;
    }
    s_acc[tid] = acc ? 1 : 0;
  }
  if (tid == 0) s_token = -1;
  __syncthreads();
  int a = k;
  for (int i = 0; i < k; ++i) {
    if (!s_acc[i]) {
      a = i;
      break;
    }
  }

  const float2 sp = stats[static_cast<int64_t>(n) * (k + 1) + a];
  ResidualRow row;
  row.p = p + (static_cast<int64_t>(n) * (k + 1) + a) * V;
  row.mp = sp.x * kLog2e;
  row.izp = 1.f / sp.y;
  row.V = V;
  row.q = nullptr;
  row.mq = 0.f;
  row.izq = 0.f;
  if (a < k) {
    const float2 sq = stats[np_rows + static_cast<int64_t>(n) * k + a];
    row.q = q + (static_cast<int64_t>(n) * k + a) * V;
    row.mq = sq.x * kLog2e;
    row.izq = 1.f / sq.y;
  }
  const float u = philox_uniform(seed, offset, n, a, kStreamResample);

  const int steps = (V + 127) / 128;
  const int per_warp = (steps + kDecideWarps - 1) / kDecideWarps;
  const int s_begin = min(warp * per_warp, steps), s_end = min(s_begin + per_warp, steps);

  // Step sums of one warp's segment: lane-local sequential sums of 4 values,
  // then a Hillis-Steele warp inclusive scan; the same code runs in both passes.
  auto step_scan = [&](int st, float (&r)[4], float& local, float& incl) {
    row.four(st * 128 + lane * 4, r);
    local = ((r[0] + r[1]) + r[2]) + r[3];
    incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
  };

  for (int attempt = 0; attempt < 2; ++attempt) {
    double wt = 0.0;
    for (int st = s_begin; st < s_end; ++st) {
      float r[4], local, incl;
      step_scan(st, r, local, incl);
      wt += static_cast<double>(__shfl_sync(0xffffffffu, incl, 31));
    }
    if (lane == 0) s_wtot[warp] = wt;
    __syncthreads();
    double Z = 0.0;
    for (int w = 0; w < kDecideWarps; ++w) Z += s_wtot[w];
    if (!(Z > 0.0) && row.q != nullptr) {
      // The residual vanished (p == q in floating point): sample from p.
      row.q = nullptr;
      __syncthreads();
      continue;
    }
    const double target = static_cast<double>(u) * Z;
    // The warp whose segment holds the target (else the last non-empty one).
    int wsel = -1, wlast = -1;
    double run = 0.0, wbase = 0.0, lastbase = 0.0;
    for (int w = 0; w < kDecideWarps; ++w) {
      if (s_wtot[w] > 0.0) {
        wlast = w;
        lastbase = run;
      }
      if (wsel < 0 && run + s_wtot[w] > target) {
        wsel = w;
        wbase = run;
      }
      run += s_wtot[w];
    }
    if (wsel < 0) {
      wsel = wlast;
      wbase = lastbase;
    }
    if (warp == wsel) {
      double running = wbase;
      int last_pos = -1;   // last token with r > 0 seen so far (fallback)
      int found = -1;
      for (int st = s_begin; st < s_end && found < 0; ++st) {
        float r[4], local, incl;
        step_scan(st, r, local, incl);
        const float step_total = __shfl_sync(0xffffffffu, incl, 31);
        int lp = -1;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (r[i] > 0.f) lp = st * 128 + lane * 4 + i;
        const unsigned has = __ballot_sync(0xffffffffu, lp >= 0);
        if (has) last_pos = __shfl_sync(0xffffffffu, lp, 31 - __clz(has));
        if (running + static_cast<double>(step_total) > target) {
          const unsigned cross = __ballot_sync(0xffffffffu, running + static_cast<double>(incl) > target);
          const int ls = __ffs(cross) - 1;
          const float excl = __shfl_up_sync(0xffffffffu, incl, 1);
          int pick = -1;
          if (lane == ls) {
            const double base = running + (lane > 0 ? static_cast<double>(excl) : 0.0);
            float part = 0.f;
            int lastpos = -1;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              part += r[i];
              if (r[i] > 0.f) lastpos = st * 128 + lane * 4 + i;
              if (pick < 0 && r[i] > 0.f && base + static_cast<double>(part) > target)
                pick = st * 128 + lane * 4 + i;
            }
            if (pick < 0) pick = lastpos;
          }
          pick = __shfl_sync(0xffffffffu, pick, ls);
          found = pick >= 0 ? pick : last_pos;
        }
        running += static_cast<double>(step_total);
      }
      if (found < 0) found = last_pos;
      if (lane == 0) s_token = found >= 0 ? found : 0;
    }
    __syncthreads();
    break;
  }

  int32_t* out = out_tokens + static_cast<int64_t>(n) * (k + 1);
  for (int i = tid; i <= k; i += blockDim.x) {
    int32_t v = -1;
    if (i < a) v = __ldg(drafts + static_cast<int64_t>(n) * k + i);
    else if (i == a) v = s_token >= 0 ? s_token : 0;
    out[i] = v;
  }
  if (tid == 0) n_accepted[n] = a;
}

}  // namespace

cudaError_t launch_spec_sample(const float* p, const float* q, const int32_t* drafts, int N, int k,
                               int V, uint64_t seed, uint32_t offset, float2* stats,
                               int32_t* out_tokens, int32_t* n_accepted, int* err,
                               cudaStream_t stream) {
  if (N == 0) return cudaSuccess;
  const int rows = N * (2 * k + 1);
  const bool vec = (V % 4 == 0) && (reinterpret_cast<uintptr_t>(p) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(q) % 16 == 0);
  if (vec) {
    row_stats_kernel<true><<<rows, kStatThreads, 0, stream>>>(p, q, N, k, V, stats);
  } else {
    row_stats_kernel<false><<<rows, kStatThreads, 0, stream>>>(p, q, N, k, V, stats);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decide_kernel<<<N, kDecideWarps * 32, 0, stream>>>(p, q, drafts, N, k, V, seed, offset, stats,
                                                      out_tokens, n_accepted, err);
  return cudaGetLastError();
}

}  // namespace s3r
