// epikv.cu -- the EPIKV score: hidden-state change between consecutive tokens, made position-free.
//
// EPIKV write-up ("方法论：EPIKV", items 1-3): instead of attention weights, a token's importance
// comes from how much the residual stream moves when it is decoded, g_l(t) = ||h_l(t) - h_l(t-1)||_2,
// at a layer of the band where that signal is positive evidence (A) and one where it is negative
// evidence (B); each signal is corrected for its positional trend by a causal rolling z-score
// z_l = (g_l - mu_l) / (sigma_l + eps), and the eviction score is z_A - z_B. The selection and the
// compaction are the ones the attention-based path uses, with one kept list per sequence shared by
// every layer and KV head (the score is a property of the token).
//
//   epikv_delta_kernel  per (block of 32 tokens, sequence, layer): rows streamed once with 16-byte
//                       loads, 16 vectors per thread in flight, the previous row kept in registers;
//                       squared differences summed in fp32, g = sqrt (HBM-bound)
//   epikv_scan_kernel   per (sequence, layer): fp64 prefix sums of g and g^2 (block scans with a
//                       running carry)
//   epikv_z_kernel      per token: the window's mean and population variance from two prefix
//                       differences in fp64, sigma and the quotient in fp32, the score, and an
//                       order-preserving unsigned key of it for the radix selection
// Readings (the write-up gives no window, eps or first-token rule): g(0) = 0 and token 0 lies in
// no window; window(t) = tokens max(1, t - W + 1) .. t; sigma is the population deviation.
#include "kvc_internal.cuh"

namespace kvc {

constexpr int kDeltaThreads = 256;
constexpr int kDeltaTokens = 32;  // tokens per CTA (one extra row read per 32)
constexpr int kZThreads = 1024;

template <typename T, int NVT>
__global__ void __launch_bounds__(kDeltaThreads, 2) epikv_delta_kernel(const T* __restrict__ hA, const T* __restrict__ hB,
                                                                     int N, int dm, float* __restrict__ g) {
  constexpr int per = 16 / (int)sizeof(T);  // elements per vector
  constexpr int kU = 16 / NVT;              // rows loaded per batch: 16 vectors per thread in flight
  __shared__ float red[kDeltaThreads / 32][kU];
  const int layer = blockIdx.z, b = blockIdx.y, B = gridDim.y;
  const int t0 = blockIdx.x * kDeltaTokens;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = dm / per;
  const uint4* h = reinterpret_cast<const uint4*>((layer ? hB : hA) + (size_t)b * N * dm);
  auto row = [&](int t) { return h + (size_t)t * nv; };
  uint4 prev[NVT];
  {
    const uint4* r = row(t0 > 0 ? t0 - 1 : 0);
#pragma unroll
    for (int i = 0; i < NVT; ++i) {
      const int j = tid + i * kDeltaThreads;
      prev[i] = j < nv ? r[j] : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  for (int tb = 0; tb < kDeltaTokens; tb += kU) {
    uint4 cur[kU][NVT];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int t = t0 + tb + u;
#pragma unroll
      for (int i = 0; i < NVT; ++i) {
        const int j = tid + i * kDeltaThreads;
        cur[u][i] = (t < N && j < nv) ? row(t)[j] : make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float part[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < NVT; ++i) {
        const T* c = reinterpret_cast<const T*>(&cur[u][i]);
        const T* p = reinterpret_cast<const T*>(u ? &cur[u - 1][i] : &prev[i]);
#pragma unroll
        for (int e = 0; e < per; ++e) {
          const float d = to_f32(c[e]) - to_f32(p[e]);
          acc = fmaf(d, d, acc);
        }
      }
      part[u] = warp_sum(acc);
    }
#pragma unroll
    for (int i = 0; i < NVT; ++i) prev[i] = cur[kU - 1][i];
    if (lane == 0)
#pragma unroll
      for (int u = 0; u < kU; ++u) red[warp][u] = part[u];
    __syncthreads();
    if (tid < kU) {
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kDeltaThreads / 32; ++w) s += red[w][tid];
      const int t = t0 + tb + tid;
      if (t < N) g[((size_t)layer * B + b) * N + t] = t == 0 ? 0.f : sqrtf(s);
    }
    __syncthreads();
  }
}

// inclusive block scan of (a, b) over kZThreads threads, fp64
__device__ __forceinline__ void block_scan2(double& a, double& b, double* sa, double* sb) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double xa = __shfl_up_sync(kFull, a, o), xb = __shfl_up_sync(kFull, b, o);
    if (lane >= o) {
      a += xa;
      b += xb;
    }
  }
  if (lane == 31) {
    sa[warp] = a;
    sb[warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    double wa = sa[lane], wb = sb[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double xa = __shfl_up_sync(kFull, wa, o), xb = __shfl_up_sync(kFull, wb, o);
      if (lane >= o) {
        wa += xa;
        wb += xb;
      }
    }
    sa[lane] = wa;  // inclusive totals of warps 0..lane
    sb[lane] = wb;
  }
  __syncthreads();
  if (warp > 0) {
    a += sa[warp - 1];
    b += sb[warp - 1];
  }
}

// Order-preserving unsigned key of a float (-0 taken as +0): larger scores, larger keys.
__device__ __forceinline__ uint32_t score_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// per (sequence, layer): fp64 prefix sums of g and g^2, pre[layer][which][b][t] = sum over tokens < t
__global__ void __launch_bounds__(kZThreads) epikv_scan_kernel(const float* __restrict__ g, int B, int N,
                                                               double* __restrict__ pre) {
  __shared__ double sa[32], sb[32], tot[2];
  griddep_wait();  // g comes from the delta kernel
  const int b = blockIdx.x, layer = blockIdx.y, tid = threadIdx.x;
  const float* gl = g + ((size_t)layer * B + b) * N;
  double* p1 = pre + (((size_t)layer * 2 + 0) * B + b) * (size_t)(N + 1);
  double* p2 = pre + (((size_t)layer * 2 + 1) * B + b) * (size_t)(N + 1);
  double c1 = 0.0, c2 = 0.0;
  if (tid == 0) p1[0] = p2[0] = 0.0;
  for (int t0 = 0; t0 < N; t0 += kZThreads) {
    const int t = t0 + tid;
    const double v = (t >= 1 && t < N) ? (double)gl[t] : 0.0;  // token 0 lies in no window
    double a = v, q = v * v;
    block_scan2(a, q, sa, sb);
    if (t < N) {
      p1[t + 1] = c1 + a;
      p2[t + 1] = c2 + q;
    }
    if (tid == kZThreads - 1) {
      tot[0] = a;
      tot[1] = q;
    }
    __syncthreads();
    c1 += tot[0];
    c2 += tot[1];
    __syncthreads();
  }
}

// per token: the window's mean and population variance from two prefix differences (fp64, where
// the cancellation is), then sigma, g - mu and the quotient in fp32; the signed score and its key
__global__ void __launch_bounds__(256) epikv_z_kernel(const float* __restrict__ g, int B, int N, int W, float eps,
                                                      const double* __restrict__ pre, float* __restrict__ score,
                                                      uint32_t* __restrict__ keys) {
  griddep_wait();  // the prefix sums come from the scan kernel
  const int b = blockIdx.y, t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= N) return;
  float z[2] = {0.f, 0.f};
  if (t >= 1) {
    const int lo = t - W + 1 > 1 ? t - W + 1 : 1;
    const double inv_n = 1.0 / (double)(t - lo + 1);
#pragma unroll
    for (int layer = 0; layer < 2; ++layer) {
      const double* p1 = pre + (((size_t)layer * 2 + 0) * B + b) * (size_t)(N + 1);
      const double* p2 = pre + (((size_t)layer * 2 + 1) * B + b) * (size_t)(N + 1);
      const double mu = (p1[t + 1] - p1[lo]) * inv_n;
      const double var = fmax((p2[t + 1] - p2[lo]) * inv_n - mu * mu, 0.0);
      const float d = (float)((double)g[((size_t)layer * B + b) * N + t] - mu);
      z[layer] = d / (sqrtf((float)var) + eps);
    }
  }
  const float s = z[0] - z[1];
  score[(size_t)b * N + t] = s;
  if (keys) keys[(size_t)b * N + t] = score_key(s);
}

int launch_epikv_score(int dtype, int B, int N, int dm, const void* hA, const void* hB, int W, double eps, float* g,
                       double* pre, float* score, uint32_t* keys, cudaStream_t s) {
  if (B == 0 || N == 0) return KVC_OK;
  const dim3 grid((N + kDeltaTokens - 1) / kDeltaTokens, B, 2);
  const int per = dtype == KVC_BF16 ? 8 : 4;
  const int nvt = (dm / per + kDeltaThreads - 1) / kDeltaThreads;  // 1..4
  if (dtype == KVC_BF16) {
    auto* a = static_cast<const __nv_bfloat16*>(hA);
    auto* b = static_cast<const __nv_bfloat16*>(hB);
    if (nvt <= 1) epikv_delta_kernel<__nv_bfloat16, 1><<<grid, kDeltaThreads, 0, s>>>(a, b, N, dm, g);
    else if (nvt <= 2) epikv_delta_kernel<__nv_bfloat16, 2><<<grid, kDeltaThreads, 0, s>>>(a, b, N, dm, g);
    else epikv_delta_kernel<__nv_bfloat16, 4><<<grid, kDeltaThreads, 0, s>>>(a, b, N, dm, g);
  } else {
    auto* a = static_cast<const float*>(hA);
    auto* b = static_cast<const float*>(hB);
    if (nvt <= 1) epikv_delta_kernel<float, 1><<<grid, kDeltaThreads, 0, s>>>(a, b, N, dm, g);
    else if (nvt <= 2) epikv_delta_kernel<float, 2><<<grid, kDeltaThreads, 0, s>>>(a, b, N, dm, g);
    else epikv_delta_kernel<float, 4><<<grid, kDeltaThreads, 0, s>>>(a, b, N, dm, g);
  }
  if (launch_ok()) return KVC_ERR_LAUNCH;
  const float* gc = g;
  const double* pc = pre;
  if (launch_pdl(epikv_scan_kernel, dim3(B, 2), dim3(kZThreads), 0, s, false, gc, B, N, pre) != cudaSuccess ||
      launch_pdl(epikv_z_kernel, dim3((N + 255) / 256, B), dim3(256), 0, s, false, gc, B, N, W, (float)eps, pc, score,
                 keys) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
