// score.cu -- kvc_score: importance of every cached key from the observation queries.
//
// BeaconKV write-up, "观察 query 集 = 最近查询 + 信标查询" (observation set = recent queries +
// beacon queries) and "打分时的 RoPE 对齐" (beacons rotated to the current step t, recent
// queries at their own positions, importance = max over the observation set of the
// attention weight). Per KV head the observation rows of its G query heads are stacked into
// one M x D tile, so the max over the GQA group is the max over that tile's rows.
//
// Launch sequence (all on the caller's stream):
//   rope_table   cos/sin of t * theta^(-2i/D) in fp64, rounded to fp32        (1 CTA)
//   build_obs    per KV head: copy recent rows, pick beacons (FPS when the buffer
//                holds more than n_b), rotate them to t, round to storage type  (heads CTAs)
//   pass1        per (key chunk, head): S = Q K^T, per-row chunk max and sum of
//                exp2, i.e. a partial log-sum-exp                             (chunks x heads)
//   combine      per head: merge the partials into lse2 per row
//   pass2        per (key chunk, head): recompute S^T = K Q^T, max over rows of
//                s*log2(e)/sqrt(D) - lse2, exp2 -> score                        (chunks x heads)
// Softmax is kept in base 2 throughout: exp(s/sqrt(D) - lse) = exp2(s*c2 - lse2).
#include "fps_warp.cuh"
#include "kvc_internal.cuh"

namespace kvc {

// ---------------------------------------------------------------------------
// small PTX helpers (legacy warp-level tensor path: ldmatrix + mma.sync)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(kFull, v, 1));
  return fmaxf(v, __shfl_xor_sync(kFull, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(kFull, v, 1);
  return v + __shfl_xor_sync(kFull, v, 2);
}

// ---------------------------------------------------------------------------
// rotary table and observation rows
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float2* rope, int D, long long t, double theta) {
  const int i = threadIdx.x;
  if (i >= D / 2) return;
  const double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
  const double ang = (double)t * inv_freq;
  double sn, cs;
  sincos(ang, &sn, &cs);
  rope[i] = make_float2((float)cs, (float)sn);
}

template <typename T>
__global__ void build_obs_kernel(ScoreArgs a, ScoreWs ws, int nw) {
  extern __shared__ float smem[];
  const int D = a.g.D, Hkv = a.g.Hkv, B = a.g.B, Hq = a.g.Hq;
  const int head = blockIdx.x;
  const int l = head / (B * Hkv), b = (head / Hkv) % B, h = head % Hkv;
  const int G = Hq / Hkv, per_q = a.n_r + a.n_b, hd = D / 2;
  T* obs = static_cast<T*>(ws.obs) + (size_t)head * a.M_pad * D;
  uint8_t* valid = ws.valid + (size_t)head * a.M_pad;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = a.qmax * (D + 1) + a.qmax;
  float* xs = smem + warp * per;
  int* pk = reinterpret_cast<int*>(xs + a.qmax * (D + 1));
  const T* qrec = static_cast<const T*>(a.q_recent);
  const T* qbuf = static_cast<const T*>(a.qbuf);

  for (int g = warp; g < G; g += nw) {
    const int hq = h * G + g;
    const size_t qh = ((size_t)l * B + b) * Hq + hq;
    T* orow = obs + (size_t)g * per_q * D;
    // recent queries: already rotated to their own positions, copied as stored (16-byte vectors)
    {
      const uint4* qr = reinterpret_cast<const uint4*>(qrec + qh * a.n_r * D);
      uint4* od = reinterpret_cast<uint4*>(orow);
      const int nv = a.n_r * D * (int)sizeof(T) / 16;
      for (int e = lane; e < nv; e += kWarp) od[e] = qr[e];
    }
    for (int r = lane; r < a.n_r; r += kWarp) valid[g * per_q + r] = 1;
    // beacons: the buffer itself when it holds at most n_b rows, else FPS down to n_b
    int c = a.qmax > 0 ? a.count[qh] : 0;
    if (c < 0 || c > a.qmax) {
      if (lane == 0) status_or(a.status, KVC_STATUS_COUNT_RANGE);
      c = c < 0 ? 0 : a.qmax;
    }
    stage_rows(qbuf + qh * a.qmax * D, c, D, xs);
    int nb;
    if (c <= a.n_b) {
      nb = c;
      for (int k = lane; k < nb; k += kWarp) pk[k] = k;
      __syncwarp();
    } else {
      nb = a.n_b;
      fps_staged(xs, c, D, nb, pk);
    }
    for (int k = 0; k < a.n_b; ++k) {
      T* dst = orow + (size_t)(a.n_r + k) * D;
      if (k < nb) {
        const float* src = xs + pk[k] * (D + 1);
        for (int i = lane; i < hd; i += kWarp) {
          const float2 cs = ws.rope[i];
          const float x0 = src[i], x1 = src[i + hd];
          // each product and the sum rounded separately (no fused multiply-add), so the
          // rounding to the storage type below is a reproducible decision
          dst[i] = from_f32<T>(__fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y)));
          dst[i + hd] = from_f32<T>(__fadd_rn(__fmul_rn(x1, cs.x), __fmul_rn(x0, cs.y)));
        }
      } else {
        for (int i = lane; i < D; i += kWarp) dst[i] = from_f32<T>(0.f);
      }
      if (lane == 0) valid[g * per_q + a.n_r + k] = k < nb ? 1 : 0;
    }
    if (a.beacon_picks)
      for (int k = lane; k < a.n_b; k += kWarp) a.beacon_picks[qh * a.n_b + k] = k < nb ? pk[k] : -1;
    __syncwarp();
  }
  // padding rows up to a multiple of 16
  for (int e = threadIdx.x; e < (a.M_pad - a.M) * D; e += blockDim.x) obs[(size_t)a.M * D + e] = from_f32<T>(0.f);
  for (int r = a.M + threadIdx.x; r < a.M_pad; r += blockDim.x) valid[r] = 0;
}

// ---------------------------------------------------------------------------
// bf16 passes (mma.sync m16n8k16, fp32 accumulate)
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void load_rows_bf16(__nv_bfloat16* sm, const __nv_bfloat16* g, int rows, int valid_rows) {
  constexpr int VPR = D / 8;
  constexpr int LDS = D + 8;
  for (int e = threadIdx.x; e < rows * VPR; e += blockDim.x) {
    const int r = e / VPR, c = e % VPR;
    __nv_bfloat16* dst = sm + r * LDS + c * 8;
    if (r < valid_rows)
      cp_async16(dst, g + (size_t)r * D + c * 8);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
}

struct HeadLoc {
  int l, bh;
};
__device__ __forceinline__ HeadLoc head_loc(const CacheGeom& g, int head) {
  return HeadLoc{head / (g.B * g.Hkv), head % (g.B * g.Hkv)};
}

template <int D>
__global__ void __launch_bounds__(128) pass1_bf16_kernel(ScoreArgs a, ScoreWs ws, float c2) {
  extern __shared__ __align__(16) unsigned char smraw[];
  constexpr int LDS = D + 8;
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smraw);
  __nv_bfloat16* Ks = Qs + a.M_pad * LDS;
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const __nv_bfloat16* Kh = static_cast<const __nv_bfloat16*>(a.K.p[hl.l]) + (size_t)hl.bh * a.g.ncap * D;
  const int j0 = chunk * kChunk;
  const int nvalid = min(kChunk, a.g.N - j0);
  load_rows_bf16<D>(Qs, static_cast<const __nv_bfloat16*>(ws.obs) + (size_t)head * a.M_pad * D, a.M_pad, a.M_pad);
  load_rows_bf16<D>(Ks, Kh + (size_t)j0 * D, kChunk, nvalid);
  cp_async_commit_wait_all();
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int mt = warp; mt < a.M_pad / 16; mt += 4) {
    uint32_t af[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(af[ks], Qs + (mt * 16 + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8);
    float acc[kChunk / 8][4];
#pragma unroll
    for (int nt = 0; nt < kChunk / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int np = 0; np < kChunk / 16; ++np) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t bf[4];
        ldsm_x4(bf, Ks + (np * 16 + ((lane >> 4) << 3) + (lane & 7)) * LDS + ks * 16 + ((lane >> 3) & 1) * 8);
        mma_bf16_16816(acc[2 * np], af[ks], bf[0], bf[1]);
        mma_bf16_16816(acc[2 * np + 1], af[ks], bf[2], bf[3]);
      }
    }
    float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = nt * 8 + 2 * (lane & 3) + e < nvalid;
        acc[nt][e] = ok ? acc[nt][e] * c2 : -INFINITY;
        acc[nt][2 + e] = ok ? acc[nt][2 + e] * c2 : -INFINITY;
        m0 = fmaxf(m0, acc[nt][e]);
        m1 = fmaxf(m1, acc[nt][2 + e]);
      }
    m0 = quad_max(m0);
    m1 = quad_max(m1);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < kChunk / 8; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        s0 += exp2f(acc[nt][e] - m0);
        s1 += exp2f(acc[nt][2 + e] - m1);
      }
    s0 = quad_sum(s0);
    s1 = quad_sum(s1);
    if ((lane & 3) == 0) {
      float2* part = ws.part + ((size_t)head * a.nchunk + chunk) * a.M_pad;
      const int r0 = mt * 16 + (lane >> 2);
      part[r0] = make_float2(m0, s0);
      part[r0 + 8] = make_float2(m1, s1);
    }
  }
}

template <int D>
__global__ void __launch_bounds__(128) pass2_bf16_kernel(ScoreArgs a, ScoreWs ws, float c2) {
  extern __shared__ __align__(16) unsigned char smraw[];
  constexpr int LDS = D + 8;
  __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(smraw);
  __nv_bfloat16* Ks = Qs + a.M_pad * LDS;
  float* L2s = reinterpret_cast<float*>(Ks + kChunk * LDS);
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const __nv_bfloat16* Kh = static_cast<const __nv_bfloat16*>(a.K.p[hl.l]) + (size_t)hl.bh * a.g.ncap * D;
  const int j0 = chunk * kChunk;
  const int nvalid = min(kChunk, a.g.N - j0);
  load_rows_bf16<D>(Qs, static_cast<const __nv_bfloat16*>(ws.obs) + (size_t)head * a.M_pad * D, a.M_pad, a.M_pad);
  load_rows_bf16<D>(Ks, Kh + (size_t)j0 * D, kChunk, nvalid);
  for (int r = threadIdx.x; r < a.M_pad; r += blockDim.x) L2s[r] = ws.lse2[(size_t)head * a.M_pad + r];
  cp_async_commit_wait_all();
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* out = a.scores + (size_t)head * a.g.N + j0;
  for (int kt = warp; kt < kChunk / 16; kt += 4) {
    if (kt * 16 >= nvalid) break;
    uint32_t af[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(af[ks], Ks + (kt * 16 + (lane & 15)) * LDS + ks * 16 + (lane >> 4) * 8);
    float b0 = -INFINITY, b1 = -INFINITY;
    for (int np = 0; np < a.M_pad / 16; ++np) {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t bf[4];
        ldsm_x4(bf, Qs + (np * 16 + ((lane >> 4) << 3) + (lane & 7)) * LDS + ks * 16 + ((lane >> 3) & 1) * 8);
        mma_bf16_16816(acc[0], af[ks], bf[0], bf[1]);
        mma_bf16_16816(acc[1], af[ks], bf[2], bf[3]);
      }
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float lb = L2s[np * 16 + t * 8 + 2 * (lane & 3) + e];
          b0 = fmaxf(b0, acc[t][e] * c2 - lb);
          b1 = fmaxf(b1, acc[t][2 + e] * c2 - lb);
        }
    }
    b0 = quad_max(b0);
    b1 = quad_max(b1);
    if ((lane & 3) == 0) {
      const int j = kt * 16 + (lane >> 2);
      if (j < nvalid) out[j] = exp2f(b0);
      if (j + 8 < nvalid) out[j + 8] = exp2f(b1);
    }
  }
}

// ---------------------------------------------------------------------------
// fp32 passes (CUDA-core FMA; fp32 storage is the small-model path)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) pass1_f32_kernel(ScoreArgs a, ScoreWs ws, float c2) {
  extern __shared__ __align__(16) float smf[];
  const int D = a.g.D, LQ = D + 1;
  float* Qs = smf;                   // [M_pad][D+1]
  float* Ks = Qs + a.M_pad * LQ;     // [kChunk][D]
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const float* Kh = static_cast<const float*>(a.K.p[hl.l]) + (size_t)hl.bh * a.g.ncap * D;
  const int j0 = chunk * kChunk;
  const int nvalid = min(kChunk, a.g.N - j0);
  const float* obs = static_cast<const float*>(ws.obs) + (size_t)head * a.M_pad * D;
  for (int e = threadIdx.x; e < a.M_pad * D; e += blockDim.x) Qs[(e / D) * LQ + e % D] = obs[e];
  for (int e = threadIdx.x; e < nvalid * D; e += blockDim.x) Ks[e] = Kh[(size_t)j0 * D + e];
  __syncthreads();
  for (int r = threadIdx.x; r < a.M_pad; r += blockDim.x) {
    float m = -INFINITY, s = 0.f;
    for (int j = 0; j < nvalid; ++j) {
      float dot = 0.f;
      for (int d = 0; d < D; ++d) dot = fmaf(Qs[r * LQ + d], Ks[j * D + d], dot);
      const float x = dot * c2;
      if (x > m) {
        s = s * exp2f(m - x) + 1.f;
        m = x;
      } else {
        s += exp2f(x - m);
      }
    }
    ws.part[((size_t)head * a.nchunk + chunk) * a.M_pad + r] = make_float2(m, s);
  }
}

__global__ void __launch_bounds__(128) pass2_f32_kernel(ScoreArgs a, ScoreWs ws, float c2) {
  extern __shared__ __align__(16) float smf[];
  const int D = a.g.D, LK = D + 1;
  float* Qs = smf;                  // [M_pad][D]
  float* Ks = Qs + a.M_pad * D;     // [kChunk][D+1]
  float* L2s = Ks + kChunk * LK;    // [M_pad]
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const float* Kh = static_cast<const float*>(a.K.p[hl.l]) + (size_t)hl.bh * a.g.ncap * D;
  const int j0 = chunk * kChunk;
  const int nvalid = min(kChunk, a.g.N - j0);
  const float* obs = static_cast<const float*>(ws.obs) + (size_t)head * a.M_pad * D;
  for (int e = threadIdx.x; e < a.M_pad * D; e += blockDim.x) Qs[e] = obs[e];
  for (int e = threadIdx.x; e < nvalid * D; e += blockDim.x) Ks[(e / D) * LK + e % D] = Kh[(size_t)j0 * D + e];
  for (int r = threadIdx.x; r < a.M_pad; r += blockDim.x) L2s[r] = ws.lse2[(size_t)head * a.M_pad + r];
  __syncthreads();
  const int j = threadIdx.x;
  if (j >= nvalid) return;
  float best = -INFINITY;
  for (int r = 0; r < a.M_pad; ++r) {
    float dot = 0.f;
    for (int d = 0; d < D; ++d) dot = fmaf(Qs[r * D + d], Ks[j * LK + d], dot);
    best = fmaxf(best, dot * c2 - L2s[r]);
  }
  a.scores[(size_t)head * a.g.N + j0 + j] = exp2f(best);
}

// ---------------------------------------------------------------------------
// merge the per-chunk partial log-sum-exps of every observation row
// ---------------------------------------------------------------------------
__global__ void combine_kernel(ScoreArgs a, ScoreWs ws) {
  const int head = blockIdx.x, r = threadIdx.x;
  if (r >= a.M_pad) return;
  const float2* p = ws.part + (size_t)head * a.nchunk * a.M_pad + r;
  float M2 = -INFINITY, S = 0.f;
  for (int c = 0; c < a.nchunk; ++c) {
    const float2 v = p[(size_t)c * a.M_pad];
    if (v.x > M2) {
      S = S * exp2f(M2 - v.x) + v.y;
      M2 = v.x;
    } else {
      S += v.y * exp2f(v.x - M2);
    }
  }
  const bool ok = ws.valid[(size_t)head * a.M_pad + r] != 0;
  ws.lse2[(size_t)head * a.M_pad + r] = ok ? M2 + log2f(S) : INFINITY;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t score_ws_bytes(const CacheGeom& g, int dtype, int n_r, int n_b, ScoreWs* carve, void* base) {
  const size_t es = dtype == KVC_BF16 ? 2 : 4;
  const size_t heads = (size_t)g.L * g.B * g.Hkv;
  const int G = g.Hq / g.Hkv;
  const int M = G * (n_r + n_b);
  const size_t M_pad = (size_t)((M + 15) / 16) * 16;
  const size_t nchunk = (size_t)(g.N + kChunk - 1) / kChunk;
  size_t off = 0;
  const size_t o_rope = off;  off += align256(sizeof(float2) * (size_t)(g.D / 2));
  const size_t o_obs = off;   off += align256(heads * M_pad * g.D * es);
  const size_t o_valid = off; off += align256(heads * M_pad);
  const size_t o_part = off;  off += align256(heads * nchunk * M_pad * sizeof(float2));
  const size_t o_lse = off;   off += align256(heads * M_pad * sizeof(float));
  if (carve) {
    char* b = static_cast<char*>(base);
    carve->rope = reinterpret_cast<float2*>(b + o_rope);
    carve->obs = b + o_obs;
    carve->valid = reinterpret_cast<uint8_t*>(b + o_valid);
    carve->part = reinterpret_cast<float2*>(b + o_part);
    carve->lse2 = reinterpret_cast<float*>(b + o_lse);
  }
  return off;
}

template <typename K>
static bool set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

int launch_score(const ScoreArgs& a, const ScoreWs& ws, cudaStream_t s) {
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  const int D = a.g.D;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  rope_table_kernel<<<1, (D / 2 + 31) / 32 * 32, 0, s>>>(ws.rope, D, a.t, a.theta);
  if (launch_ok()) return KVC_ERR_LAUNCH;

  // observation rows: one warp per query head of the group
  const int G = a.g.Hq / a.g.Hkv;
  const size_t per_warp = sizeof(float) * (size_t)(a.qmax * (D + 1) + a.qmax);
  int nw = G < 8 ? G : 8;
  while (nw > 1 && per_warp * nw > 200u * 1024u) --nw;
  const size_t obs_smem = per_warp * nw;
  if (a.dtype == KVC_BF16) {
    if (!set_smem(build_obs_kernel<__nv_bfloat16>, obs_smem)) return KVC_ERR_LAUNCH;
    build_obs_kernel<__nv_bfloat16><<<heads, 32 * nw, obs_smem, s>>>(a, ws, nw);
  } else {
    if (!set_smem(build_obs_kernel<float>, obs_smem)) return KVC_ERR_LAUNCH;
    build_obs_kernel<float><<<heads, 32 * nw, obs_smem, s>>>(a, ws, nw);
  }
  if (launch_ok()) return KVC_ERR_LAUNCH;

  const dim3 grid(a.nchunk, heads);
  if (a.dtype == KVC_BF16) {
    const size_t sm1 = (size_t)(a.M_pad + kChunk) * (D + 8) * 2;
    const size_t sm2 = sm1 + (size_t)a.M_pad * 4;
    if (D == 128) {
      if (!set_smem(pass1_bf16_kernel<128>, sm1) || !set_smem(pass2_bf16_kernel<128>, sm2)) return KVC_ERR_LAUNCH;
      pass1_bf16_kernel<128><<<grid, 128, sm1, s>>>(a, ws, c2);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      combine_kernel<<<heads, (a.M_pad + 31) / 32 * 32, 0, s>>>(a, ws);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      pass2_bf16_kernel<128><<<grid, 128, sm2, s>>>(a, ws, c2);
    } else {
      if (!set_smem(pass1_bf16_kernel<64>, sm1) || !set_smem(pass2_bf16_kernel<64>, sm2)) return KVC_ERR_LAUNCH;
      pass1_bf16_kernel<64><<<grid, 128, sm1, s>>>(a, ws, c2);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      combine_kernel<<<heads, (a.M_pad + 31) / 32 * 32, 0, s>>>(a, ws);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      pass2_bf16_kernel<64><<<grid, 128, sm2, s>>>(a, ws, c2);
    }
  } else {
    const size_t sm1 = sizeof(float) * ((size_t)a.M_pad * (D + 1) + (size_t)kChunk * D);
    const size_t sm2 = sizeof(float) * ((size_t)a.M_pad * D + (size_t)kChunk * (D + 1) + a.M_pad);
    if (!set_smem(pass1_f32_kernel, sm1) || !set_smem(pass2_f32_kernel, sm2)) return KVC_ERR_LAUNCH;
    pass1_f32_kernel<<<grid, 128, sm1, s>>>(a, ws, c2);
    if (launch_ok()) return KVC_ERR_LAUNCH;
    combine_kernel<<<heads, (a.M_pad + 31) / 32 * 32, 0, s>>>(a, ws);
    if (launch_ok()) return KVC_ERR_LAUNCH;
    pass2_f32_kernel<<<grid, 128, sm2, s>>>(a, ws, c2);
  }
  return launch_ok();
}

}  // namespace kvc
