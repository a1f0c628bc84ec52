// score.cu -- kvc_score: importance of every cached key from the observation queries.
//
// BeaconKV write-up, "观察 query 集 = 最近查询 + 信标查询" (observation set = recent queries +
// beacon queries) and "打分时的 RoPE 对齐" (beacons rotated to the current step t, recent
// queries at their own positions, importance = max over the observation set of the
// attention weight). Per KV head the observation rows of its G query heads are stacked into
// one M x D tile, so the max over the GQA group is the max over that tile's rows.
//
// Launch sequence (all on the caller's stream):
//   (host)       cos/sin of t * theta^(-2i/D) in fp64, rounded to fp32, passed as a parameter
//   build_obs    per KV head: copy recent rows, pick beacons (FPS when the buffer
//                holds more than n_b), rotate them to t, round to storage type  (heads CTAs)
//   pass1        per (key chunk, head): S = Q K^T, per-row chunk max and sum of
//                exp2, i.e. a partial log-sum-exp                             (chunks x heads)
//   combine      per head: merge the partials into lse2 per row
//   pass2        per (key chunk, head): recompute S^T = K Q^T, max over rows of
//                s*log2(e)/sqrt(D) - lse2, exp2 -> score                        (chunks x heads)
// Softmax is kept in base 2 throughout: exp(s/sqrt(D) - lse) = exp2(s*c2 - lse2).
#include <cudaTypedefs.h>

#include "fps_warp.cuh"
#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {

// ---------------------------------------------------------------------------
// rotary table and observation rows
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void build_obs_kernel(ScoreArgs a, ScoreWs ws, int nw) {
  extern __shared__ float smem[];
  const int Hkv = a.g.Hkv, B = a.g.B, Hq = a.g.Hq;
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
    stage_rows<T, D>(qbuf + qh * a.qmax * D, c, xs);
    int nb;
    if (c <= a.n_b) {
      nb = c;
      for (int k = lane; k < nb; k += kWarp) pk[k] = k;
      __syncwarp();
    } else {
      nb = a.n_b;
      fps_staged<D>(xs, c, nb, pk);
    }
    for (int k = 0; k < a.n_b; ++k) {
      T* dst = orow + (size_t)(a.n_r + k) * D;
      if (k < nb) {
        const float* src = xs + pk[k] * (D + 1);
        for (int i = lane; i < hd; i += kWarp) {
          const float2 cs = a.rope[i];
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
// bf16 passes on the 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM)
//
// Shared memory holds the observation tile Q [D/64][M_pad rows][128 B] and one key chunk
// K [D/64][128 rows][128 B], both written by TMA in the 128-byte-swizzled K-major layout the
// UMMA descriptors read. Pass 1 computes S = Q K^T (TMEM lane = observation row, column =
// key), so each epilogue thread owns one row and folds its chunk max and exp2-sum in
// registers. Pass 2 computes S^T = K Q^T (lane = key, column = row), so each thread owns one
// key and takes the max over rows in registers.
// ---------------------------------------------------------------------------
struct HeadLoc {
  int l, bh;
};
__device__ __forceinline__ HeadLoc head_loc(const CacheGeom& g, int head) {
  return HeadLoc{head / (g.B * g.Hkv), head % (g.B * g.Hkv)};
}

struct TcMaps {
  CUtensorMap k[KVC_MAX_LAYERS];  // per layer: dims {D, ncap, B*Hkv}, box {64, 128, 1}
  CUtensorMap q;                  // observation rows: dims {D, heads*M_pad}, box {64, 128}
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

// Load the observation tile and key chunk with TMA, wait, and (thread 0) issue the MMAs.
// Returns the shared flag telling every thread whether the accumulator will arrive.
template <int D>
__device__ __forceinline__ bool tc_load_and_mma(const TcMaps& maps, const ScoreArgs& a, int head, const HeadLoc& hl,
                                                int j0, uint8_t* Qs, uint8_t* Ks, uint64_t* bars, uint32_t tmem,
                                                int pass, int* s_ok) {
  constexpr int HALVES = D / 64;
  const int MT = a.M_pad >> 7;
  if (threadIdx.x == 0) {
    int ok = 1;
    tc::mbar_expect_tx(&bars[0], (uint32_t)((a.M_pad + kChunk) * D * 2));
#pragma unroll
    for (int h = 0; h < HALVES; ++h) {
      for (int mt = 0; mt < MT; ++mt)
        tc::tma_load_2d(Qs + h * a.M_pad * 128 + mt * 16384, &maps.q, &bars[0], h * 64, head * a.M_pad + mt * 128);
      tc::tma_load_3d(Ks + h * 16384, &maps.k[hl.l], &bars[0], h * 64, j0, hl.bh);
    }
    if (!tc::mbar_wait(&bars[0], 0)) {
      ok = 0;
      status_or(a.status, KVC_STATUS_TIMEOUT);
      tc::mbar_wait(&bars[0], 0);  // give the copies in flight one more bounded chance to land
    } else {
      tc::fence_after_sync();
      const uint32_t qb = tc::smem_u32(Qs), kb = tc::smem_u32(Ks);
      if (pass == 1) {  // S[row][key]: A = Q M-tile, B = K chunk
        const uint32_t idesc = tc::idesc_bf16(128, kChunk);
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc::umma_bf16(tmem + mt * kChunk,
                          tc::desc_k_sw128(qb + (ks >> 2) * a.M_pad * 128 + mt * 16384 + (ks & 3) * 32),
                          tc::desc_k_sw128(kb + (ks >> 2) * 16384 + (ks & 3) * 32), idesc, ks > 0);
      } else {  // S^T[key][row]: A = K chunk, B = Q (N = M_n rows)
        const uint32_t idesc = tc::idesc_bf16(128, a.M_n);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc::umma_bf16(tmem, tc::desc_k_sw128(kb + (ks >> 2) * 16384 + (ks & 3) * 32),
                        tc::desc_k_sw128(qb + (ks >> 2) * a.M_pad * 128 + (ks & 3) * 32), idesc, ks > 0);
      }
      tc::umma_commit(&bars[1]);
    }
    *s_ok = ok;
  }
  __syncthreads();
  bool ok = *s_ok != 0;
  if (ok && !tc::mbar_wait(&bars[1], 0)) {
    status_or(a.status, KVC_STATUS_TIMEOUT);
    ok = false;
  }
  tc::fence_after_sync();
  return ok;
}

template <int D>
__global__ void __launch_bounds__(256) pass1_tc_kernel(const __grid_constant__ TcMaps maps, ScoreArgs a, ScoreWs ws,
                                                       float c2) {
  extern __shared__ uint8_t smraw[];
  uint8_t* Qs = align1024(smraw);
  uint8_t* Ks = Qs + (size_t)a.M_pad * D * 2;
  uint64_t* bars = reinterpret_cast<uint64_t*>(Ks + kChunk * D * 2);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 2);
  int* s_ok = reinterpret_cast<int*>(slot + 1);
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const int j0 = chunk * kChunk;
  const int nvalid = min(kChunk, a.g.N - j0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = (uint32_t)(a.M_pad >> 7) * kChunk;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::mbar_fence_init();
  }
  if (warp == 0) tc::tmem_alloc(slot, ncols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  if (tc_load_and_mma<D>(maps, a, head, hl, j0, Qs, Ks, bars, tmem, 1, s_ok)) {
    const int mt = warp >> 2, q = warp & 3;
    const int r = mt * 128 + q * 32 + lane;
    float m = -INFINITY, s = 0.f;
#pragma unroll 1
    for (int cs = 0; cs < kChunk / 32; ++cs) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(mt * kChunk + cs * 32), v);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v[i] = (cs * 32 + i < nvalid) ? v[i] * c2 : -INFINITY;
        mx = fmaxf(mx, v[i]);
      }
      if (mx > -INFINITY) {
        const float mn = fmaxf(m, mx);
        s *= exp2f(m - mn);
#pragma unroll
        for (int i = 0; i < 32; ++i) s += exp2f(v[i] - mn);
        m = mn;
      }
    }
    ws.part[((size_t)head * a.nchunk + chunk) * a.M_pad + r] = make_float2(m, s);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, ncols);
}

template <int D>
__global__ void __launch_bounds__(128) pass2_tc_kernel(const __grid_constant__ TcMaps maps, ScoreArgs a, ScoreWs ws,
                                                       float c2) {
  extern __shared__ uint8_t smraw[];
  uint8_t* Qs = align1024(smraw);
  uint8_t* Ks = Qs + (size_t)a.M_pad * D * 2;
  uint64_t* bars = reinterpret_cast<uint64_t*>(Ks + kChunk * D * 2);
  uint32_t* slot = reinterpret_cast<uint32_t*>(bars + 2);
  int* s_ok = reinterpret_cast<int*>(slot + 1);
  float* L2s = reinterpret_cast<float*>(slot + 4);
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const int j0 = chunk * kChunk;
  const int nvalid = min(kChunk, a.g.N - j0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ncols = a.M_n <= 128 ? 128u : 256u;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::mbar_fence_init();
  }
  for (int r = threadIdx.x; r < a.M_pad; r += blockDim.x) L2s[r] = ws.lse2[(size_t)head * a.M_pad + r];
  if (warp == 0) tc::tmem_alloc(slot, ncols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  if (tc_load_and_mma<D>(maps, a, head, hl, j0, Qs, Ks, bars, tmem, 2, s_ok)) {
    const int key = warp * 32 + lane;
    float best = -INFINITY;
    const int nslice = (a.M_n + 31) >> 5;
#pragma unroll 1
    for (int cs = 0; cs < nslice; ++cs) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(cs * 32), v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = cs * 32 + i;
        if (r < a.M_n) best = fmaxf(best, v[i] * c2 - L2s[r]);
      }
    }
    if (key < nvalid) a.scores[(size_t)head * a.g.N + j0 + key] = exp2f(best);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, ncols);
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

int obs_rows(int M, int dtype) {
  if (dtype == KVC_BF16) return M <= 128 ? 128 : 256;  // whole 128-row MMA tiles
  return (M + 15) / 16 * 16;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;  // resolved once from the driver
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

static bool encode_maps(TcMaps* m, const ScoreArgs& a, const ScoreWs& ws) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int D = a.g.D;
  const cuuint32_t es[3] = {1, 1, 1};
  for (int l = 0; l < a.g.L; ++l) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.g.ncap, (cuuint64_t)a.g.B * a.g.Hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.g.ncap * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kChunk, 1};
    if (enc(&m->k[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K.p[l], dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  const cuuint64_t qdims[2] = {(cuuint64_t)D, (cuuint64_t)heads * a.M_pad};
  const cuuint64_t qstrides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t qbox[2] = {64, 128};
  return enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws.obs, qdims, qstrides, qbox, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t score_ws_bytes(const CacheGeom& g, int dtype, int n_r, int n_b, ScoreWs* carve, void* base) {
  const size_t es = dtype == KVC_BF16 ? 2 : 4;
  const size_t heads = (size_t)g.L * g.B * g.Hkv;
  const int G = g.Hq / g.Hkv;
  const int M = G * (n_r + n_b);
  const size_t M_pad = (size_t)obs_rows(M, dtype);
  const size_t nchunk = (size_t)(g.N + kChunk - 1) / kChunk;
  size_t off = 0;
  const size_t o_obs = off;   off += align256(heads * M_pad * g.D * es);
  const size_t o_valid = off; off += align256(heads * M_pad);
  const size_t o_part = off;  off += align256(heads * nchunk * M_pad * sizeof(float2));
  const size_t o_lse = off;   off += align256(heads * M_pad * sizeof(float));
  if (carve) {
    char* b = static_cast<char*>(base);
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
  // observation rows: one warp per query head of the group
  const int G = a.g.Hq / a.g.Hkv;
  const size_t per_warp = sizeof(float) * (size_t)(a.qmax * (D + 1) + a.qmax);
  int nw = G < 8 ? G : 8;
  while (nw > 1 && per_warp * nw > 200u * 1024u) --nw;
  const size_t obs_smem = per_warp * nw;
  {
    bool ok;
    if (a.dtype == KVC_BF16) {
      auto k = D == 128 ? build_obs_kernel<__nv_bfloat16, 128> : build_obs_kernel<__nv_bfloat16, 64>;
      ok = set_smem(k, obs_smem);
      if (ok) k<<<heads, 32 * nw, obs_smem, s>>>(a, ws, nw);
    } else {
      auto k = D == 128 ? build_obs_kernel<float, 128> : build_obs_kernel<float, 64>;
      ok = set_smem(k, obs_smem);
      if (ok) k<<<heads, 32 * nw, obs_smem, s>>>(a, ws, nw);
    }
    if (!ok) return KVC_ERR_LAUNCH;
  }
  if (launch_ok()) return KVC_ERR_LAUNCH;

  const dim3 grid(a.nchunk, heads);
  if (a.dtype == KVC_BF16) {
    TcMaps maps;  // host staging for the kernel parameter (copied at launch)
    if (!encode_maps(&maps, a, ws)) return KVC_ERR_LAUNCH;
    const int MT = a.M_pad >> 7;
    const size_t tail = 64 + (size_t)a.M_pad * 4;  // barriers, TMEM slot, flag, lse2 copy
    size_t sm = 1024 + (size_t)(a.M_pad + kChunk) * D * 2 + tail;
    // Never let more CTAs share an SM than its 512 TMEM columns can serve at once: ask for
    // enough shared memory that one more CTA would not fit.
    int dev = 0, smem_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    const int cols = (a.M_pad > 128 || a.M_n > 128) ? 256 : 128;
    const size_t floor_sm = (size_t)smem_sm / (size_t)(512 / cols + 1) + 1024;
    if (sm < floor_sm) sm = floor_sm;
    if (D == 128) {
      if (!set_smem(pass1_tc_kernel<128>, sm) || !set_smem(pass2_tc_kernel<128>, sm)) return KVC_ERR_LAUNCH;
      pass1_tc_kernel<128><<<grid, 128 * MT, sm, s>>>(maps, a, ws, c2);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      combine_kernel<<<heads, (a.M_pad + 31) / 32 * 32, 0, s>>>(a, ws);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      pass2_tc_kernel<128><<<grid, 128, sm, s>>>(maps, a, ws, c2);
    } else {
      if (!set_smem(pass1_tc_kernel<64>, sm) || !set_smem(pass2_tc_kernel<64>, sm)) return KVC_ERR_LAUNCH;
      pass1_tc_kernel<64><<<grid, 128 * MT, sm, s>>>(maps, a, ws, c2);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      combine_kernel<<<heads, (a.M_pad + 31) / 32 * 32, 0, s>>>(a, ws);
      if (launch_ok()) return KVC_ERR_LAUNCH;
      pass2_tc_kernel<64><<<grid, 128, sm, s>>>(maps, a, ws, c2);
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
