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
//   bf16 caches: both passes on the tensor cores in one persistent kernel:
//                score_resident (score_resident.cu) when the observation tile is one
//                128-row MMA tile and a head spreads over at most one CTA per SM in
//                256-key pieces (pass-1 logits kept in TMEM, every key read once);
//                otherwise score_fused (score_fused.cu), which reads the keys twice
//   fp32 caches of at most 1024 keys per head: score_small (score_small.cu), one cluster launch
//                that also builds the observation rows (no build_obs launch)
//   other fp32 caches: pass1 / combine / pass2 below on CUDA cores:
//     pass1      per (key chunk, head): per-row chunk max and sum of exp2
//     combine    per head: merge the partials into lse2 per row
//     pass2      per (key chunk, head): max over rows of s*log2(e)/sqrt(D) - lse2, exp2
// Softmax is kept in base 2 throughout: exp(s/sqrt(D) - lse) = exp2(s*c2 - lse2).
#include <stdlib.h>
#include <string.h>

#include "obs_rows.cuh"

namespace kvc {

// ---------------------------------------------------------------------------
// rotary table and observation rows
// ---------------------------------------------------------------------------
// The order in which kvc_evict's selection-and-compaction CTAs take the heads when each head has its
// own budget: largest budget first, so that the longest moves start in the launch's first wave
// instead of trailing it (one warp moves a head's K, another its V; a head of many scattered kept
// rows is the slowest). Heads go into 128 buckets, four per octave of the budget clamped to [1, N],
// largest first; heads within a bucket in any order. Run by one whole CTA.
__device__ void head_order_cta(const int32_t* budget, int heads, int N, int32_t* order) {
  __shared__ int cnt[128];
  auto bucket = [&](int h) {
    int b = budget[h];
    b = b < 1 ? 1 : (b > N ? N : b);
    const int e = 31 - __clz(b);                                   // floor(log2 b)
    const int f = e >= 2 ? (b >> (e - 2)) & 3 : (b << (2 - e)) & 3;  // the next two bits
    const int k = 4 * e + f;
    return 127 - (k < 127 ? k : 127);
  };
  for (int i = threadIdx.x; i < 128; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int h = threadIdx.x; h < heads; h += blockDim.x) atomicAdd(&cnt[bucket(h)], 1);
  __syncthreads();
  if (threadIdx.x == 0) {  // bucket counts -> first positions
    int sum = 0;
    for (int i = 0; i < 128; ++i) {
      const int c = cnt[i];
      cnt[i] = sum;
      sum += c;
    }
  }
  __syncthreads();
  for (int h = threadIdx.x; h < heads; h += blockDim.x) order[atomicAdd(&cnt[bucket(h)], 1)] = h;
  __syncthreads();
}

template <typename T, int D>
__global__ void build_obs_kernel(ScoreArgs a, ScoreWs ws, int nw) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_nvalid;  // valid observation rows of this KV head (for the entropy's mean)
  const int head = blockIdx.x;
  if (a.order && head == 0) head_order_cta(a.order_budget, a.g.L * a.g.B * a.g.Hkv, a.g.N, a.order);
  const int G = a.g.Hq / a.g.Hkv, qs = a.qstride;
  T* obs = static_cast<T*>(ws.obs) + (size_t)head * a.M_pad * D;
  uint8_t* valid = ws.valid + (size_t)head * a.M_pad;
  // the CTA's nw warps (nw <= G, so every warp has a query head and reaches the shared step of the
  // first one)
  obs_group_rows<T, D>(a, ws, head, nw, smem_raw, obs, valid, &s_nvalid);
  obs_padding<T, D>(a, obs, valid);
  const bool mean_w = a.ext && a.row_agg == KVC_AGG_MEAN;
  if (a.ext) {
    if (mean_w)
      for (int r = (G - 1) * qs + qs + threadIdx.x; r < a.M_pad; r += blockDim.x) ws.rw[(size_t)head * a.M_pad + r] = 0.f;
    __syncthreads();
    if (threadIdx.x == 0) {
      // the scoring kernel adds -sum p log2 p of its rows and keys, times this scale, into entropy
      const int nv = s_nvalid;
      ws.escale[head] = (nv > 0 && a.g.N > 1) ? 1.f / ((float)nv * log2f((float)a.g.N)) : 0.f;
      if (a.entropy) a.entropy[head] = 0.f;
    }
  }
}

struct HeadLoc {
  int l, bh;
};
__device__ __forceinline__ HeadLoc head_loc(const CacheGeom& g, int head) {
  return HeadLoc{head / (g.B * g.Hkv), head % (g.B * g.Hkv)};
}

// ---------------------------------------------------------------------------
// fp32 passes (CUDA-core FMA; fp32 storage is the small-model path)
// ---------------------------------------------------------------------------
// q . k over D floats with four independent accumulators (the loop fully unrolled, so the shared
// memory loads of later terms are in flight while earlier products accumulate)
template <int D>
__device__ __forceinline__ float dot_f32(const float* __restrict__ q, const float* __restrict__ k) {
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int d = 0; d < D; d += 4) {
#pragma unroll
    for (int u = 0; u < 4; ++u) acc[u] = fmaf(q[d + u], k[d + u], acc[u]);
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// fp32 caches are scored in chunks of 32 keys (one row per thread in pass 1, one key per thread
// in pass 2), so that even a small cache spreads over many CTAs
constexpr int kF32Chunk = 32;

template <int D>
__global__ void __launch_bounds__(128) pass1_f32_kernel(ScoreArgs a, ScoreWs ws, float c2) {
  extern __shared__ __align__(16) float smf[];
  constexpr int LQ = D + 1;
  float* Qs = smf;                   // [M_pad][D+1]
  float* Ks = Qs + a.M_pad * LQ;     // [kF32Chunk][D]
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const float* Kh = static_cast<const float*>(a.K.p[hl.l]) + (size_t)hl.bh * a.g.ncap * D;
  const int j0 = chunk * kF32Chunk;
  const int nvalid = min(kF32Chunk, a.g.N - j0);
  const float* obs = static_cast<const float*>(ws.obs) + (size_t)head * a.M_pad * D;
  for (int e = threadIdx.x; e < a.M_pad * D; e += blockDim.x) Qs[(e / D) * LQ + e % D] = obs[e];
  for (int e = threadIdx.x; e < nvalid * D; e += blockDim.x) Ks[e] = Kh[(size_t)j0 * D + e];
  __syncthreads();
  for (int r = threadIdx.x; r < a.M_pad; r += blockDim.x) {
    float m = -INFINITY, s = 0.f;
    for (int j = 0; j < nvalid; ++j) {
      const float x = dot_f32<D>(Qs + r * LQ, Ks + j * D) * c2;
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

template <int D>
__global__ void __launch_bounds__(128) pass2_f32_kernel(ScoreArgs a, ScoreWs ws, float c2) {
  extern __shared__ __align__(16) float smf[];
  constexpr int LK = D + 1;
  float* Qs = smf;                  // [M_pad][D]
  float* Ks = Qs + a.M_pad * D;     // [kF32Chunk][D+1]
  float* L2s = Ks + kF32Chunk * LK; // [M_pad]
  float* RWs = L2s + a.M_pad;       // [M_pad] row weights (extended epilogue, mean over rows)
  const int chunk = blockIdx.x, head = blockIdx.y;
  const HeadLoc hl = head_loc(a.g, head);
  const float* Kh = static_cast<const float*>(a.K.p[hl.l]) + (size_t)hl.bh * a.g.ncap * D;
  const int j0 = chunk * kF32Chunk;
  const int nvalid = min(kF32Chunk, a.g.N - j0);
  const float* obs = static_cast<const float*>(ws.obs) + (size_t)head * a.M_pad * D;
  const bool mean = a.ext && a.row_agg == KVC_AGG_MEAN;
  for (int e = threadIdx.x; e < a.M_pad * D; e += blockDim.x) Qs[e] = obs[e];
  for (int e = threadIdx.x; e < nvalid * D; e += blockDim.x) Ks[(e / D) * LK + e % D] = Kh[(size_t)j0 * D + e];
  for (int r = threadIdx.x; r < a.M_pad; r += blockDim.x) {
    L2s[r] = ws.lse2[(size_t)head * a.M_pad + r];
    if (mean) RWs[r] = ws.rw[(size_t)head * a.M_pad + r];
  }
  __syncthreads();
  const int j = threadIdx.x;
  if (!a.ext) {
    if (j >= nvalid) return;
    float best = -INFINITY;
    for (int r = 0; r < a.M_pad; ++r) best = fmaxf(best, dot_f32<D>(Qs + r * D, Ks + j * LK) * c2 - L2s[r]);
    a.scores[(size_t)head * a.g.N + j0 + j] = exp2f(best);
    return;
  }
  // Extended epilogue: p = exp2(s*c2 - lse2) per row; the max (or row-weighted sum) over each
  // query head's rows (rows of head g start at g * qstride), then the max or sum over heads;
  // -sum p log2 p over rows and keys for the entropy.
  const bool gsum = a.group_agg == KVC_AGG_SUM;
  float hacc = 0.f, gacc = 0.f, cv = 0.f;  // values >= 0: 0 is the identity of max and sum
  int cur = -1;
  if (j < nvalid) {
    for (int r = 0; r < a.M_pad; ++r) {
      const float y = dot_f32<D>(Qs + r * D, Ks + j * LK) * c2 - fminf(L2s[r], 1e30f);  // unused rows: p = 0
      const float e = exp2f(y);
      hacc = fmaf(e, y, hacc);
      const int sg = r / a.qstride;
      const float v = mean ? RWs[r] * e : e;
      if (sg != cur) {
        if (cur >= 0) gacc = gsum ? gacc + cv : fmaxf(gacc, cv);
        cur = sg;
        cv = v;
      } else {
        cv = mean ? cv + v : fmaxf(cv, v);
      }
    }
    gacc = gsum ? gacc + cv : fmaxf(gacc, cv);
    a.scores[(size_t)head * a.g.N + j0 + j] = gacc;
  }
  if (a.entropy) {
    const float h = warp_sum(hacc);
    if ((threadIdx.x & 31) == 0) atomicAdd(&a.entropy[head], -h * ws.escale[head]);
  }
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

size_t score_ws_bytes(const CacheGeom& g, int dtype, int n_r, int n_b, bool ext, ScoreWs* carve, void* base) {
  const size_t es = dtype == KVC_BF16 ? 2 : 4;
  const size_t heads = (size_t)g.L * g.B * g.Hkv;
  const int G = g.Hq / g.Hkv;
  const int M = obs_rows_used(G, n_r, n_b, ext);
  const size_t M_pad = (size_t)obs_rows(M, dtype);
  const size_t nchunk = dtype == KVC_BF16 ? (size_t)(g.N + kChunk - 1) / kChunk : (size_t)(g.N + kF32Chunk - 1) / kF32Chunk;
  size_t off = 0;
  const size_t o_obs = off;   off += align256(heads * M_pad * g.D * es);
  const size_t o_valid = off; off += align256(heads * M_pad);
  // fp32 caches keep per-chunk partials; bf16 caches exchange per-range partials in the fused kernel
  // (twice that with the extended options: the single-read kernel then also publishes each row's mean logit)
  const size_t part_bytes = dtype == KVC_BF16 ? fused_xch_bytes((int)M_pad) * (ext ? 2 : 1)
                                              : heads * nchunk * M_pad * sizeof(float2);
  const size_t o_part = off;  off += align256(part_bytes);
  const size_t o_lse = off;   off += align256(heads * M_pad * sizeof(float));
  const size_t o_rw = off;    off += ext ? align256(heads * M_pad * sizeof(float)) : 0;
  const size_t o_esc = off;   off += ext ? align256(heads * sizeof(float)) : 0;
  const size_t o_ent = off;   off += ext ? align256(heads * sizeof(float)) : 0;
  // the two-pass streaming kernels' per-range partials and the wide kernel's fallback list (bf16,
  // default options only)
  const size_t ranges = (size_t)split_ranges((int)nchunk, (int)M_pad);
  const size_t o_l2p = off;
  if (dtype == KVC_BF16 && !ext) off += align256(heads * ranges * M_pad * sizeof(float));
  const size_t o_fb = off;
  if (dtype == KVC_BF16 && !ext) off += align256((1 + heads * ranges) * sizeof(int32_t));
  if (carve) {
    char* b = static_cast<char*>(base);
    carve->obs = b + o_obs;
    carve->valid = reinterpret_cast<uint8_t*>(b + o_valid);
    carve->part = reinterpret_cast<float2*>(b + o_part);
    carve->lse2 = reinterpret_cast<float*>(b + o_lse);
    carve->rw = ext ? reinterpret_cast<float*>(b + o_rw) : nullptr;
    carve->escale = ext ? reinterpret_cast<float*>(b + o_esc) : nullptr;
    carve->ent = ext ? reinterpret_cast<float*>(b + o_ent) : nullptr;
    carve->lse2p = (dtype == KVC_BF16 && !ext) ? reinterpret_cast<float*>(b + o_l2p) : nullptr;
    carve->fb = (dtype == KVC_BF16 && !ext) ? reinterpret_cast<int32_t*>(b + o_fb) : nullptr;
  }
  return off;
}

template <typename K>
static bool set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

// Which bf16 scoring kernel runs (sets a->tiles); 0 = fp32 passes.
enum ScorePath { kPathF32 = 0, kPathResident = 1, kPathSplit = 2, kPathFused = 3, kPathWide = 4, kPathSmall = 5 };
static ScorePath choose_score(ScoreArgs* a, FusedPlan* rp, size_t* rsmem, SplitPlan* sp, size_t* ssmem,
                              WidePlan* wp, size_t* wsmem, bool evict = false) {
  a->tiles = 1;
  // fp32: one cluster launch for short caches (score_small.cu) unless the streaming passes are asked for
  if (a->dtype != KVC_BF16)
    return (a->kernel != KVC_KERNEL_SPLIT && score_small_plan(*a, ssmem, evict)) ? kPathSmall : kPathF32;
  // A 256-row observation tile goes to the single-read kernel as two 128-row tiles when no query
  // head's rows cross the tile boundary (or the aggregation is max over everything, where heads do
  // not matter).
  if (a->M_pad == 2 * 128) {
    bool straddle = false;
    const int per_q = a->n_r + a->n_b, G = a->g.Hq / a->g.Hkv;
    if (a->row_agg != KVC_AGG_MAX || a->group_agg != KVC_AGG_MAX)
      for (int g = 0; g < G; ++g) straddle |= (g * a->qstride) / 128 != (g * a->qstride + per_q - 1) / 128;
    if (!straddle) a->tiles = 2;
  }
  bool resident = score_resident_plan(*a, rp, rsmem);
  // The two-pass streaming kernel takes over where the single-read kernel's per-round meetings
  // would involve many CTAs (more than 16 per head, i.e. more than 4096 keys) or two row tiles.
  bool split = score_split_plan(*a, sp, ssmem);
  const int path = a->kernel;  // KVC_KERNEL_*: forced by the caller (tests, profiling) or automatic
  if (split && path == KVC_KERNEL_AUTO) split = !resident || a->M_pad > 128 || rp->group_size > 16;
  if (split && path != KVC_KERNEL_AUTO) split = path == KVC_KERNEL_SPLIT;
  if (resident && path == KVC_KERNEL_FUSED) resident = false;
  // Tiles of more than 128 rows with default options go to the wide kernel (keys on the TMEM lanes,
  // one MMA chain per chunk over every row), unless another kernel is asked for.
  const bool wide = score_wide_plan(*a, wp, wsmem) &&
                    (path == KVC_KERNEL_WIDE || (path == KVC_KERNEL_AUTO && split && a->M_pad > 128));
  if (wide) {
    a->tiles = 1;
    return kPathWide;
  }
  if (split) resident = false;
  if (!resident) a->tiles = 1;
  return resident ? kPathResident : (split ? kPathSplit : kPathFused);
}

int score_launches(const CacheGeom& g, int dtype, int n_r, int n_b, bool ext) {
  ScoreArgs a;
  memset(&a, 0, sizeof(a));
  a.g = g;
  a.dtype = dtype;
  a.n_r = n_r;
  a.n_b = n_b;
  a.ext = ext ? 1 : 0;
  a.qstride = obs_qstride(n_r, n_b, ext);
  a.M = obs_rows_used(g.Hq / g.Hkv, n_r, n_b, ext);
  a.M_pad = obs_rows(a.M, dtype);
  a.M_n = (a.M + 15) / 16 * 16;  // the wide kernel's plan reads it
  a.qmax = 2 * n_b;
  a.nchunk = (g.N + kChunk - 1) / kChunk;
  FusedPlan rp;
  SplitPlan sp;
  WidePlan wp;
  size_t r1 = 0, r2 = 0, r3 = 0;
  switch (choose_score(&a, &rp, &r1, &sp, &r2, &wp, &r3)) {
    case kPathF32: return 4;    // observation rows, pass 1, combine, pass 2
    case kPathSmall: return 1;  // one cluster kernel (observation rows included)
    case kPathSplit: return 4;  // observation rows, pass 1, combine, pass 2
    case kPathWide: return 5;   // observation rows, pass 1, exact fallback, combine, pass 2
    default: return 2;          // observation rows, one scoring kernel
  }
}

bool evict_fused_small(const CacheGeom& g, int dtype, int n_r, int n_b) {
  ScoreArgs a;
  memset(&a, 0, sizeof(a));
  a.g = g;
  a.dtype = dtype;
  a.n_r = n_r;
  a.n_b = n_b;
  a.qstride = obs_qstride(n_r, n_b, false);
  a.M = obs_rows_used(g.Hq / g.Hkv, n_r, n_b, false);
  a.M_pad = obs_rows(a.M, dtype);
  a.qmax = 2 * n_b;  // the continual-FPS buffer of twice the beacons
  size_t smem = 0;
  return dtype == KVC_F32 && score_small_plan(a, &smem, true);
}

int launch_score(const ScoreArgs& a_in, const ScoreWs& ws, cudaStream_t s, const SmallEvict* ev, bool* fused) {
  ScoreArgs a = a_in;
  if (fused) *fused = false;
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  // the single-read kernel's plan is fixed first: the observation kernel zeroes its exchange words.
  FusedPlan rp;
  SplitPlan sp;
  WidePlan wp;
  size_t rsmem = 0, ssmem = 0, wsmem = 0;
  const ScorePath path = choose_score(&a, &rp, &rsmem, &sp, &ssmem, &wp, &wsmem, ev != nullptr);
  if (path == kPathSmall) {  // the cluster kernel builds the observation rows itself
    a.xch_zero = nullptr;
    a.xch_zero_words = 0;
    if (ev && fused) *fused = true;
    return launch_score_small(a, ws, s, ev && fused ? ev : nullptr);
  }
  const bool resident = path == kPathResident, split = path == kPathSplit, wide = path == kPathWide;
  // the observation kernel zeroes the single-read kernel's exchange words, or the wide kernel's
  // fallback count
  a.xch_zero = resident ? reinterpret_cast<unsigned long long*>(ws.part)
                        : (wide ? reinterpret_cast<unsigned long long*>(ws.fb) : nullptr);
  a.xch_zero_words = resident ? score_resident_words(rp, a.entropy != nullptr) : (wide ? 1 : 0);
  const int D = a.g.D;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  // observation rows: one warp per query head of the group
  const int G = a.g.Hq / a.g.Hkv;
  const int npad = (a.qmax + 15) & ~15;
  const size_t raw = a.dtype == KVC_BF16
                         ? (D == 128 ? fps_scratch_bytes<__nv_bfloat16, 128>(npad) : fps_scratch_bytes<__nv_bfloat16, 64>(npad))
                         : (D == 128 ? fps_scratch_bytes<float, 128>(npad) : fps_scratch_bytes<float, 64>(npad));
  const size_t per_warp = (raw + 15) & ~(size_t)15;
  int nw = G < 8 ? G : 8;
  while (nw > 1 && per_warp * nw > 200u * 1024u) --nw;
  const size_t obs_smem = per_warp * nw + 64 * sizeof(float2);  // + the rotation table
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
    if (resident) return launch_score_resident(a, ws, rp, rsmem, s);
    if (wide) return launch_score_wide(a, ws, wp, wsmem, s);
    if (split) return launch_score_split(a, ws, sp, ssmem, s);
    return launch_score_fused(a, ws, ws.part, s);
  } else {
    a.nchunk = (a.g.N + kF32Chunk - 1) / kF32Chunk;
    const dim3 fgrid(a.nchunk, heads);
    const size_t sm1 = sizeof(float) * ((size_t)a.M_pad * (D + 1) + (size_t)kF32Chunk * D);
    const size_t sm2 = sizeof(float) * ((size_t)a.M_pad * D + (size_t)kF32Chunk * (D + 1) + 2 * (size_t)a.M_pad);
    auto p1 = D == 128 ? pass1_f32_kernel<128> : pass1_f32_kernel<64>;
    auto p2 = D == 128 ? pass2_f32_kernel<128> : pass2_f32_kernel<64>;
    if (!set_smem(p1, sm1) || !set_smem(p2, sm2)) return KVC_ERR_LAUNCH;
    p1<<<fgrid, 128, sm1, s>>>(a, ws, c2);
    if (launch_ok()) return KVC_ERR_LAUNCH;
    combine_kernel<<<heads, (a.M_pad + 31) / 32 * 32, 0, s>>>(a, ws);
    if (launch_ok()) return KVC_ERR_LAUNCH;
    p2<<<fgrid, kF32Chunk, sm2, s>>>(a, ws, c2);
  }
  return launch_ok();
}

}  // namespace kvc
