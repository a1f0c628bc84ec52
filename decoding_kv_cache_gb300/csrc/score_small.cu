// score_small.cu -- fp32 scoring of short caches in one launch: a thread-block cluster per KV head.
//
// What it computes is kvc_score's definition (BeaconKV write-up, "打分时的 RoPE 对齐": a key's
// importance is the max over the observation rows of its softmax weight over all cached keys),
// the same as the observation kernel and the fp32 streaming passes of score.cu, for caches short
// enough that a head's keys spread over at most eight CTAs of at most 128 keys each:
//   every CTA of the head's cluster starts the copies of its own keys into shared memory and, while
//   they are in flight, builds the head's observation tile there itself (obs_rows.cuh: recent rows,
//   FPS beacons rotated to t; each CTA of the cluster repeats this small step instead of waiting for
//   another kernel); it forms its block of logits s c2 once (CUDA-core fp32 FMA, kept in shared
//   memory) and reduces each row to a partial (max, sum of exp2) over its keys;
//   after a cluster barrier every CTA reads the cluster's partials of each row from distributed
//   shared memory and merges them in rank order (every CTA forms the same lse2);
//   each CTA then writes exp2(max over rows of s c2 - lse2) for its keys.
// K is read once and the step is one launch. Called from kvc_evict, the same launch also selects
// and compacts:
//   every CTA also stages its keys' V rows at the start; after a cluster barrier every CTA gathers
//   the head's scores from the cluster as order-preserving keys (select_head.cuh's score_key) and
//   ranks its own middle keys against them (kept: fewer than kmid middle keys rank above, ties to
//   the lower index, which is kvc_select's set); the CTAs' kept counts give each kept key its slot,
//   and every CTA writes its kept keys' indices and rows there from shared memory. Every CTA has
//   read its rows before the first barrier, so the in-place moves cannot overwrite a row still to
//   be read.
#include <string.h>

#include "obs_rows.cuh"
#include "select_head.cuh"

namespace kvc {

struct SmallPlan {
  int C;        // CTAs per head (the cluster)
  int kpc;      // keys per CTA
  int kpad;     // kpc rounded up to even
  int nw;       // warps building the observation rows
  int ufloats;  // floats of the region shared by the FPS scratch and the logits
};

constexpr int kSmallThreads = 256;
constexpr int kSmallMaxKeys = 128;  // keys per CTA
constexpr int kSmallMaxCluster = 8;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// every thread of the cluster: this CTA's shared-memory writes before the barrier are visible to
// the cluster's reads after it
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ float2 ld_cluster_f2(const float2* p, uint32_t rank) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"(a), "r"(rank));
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(ra) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(ra) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
  return ra;
}
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_i32(const int* p, uint32_t rank) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];\n" : "=r"(v) : "r"(cluster_addr(p, rank)) : "memory");
  return v;
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}

template <int D>
__global__ void __launch_bounds__(kSmallThreads)
    score_small_f32_kernel(ScoreArgs a, ScoreWs ws, SmallPlan p, float c2, SmallEvict ev, int evict) {
  extern __shared__ __align__(16) float sm[];
  __shared__ int s_nvalid;
  constexpr int LD = D + 4;  // key row stride: 16-byte rows, eight consecutive rows on distinct bank groups
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();
  const int head = blockIdx.x / p.C;
  const int Mp = a.M_pad;
  const int LS = p.kpad + 1;  // logit row stride (odd: a thread per row reads without conflicts)
  float* Qs = sm;                                      // [Mp][D] observation rows
  float* Ks = Qs + Mp * D;                             // [kpad][LD] this CTA's keys
  float* Vs = Ks + p.kpad * LD;                        // [kpad][D] their values (evict only)
  float* U = Vs + (evict ? p.kpad * D : 0);            // the FPS scratch, later the logits and partials
  uint8_t* validS = reinterpret_cast<uint8_t*>(U + p.ufloats);  // [Mp] observation row flags
  float* Ss = U;                                       // [Mp][LS] logits times c2
  float2* part = reinterpret_cast<float2*>(Ss + ((Mp * LS + 1) & ~1));  // [Mp] (max, sum) over this CTA's keys
  float* lse = reinterpret_cast<float*>(part + Mp);    // [Mp] lse2 of the row (+inf: no observation)
  float* red = lse + Mp;                               // [8][kpad] per-slice maxima
  float* own = red + 8 * p.kpad;                       // [kpad] this CTA's scores (evict)
  int* pos_s = reinterpret_cast<int*>(own + p.kpad);   // [kpad] kept slot of each key, or -1 (evict)
  int* wtot = pos_s + p.kpad;                          // [8] kept keys per warp (evict)
  int* my_count = wtot + 8;                            // kept keys of this CTA (evict)
  const int j0 = (int)rank * p.kpc;
  const int nk = max(0, min(p.kpc, a.g.N - j0));

  // everything this kernel reads may come from the previous kernel on the stream
  griddep_wait();
  const int l = head / (a.g.B * a.g.Hkv), bh = head % (a.g.B * a.g.Hkv);
  const float* Kh = static_cast<const float*>(a.K.p[l]) + ((size_t)bh * a.g.ncap + j0) * D;
  constexpr int V = D / 4;  // 16-byte vectors per row
  for (int e = tid; e < p.kpad * V; e += kSmallThreads) {
    const int r = e / V, v = e % V;
    if (r < nk) cp_async16(Ks + r * LD + 4 * v, Kh + (size_t)r * D + 4 * v);
    else *reinterpret_cast<float4*>(Ks + r * LD + 4 * v) = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (evict) {
    const float* Vh = static_cast<const float*>(ev.V.p[l]) + ((size_t)bh * a.g.ncap + j0) * D;
    for (int e = tid; e < nk * V; e += kSmallThreads) cp_async16(Vs + 4 * e, Vh + 4 * (size_t)e);
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  // the observation rows, built by every CTA of the cluster for itself (the first p.nw warps take
  // the query heads; one CTA reports the beacon picks)
  if ((int)(tid >> 5) < p.nw)
    obs_group_rows<float, D>(a, ws, head, p.nw, reinterpret_cast<unsigned char*>(U), Qs, validS, &s_nvalid, rank == 0);
  obs_padding<float, D>(a, Qs, validS);
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
  __syncthreads();

  // logits: a thread forms 4 rows x 2 keys at a time, 16-byte reads along D
  const int nkg = p.kpad / 2;
  for (int mt = tid; mt < (Mp / 4) * nkg; mt += kSmallThreads) {
    const int rg = mt / nkg, kg = mt % nkg;
    const float* q0 = Qs + 4 * rg * D;
    const float* k0 = Ks + 2 * kg * LD;
    float acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = 0.f;
#pragma unroll
    for (int d = 0; d < D; d += 4) {
      const float4 ka = *reinterpret_cast<const float4*>(k0 + d);
      const float4 kb = *reinterpret_cast<const float4*>(k0 + LD + d);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 q = *reinterpret_cast<const float4*>(q0 + i * D + d);  // one address per 8 lanes
        acc[i][0] = fmaf(q.w, ka.w, fmaf(q.z, ka.z, fmaf(q.y, ka.y, fmaf(q.x, ka.x, acc[i][0]))));
        acc[i][1] = fmaf(q.w, kb.w, fmaf(q.z, kb.z, fmaf(q.y, kb.y, fmaf(q.x, kb.x, acc[i][1]))));
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      Ss[(4 * rg + i) * LS + 2 * kg] = acc[i][0] * c2;
      Ss[(4 * rg + i) * LS + 2 * kg + 1] = acc[i][1] * c2;
    }
  }
  __syncthreads();

  // each row's (max, sum of exp2) over this CTA's keys
  for (int r = tid; r < Mp; r += kSmallThreads) {
    const float* sr = Ss + r * LS;
    float m = -INFINITY;
    for (int j = 0; j < nk; ++j) m = fmaxf(m, sr[j]);
    float s = 0.f;
    if (m > -INFINITY)
      for (int j = 0; j < nk; ++j) s += exp2f(sr[j] - m);
    part[r] = make_float2(m, s);
  }
  cluster_sync_all();

  // the head's lse2 per row: the cluster's partials merged in rank order
  for (int r = tid; r < Mp; r += kSmallThreads) {
    float2 pv[kSmallMaxCluster];  // every remote read in flight before the merge
#pragma unroll
    for (int c = 0; c < kSmallMaxCluster; ++c)
      pv[c] = c < p.C ? ld_cluster_f2(part + r, (uint32_t)c) : make_float2(-INFINITY, 0.f);
    float M2 = -INFINITY, S = 0.f;
#pragma unroll
    for (int c = 0; c < kSmallMaxCluster; ++c) {
      const float2 v = pv[c];
      if (v.x > M2) {
        S = S * exp2f(M2 - v.x) + v.y;
        M2 = v.x;
      } else if (v.x > -INFINITY) {
        S += v.y * exp2f(v.x - M2);
      }
    }
    const bool ok = validS[r] != 0;
    lse[r] = ok ? M2 + log2f(S) : INFINITY;
  }
  // every remote read of `part` is done before any CTA of the cluster may exit, and lse is
  // visible to the whole CTA
  cluster_sync_all();

  // scores: eight slices of the rows per key, then the max of the slices
  for (int e = tid; e < 8 * p.kpad; e += kSmallThreads) {
    const int j = e % p.kpad, sl = e / p.kpad;
    float best = -INFINITY;
    for (int r = sl; r < Mp; r += 8) best = fmaxf(best, Ss[r * LS + j] - lse[r]);
    red[sl * p.kpad + j] = best;
  }
  __syncthreads();
  for (int j = tid; j < nk; j += kSmallThreads) {
    float best = red[j];
#pragma unroll
    for (int sl = 1; sl < 8; ++sl) best = fmaxf(best, red[sl * p.kpad + j]);
    const float sc = exp2f(best);
    a.scores[(size_t)head * a.g.N + j0 + j] = sc;
    own[j] = sc;
  }
  if (!evict) return;

  // ---- selection: the prefix and recent windows are kept, and of the middle the kmid keys of
  // highest score, ties to the lower index (the order of kvc_select). Every CTA gathers the head's
  // scores as order-preserving keys from the cluster and ranks its own middle keys against them.
  const int N = a.g.N, P = ev.P, R = ev.R;
  const int b = ev.budget ? ev.budget[head] : ev.budget_all;
  const bool keep_all = b >= N || b < P + R;  // out-of-range budgets keep everything and are flagged
  if (keep_all && b < N && rank == 0 && tid == 0) status_or(a.status, KVC_STATUS_BUDGET_RANGE);
  const int lo = P, hi = N - R, kmid = b - P - R;
  uint32_t* allK = reinterpret_cast<uint32_t*>(Ss);  // [N] (the logits are no longer needed)
  int* cnt = reinterpret_cast<int*>(red);            // [nsl][kpad] partial counts
  cluster_sync_all();  // every CTA's scores are in its `own`
  if (!keep_all)
    for (int k = tid; k < N; k += kSmallThreads)
      allK[k] = score_key(__float_as_uint(ld_cluster_f32(own + k % p.kpc, (uint32_t)(k / p.kpc))));
  __syncthreads();
  int nsl = kSmallThreads / p.kpad;
  nsl = nsl < 1 ? 1 : (nsl > 8 ? 8 : nsl);
  if (!keep_all)
    for (int e = tid; e < nsl * p.kpad; e += kSmallThreads) {
      const int j = e % p.kpad, sl = e / p.kpad, jj = j0 + j;
      int c = 0;  // middle keys ranked above key jj: a larger key, or an equal key at a lower index
      if (j < nk && jj >= lo && jj < hi) {
        const uint32_t kj = allK[jj];
        for (int k = lo + sl; k < hi; k += nsl) {
          const uint32_t kk = allK[k];
          c += (kk > kj || (kk == kj && k < jj)) ? 1 : 0;
        }
      }
      cnt[sl * p.kpad + j] = c;
    }
  __syncthreads();
  // this CTA's kept keys in index order (a thread per key: kpad <= 128 < the CTA's threads)
  bool kept = false;
  if (tid < nk) {
    const int jj = j0 + tid;
    if (keep_all || jj < lo || jj >= hi) {
      kept = true;
    } else {
      int c = 0;
      for (int sl = 0; sl < nsl; ++sl) c += cnt[sl * p.kpad + tid];
      kept = c < kmid;
    }
  }
  const int lane = tid & 31, warp = tid >> 5;
  const unsigned bal = __ballot_sync(kFull, kept);
  if (lane == 0) wtot[warp] = __popc(bal);
  __syncthreads();
  int before = __popc(bal & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) before += wtot[w];
  if (tid == 0) {
    int t = 0;
    for (int w = 0; w < kSmallThreads / 32; ++w) t += wtot[w];
    *my_count = t;
  }
  cluster_sync_all();  // every CTA's count is visible
  int cc[kSmallMaxCluster];
#pragma unroll
  for (int c = 0; c < kSmallMaxCluster; ++c) cc[c] = c < p.C ? ld_cluster_i32(my_count, (uint32_t)c) : 0;
  int base = 0, total = 0;
#pragma unroll
  for (int c = 0; c < kSmallMaxCluster; ++c) {
    total += cc[c];
    base += c < (int)rank ? cc[c] : 0;
  }
  // after this barrier no CTA reads another's shared memory, and every CTA read its own rows at the
  // start: the in-place moves below overwrite nothing still to be read
  cluster_sync_all();
  int32_t* ki = ev.kept_idx + (size_t)head * N;
  if (tid < p.kpad) pos_s[tid] = kept ? base + before : -1;
  if (kept) ki[base + before] = j0 + tid;
  if (rank == 0 && tid == 0) ev.kept_len[head] = total;
  __syncthreads();
  // ---- compaction: this CTA's kept rows to their slots, from shared memory (rows in place stay)
  float* Kd = static_cast<float*>(a.K.p[l]) + (size_t)bh * a.g.ncap * D;
  float* Vd = static_cast<float*>(ev.V.p[l]) + (size_t)bh * a.g.ncap * D;
  for (int e = tid; e < nk * V; e += kSmallThreads) {
    const int j = e / V, v = e % V;
    const int pos = pos_s[j];
    if (pos >= 0 && pos != j0 + j) {
      *reinterpret_cast<float4*>(Kd + (size_t)pos * D + 4 * v) = *reinterpret_cast<const float4*>(Ks + j * LD + 4 * v);
      *reinterpret_cast<float4*>(Vd + (size_t)pos * D + 4 * v) = *reinterpret_cast<const float4*>(Vs + j * D + 4 * v);
    }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static size_t small_smem(const ScoreArgs& a, SmallPlan* p, bool evict) {
  const size_t Mp = (size_t)a.M_pad, D = (size_t)a.g.D, LD = D + 4, LS = (size_t)p->kpad + 1;
  const int npad = (a.qmax + 15) & ~15;
  const size_t warp_bytes = ((D == 128 ? fps_scratch_bytes<float, 128>(npad) : fps_scratch_bytes<float, 64>(npad)) + 15) &
                            ~(size_t)15;
  const size_t fps = (size_t)p->nw * warp_bytes + (D / 2) * sizeof(float2);
  // logits, partials, lse2, slice maxima, and (kvc_evict) own scores, slots, warp counts
  const size_t logits = (((Mp * LS + 1) & ~(size_t)1) + 2 * Mp + Mp + 10 * (size_t)p->kpad + 16) * sizeof(float);
  const size_t u = (fps > logits ? fps : logits) + 15;
  p->ufloats = (int)(u / sizeof(float)) & ~3;
  return Mp * D * sizeof(float) + (size_t)p->kpad * LD * sizeof(float) + (evict ? (size_t)p->kpad * D * sizeof(float) : 0) +
         (size_t)p->ufloats * sizeof(float) + ((Mp + 15) & ~(size_t)15);
}

// the plan, or false when the cluster kernel does not apply (the streaming passes run instead)
static bool small_plan(const ScoreArgs& a, bool evict, SmallPlan* p, size_t* smem) {
  if (a.dtype != KVC_F32 || a.ext || a.g.N < 1 || a.M_pad > kMaxRows || (a.g.D != 64 && a.g.D != 128)) return false;
  p->C = (a.g.N + 31) / 32;
  if (p->C > kSmallMaxCluster) p->C = kSmallMaxCluster;
  p->kpc = (a.g.N + p->C - 1) / p->C;
  if (p->kpc > kSmallMaxKeys) return false;
  p->kpad = (p->kpc + 1) & ~1;
  int dev = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  // the selection's and the row count's own shared arrays come on top of the dynamic part
  const size_t limit = (size_t)optin - 8192;
  const int G = a.g.Hq / a.g.Hkv;
  for (p->nw = G < 8 ? G : 8; p->nw >= 1; --p->nw) {
    const size_t bytes = small_smem(a, p, evict);
    if (bytes <= limit) {
      *smem = bytes;
      return true;
    }
  }
  return false;
}

bool score_small_plan(const ScoreArgs& a, size_t* smem, bool evict) {
  SmallPlan p;
  size_t bytes = 0;
  if (!small_plan(a, evict, &p, &bytes)) return false;
  if (smem) *smem = bytes;
  return true;
}

int launch_score_small(const ScoreArgs& a, const ScoreWs& ws, cudaStream_t s, const SmallEvict* ev) {
  SmallPlan p;
  size_t smem = 0;
  if (!small_plan(a, ev != nullptr, &p, &smem)) return KVC_ERR_LAUNCH;
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)a.g.D));
  auto kern = a.g.D == 128 ? score_small_f32_kernel<128> : score_small_f32_kernel<64>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(heads * p.C));
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  ScoreArgs aa = a;
  ScoreWs wss = ws;
  float cc = c2;
  SmallEvict e;
  memset(&e, 0, sizeof(e));
  if (ev) e = *ev;
  int on = ev ? 1 : 0;
  cudaError_t err = cudaLaunchKernelEx(&cfg, kern, aa, wss, p, cc, e, on);
  if (err != cudaSuccess) {  // without programmatic serialisation
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kern, aa, wss, p, cc, e, on);
  }
  return err == cudaSuccess ? KVC_OK : KVC_ERR_LAUNCH;
}

}  // namespace kvc
