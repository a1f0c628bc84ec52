// kvc_internal.cuh -- device helpers and launch parameters shared by libkvc's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvc.h"

namespace kvc {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kChunk = 128;     // keys per scoring CTA
constexpr int kMaxRows = 256;   // observation rows per KV head (G * (n_r + n_b), padded to 16)
constexpr int kMaxQmax = 64;    // FPS buffer capacity
constexpr int kMaxSMs = 256;    // bound on the SM count used to size the fused kernel's exchange
constexpr float kLog2e = 1.4426950408889634f;

// ---- storage access -------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// ---- warp reductions --------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ void status_or(int32_t* status, unsigned bits) {
  if (status) atomicOr(reinterpret_cast<unsigned*>(status), bits);
}

// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with programmatic stream serialisation may start while the previous
// kernel in the stream is still running; griddep_wait() returns once that kernel has
// completed and its memory operations are visible (immediately when launched normally).
// No kernel here signals early completion: dependents are released when their predecessor
// exits (an early signal let waiting CTAs sit beside the scoring kernel and slowed it), so
// the overlap is the launch's own latency and the waiting roles' prologue.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Launch with programmatic stream serialisation (and cooperatively if asked); when the
// runtime refuses the attribute, launch again without it.
template <typename... Params, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool coop,
                              Args... args) {
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (coop) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    cfg.numAttrs = na - 1;
    e = cudaLaunchKernelEx(&cfg, kern, args...);
  }
  return e;
}

// ---- per-layer pointer tables passed by value -------------------------------
struct LayerPtrs {
  void* p[KVC_MAX_LAYERS];
};

// Geometry of one cache, as the kernels see it.
struct CacheGeom {
  int L, B, Hq, Hkv, D, N;
  long long ncap;
};

// ---- launchers (host) ---------------------------------------------------------
// Each returns KVC_OK or KVC_ERR_LAUNCH; arguments are already validated.
struct AppendArgs {         // kvc_append, flattened over query heads
  const void* q_pre;        // [nheads][D] pre-RoPE query of this step
  const void* q_post;       // [nheads][D] post-RoPE query, or null (then q_pre is turned to t)
  void* qbuf;               // [nheads][qmax][D]
  int32_t* count;           // [nheads]
  void* q_recent;           // [nheads][n_r][D] ring
  int32_t* picks;           // [nheads][qmax/2] or null
  int32_t* status;
  int nheads, qmax, n_r;
  int ring_slot;            // t mod n_r
  float2 rope[64];          // (cos, sin) of t * theta^(-2i/D), i < D/2, from fp64 (when q_post is null)
};
int launch_append(const AppendArgs& a, int dtype, int D, cudaStream_t s);

int launch_fps_update(int dtype, int nheads_q, int D, void* qbuf, int qmax, int32_t* count, int32_t* picks,
                      int32_t* status, cudaStream_t s);

struct ScoreWs {            // carved out of the caller's workspace
  void* obs;                // [heads][M_pad][D] storage type
  uint8_t* valid;           // [heads][M_pad]
  float2* part;             // fp32: [heads][nchunk][M_pad] partial (max, sum) in base 2; bf16: fused exchange
  float* lse2;              // [heads][M_pad] log2-sum-exp2, +inf for unused rows
  float* rw;                // [heads][M_pad] row weight of a mean over the query head's rows (0: no row)
  float* escale;            // [heads] 1 / (valid rows * log2 N): entropy in bits -> normalised mean
  float* ent;               // [heads] entropy accumulator when the caller keeps none (kvc_evict)
  float* lse2p;             // bf16 two-pass streaming kernels: [heads][ranges][M_pad] log2-sum-exp2 per key range
  int32_t* fb;              // wide kernel: [0] items listed for the exact fallback, [1..] the items (zeroed by build_obs)
};

struct ScoreArgs {
  CacheGeom g;
  int dtype;
  LayerPtrs K;
  const void* q_recent;
  int n_r;
  const void* qbuf;
  const int32_t* count;
  int qmax, n_b;
  long long t;
  double theta;
  float* scores;
  int32_t* beacon_picks;
  int32_t* status;
  int M, M_pad, M_n, nchunk;  // rows, rows stored per head, rows rounded to 16, key chunks
  float2 rope[64];            // (cos, sin) of t * theta^(-2i/D), i < D/2, from fp64
  unsigned long long* xch_zero;  // words the observation kernel zeroes for the scoring kernel, or null
  long long xch_zero_words;
  // kvc_evict with per-head budgets: the observation kernel's first CTA also writes the order in
  // which the selection-and-compaction CTAs take the heads (head_order_cta), or null
  const int32_t* order_budget;
  int32_t* order;
  int debug_fault;               // kvc_debug_fault mode at launch (0 in normal use)
  int kernel;                    // KVC_KERNEL_*: the bf16 scoring kernel asked for (0 = automatic)
  // Variants: an aggregation other than max/max or an entropy output runs the kernels'
  // extended epilogue (ext = 1). Rows of query head g then start at g * qstride, a multiple
  // of 16, so every 16-row block of the tile belongs to one query head.
  int ext;
  int qstride;                   // rows per query head in the tile (n_r + n_b, or rounded up to 16)
  int row_agg, group_agg;        // KVC_AGG_* (ext only)
  float* entropy;                // [heads] normalised entropy, accumulated (zeroed by build_obs), or null
  int tiles;                     // 128-row tiles scored apart per head by the single-read kernel (1 or 2);
                                 // with 2, build_obs zeroes the scores and the tiles combine atomically
};

// kvc_evict's selection and compaction arguments, for the fp32 cluster kernel that runs them
// itself (launch_score_small)
struct SmallEvict {
  LayerPtrs V;
  int P, R, budget_all;
  const int32_t* budget;  // [heads] or null
  int32_t* kept_idx;      // [heads][N]
  int32_t* kept_len;      // [heads]
};

// Row stride of a query head and row count of the observation tile for a mode.
inline int obs_qstride(int n_r, int n_b, bool ext) { return ext ? (n_r + n_b + 15) / 16 * 16 : n_r + n_b; }
inline int obs_rows_used(int G, int n_r, int n_b, bool ext) { return (G - 1) * obs_qstride(n_r, n_b, ext) + n_r + n_b; }

int obs_rows(int M, int dtype);

size_t score_ws_bytes(const CacheGeom& g, int dtype, int n_r, int n_b, bool ext, ScoreWs* carve, void* base);
// ev: kvc_evict's selection and compaction, taken into the scoring launch where the fp32 cluster
// kernel runs (then *fused is set; else the caller launches them)
int launch_score(const ScoreArgs& a, const ScoreWs& ws, cudaStream_t s, const SmallEvict* ev = nullptr,
                 bool* fused = nullptr);
size_t fused_xch_bytes(int M_pad);
int launch_score_fused(const ScoreArgs& a, const ScoreWs& ws, void* xch_base, cudaStream_t s);
// Single-read kernel (bf16, 128 observation rows, at most 256 keys per SM per head): the plan, or
// false when it does not apply; the exchange words it needs zeroed (in ws.part); the launch.
struct FusedPlan {
  int group_size;      // CTAs per head
  int ngroups;         // heads processed at once
  int chunks_per_cta;  // key chunks per CTA per head
  int stages;          // K ring depth
  int qbytes;          // one observation tile: M_pad * D * 2
};
bool score_resident_plan(const ScoreArgs& a, FusedPlan* p, size_t* smem);
long long score_resident_words(const FusedPlan& p, bool entropy);
int launch_score_resident(const ScoreArgs& a, const ScoreWs& ws, const FusedPlan& p, size_t smem, cudaStream_t s);

// Two-pass streaming kernel (bf16, max/max, 128- or 256-row tiles): every (head, key range) is an
// independent work item of both passes; a combine kernel between them forms lse2.
struct SplitPlan {
  int rk;      // 128-key chunks per range
  int R;       // ranges per head
  int items;   // heads * R
  int grid;    // CTAs (one per SM)
  int stages;  // K ring depth
  const int32_t* list;  // null: every item; else [0] = count, [1..] = the items (device, written by the
                        // previous kernel on the stream)
};
// The wide kernel's exact fallback recomputes each of its n listed items as this many sub-ranges on
// separate CTAs (at most grid CTAs in all, kFallbackSub sub-ranges an item, at least one key chunk
// each), so that a few listed items of many chunks do not run one chunk after another on one CTA:
// sub-range 0 writes the item's partial, the others theirs into the workspace's exchange area, and
// the combine kernel merges them (one batch of reads per listed item).
constexpr int kFallbackSub = 16;
__host__ __device__ inline int fallback_sub(int n, int grid, int rk) {
  if (n <= 0 || n > kMaxSMs / 2) return 1;
  int s = grid / n;
  if (s > kFallbackSub) s = kFallbackSub;
  if (s > rk) s = rk;
  return s < 1 ? 1 : s;
}
// Pass 1 of the two-pass streaming kernel over a device list of items (the wide kernel's fallback),
// with the listing kernel's ranges: item = head * R + range, rk key chunks per range; grid CTAs.
int launch_score_split_pass1_list(const ScoreArgs& a, const ScoreWs& ws, const int32_t* list, int rk, int R,
                                  int grid, cudaStream_t s);
int split_ranges(int nchunk, int M_pad);
bool score_split_plan(const ScoreArgs& a, SplitPlan* p, size_t* smem);
int launch_score_split(const ScoreArgs& a, const ScoreWs& ws, const SplitPlan& p, size_t smem, cudaStream_t s);
__global__ void split_combine_kernel(ScoreArgs a, ScoreWs ws, SplitPlan p);

// Two-pass kernel with the keys on the TMEM lanes (bf16, default options, more than 128 rows): the
// same work items as the two-pass streaming kernel; an exact fallback for items whose logits spread
// too far for its one-reference sums, then the combine, between the passes.
struct WidePlan {
  int rk, R, items, grid, stages;
};
bool score_wide_plan(const ScoreArgs& a, WidePlan* p, size_t* smem);
int launch_score_wide(const ScoreArgs& a, const ScoreWs& ws, const WidePlan& p, size_t smem, cudaStream_t s);
// fp32 caches of at most eight CTAs of 128 keys per head (default options): the whole scoring
// (observation rows included) in one launch, a thread-block cluster per head; kvc_evict's
// selection and compaction can run in the same launch (SmallEvict).
bool score_small_plan(const ScoreArgs& a, size_t* smem, bool evict);
int launch_score_small(const ScoreArgs& a, const ScoreWs& ws, cudaStream_t s, const SmallEvict* ev);
// kernels launch_score starts for these arguments (host only; default options when !ext)
int score_launches(const CacheGeom& g, int dtype, int n_r, int n_b, bool ext);
// whether kvc_evict (default options, given budgets, a buffer of 2 n_b rows) selects and compacts
// inside the scoring launch
bool evict_fused_small(const CacheGeom& g, int dtype, int n_r, int n_b);

// entropy non-null: each (layer, sequence)'s budgets are reallocated over its Hkv heads first;
// keyed: `scores` holds order-preserving unsigned keys already (EPIKV), not fp32 scores
int launch_select(const float* scores, int heads, int N, int P, int R, const int32_t* budget, int budget_all,
                  const float* entropy, int Hkv, int32_t* kept_idx, int32_t* kept_len, int32_t* status,
                  cudaStream_t s, bool keyed = false);
int launch_head_budget(const float* entropy, int groups, int Hkv, int N, int P, int R, const int32_t* budget,
                       int budget_all, int32_t* budget_out, int32_t* status, cudaStream_t s);

// kvc_evict's selection and compaction in one launch (one CTA per head; N <= kSelectCompactMaxN)
constexpr int kSelectCompactMaxN = 65536;
// order: the head each CTA takes (a permutation of the heads, written by head_order_cta), or null
int launch_select_compact(const int32_t* order, const float* scores, const CacheGeom& g, int dtype, const LayerPtrs& K,
                          const LayerPtrs& V, int P, int R, const int32_t* budget, int budget_all, const float* entropy, int32_t* kept_idx,
                          int32_t* kept_len, int32_t* status, cudaStream_t s);

// list_per_seq: kept_idx [B][N] / kept_len [B], one list per sequence for all its layers and heads
int launch_compact(const CacheGeom& g, int dtype, const LayerPtrs& K, const LayerPtrs& V, const int32_t* kept_idx,
                   const int32_t* kept_len, int32_t* status, bool validate, cudaStream_t s, bool list_per_seq = false);

// EPIKV: signals g [2][B][N] (layer A, layer B), prefix sums pre [2][2][B][N+1] fp64, signed
// scores [B][N] and (if keys) their order-preserving unsigned keys [B][N] for the radix selection
int launch_epikv_score(int dtype, int B, int N, int dm, const void* hA, const void* hB, int W, double eps, float* g,
                       double* pre, float* score, uint32_t* keys, cudaStream_t s);

inline int launch_ok() { return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_LAUNCH; }

}  // namespace kvc
