// select.cu -- kvc_select: which tokens each head keeps.
//
// BeaconKV write-up, end of "打分时的 RoPE 对齐": prefix tokens and the most recent tokens
// are always kept, the rest of the budget is filled by top score; "实验": the cache drops to
// 7/8 of B_KV^max. ReasonAlloc note, "Core Mechanism": the budget may differ per head.
//
// One CTA per head (256 or 1024 threads, each holding 8 consecutive tokens of a tile; a head of
// one tile stays in registers). Each fp32 score becomes an unsigned key that orders like the
// value (sign bit set: all bits flipped; else the sign bit set; -0 taken as +0), so any finite
// score, negative ones included, ranks as its value does (a NaN with the sign bit clear ranks
// above +inf, one with it set below -inf); EPIKV hands over such keys already made. A radix
// select finds the key T of the k-th largest middle score and
// how many copies of T must be kept. The leading bits shared by every middle score (from their
// minimum and maximum) are skipped; then 8-bit digits, one shared-memory histogram pass each (two
// barriers, the next pass's bins cleared during this one), stopping early once the rank's bucket
// is kept whole (T is then a prefix and ties are compared on the bits resolved so far). A final
// ordered sweep keeps every middle score above T and the lowest-index copies of T, which is the
// same set as sorting by (score descending, index ascending).
//
// Online head budgets (ReasonAlloc note, "Core Mechanism" and "Key Concepts"): with an
// entropy array, the budgets of the Hkv heads of one (layer, sequence) are first reallocated
// by head_budget_warp (select_head.cuh, with the selection itself); kvc_head_budget runs the same
// function on its own.
#include "compact.cuh"
#include "select_head.cuh"

namespace kvc {

// kvc_head_budget: one warp per (layer, sequence) (budget_out may alias budget: the warp reads
// its slice before writing it).
__global__ void head_budget_kernel(const float* __restrict__ entropy, int Hkv, int N, int P, int R,
                                   const int32_t* budget, int budget_all, int32_t* budget_out, int32_t* status) {
  __shared__ int32_t sout[kMaxBudgetHeads];
  griddep_wait();
  const int lb = blockIdx.x;
  const int32_t* given = budget ? budget + (size_t)lb * Hkv : nullptr;
  if (!head_budget_warp(entropy + (size_t)lb * Hkv, given, budget_all, Hkv, N, P, R, sout)) {
    if (threadIdx.x == 0) status_or(status, KVC_STATUS_BUDGET_RANGE);
    for (int h = threadIdx.x; h < Hkv; h += 32) sout[h] = given ? given[h] : budget_all;
  }
  __syncwarp();
  for (int h = threadIdx.x; h < Hkv; h += 32) budget_out[(size_t)lb * Hkv + h] = sout[h];
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) select_kernel(const float* __restrict__ scores, int N, int P, int R,
                                                             const int32_t* __restrict__ budget, int budget_all,
                                                             const float* __restrict__ entropy, int Hkv,
                                                             int32_t* __restrict__ kept_idx,
                                                             int32_t* __restrict__ kept_len, int32_t* status,
                                                             int use_smem, int keyed) {
  extern __shared__ __align__(16) uint32_t sh_bits[];
  griddep_wait();  // the scores (and entropies) come from the previous kernel
  select_head<kThreads>(blockIdx.x, scores, N, P, R, budget, budget_all, entropy, Hkv, kept_idx, kept_len, status,
                        use_smem, keyed, sh_bits);
}

// Selection and compaction of one head per CTA (256 threads, heads of at most kSelectCompactMaxN
// tokens): the CTA selects, then two of its warps move the head's kept K and V rows (compact_warp).
// One launch instead of two, and each head's selection overlaps the other heads' moves (two CTAs
// fit on an SM). CTA b takes head order[b] (largest budget first, when the heads' budgets differ)
// or head b. The dynamic shared memory stages the scores of a head of more than one tile (when
// they fit), then serves as the two warps' rings.
__global__ void __launch_bounds__(256) select_compact_kernel(const int32_t* __restrict__ order,
                                                             const float* __restrict__ scores, int N, int P, int R,
                                                             const int32_t* __restrict__ budget, int budget_all,
                                                             const float* __restrict__ entropy, int Hkv,
                                                             int32_t* __restrict__ kept_idx,
                                                             int32_t* __restrict__ kept_len, int32_t* status,
                                                             int use_smem, CompactArgs ca) {
  extern __shared__ __align__(128) uint8_t smc[];
  griddep_wait();  // the scores (and entropies) come from the previous kernel
  const int head = order ? order[blockIdx.x] : (int)blockIdx.x;
  select_head<256>(head, scores, N, P, R, budget, budget_all, entropy, Hkv, kept_idx, kept_len, status, use_smem,
                   0, reinterpret_cast<uint32_t*>(smc));
  // the head's kept list, written by this CTA, is visible to all its threads, and the staging area is free
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if (warp < 2) compact_warp(ca, head, warp, smc + warp * kCompactWarpSmem);
}

int launch_select_compact(const int32_t* order, const float* scores, const CacheGeom& g, int dtype, const LayerPtrs& K,
                          const LayerPtrs& V, int P, int R, const int32_t* budget, int budget_all, const float* entropy, int32_t* kept_idx,
                          int32_t* kept_len, int32_t* status, cudaStream_t s) {
  const int heads = g.L * g.B * g.Hkv, N = g.N;
  if (heads == 0) return KVC_OK;
  CompactArgs ca;
  ca.g = g;
  ca.K = K;
  ca.V = V;
  ca.kept_idx = kept_idx;
  ca.kept_len = kept_len;
  ca.status = status;
  ca.rowbytes = g.D * (dtype == KVC_BF16 ? 2 : 4);
  ca.validate = 0;
  ca.list_seq = 0;
  // a head of more than one tile is staged in shared memory when it fits in the two warps' rings
  // (the CTA's footprint stays at two per SM, so one CTA's selection runs beside another's moves);
  // a longer head is read from global memory (L2) on every pass
  const size_t stage = (size_t)(N + kSweep - 1) / kSweep * kSweep * 4;
  const size_t smem = 2 * (size_t)kCompactWarpSmem;
  const int use_smem = (N > kSweep * 256 && stage <= smem) ? 1 : 0;
  if (cudaFuncSetAttribute(select_compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (launch_pdl(select_compact_kernel, dim3(heads), dim3(256), smem, s, false, order, scores, N, P, R, budget, budget_all,
                 entropy, g.Hkv, kept_idx, kept_len, status, use_smem, ca) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

int launch_select(const float* scores, int heads, int N, int P, int R, const int32_t* budget, int budget_all,
                  const float* entropy, int Hkv, int32_t* kept_idx, int32_t* kept_len, int32_t* status,
                  cudaStream_t s, bool keyed) {
  if (heads == 0) return KVC_OK;
  // A head's scores up to 64 KB: 256 threads, so that several heads share an SM and each barrier
  // spans 8 warps (R1-Qwen-7B-shaped heads of 8192 keys: 88 -> 58 us); longer heads fill an SM's
  // shared memory alone and need 1024 threads (Qwen3-14B-shaped, 32768 keys: 0.81 ms vs 2.4 ms).
  auto kern = N <= 16384 ? select_kernel<256> : select_kernel<kSelThreads>;
  const int threads = N <= 16384 ? 256 : kSelThreads;
  // one tile (kSweep tokens per thread) stays in registers; longer heads are staged in shared
  // memory when they fit
  const size_t bytes = (size_t)(N + kSweep - 1) / kSweep * kSweep * 4;
  const int use_smem = N > kSweep * threads && bytes <= 200u * 1024u ? 1 : 0;
  const size_t smem = use_smem ? bytes : 0;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (launch_pdl(kern, dim3(heads), dim3(threads), smem, s, false, scores, N, P, R, budget, budget_all,
                 entropy, Hkv, kept_idx, kept_len, status, use_smem, keyed ? 1 : 0) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

int launch_head_budget(const float* entropy, int groups, int Hkv, int N, int P, int R, const int32_t* budget,
                       int budget_all, int32_t* budget_out, int32_t* status, cudaStream_t s) {
  if (groups == 0) return KVC_OK;
  if (launch_pdl(head_budget_kernel, dim3(groups), dim3(32), 0, s, false, entropy, Hkv, N, P, R, budget, budget_all,
                 budget_out, status) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
