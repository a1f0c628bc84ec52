// select.cu -- kvc_select: which tokens each head keeps.
//
// BeaconKV write-up, end of "打分时的 RoPE 对齐": prefix tokens and the most recent tokens
// are always kept, the rest of the budget is filled by top score; "实验": the cache drops to
// 7/8 of B_KV^max. ReasonAlloc note, "Core Mechanism": the budget may differ per head.
//
// One CTA per head. Scores are non-negative fp32, so their IEEE bit patterns order like
// the values; a 4-pass radix select (8-bit digits, shared-memory histograms) finds the
// bit pattern T of the k-th largest middle score and how many copies of T must be kept.
// A final ordered sweep keeps every middle score above T and the lowest-index copies of T,
// which is the same set as sorting by (score descending, index ascending).
#include "kvc_internal.cuh"

namespace kvc {

constexpr int kSelThreads = 1024;

// Block-wide exclusive prefix count of a flag, in thread order. Returns this thread's
// prefix; *total receives the block total. Uses warp ballots and one shared array.
__device__ __forceinline__ int block_excl_count(bool flag, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(kFull, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int v = wsum[lane];
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += u;
    }
    wsum[lane] = inc - v;       // exclusive
    if (lane == 31) wsum[32] = inc;
  }
  __syncthreads();
  const int r = wsum[warp] + in_warp;
  *total = wsum[32];
  __syncthreads();  // wsum is reused by the next call
  return r;
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const float* __restrict__ scores, int N, int P, int R,
                                                             const int32_t* __restrict__ budget, int budget_all,
                                                             int32_t* __restrict__ kept_idx,
                                                             int32_t* __restrict__ kept_len, int32_t* status,
                                                             int use_smem) {
  extern __shared__ uint32_t sh_bits[];
  __shared__ unsigned hist[256];
  __shared__ int wsum[33];
  __shared__ unsigned s_digit, s_k;
  const int head = blockIdx.x, tid = threadIdx.x;
  griddep_wait();  // the scores come from the previous kernel
  const float* sc = scores + (size_t)head * N;
  int32_t* out = kept_idx + (size_t)head * N;
  const int b = budget ? budget[head] : budget_all;
  if (b >= N || b < P + R) {  // keep everything (out-of-range budgets are flagged)
    if (b < N && tid == 0) status_or(status, KVC_STATUS_BUDGET_RANGE);
    for (int j = tid; j < N; j += blockDim.x) out[j] = j;
    if (tid == 0) kept_len[head] = N;
    return;
  }
  const uint32_t* bits = reinterpret_cast<const uint32_t*>(sc);
  if (use_smem) {
    for (int j = tid; j < N; j += blockDim.x) sh_bits[j] = __float_as_uint(sc[j]);
    __syncthreads();
    bits = sh_bits;
  }
  const int lo = P, hi = N - R, kmid = b - P - R;
  uint32_t T = 0xffffffffu;  // with kmid == 0 nothing of the middle passes "> T" or "== T, rank < 0"
  unsigned keq = 0;
  if (kmid > 0) {
    uint32_t prefix = 0, mask = 0;
    unsigned k = (unsigned)kmid;  // rank (1-based, from the top) still to locate
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      for (int j = lo + tid; j < hi; j += blockDim.x) {
        const uint32_t u = bits[j];
        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (tid < 32) {
        // lane l holds digits 255-8l ... 248-8l, so lane order is descending digit order
        unsigned c[8], local = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          c[q] = hist[255 - 8 * tid - q];
          local += c[q];
        }
        unsigned inc = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned u = __shfl_up_sync(kFull, inc, o);
          if (tid >= o) inc += u;
        }
        const unsigned found = __ballot_sync(kFull, inc >= k);
        if (tid == __ffs(found) - 1) {
          unsigned cum = inc - local;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (cum + c[q] >= k) {
              s_digit = 255u - 8u * tid - q;
              s_k = k - cum;
              break;
            }
            cum += c[q];
          }
        }
      }
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= 255u << shift;
      k = s_k;
      __syncthreads();
    }
    T = prefix;
    keq = k;
  }
  // ordered sweep: write kept indices ascending
  int base_out = 0, base_eq = 0;
  for (int j0 = 0; j0 < N; j0 += blockDim.x) {
    const int j = j0 + tid;
    const bool live = j < N;
    const uint32_t u = live ? bits[j] : 0u;
    const bool mid = live && j >= lo && j < hi;
    const bool eq = mid && u == T;
    int eq_tot;
    const int eq_rank = base_eq + block_excl_count(eq, wsum, &eq_tot);
    const bool keep = live && (!mid || u > T || (eq && (unsigned)eq_rank < keq));
    int keep_tot;
    const int pos = base_out + block_excl_count(keep, wsum, &keep_tot);
    if (keep) out[pos] = j;
    base_eq += eq_tot;
    base_out += keep_tot;
  }
  if (tid == 0) kept_len[head] = base_out;
}

int launch_select(const float* scores, int heads, int N, int P, int R, const int32_t* budget, int budget_all,
                  int32_t* kept_idx, int32_t* kept_len, int32_t* status, cudaStream_t s) {
  if (heads == 0) return KVC_OK;
  const size_t bytes = (size_t)N * 4;
  const int use_smem = bytes <= 200u * 1024u ? 1 : 0;
  const size_t smem = use_smem ? bytes : 0;
  if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (launch_pdl(select_kernel, dim3(heads), dim3(kSelThreads), smem, s, false, scores, N, P, R, budget, budget_all,
                 kept_idx, kept_len, status, use_smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
