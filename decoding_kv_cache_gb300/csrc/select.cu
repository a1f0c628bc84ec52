// select.cu -- kvc_select: which tokens each head keeps.
//
// BeaconKV write-up, end of "打分时的 RoPE 对齐": prefix tokens and the most recent tokens
// are always kept, the rest of the budget is filled by top score; "实验": the cache drops to
// 7/8 of B_KV^max. ReasonAlloc note, "Core Mechanism": the budget may differ per head.
//
// One CTA per head (256 or 1024 threads). Scores are non-negative fp32, so their IEEE bit patterns order like
// the values; a 4-pass radix select (8-bit digits, shared-memory histograms) finds the
// bit pattern T of the k-th largest middle score and how many copies of T must be kept.
// A final ordered sweep keeps every middle score above T and the lowest-index copies of T,
// which is the same set as sorting by (score descending, index ascending).
//
// Online head budgets (ReasonAlloc note, "Core Mechanism" and "Key Concepts"): with an
// entropy array, the budgets of the Hkv heads of one (layer, sequence) are first reallocated
// by head_budget_alloc below; kvc_head_budget runs the same function on its own.
#include "kvc_internal.cuh"

namespace kvc {

constexpr int kSelThreads = 1024;  // the most a select CTA is launched with
constexpr int kMaxBudgetHeads = 64;

// Reallocation of one (layer, sequence)'s budget total over its H heads by normalised entropy
// (low entropy, more budget). Floors f = P + R; the E = T - H f slots above them go in
// proportion to the utility u = 1 - entropy (clipped to [0, 1]) held as the 24-bit fixed-point
// integer w = floor(u * 2^24) (equal shares when every remaining w is 0); a share above the cap
// N - f is cut to it and the rest shared again (water-filling); integers by largest remainder,
// ties to the lower head. After w everything is exact integer arithmetic (E <= 2^36, w <= 2^24,
// so E w and cap W stay below 2^61), so the result is a fixed function of the fp32 entropies.
// One warp: lanes hold heads lane and lane + 32 (H <= 64, N <= 2^30). Returns false (out
// untouched) when some given budget is below f; with N <= f or T >= H N, out = min(given, N).
__device__ __forceinline__ long long warp_sum64(long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ bool head_budget_warp(const float* ent, const int32_t* given, int given_all, int H, int N, int P, int R,
                                 int32_t* out) {
  const int lane = threadIdx.x & 31, f = P + R;
  const int h0 = lane, h1 = lane + 32;
  const bool in0 = h0 < H, in1 = h1 < H;
  const int g0 = in0 ? (given ? given[h0] : given_all) : f, g1 = in1 ? (given ? given[h1] : given_all) : f;
  if (__any_sync(kFull, g0 < f || g1 < f)) return false;
  const long long T = warp_sum64((in0 ? (g0 < N ? g0 : N) : 0) + (in1 ? (g1 < N ? g1 : N) : 0));
  if (N <= f || T >= (long long)H * N) {
    if (in0) out[h0] = g0 < N ? g0 : N;
    if (in1) out[h1] = g1 < N ? g1 : N;
    return true;
  }
  const unsigned long long cap = (unsigned long long)(N - f), E = (unsigned long long)(T - (long long)H * f);
  auto weight = [&](int h) -> unsigned long long {
    double u = __dsub_rn(1.0, (double)ent[h]);
    if (!(u > 0.0)) u = 0.0;  // NaN too
    if (u > 1.0) u = 1.0;
    return (unsigned long long)floor(__dmul_rn(u, 16777216.0));
  };
  const unsigned long long w0 = in0 ? weight(h0) : 0ull, w1 = in1 ? weight(h1) : 0ull;
  bool a0 = in0, a1 = in1;  // still sharing (not capped)
  unsigned long long Erem = E;
  for (int pass = 0; pass <= H; ++pass) {
    const unsigned long long W = (unsigned long long)warp_sum64((long long)((a0 ? w0 : 0ull) + (a1 ? w1 : 0ull)));
    const int na = __popc(__ballot_sync(kFull, a0)) + __popc(__ballot_sync(kFull, a1));
    if (na == 0) break;
    // share > cap  <=>  Erem w > cap W (or Erem > cap na for the equal split)
    const bool o0 = a0 && (W > 0 ? Erem * w0 > cap * W : Erem > cap * (unsigned long long)na);
    const bool o1 = a1 && (W > 0 ? Erem * w1 > cap * W : Erem > cap * (unsigned long long)na);
    const int nc = __popc(__ballot_sync(kFull, o0)) + __popc(__ballot_sync(kFull, o1));
    if (nc == 0) break;
    a0 = a0 && !o0;
    a1 = a1 && !o1;
    const int ncap_all = H - (__popc(__ballot_sync(kFull, a0)) + __popc(__ballot_sync(kFull, a1)));
    Erem = E - (unsigned long long)ncap_all * cap;
  }
  const unsigned long long W = (unsigned long long)warp_sum64((long long)((a0 ? w0 : 0ull) + (a1 ? w1 : 0ull)));
  const unsigned long long na = (unsigned long long)(__popc(__ballot_sync(kFull, a0)) + __popc(__ballot_sync(kFull, a1)));
  unsigned long long x0 = in0 ? cap : 0ull, x1 = in1 ? cap : 0ull, r0 = 0ull, r1 = 0ull;
  if (a0) {
    const unsigned long long num = W > 0 ? Erem * w0 : Erem, den = W > 0 ? W : na;
    x0 = num / den;
    r0 = num % den;  // the active heads' remainders share the denominator
  }
  if (a1) {
    const unsigned long long num = W > 0 ? Erem * w1 : Erem, den = W > 0 ? W : na;
    x1 = num / den;
    r1 = num % den;
  }
  const long long left = (long long)E - warp_sum64((long long)((in0 ? x0 : 0ull) + (in1 ? x1 : 0ull)));
  // one more slot for the `left` eligible heads ranked first by (remainder desc, head asc)
  const bool e0 = a0 && x0 < cap, e1 = a1 && x1 < cap;
  int rank0 = 0, rank1 = 0;
  for (int src = 0; src < 32; ++src) {
    const unsigned long long q0 = __shfl_sync(kFull, r0, src), q1 = __shfl_sync(kFull, r1, src);
    const bool f0 = __shfl_sync(kFull, e0, src), f1 = __shfl_sync(kFull, e1, src);
    // head src (rank before every head above it on a tie) and head src + 32
    rank0 += (f0 && (q0 > r0 || (q0 == r0 && src < h0))) + (f1 && (q1 > r0 || (q1 == r0 && src + 32 < h0)));
    rank1 += (f0 && (q0 > r1 || (q0 == r1 && src < h1))) + (f1 && (q1 > r1 || (q1 == r1 && src + 32 < h1)));
  }
  if (in0) out[h0] = f + (int)(x0 + (e0 && rank0 < left ? 1 : 0));
  if (in1) out[h1] = f + (int)(x1 + (e1 && rank1 < left ? 1 : 0));
  return true;
}

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

// Block-wide exclusive prefix count of a flag, in thread order. Returns this thread's
// prefix; *total receives the block total. Uses warp ballots and one shared array.
__device__ __forceinline__ int block_excl_count(bool flag, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(kFull, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) wsum[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int v = lane < (int)(blockDim.x >> 5) ? wsum[lane] : 0;  // entries past the block's warps are unset
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

template <int kThreads>
__global__ void __launch_bounds__(kThreads) select_kernel(const float* __restrict__ scores, int N, int P, int R,
                                                             const int32_t* __restrict__ budget, int budget_all,
                                                             const float* __restrict__ entropy, int Hkv,
                                                             int32_t* __restrict__ kept_idx,
                                                             int32_t* __restrict__ kept_len, int32_t* status,
                                                             int use_smem) {
  extern __shared__ uint32_t sh_bits[];
  __shared__ unsigned hist[256];
  __shared__ int wsum[33];
  __shared__ unsigned s_digit, s_k;
  __shared__ int32_t s_alloc[kMaxBudgetHeads];
  const int head = blockIdx.x, tid = threadIdx.x;
  griddep_wait();  // the scores (and entropies) come from the previous kernel
  const float* sc = scores + (size_t)head * N;
  int32_t* out = kept_idx + (size_t)head * N;
  int b = budget ? budget[head] : budget_all;
  if (entropy) {  // this head's share of its (layer, sequence)'s reallocated total (warp 0)
    const int lb = head / Hkv, h = head % Hkv;
    if (tid < 32 && !head_budget_warp(entropy + (size_t)lb * Hkv, budget ? budget + (size_t)lb * Hkv : nullptr,
                                      budget_all, Hkv, N, P, R, s_alloc) && tid == 0)
      s_alloc[h] = b;  // a given budget below prefix + recent: the given budgets stand
    __syncthreads();
    b = s_alloc[h];
  }
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
                  const float* entropy, int Hkv, int32_t* kept_idx, int32_t* kept_len, int32_t* status,
                  cudaStream_t s) {
  if (heads == 0) return KVC_OK;
  const size_t bytes = (size_t)N * 4;
  const int use_smem = bytes <= 200u * 1024u ? 1 : 0;
  const size_t smem = use_smem ? bytes : 0;
  // A head's scores up to 64 KB: 256 threads, so that several heads share an SM and each barrier
  // spans 8 warps (R1-Qwen-7B-shaped heads of 8192 keys: 88 -> 58 us); longer heads fill an SM's
  // shared memory alone and need 1024 threads (Qwen3-14B-shaped, 32768 keys: 0.81 ms vs 2.4 ms).
  auto kern = N <= 16384 ? select_kernel<256> : select_kernel<kSelThreads>;
  const int threads = N <= 16384 ? 256 : kSelThreads;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (launch_pdl(kern, dim3(heads), dim3(threads), smem, s, false, scores, N, P, R, budget, budget_all,
                 entropy, Hkv, kept_idx, kept_len, status, use_smem) != cudaSuccess)
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
