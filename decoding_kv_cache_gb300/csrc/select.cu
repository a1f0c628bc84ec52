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
//
// Online head budgets (ReasonAlloc note, "Core Mechanism" and "Key Concepts"): with an
// entropy array, the budgets of the Hkv heads of one (layer, sequence) are first reallocated
// by head_budget_alloc below; kvc_head_budget runs the same function on its own.
#include "kvc_internal.cuh"

namespace kvc {

constexpr int kSelThreads = 1024;
constexpr int kMaxBudgetHeads = 64;

// Reallocation of one (layer, sequence)'s budget total over its H heads by normalised entropy
// (low entropy, more budget): floors f = P + R, the T - H f slots above them in proportion to
// u = 1 - entropy (clipped to [0, 1]; equal shares when every remaining u is 0), shares above
// the cap N - f cut to it and the rest shared again (water-filling), then integers by largest
// remainder with ties to the lower head. fp64 with every operation rounded on its own, heads in
// order, so the integer outcome is a fixed function of the fp32 entropies. Returns false (out
// untouched) when some given budget is below f; with N <= f or T >= H N, out = min(given, N).
// One thread; H <= kMaxBudgetHeads; u and share are H doubles of scratch (shared memory).
__device__ bool head_budget_alloc(const float* ent, const int32_t* given, int given_all, int H, int N, int P, int R,
                                  double* u, double* share, int32_t* out) {
  const int f = P + R;
  long long T = 0;
  for (int h = 0; h < H; ++h) {
    const int g = given ? given[h] : given_all;
    if (g < f) return false;
    T += g < N ? g : N;
  }
  if (N <= f || T >= (long long)H * N) {
    for (int h = 0; h < H; ++h) {
      const int g = given ? given[h] : given_all;
      out[h] = g < N ? g : N;
    }
    return true;
  }
  const int cap = N - f;
  const long long E = T - (long long)H * f;
  uint64_t active = 0;
  for (int h = 0; h < H; ++h) {
    double v = __dsub_rn(1.0, (double)ent[h]);
    if (!(v > 0.0)) v = 0.0;  // NaN too
    if (v > 1.0) v = 1.0;
    u[h] = v;
    share[h] = 0.0;
    active |= 1ull << h;
  }
  double Erem = (double)E;
  for (int pass = 0; pass <= H; ++pass) {  // each pass caps a head or ends
    double U = 0.0;
    int na = 0;
    for (int h = 0; h < H; ++h)
      if (active >> h & 1) {
        U = __dadd_rn(U, u[h]);
        ++na;
      }
    if (na == 0) break;
    for (int h = 0; h < H; ++h)
      if (active >> h & 1) share[h] = U > 0.0 ? __ddiv_rn(__dmul_rn(Erem, u[h]), U) : __ddiv_rn(Erem, (double)na);
    bool capped = false;
    for (int h = 0; h < H; ++h)
      if ((active >> h & 1) && share[h] > (double)cap) {
        share[h] = (double)cap;
        active &= ~(1ull << h);
        Erem = __dsub_rn(Erem, (double)cap);
        capped = true;
      }
    if (!capped) break;
  }
  long long sum = 0;
  for (int h = 0; h < H; ++h) {  // out holds the integer shares until the end
    int x = (active >> h & 1) ? (int)floor(share[h]) : cap;
    if (x > cap) x = cap;
    out[h] = x;
    sum += x;
  }
  uint64_t bonus = 0;
  for (long long left = E - sum; left > 0; --left) {  // largest remainders, ties to the lower head
    int best = -1;
    double bf = -1.0;
    for (int h = 0; h < H; ++h) {
      if ((bonus >> h & 1) || out[h] >= cap) continue;
      const double fr = __dsub_rn(share[h], (double)out[h]);
      if (fr > bf) {
        bf = fr;
        best = h;
      }
    }
    if (best < 0) break;
    bonus |= 1ull << best;
    out[best] += 1;
  }
  for (int h = 0; h < H; ++h) out[h] += f;
  return true;
}

// kvc_head_budget: one warp per (layer, sequence), its first thread allocates (budget_out may
// alias budget: a warp reads its slice before writing it).
__global__ void head_budget_kernel(const float* __restrict__ entropy, int Hkv, int N, int P, int R,
                                   const int32_t* budget, int budget_all, int32_t* budget_out,
                                   int32_t* status) {
  __shared__ double su[kMaxBudgetHeads], sshare[kMaxBudgetHeads];
  __shared__ int32_t sout[kMaxBudgetHeads];
  griddep_wait();
  const int lb = blockIdx.x;
  const int32_t* given = budget ? budget + (size_t)lb * Hkv : nullptr;
  if (threadIdx.x == 0 &&
      !head_budget_alloc(entropy + (size_t)lb * Hkv, given, budget_all, Hkv, N, P, R, su, sshare, sout)) {
    status_or(status, KVC_STATUS_BUDGET_RANGE);
    for (int h = 0; h < Hkv; ++h) sout[h] = given ? given[h] : budget_all;
  }
  __syncwarp();
  for (int h = threadIdx.x; h < Hkv; h += blockDim.x) budget_out[(size_t)lb * Hkv + h] = sout[h];
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
                                                             const float* __restrict__ entropy, int Hkv,
                                                             int32_t* __restrict__ kept_idx,
                                                             int32_t* __restrict__ kept_len, int32_t* status,
                                                             int use_smem) {
  extern __shared__ uint32_t sh_bits[];
  __shared__ unsigned hist[256];
  __shared__ int wsum[33];
  __shared__ unsigned s_digit, s_k;
  __shared__ int s_budget;
  __shared__ double s_u[kMaxBudgetHeads], s_share[kMaxBudgetHeads];
  __shared__ int32_t s_alloc[kMaxBudgetHeads];
  const int head = blockIdx.x, tid = threadIdx.x;
  griddep_wait();  // the scores (and entropies) come from the previous kernel
  const float* sc = scores + (size_t)head * N;
  int32_t* out = kept_idx + (size_t)head * N;
  int b = budget ? budget[head] : budget_all;
  if (entropy) {  // this head's share of its (layer, sequence)'s reallocated total
    if (tid == 0) {
      const int lb = head / Hkv, h = head % Hkv;
      s_budget = head_budget_alloc(entropy + (size_t)lb * Hkv, budget ? budget + (size_t)lb * Hkv : nullptr,
                                   budget_all, Hkv, N, P, R, s_u, s_share, s_alloc)
                     ? s_alloc[h]
                     : b;
    }
    __syncthreads();
    b = s_budget;
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
  if (cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (launch_pdl(select_kernel, dim3(heads), dim3(kSelThreads), smem, s, false, scores, N, P, R, budget, budget_all,
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
