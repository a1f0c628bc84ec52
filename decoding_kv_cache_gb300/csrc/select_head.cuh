// select_head.cuh -- the per-head selection (radix select over order-preserving keys) and the
// online head-budget rule, as device functions: select.cu's kernels and the fp32 cluster kernel
// (score_small.cu) run them. What they compute is described at the top of select.cu.
#pragma once

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

static __device__ bool head_budget_warp(const float* ent, const int32_t* given, int given_all, int H, int N, int P, int R,
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

// Block-wide exclusive prefix sum, in thread order, of two counts packed in one 64-bit word (each
// half stays below 2^32, so the halves never carry into each other). Returns this thread's prefix;
// *total receives the block total. wsum holds 33 words; every thread of the block calls it.
__device__ __forceinline__ unsigned long long block_excl_scan64(unsigned long long v, unsigned long long* wsum,
                                                                unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
  unsigned long long inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long u = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += u;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = lane < nw ? wsum[lane] : 0ull;  // entries past the block's warps are unset
    unsigned long long winc = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long u = __shfl_up_sync(kFull, winc, o);
      if (lane >= o) winc += u;
    }
    wsum[lane] = winc - w;  // exclusive over warps
    if (lane == 31) wsum[32] = winc;
  }
  __syncthreads();
  const unsigned long long r = wsum[warp] + (inc - v);
  *total = wsum[32];
  __syncthreads();  // wsum is reused by the next call
  return r;
}

constexpr int kSweep = 8;  // consecutive tokens per thread: a tile is kSweep * threads tokens

// Order-preserving key of an fp32 score's bits (-0 as +0).
__device__ __forceinline__ uint32_t score_key(uint32_t u) {
  u = u == 0x80000000u ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// This thread's kSweep consecutive tokens from j as keys: two 16-byte loads where the source
// allows (vec: base 16-byte aligned and j a multiple of kSweep), else element by element; tokens
// past N read as 0 (they lie outside the middle). keyed: the words are keys already.
__device__ __forceinline__ void load_group(const uint32_t* p, int j, int N, bool vec, bool keyed,
                                           uint32_t (&w)[kSweep]) {
  if (vec && j + kSweep <= N) {
    const uint4 x = *reinterpret_cast<const uint4*>(p + j), y = *reinterpret_cast<const uint4*>(p + j + 4);
    w[0] = x.x, w[1] = x.y, w[2] = x.z, w[3] = x.w, w[4] = y.x, w[5] = y.y, w[6] = y.z, w[7] = y.w;
  } else {
#pragma unroll
    for (int e = 0; e < kSweep; ++e) w[e] = j + e < N ? p[j + e] : 0u;
  }
  if (!keyed)
#pragma unroll
    for (int e = 0; e < kSweep; ++e) w[e] = score_key(w[e]);
}

// The selection of one head by the whole CTA (kThreads threads); sh_bits is the dynamic shared
// memory used to stage a head of more than one tile (use_smem). Every thread returns.
template <int kThreads>
__device__ __forceinline__ void select_head(int head, const float* __restrict__ scores, int N, int P, int R,
                                            const int32_t* __restrict__ budget, int budget_all,
                                            const float* __restrict__ entropy, int Hkv, int32_t* __restrict__ kept_idx,
                                            int32_t* __restrict__ kept_len, int32_t* status, int use_smem, int keyed,
                                            uint32_t* sh_bits) {
  constexpr int kWarps = kThreads / 32;
  constexpr int kTile = kSweep * kThreads;
  __shared__ __align__(16) unsigned hist[2][256];
  __shared__ unsigned long long wsum[33];
  __shared__ uint32_t s_min[kWarps], s_max[kWarps];
  __shared__ unsigned s_digit, s_k, s_cnt;
  __shared__ int32_t s_alloc[kMaxBudgetHeads];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* sc = scores + (size_t)head * N;
  int32_t* out = kept_idx + (size_t)head * N;
  // Where the tokens come from: one tile is held in registers for the whole kernel, its loads
  // issued before the budget is known (they do not depend on it, so the two round trips overlap);
  // longer heads are staged in shared memory (or read from global memory when too long) tile by tile.
  const int ntiles = (N + kTile - 1) / kTile;
  const uint32_t* bits = reinterpret_cast<const uint32_t*>(sc);
  bool vec = (N & 3) == 0 && (reinterpret_cast<uintptr_t>(sc) & 15) == 0;
  uint32_t w[kSweep];
  if (ntiles == 1) load_group(bits, tid * kSweep, N, vec, keyed, w);
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
  if (ntiles > 1 && use_smem) {
    if (vec) {
      const uint4* s4 = reinterpret_cast<const uint4*>(sc);
      uint4* d4 = reinterpret_cast<uint4*>(sh_bits);
#pragma unroll 4
      for (int i = tid; i < N / 4; i += kThreads) d4[i] = s4[i];
    } else {
#pragma unroll 4
      for (int j = tid; j < N; j += kThreads) sh_bits[j] = bits[j];
    }
    bits = sh_bits;
    vec = true;
  }
  auto tile_load = [&](int j0) {
    if (ntiles > 1) load_group(bits, j0 + tid * kSweep, N, vec, keyed, w);
  };
  for (int i = tid; i < 256; i += kThreads) hist[0][i] = 0;

  const int lo = P, hi = N - R, kmid = b - P - R;
  // Threshold on the bits under `mask`: a middle token whose masked bits exceed T is kept, and of
  // those equal to T the keq of lowest index. With kmid == 0 nothing of the middle is kept.
  uint32_t T = 0xffffffffu, mask = 0xffffffffu;
  unsigned keq = 0;
  if (kmid > 0) {
    // the leading bits that every middle token shares (from their minimum and maximum) need no
    // digit pass: the keys of scores in (0, 1] share several, and a digit over them would fill
    // one bin
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (int j0 = 0; j0 < N; j0 += kTile) {
      tile_load(j0);
#pragma unroll
      for (int e = 0; e < kSweep; ++e) {
        const int j = j0 + tid * kSweep + e;
        if (j >= lo && j < hi) {
          mn = min(mn, w[e]);
          mx = max(mx, w[e]);
        }
      }
    }
    mn = __reduce_min_sync(kFull, mn);
    mx = __reduce_max_sync(kFull, mx);
    if (lane == 0) {
      s_min[warp] = mn;
      s_max[warp] = mx;
    }
    __syncthreads();  // also orders the zeroing of hist[0] before the first pass
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      mn = min(mn, s_min[i]);
      mx = max(mx, s_max[i]);
    }
    int rem = (mn ^ mx) ? 32 - __clz(mn ^ mx) : 0;  // bits below the shared prefix
    mask = rem >= 32 ? 0u : ~((1u << rem) - 1u);
    uint32_t prefix = mn & mask;
    unsigned k = (unsigned)kmid;  // rank (1-based, from the top) still to locate
    int cur = 0;
    while (rem > 0) {
      const int width = rem < 8 ? rem : 8;
      const int shift = rem - width;
      const uint32_t dmask = (1u << width) - 1u;
      for (int i = tid; i < 256; i += kThreads) hist[cur ^ 1][i] = 0;  // the next pass's bins
      for (int j0 = 0; j0 < N; j0 += kTile) {
        tile_load(j0);
#pragma unroll
        for (int e = 0; e < kSweep; ++e) {
          const int j = j0 + tid * kSweep + e;
          if (j >= lo && j < hi && (w[e] & mask) == prefix) atomicAdd(&hist[cur][(w[e] >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      if (tid < 32) {
        // lane l holds digits 255-8l ... 248-8l, so lane order is descending digit order
        const uint4 x = *reinterpret_cast<const uint4*>(&hist[cur][248 - 8 * tid]);
        const uint4 y = *reinterpret_cast<const uint4*>(&hist[cur][252 - 8 * tid]);
        const unsigned c[8] = {y.w, y.z, y.y, y.x, x.w, x.z, x.y, x.x};  // digits 255-8l-q
        unsigned local = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q) local += c[q];
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
              s_cnt = c[q];
              break;
            }
            cum += c[q];
          }
        }
      }
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= dmask << shift;
      k = s_k;
      rem = shift;
      cur ^= 1;
      if (s_k == s_cnt) break;  // the rank's bucket is kept whole: its lower bits do not matter
    }
    T = prefix;
    keq = k;
  }
  // Ordered sweep: one scan per tile gives every token the number of kept tokens above the
  // threshold and of tied tokens before it. The kept tied tokens are the first keq, so a kept
  // token's slot is nk + min(neq, keq).
  int base_k = 0, base_eq = 0;  // totals of the earlier tiles
  for (int j0 = 0; j0 < N; j0 += kTile) {
    tile_load(j0);
    const int jt = j0 + tid * kSweep;
    unsigned gt = 0, eqm = 0;
#pragma unroll
    for (int e = 0; e < kSweep; ++e) {
      const int j = jt + e;
      if (j < N) {
        const uint32_t v = w[e] & mask;
        if (j < lo || j >= hi || v > T) gt |= 1u << e;
        else if (v == T) eqm |= 1u << e;
      }
    }
    unsigned long long tot;
    const unsigned long long ex =
        block_excl_scan64(((unsigned long long)__popc(eqm) << 32) | (unsigned)__popc(gt), wsum, &tot);
    int nk = base_k + (int)(ex & 0xffffffffull), neq = base_eq + (int)(ex >> 32);
#pragma unroll
    for (int e = 0; e < kSweep; ++e) {
      const bool is_gt = (gt >> e) & 1u, is_eq = (eqm >> e) & 1u;
      if (is_gt || (is_eq && neq < (int)keq)) out[nk + min(neq, (int)keq)] = jt + e;
      nk += is_gt;
      neq += is_eq;
    }
    base_k += (int)(tot & 0xffffffffull);
    base_eq += (int)(tot >> 32);
  }
  if (tid == 0) kept_len[head] = base_k + min(base_eq, (int)keq);
}

}  // namespace kvc
