// fps_warp.cuh -- one warp runs greedy farthest-point sampling over a small query buffer.
//
// BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": FPS greedily picks the
// m mutually most dissimilar points of the buffer. Here: cosine distance 1 - cos on the
// (pre-RoPE) rows, start from the oldest row (index 0), each step adds the candidate with
// the largest distance to the chosen set, ties to the lower row. Distances are fp32.
// A query head's buffer is staged once into shared memory; everything after reads it there.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

// Stage rows [0, n) of x (global, storage type T, row length D) into the warp's shared
// scratch xs[n][D+1] as fp32 with coalesced 16-byte loads (the +1 keeps lane-per-row reads
// conflict-free). Requires D % 8 == 0 and a 16-byte aligned x.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(const T* __restrict__ x, int n, float* xs) {
  const int lane = threadIdx.x & 31;
  constexpr int per = 16 / sizeof(T);
  constexpr int vpr = D / per;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  for (int e = lane; e < n * vpr; e += kWarp) {
    const uint4 v = src[e];
    const int r = e / vpr, c0 = (e % vpr) * per;
    const T* t = reinterpret_cast<const T*>(&v);
#pragma unroll
    for (int q = 0; q < per; ++q) xs[r * (D + 1) + c0 + q] = to_f32(t[q]);
  }
  __syncwarp();
}

// Dot product of two staged rows with four independent accumulators (the loads are
// independent, so the FMA chain is the latency that matters).
template <int D>
__device__ __forceinline__ float dot_rows(const float* a, const float* b) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int d = 0; d < D; d += 4) {
    s0 = fmaf(a[d], b[d], s0);
    s1 = fmaf(a[d + 1], b[d + 1], s1);
    s2 = fmaf(a[d + 2], b[d + 2], s2);
    s3 = fmaf(a[d + 3], b[d + 3], s3);
  }
  return (s0 + s1) + (s2 + s3);
}

// Greedy FPS over the n <= 64 rows already staged in xs[n][D+1] (fp32, unnormalised):
// m picks, written ascending to picks[0..m) (warp-shared). Lane l owns candidates l and
// l+32; cosine distances use per-row inverse norms (a zero row has inverse norm 0, which
// puts it at distance 1 from everything). All 32 lanes must call it.
template <int D>
__device__ __forceinline__ void fps_staged(const float* xs, int n, int m, int* picks) {
  const int lane = threadIdx.x & 31;
  constexpr int ld = D + 1;
  float inv[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int i = lane + kWarp * c;
    float ss = 0.f;
    if (i < n) ss = dot_rows<D>(xs + i * ld, xs + i * ld);
    inv[c] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
  }
  // inverse norm of the row just chosen, fetched from its owning lane
  auto inv_of = [&](int j) {
    const float a = __shfl_sync(kFull, inv[0], j & 31);
    const float b = __shfl_sync(kFull, inv[1], j & 31);
    return j < kWarp ? a : b;
  };
  auto dist = [&](int c, int i, int j, float invj) {
    return 1.f - dot_rows<D>(xs + i * ld, xs + j * ld) * inv[c] * invj;
  };

  float md[2];
  bool live[2], chosen[2];
  const float inv0 = inv_of(0);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int i = lane + kWarp * c;
    live[c] = i < n;
    chosen[c] = (i == 0);
    const float d0 = live[c] ? dist(c, i, 0, inv0) : -INFINITY;
    md[c] = d0 == d0 ? d0 : -INFINITY;  // a NaN row can still be picked last, never out of range
  }
  for (int k = 1; k < m; ++k) {
    float bv = -INFINITY;
    int bi = 1 << 30;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int i = lane + kWarp * c;
      if (live[c] && !chosen[c] && (md[c] > bv || (md[c] == bv && i < bi))) {
        bv = md[c];
        bi = i;
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    const float invj = inv_of(bi);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int i = lane + kWarp * c;
      if (i == bi) chosen[c] = true;
      if (live[c] && !chosen[c]) md[c] = fminf(md[c], dist(c, i, bi, invj));
    }
  }
  // ascending output: position = number of chosen rows below this one
  const unsigned m0 = __ballot_sync(kFull, live[0] && chosen[0]);
  const unsigned m1 = __ballot_sync(kFull, live[1] && chosen[1]);
  const unsigned below = (1u << lane) - 1u;
  if (live[0] && chosen[0]) picks[__popc(m0 & below)] = lane;
  if (live[1] && chosen[1]) picks[__popc(m0) + __popc(m1 & below)] = lane + kWarp;
  __syncwarp();
}

}  // namespace kvc
