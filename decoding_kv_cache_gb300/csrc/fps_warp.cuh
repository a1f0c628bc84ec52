// fps_warp.cuh -- one warp runs greedy farthest-point sampling over a small query buffer.
//
// BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": FPS greedily picks the
// m mutually most dissimilar points of the buffer. Here: cosine distance 1 - cos on the
// (pre-RoPE) rows, start from the oldest row (index 0), each step adds the candidate with
// the largest distance to the chosen set, ties to the lower row. Distances are fp32.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

// Rows of x (global, storage type T, row length D, n <= 64 rows) are normalised into the
// warp's shared scratch xs[n][D+1] (the +1 keeps lane-per-row reads conflict-free). Lane l
// owns candidates l and l+32. On return picks[0..m) (warp-shared) holds the chosen rows in
// ascending order. All 32 lanes must call it.
template <typename T>
__device__ void fps_warp(const T* __restrict__ x, int n, int D, int m, float* xs, int* picks) {
  const int lane = threadIdx.x & 31;
  const int ld = D + 1;
  for (int i = 0; i < n; ++i) {
    float ss = 0.f;
    for (int d = lane; d < D; d += kWarp) {
      const float v = to_f32(x[(size_t)i * D + d]);
      xs[i * ld + d] = v;
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;  // a zero row stays zero: distance 1 to all
    for (int d = lane; d < D; d += kWarp) xs[i * ld + d] *= inv;
  }
  __syncwarp();

  auto dist = [&](int i, int j) {
    float s = 0.f;
    const float* a = xs + i * ld;
    const float* b = xs + j * ld;
    for (int d = 0; d < D; ++d) s = fmaf(a[d], b[d], s);
    return 1.f - s;
  };

  float md[2];
  bool live[2], chosen[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int i = lane + kWarp * c;
    live[c] = i < n;
    chosen[c] = (i == 0);
    const float d0 = live[c] ? dist(i, 0) : -INFINITY;
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
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int i = lane + kWarp * c;
      if (i == bi) chosen[c] = true;
      if (live[c] && !chosen[c]) md[c] = fminf(md[c], dist(i, bi));
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
