// fps_warp.cuh -- one warp runs greedy farthest-point sampling over a small query buffer.
//
// BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": FPS greedily picks the
// m mutually most dissimilar points of the buffer. Here: cosine distance 1 - cos on the
// (pre-RoPE) rows, start from the oldest row (index 0), each step adds the candidate with
// the largest distance to the chosen set, ties to the lower row. Distances are fp32.
//
// A query head's buffer (n <= 64 rows) is staged once into shared memory in its storage
// type, its Gram matrix G = X X^T is formed once (warp-level bf16 MMA with fp32 accumulate,
// whose products are exact; plain FMAs for fp32 rows), and each greedy step then needs one
// G entry per candidate: cos(i, j) = G_ij / sqrt(G_ii G_jj).
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

template <typename T, int D>
struct Staging;
template <int D>
struct Staging<__nv_bfloat16, D> {
  static constexpr int LD = D + 8;  // keeps 8-row ldmatrix reads conflict-free
};
template <int D>
struct Staging<float, D> {
  static constexpr int LD = D + 1;  // keeps lane-per-row reads conflict-free
};

// Shared scratch one warp needs for a buffer of up to npad rows (npad a multiple of 16).
template <typename T, int D>
__host__ __device__ constexpr size_t fps_scratch_bytes(int npad) {
  return (size_t)npad * Staging<T, D>::LD * sizeof(T) + (size_t)npad * (npad + 1) * sizeof(float) +
         (size_t)npad * sizeof(int);
}

// Copy rows [0, n) of x (global, 16-byte aligned) into xs[npad][LD]; rows [n, npad) become zero.
template <typename T, int D>
__device__ __forceinline__ void stage_rows(const T* __restrict__ x, int n, int npad, T* xs) {
  const int lane = threadIdx.x & 31;
  constexpr int per = 16 / sizeof(T);
  constexpr int vpr = D / per;
  constexpr int LD = Staging<T, D>::LD;
  const uint4* src = reinterpret_cast<const uint4*>(x);
  for (int e = lane; e < npad * vpr; e += kWarp) {
    const int r = e / vpr, c0 = (e % vpr) * per;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r < n) v = src[e];
    if constexpr (sizeof(T) == 2) {
      *reinterpret_cast<uint4*>(xs + r * LD + c0) = v;  // LD*2 is a multiple of 16 bytes
    } else {
      const T* t = reinterpret_cast<const T*>(&v);
#pragma unroll
      for (int q = 0; q < per; ++q) xs[r * LD + c0 + q] = t[q];
    }
  }
  __syncwarp();
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// G[i][j] (ld = npad + 1) = row_i . row_j over the staged bf16 rows, npad a multiple of 16.
template <int D>
__device__ __forceinline__ void gram_rows(const __nv_bfloat16* xs, int npad, float* G) {
  const int lane = threadIdx.x & 31;
  constexpr int LD = Staging<__nv_bfloat16, D>::LD;
  const int ldg = npad + 1;
  for (int mt = 0; mt < npad / 16; ++mt)
    for (int np = 0; np < npad / 16; ++np) {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t af[4], bf[4];
        ldsm_x4(af, xs + (mt * 16 + (lane & 15)) * LD + ks * 16 + (lane >> 4) * 8);
        ldsm_x4(bf, xs + (np * 16 + ((lane >> 4) << 3) + (lane & 7)) * LD + ks * 16 + ((lane >> 3) & 1) * 8);
        mma_16816(acc[0], af, bf[0], bf[1]);
        mma_16816(acc[1], af, bf[2], bf[3]);
      }
      const int r0 = mt * 16 + (lane >> 2), cb = np * 16 + 2 * (lane & 3);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        G[r0 * ldg + cb + 8 * t] = acc[t][0];
        G[r0 * ldg + cb + 8 * t + 1] = acc[t][1];
        G[(r0 + 8) * ldg + cb + 8 * t] = acc[t][2];
        G[(r0 + 8) * ldg + cb + 8 * t + 1] = acc[t][3];
      }
    }
  __syncwarp();
}

template <int D>
__device__ __forceinline__ void gram_rows(const float* xs, int npad, float* G) {
  const int lane = threadIdx.x & 31;
  constexpr int LD = Staging<float, D>::LD;
  const int ldg = npad + 1;
  for (int i = lane; i < npad; i += kWarp)
    for (int j = 0; j < npad; ++j) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll 8
      for (int d = 0; d < D; d += 2) {
        s0 = fmaf(xs[i * LD + d], xs[j * LD + d], s0);
        s1 = fmaf(xs[i * LD + d + 1], xs[j * LD + d + 1], s1);
      }
      G[i * ldg + j] = s0 + s1;
    }
  __syncwarp();
}

// Greedy FPS from the Gram matrix of n <= 64 rows: m picks, written ascending to picks[0..m)
// (warp-shared). Lane l owns candidates l and l+32. A zero row (G_ii = 0) has inverse norm 0,
// which puts it at distance 1 from everything. All 32 lanes must call it.
__device__ __forceinline__ void fps_gram(const float* G, int ldg, int n, int m, int* picks) {
  const int lane = threadIdx.x & 31;
  float inv[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int i = lane + kWarp * c;
    const float ss = i < n ? G[i * ldg + i] : 0.f;
    inv[c] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
  }
  // inverse norm of the row just chosen, fetched from its owning lane
  auto inv_of = [&](int j) {
    const float a = __shfl_sync(kFull, inv[0], j & 31);
    const float b = __shfl_sync(kFull, inv[1], j & 31);
    return j < kWarp ? a : b;
  };
  float md[2];
  bool live[2], chosen[2];
  const float inv0 = inv_of(0);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int i = lane + kWarp * c;
    live[c] = i < n;
    chosen[c] = (i == 0);
    const float d0 = live[c] ? 1.f - G[i * ldg] * inv[c] * inv0 : -INFINITY;
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
      if (live[c] && !chosen[c]) md[c] = fminf(md[c], 1.f - G[i * ldg + bi] * inv[c] * invj);
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

// Stage rows [0, n) of x, form their Gram matrix and run FPS for m picks (all n rows are
// picked when m >= n). Scratch layout: staged rows, then G, then picks (fps_scratch_bytes).
// Returns the staged rows; *picks_out points at the picks.
template <typename T, int D>
__device__ __forceinline__ T* fps_buffer(const T* __restrict__ x, int n, int m, int npad, void* scratch,
                                         int** picks_out) {
  T* xs = reinterpret_cast<T*>(scratch);
  float* G = reinterpret_cast<float*>(xs + (size_t)npad * Staging<T, D>::LD);
  int* picks = reinterpret_cast<int*>(G + (size_t)npad * (npad + 1));
  *picks_out = picks;
  stage_rows<T, D>(x, n, npad, xs);
  if (m < n) {
    gram_rows<D>(xs, npad, G);
    fps_gram(G, npad + 1, n, m, picks);
  } else {
    for (int k = threadIdx.x & 31; k < n; k += kWarp) picks[k] = k;
    __syncwarp();
  }
  return xs;
}

}  // namespace kvc
