// fps_warp.cuh -- one warp runs greedy farthest-point sampling over a small query buffer.
//
// BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": FPS greedily picks the
// m mutually most dissimilar points of the buffer. Here: cosine distance 1 - cos on the
// (pre-RoPE) rows, start from the oldest row (index 0), each step adds the candidate with
// the largest distance to the chosen set, ties to the lower row. Distances are fp32.
//
// A query head's buffer (n <= 64 rows) is staged once into shared memory in its storage
// type; each greedy step needs one dot product per candidate, cos(i, j) = G_ij / sqrt(G_ii G_jj).
// bf16 rows: the Gram matrix G = X X^T is formed once (warp-level bf16 MMA with fp32 accumulate,
// whose products are exact). fp32 rows: the dot products are formed as the steps need them (plain
// FMAs), which is fewer than the whole matrix when m < n.
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
  static constexpr int LD = D + 4;  // 16-byte rows; eight consecutive rows on distinct bank groups
};

// Shared scratch one warp needs for a buffer of up to npad rows (npad a multiple of 16):
// staged rows, Gram matrix and picks (offsets stay multiples of 16).
template <typename T, int D>
__host__ __device__ constexpr size_t fps_scratch_bytes(int npad) {
  return (size_t)npad * Staging<T, D>::LD * sizeof(T) + (size_t)npad * (npad + 1) * sizeof(float) +
         (size_t)npad * sizeof(int);
}

// Copy rows [0, n) of x (global, 16-byte aligned) into xs[npad][LD]; rows [n, npad) become zero.
// Rows go straight to shared memory as 16-byte cp.async copies (LD times the element size is a
// multiple of 16 bytes for both storage types), eight or sixteen per lane for a 32-row buffer (one
// bulk copy per row instead issued 32 copies one after another, ~3k cycles): stage_rows_issue only
// starts them and stage_rows_wait completes them, so other memory work can overlap.
template <typename T, int D>
__device__ __forceinline__ void stage_rows_issue(const T* __restrict__ x, int n, int npad, T* xs) {
  const int lane = threadIdx.x & 31;
  constexpr int LD = Staging<T, D>::LD;
  constexpr int per = 16 / (int)sizeof(T);
  constexpr int vpr = D / per;  // 16-byte vectors per row
  for (int e = lane; e < n * vpr; e += kWarp) {
    const int r = e / vpr, v = e % vpr;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(xs + r * LD + v * per)),
                 "l"(x + (size_t)r * D + v * per)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;\n" ::: "memory");
  for (int e = lane; e < (npad - n) * vpr; e += kWarp)  // zero rows past n
    *reinterpret_cast<uint4*>(xs + (n + e / vpr) * LD + (e % vpr) * per) = make_uint4(0u, 0u, 0u, 0u);
}

// Complete the staging started by stage_rows_issue (this lane's copies, then the warp's: the
// rows are read by other lanes). The copies depend on nothing else, so the wait always ends.
template <typename T>
__device__ __forceinline__ void stage_rows_wait() {
  asm volatile("cp.async.wait_group 0;\n" ::: "memory");
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

// G[i][j] (ld = npad + 1) = row_i . row_j over the staged bf16 rows, npad a multiple of 16 (<= 64).
// Only tiles on or above the diagonal are formed (the A fragment of a tile row is loaded once and
// shared by that row's tiles); an off-diagonal tile is also written mirrored.
template <int D>
__device__ __forceinline__ void gram_rows(const __nv_bfloat16* xs, int npad, float* G) {
  const int lane = threadIdx.x & 31;
  constexpr int LD = Staging<__nv_bfloat16, D>::LD;
  const int ldg = npad + 1;
  const int nt = npad / 16;
  if (nt == 2) {
    // 32 rows: the three upper tiles (0,0), (0,1), (1,1) in one pass over D, six independent
    // accumulation chains (tile row by tile row, the chains of the second row waited on the first)
    float acc[3][2][4];
#pragma unroll
    for (int t = 0; t < 3; ++t)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[t][h][k] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t af[2][4], bf[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        ldsm_x4(af[m], xs + (m * 16 + (lane & 15)) * LD + ks * 16 + (lane >> 4) * 8);
        ldsm_x4(bf[m], xs + (m * 16 + ((lane >> 4) << 3) + (lane & 7)) * LD + ks * 16 + ((lane >> 3) & 1) * 8);
      }
      const int tm[3] = {0, 0, 1}, tn[3] = {0, 1, 1};
#pragma unroll
      for (int t = 0; t < 3; ++t) {
        mma_16816(acc[t][0], af[tm[t]], bf[tn[t]][0], bf[tn[t]][1]);
        mma_16816(acc[t][1], af[tm[t]], bf[tn[t]][2], bf[tn[t]][3]);
      }
    }
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      const int mt = t == 2 ? 1 : 0, ct = t == 0 ? 0 : 1;
      const int r0 = mt * 16 + (lane >> 2);
      const int cb = ct * 16 + 2 * (lane & 3);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = cb + 8 * h;
        G[r0 * ldg + c] = acc[t][h][0];
        G[r0 * ldg + c + 1] = acc[t][h][1];
        G[(r0 + 8) * ldg + c] = acc[t][h][2];
        G[(r0 + 8) * ldg + c + 1] = acc[t][h][3];
        if (mt != ct) {
          G[c * ldg + r0] = acc[t][h][0];
          G[(c + 1) * ldg + r0] = acc[t][h][1];
          G[c * ldg + r0 + 8] = acc[t][h][2];
          G[(c + 1) * ldg + r0 + 8] = acc[t][h][3];
        }
      }
    }
    __syncwarp();
    return;
  }
  for (int mt = 0; mt < nt; ++mt) {
    float acc[4][2][4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[t][h][k] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t af[4];
      ldsm_x4(af, xs + (mt * 16 + (lane & 15)) * LD + ks * 16 + (lane >> 4) * 8);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (mt + t < nt) {
          uint32_t bf[4];
          ldsm_x4(bf, xs + ((mt + t) * 16 + ((lane >> 4) << 3) + (lane & 7)) * LD + ks * 16 + ((lane >> 3) & 1) * 8);
          mma_16816(acc[t][0], af, bf[0], bf[1]);
          mma_16816(acc[t][1], af, bf[2], bf[3]);
        }
    }
    const int r0 = mt * 16 + (lane >> 2);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (mt + t < nt) {
        const int cb = (mt + t) * 16 + 2 * (lane & 3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = cb + 8 * h;
          G[r0 * ldg + c] = acc[t][h][0];
          G[r0 * ldg + c + 1] = acc[t][h][1];
          G[(r0 + 8) * ldg + c] = acc[t][h][2];
          G[(r0 + 8) * ldg + c + 1] = acc[t][h][3];
          if (t > 0) {
            G[c * ldg + r0] = acc[t][h][0];
            G[(c + 1) * ldg + r0] = acc[t][h][1];
            G[c * ldg + r0 + 8] = acc[t][h][2];
            G[(c + 1) * ldg + r0 + 8] = acc[t][h][3];
          }
        }
      }
  }
  __syncwarp();
}

// Unsigned key with the order of the float (NaN excluded); -0 is first made +0 so that equal
// floats give equal keys.
__device__ __forceinline__ uint32_t ordered_key(float f) {
  const uint32_t b = __float_as_uint(f + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Greedy FPS over n <= 64 rows given their dot products g(i, j) = row_i . row_j (called by the lane
// that owns candidate i, for i < n): m picks, written ascending to picks[0..m) (warp-shared). Lane
// l owns candidates l and l+32. A zero row (g(i, i) = 0) has inverse norm 0, which puts it at
// distance 1 from everything. All 32 lanes must call it.
template <typename GF>
__device__ __forceinline__ void fps_greedy(GF g, int n, int m, int* picks) {
  const int lane = threadIdx.x & 31;
  float inv[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int i = lane + kWarp * c;
    const float ss = i < n ? g(i, i) : 0.f;
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
    const float d0 = live[c] ? 1.f - g(i, 0) * inv[c] * inv0 : -INFINITY;
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
    // warp argmax, ties to the lower row: the largest order-preserving key, then the lowest row
    // among the lanes holding it (two warp reductions instead of a five-step shuffle tree)
    const uint32_t key = ordered_key(bv);
    const uint32_t kmax = __reduce_max_sync(kFull, key);
    bi = (int)__reduce_min_sync(kFull, key == kmax ? (uint32_t)bi : 0xffffffffu);
    const float invj = inv_of(bi);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int i = lane + kWarp * c;
      if (i == bi) chosen[c] = true;
      if (live[c] && !chosen[c]) md[c] = fminf(md[c], 1.f - g(i, bi) * inv[c] * invj);
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

// Greedy FPS from a Gram matrix G (leading dimension ldg).
__device__ __forceinline__ void fps_gram(const float* G, int ldg, int n, int m, int* picks) {
  fps_greedy([&](int i, int j) { return G[i * ldg + j]; }, n, m, picks);
}

// row_i . row_j of staged fp32 rows: 16-byte reads (row i differs per lane, row j is one address for
// the warp), four FMA chains
template <int D>
__device__ __forceinline__ float dot_rows_f32(const float* xs, int i, int j) {
  constexpr int LD = Staging<float, D>::LD;
  const float4* a = reinterpret_cast<const float4*>(xs + i * LD);
  const float4* b = reinterpret_cast<const float4*>(xs + j * LD);
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  auto step = [&](int u) {
    const float4 x = a[u], y = b[u];
    a0 = fmaf(x.x, y.x, a0);
    a1 = fmaf(x.y, y.y, a1);
    a2 = fmaf(x.z, y.z, a2);
    a3 = fmaf(x.w, y.w, a3);
  };
  if constexpr (D <= 64) {  // every read in flight at once (the greedy steps wait on this product)
#pragma unroll
    for (int u = 0; u < D / 4; ++u) step(u);
  } else {  // D = 128: in batches of eight, so that the cluster kernel stays within its registers
#pragma unroll 8
    for (int u = 0; u < D / 4; ++u) step(u);
  }
  return (a0 + a1) + (a2 + a3);
}

// FPS picks over n staged rows. bf16 rows: the whole Gram matrix on warp MMAs (exact products)
// into G first. fp32 rows: only the dot products FPS reads (each candidate's norm and its product
// with every chosen row), formed when needed: m + 1 per candidate instead of n (G unused).
template <typename T, int D>
__device__ __forceinline__ void fps_rows(const T* xs, float* G, int n, int npad, int m, int* picks) {
  if constexpr (sizeof(T) == 2) {
    gram_rows<D>(xs, npad, G);
    fps_gram(G, npad + 1, n, m, picks);
  } else {
    fps_greedy([&](int i, int j) { return dot_rows_f32<D>(xs, i, j); }, n, m, picks);
  }
}

// FPS over a staged buffer. Scratch layout: staged rows, then G, then picks (fps_scratch_bytes).
// fps_buffer_issue starts staging rows [0, n) of x; fps_buffer_finish completes it, forms the Gram
// matrix and runs FPS for m picks (all n rows are picked when m >= n). finish returns the staged
// rows (*picks_out points at the picks).
template <typename T, int D>
__device__ __forceinline__ void fps_buffer_issue(const T* __restrict__ x, int n, int npad, void* scratch) {
  stage_rows_issue<T, D>(x, n, npad, reinterpret_cast<T*>(scratch));
}

template <typename T, int D>
__device__ __forceinline__ T* fps_buffer_finish(int n, int m, int npad, void* scratch, int** picks_out) {
  T* xs = reinterpret_cast<T*>(scratch);
  float* G = reinterpret_cast<float*>(xs + (size_t)npad * Staging<T, D>::LD);
  int* picks = reinterpret_cast<int*>(G + (size_t)npad * (npad + 1));
  *picks_out = picks;
  stage_rows_wait<T>();
  if (m < n) {
    fps_rows<T, D>(xs, G, n, npad, m, picks);
  } else {
    for (int k = threadIdx.x & 31; k < n; k += kWarp) picks[k] = k;
    __syncwarp();
  }
  return xs;
}

template <typename T, int D>
__device__ __forceinline__ T* fps_buffer(const T* __restrict__ x, int n, int m, int npad, void* scratch,
                                         int** picks_out) {
  fps_buffer_issue<T, D>(x, n, npad, scratch);
  return fps_buffer_finish<T, D>(n, m, npad, scratch, picks_out);
}

}  // namespace kvc
