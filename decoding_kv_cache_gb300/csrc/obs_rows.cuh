// obs_rows.cuh -- the observation rows of a KV head's GQA group, as device functions run by the
// observation kernel (score.cu) and the fp32 cluster kernel (score_small.cu).
//
// BeaconKV write-up, "观察 query 集 = 最近查询 + 信标查询" (observation set = recent queries +
// beacon queries) and "打分时的 RoPE 对齐" (beacons rotated to the current step t, recent queries
// at their own positions): per query head of the group, its recent rows as stored, then its
// beacons (the buffer itself when it holds at most n_b rows, else FPS down to n_b) rotated to t
// and rounded to the storage type.
#pragma once

#include "fps_warp.cuh"

namespace kvc {

// The observation rows of one KV head's group: the first nw warps of the CTA take its query heads,
// one warp at a time each. obs / valid point at the head's tile (global memory for build_obs_kernel,
// shared memory in the fp32 cluster kernel of score_small.cu); smem_raw holds nw FPS scratch areas,
// then the rotation table; s_nvalid counts the valid rows (extended options); write_picks: this CTA
// reports the beacon picks (when the caller asked for them).
template <typename T, int D>
__device__ __forceinline__ void obs_group_rows(const ScoreArgs& a, const ScoreWs& ws, int head, int nw,
                                               unsigned char* smem_raw, T* obs, uint8_t* valid, int* s_nvalid,
                                               bool write_picks = true) {
  const int Hkv = a.g.Hkv, B = a.g.B, Hq = a.g.Hq;
  const int l = head / (B * Hkv), b = (head / Hkv) % B, h = head % Hkv;
  const int G = Hq / Hkv, per_q = a.n_r + a.n_b, hd = D / 2;
  const int qs = a.qstride;  // rows of query head g start at g * qs
  constexpr int LD = Staging<T, D>::LD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nthr = nw * kWarp;  // the participating threads: warps 0 .. nw-1
  const int npad = (a.qmax + 15) & ~15;
  void* scratch = smem_raw + warp * ((fps_scratch_bytes<T, D>(npad) + 15) & ~(size_t)15);
  const T* qrec = static_cast<const T*>(a.q_recent);
  const T* qbuf = static_cast<const T*>(a.qbuf);

  constexpr int per = 16 / (int)sizeof(T);
  constexpr int lpr = (D / 2) / per;  // rotation: lanes per beacon row, `per` pairs (i, i + D/2) each
  constexpr int rpi = kWarp / lpr;
  const int i0 = (lane % lpr) * per, rsel = lane / lpr;
  float2* rope_s = reinterpret_cast<float2*>(smem_raw + (size_t)nw * ((fps_scratch_bytes<T, D>(npad) + 15) & ~(size_t)15));
  const bool mean_w = a.ext && a.row_agg == KVC_AGG_MEAN;

  // every participating warp has at least one query head (nw <= G), so the step shared by the nw
  // warps in the first iteration is reached by all of them
  for (int g = warp, it = 0; g < G; g += nw, ++it) {
    const int hq = h * G + g;
    const size_t qh = ((size_t)l * B + b) * Hq + hq;
    T* orow = obs + (size_t)g * qs * D;
    // Issue this query head's global reads first: stage the whole buffer (rows at or past its
    // count are staged too but never read: FPS and the Gram entries it uses involve live rows
    // only), the count, and the first batch of recent rows.
    fps_buffer_issue<T, D>(qbuf + qh * a.qmax * D, a.qmax, npad, scratch);
    int c = a.qmax > 0 ? a.count[qh] : 0;
    const uint4* qr = reinterpret_cast<const uint4*>(qrec + qh * a.n_r * D);
    uint4* od = reinterpret_cast<uint4*>(orow);
    const int nv = a.n_r * D * (int)sizeof(T) / 16;  // recent rows, 16-byte vectors
    uint4 rv[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (u * kWarp + lane < nv) rv[u] = qr[u * kWarp + lane];
    if (it == 0) {
      // while those are in flight: this CTA's share of the scoring kernel's exchange words (they
      // start at zero) and the rotation table in shared memory, read from the parameter block at
      // warp-uniform indices (a per-lane index there serialises; the rotation reads it per lane)
      if (a.xch_zero) {
        const long long share = (a.xch_zero_words + gridDim.x - 1) / gridDim.x;
        const long long lo = (long long)blockIdx.x * share;
        const long long hi = lo + share < a.xch_zero_words ? lo + share : a.xch_zero_words;
        for (long long w = lo + threadIdx.x; w < hi; w += nthr) a.xch_zero[w] = 0ull;
      }
      for (int i = warp; i < hd; i += nw)  // warp-uniform indices: broadcast parameter reads
        if (lane == 0) rope_s[i] = a.rope[i];
      // the scoring kernel combines a head's tiles into its scores with atomics: start at zero
      if (a.tiles > 1)
        for (int j = threadIdx.x; j < a.g.N; j += nthr) a.scores[(size_t)head * a.g.N + j] = 0.f;
      if (threadIdx.x == 0) *s_nvalid = 0;
      asm volatile("bar.sync 1, %0;\n" ::"r"(nthr) : "memory");  // the nw warps
    }
    if (c < 0 || c > a.qmax) {
      if (lane == 0) status_or(a.status, KVC_STATUS_COUNT_RANGE);
      c = c < 0 ? 0 : a.qmax;
    }
    // recent queries: already rotated to their own positions, copied as stored
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (u * kWarp + lane < nv) od[u * kWarp + lane] = rv[u];
    for (int e0 = 8 * kWarp; e0 < nv; e0 += 8 * kWarp) {  // more than 8 vectors per lane: further batches
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * kWarp + lane < nv) v[u] = qr[e0 + u * kWarp + lane];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (e0 + u * kWarp + lane < nv) od[e0 + u * kWarp + lane] = v[u];
    }
    for (int r = lane; r < a.n_r; r += kWarp) valid[g * qs + r] = 1;
    // beacons: the buffer itself when it holds at most n_b rows, else FPS down to n_b
    int* pk;
    const T* xs = fps_buffer_finish<T, D>(c, a.n_b, npad, scratch, &pk);
    const int nb = c < a.n_b ? c : a.n_b;
    if (a.ext) {
      if (lane == 0) atomicAdd(s_nvalid, a.n_r + nb);
      // the mean over this query head's rows weighs each valid row 1 / (its valid rows)
      if (mean_w) {
        const float w = a.n_r + nb > 0 ? 1.f / (float)(a.n_r + nb) : 0.f;
        for (int r = lane; r < qs && g * qs + r < a.M_pad; r += kWarp)
          ws.rw[(size_t)head * a.M_pad + g * qs + r] = r < a.n_r + nb ? w : 0.f;
      }
      // rows between this query head's last row and the next head's first
      if (g + 1 < G)
        for (int e = lane; e < (qs - per_q) * D; e += kWarp) orow[(size_t)per_q * D + e] = from_f32<T>(0.f);
      for (int r = per_q + lane; r < qs && g + 1 < G; r += kWarp) valid[g * qs + r] = 0;
    }
    // the lane's `per` pairs of the rotation table (the same for every beacon row), in 16-byte reads
    alignas(16) float2 csv[per];
#pragma unroll
    for (int q2 = 0; q2 < per / 2; ++q2)
      reinterpret_cast<float4*>(csv)[q2] = reinterpret_cast<const float4*>(rope_s + i0)[q2];
    for (int k0 = 0; k0 < a.n_b; k0 += rpi) {
      const int k = k0 + rsel;
      if (k >= a.n_b) continue;
      T* dst = orow + (size_t)(a.n_r + k) * D;
      alignas(16) T o1[per];
      alignas(16) T o2[per];
      if (k < nb) {
        // the lane's `per` pairs: one 16-byte read per half (the staged rows' stride LD and i0 are
        // multiples of 16 bytes for both storage types)
        const T* src = xs + pk[k] * LD;
        alignas(16) T xa[per];
        alignas(16) T xb[per];
        *reinterpret_cast<uint4*>(xa) = *reinterpret_cast<const uint4*>(src + i0);
        *reinterpret_cast<uint4*>(xb) = *reinterpret_cast<const uint4*>(src + i0 + hd);
#pragma unroll
        for (int u = 0; u < per; ++u) {
          const float2 cs = csv[u];
          const float x0 = to_f32(xa[u]), x1 = to_f32(xb[u]);
          // each product and the sum rounded separately (no fused multiply-add), so the
          // rounding to the storage type below is a reproducible decision
          o1[u] = from_f32<T>(__fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y)));
          o2[u] = from_f32<T>(__fadd_rn(__fmul_rn(x1, cs.x), __fmul_rn(x0, cs.y)));
        }
      } else {
#pragma unroll
        for (int u = 0; u < per; ++u) o1[u] = o2[u] = from_f32<T>(0.f);
      }
      *reinterpret_cast<uint4*>(dst + i0) = *reinterpret_cast<const uint4*>(o1);
      *reinterpret_cast<uint4*>(dst + i0 + hd) = *reinterpret_cast<const uint4*>(o2);
      if (i0 == 0) valid[g * qs + a.n_r + k] = k < nb ? 1 : 0;
    }
    if (a.beacon_picks && write_picks)
      for (int k = lane; k < a.n_b; k += kWarp) a.beacon_picks[qh * a.n_b + k] = k < nb ? pk[k] : -1;
    __syncwarp();
  }
}

// padding rows of a head's tile up to the stored row count (every thread of the CTA)
template <typename T, int D>
__device__ __forceinline__ void obs_padding(const ScoreArgs& a, T* obs, uint8_t* valid) {
  for (int e = threadIdx.x; e < (a.M_pad - a.M) * D; e += blockDim.x) obs[(size_t)a.M * D + e] = from_f32<T>(0.f);
  for (int r = a.M + threadIdx.x; r < a.M_pad; r += blockDim.x) valid[r] = 0;
}

}  // namespace kvc
