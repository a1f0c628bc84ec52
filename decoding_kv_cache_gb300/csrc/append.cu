// append.cu -- kvc_append: one decode step's queries into the observation state.
//
// BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": every attention head keeps a
// bounded buffer of pre-RoPE queries that grows to B_Q^max and is cut back to B_Q^min by
// farthest-point sampling, so beacons keep evolving while memory stays bounded; "观察 query 集 =
// 最近查询 + 信标查询": the recent part of the observation set is the latest n_r queries at
// their own positions. One warp per query head:
//   ring     row t mod n_r of the head's recent ring takes the post-RoPE query (or the pre-RoPE
//            query turned to position t, rounded to the storage type as beacons are)
//   buffer   a buffer full on entry is compressed first; the pre-RoPE query goes to row count;
//            a buffer that has just become full is compressed. Compression = greedy FPS under
//            cosine distance from the oldest row, qmax/2 survivors moved to the front in time
//            order. Rows past the new count keep whatever they held.
// Most steps only append (two short row writes); the staging and the FPS run on the steps that
// fill a buffer, one in qmax/2.
#include "fps_warp.cuh"
#include "kvc_internal.cuh"

namespace kvc {

template <typename T, int D>
__global__ void append_kernel(AppendArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int npad = (a.qmax + 15) & ~15;
  const size_t per_warp = (fps_scratch_bytes<T, D>(npad) + 15) & ~(size_t)15;
  void* scratch = smem_raw + warp * per_warp;
  const int qh = blockIdx.x * wpb + warp;
  if (qh >= a.nheads) return;  // the whole warp leaves together
  constexpr int per = 16 / (int)sizeof(T);  // elements per 16-byte vector
  constexpr int vpr = D / per;              // vectors per row (8 .. 32)
  constexpr int hd = D / 2;
  const int m = a.qmax / 2;

  // every global read of this head in flight first: the new query (vector lane of the row), the
  // post-RoPE query when given, and the buffer's count
  const T* qp = static_cast<const T*>(a.q_pre) + (size_t)qh * D;
  uint4 vpre = make_uint4(0u, 0u, 0u, 0u), vpost = vpre;
  if (lane < vpr) vpre = reinterpret_cast<const uint4*>(qp)[lane];
  if (a.q_post && lane < vpr) vpost = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q_post) + (size_t)qh * D)[lane];
  const int c0 = a.count[qh];

  // ---- recent ring -------------------------------------------------------------------------
  if (a.n_r > 0) {
    T* dst = static_cast<T*>(a.q_recent) + ((size_t)qh * a.n_r + a.ring_slot) * D;
    if (a.q_post) {
      if (lane < vpr) reinterpret_cast<uint4*>(dst)[lane] = vpost;
    } else {
      // lane owns pairs (i, i + D/2) for i in [lane*per, lane*per + per); its second half comes
      // from the lane holding vector lane + vpr/2 (the branch is uniform over the warp)
      const int from = (lane + vpr / 2) & 31;
      uint4 hi;
      hi.x = __shfl_sync(kFull, vpre.x, from);
      hi.y = __shfl_sync(kFull, vpre.y, from);
      hi.z = __shfl_sync(kFull, vpre.z, from);
      hi.w = __shfl_sync(kFull, vpre.w, from);
      // this lane's (cos, sin) pairs, read with warp-uniform indices (a per-lane index into the
      // parameter block would serialise the warp's constant loads)
      float2 cs[per];
#pragma unroll
      for (int i = 0; i < hd; ++i) {
        const float2 v = a.rope[i];
        if (lane == i / per) cs[i % per] = v;
      }
      if (lane < hd / per) {
        const T* lo_e = reinterpret_cast<const T*>(&vpre);
        const T* hi_e = reinterpret_cast<const T*>(&hi);
        alignas(16) T o1[per];
        alignas(16) T o2[per];
#pragma unroll
        for (int u = 0; u < per; ++u) {
          const float x0 = to_f32(lo_e[u]), x1 = to_f32(hi_e[u]);
          // each product and the sum rounded on its own (no fused multiply-add), as for beacons
          o1[u] = from_f32<T>(__fsub_rn(__fmul_rn(x0, cs[u].x), __fmul_rn(x1, cs[u].y)));
          o2[u] = from_f32<T>(__fadd_rn(__fmul_rn(x1, cs[u].x), __fmul_rn(x0, cs[u].y)));
        }
        reinterpret_cast<uint4*>(dst)[lane] = *reinterpret_cast<const uint4*>(o1);
        reinterpret_cast<uint4*>(dst)[lane + vpr / 2] = *reinterpret_cast<const uint4*>(o2);
      }
    }
  }

  // ---- pre-RoPE buffer -----------------------------------------------------------------------
  T* x = static_cast<T*>(a.qbuf) + (size_t)qh * a.qmax * D;
  int32_t* pick_out = a.picks ? a.picks + (size_t)qh * m : nullptr;
  if (c0 < 0 || c0 > a.qmax) {
    if (lane == 0) status_or(a.status, KVC_STATUS_COUNT_RANGE);
    if (pick_out)
      for (int k = lane; k < m; k += kWarp) pick_out[k] = -1;
    return;
  }
  if (c0 + 1 < a.qmax) {  // the common step: append only
    if (lane < vpr) reinterpret_cast<uint4*>(x + (size_t)c0 * D)[lane] = vpre;
    __syncwarp();
    if (lane == 0) a.count[qh] = c0 + 1;
    if (pick_out)
      for (int k = lane; k < m; k += kWarp) pick_out[k] = -1;
    return;
  }

  // This step fills the buffer (c0 == qmax - 1) or finds it full (c0 == qmax): stage its rows.
  constexpr int LD = Staging<T, D>::LD;
  T* xs = reinterpret_cast<T*>(scratch);
  float* G = reinterpret_cast<float*>(xs + (size_t)npad * LD);
  int* pk = reinterpret_cast<int*>(G + (size_t)npad * (npad + 1));
  stage_rows_issue<T, D>(x, c0, npad, xs);
  // the new row's global copy (not among the staged rows: it goes to row c0 < qmax when the
  // buffer is filling, to row qmax/2 after a compression when it was full)
  const int new_row = c0 == a.qmax ? m : c0;
  stage_rows_wait<T>();
  int c = c0;
  int compressions = 0;
  // one compression of the c == qmax staged rows: FPS picks, survivors to global rows [0, m)
  // from the staged copy, and the staged rows compacted the same way when more work follows
  auto compress = [&](bool more) {
    fps_rows<T, D>(xs, G, a.qmax, npad, m, pk);  // pk[0..m) ascending; pk[0] = 0
    for (int e = lane; e < m * vpr; e += kWarp) {
      const int k = e / vpr, v = e % vpr;
      const int src = pk[k];
      if (src != k) {
        const T* s = xs + (size_t)src * LD + v * per;
        T* d = x + (size_t)k * D + v * per;
        if constexpr (sizeof(T) == 2) {
          *reinterpret_cast<uint4*>(d) = *reinterpret_cast<const uint4*>(s);  // LD*2 is a multiple of 16
        } else {
#pragma unroll
          for (int u = 0; u < per; ++u) d[u] = s[u];
        }
      }
    }
    __syncwarp();
    if (more) {
      // in place, in row order: a source row pk[k] >= k is never overwritten before it is read
      for (int k = 1; k < m; ++k) {
        const int src = pk[k];
        if (src != k)
          for (int d = lane; d < D; d += kWarp) xs[(size_t)k * LD + d] = xs[(size_t)src * LD + d];
        __syncwarp();
      }
      for (int e = lane; e < (npad - m) * D; e += kWarp) xs[(size_t)(m + e / D) * LD + e % D] = from_f32<T>(0.f);
    }
    __syncwarp();
    c = m;
    ++compressions;
  };
  if (c == a.qmax) compress(true);
  // the new row: staged (for a compression that follows) and written to its global row
  {
    const T* e = reinterpret_cast<const T*>(&vpre);
    if (lane < vpr)
      for (int u = 0; u < per; ++u) xs[(size_t)c * LD + lane * per + u] = e[u];
    if (lane < vpr) reinterpret_cast<uint4*>(x + (size_t)new_row * D)[lane] = vpre;
    __syncwarp();
    c += 1;
  }
  if (c == a.qmax) compress(false);
  if (lane == 0) a.count[qh] = c;
  if (pick_out)
    for (int k = lane; k < m; k += kWarp) pick_out[k] = compressions ? pk[k] : -1;
}

int launch_append(const AppendArgs& a, int dtype, int D, cudaStream_t s) {
  if (a.nheads == 0) return KVC_OK;
  const int npad = (a.qmax + 15) & ~15;
  auto go = [&](auto kernel, size_t per_warp) -> int {
    per_warp = (per_warp + 15) & ~(size_t)15;
    int wpb = (int)((200u * 1024u) / per_warp);
    wpb = wpb < 1 ? 1 : (wpb > 4 ? 4 : wpb);
    const size_t smem = per_warp * wpb;
    const int grid = (a.nheads + wpb - 1) / wpb;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    kernel<<<grid, 32 * wpb, smem, s>>>(a);
    return KVC_OK;
  };
  int rc;
  if (dtype == KVC_BF16)
    rc = D == 128 ? go(append_kernel<__nv_bfloat16, 128>, fps_scratch_bytes<__nv_bfloat16, 128>(npad))
                  : go(append_kernel<__nv_bfloat16, 64>, fps_scratch_bytes<__nv_bfloat16, 64>(npad));
  else
    rc = D == 128 ? go(append_kernel<float, 128>, fps_scratch_bytes<float, 128>(npad))
                  : go(append_kernel<float, 64>, fps_scratch_bytes<float, 64>(npad));
  if (rc) return rc;
  return launch_ok();
}

}  // namespace kvc
