// fps.cu -- kvc_fps_update: continual farthest-point compression of the beacon buffers.
//
// BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": each head's bounded buffer of
// pre-RoPE queries is filled to B_Q^max and then cut back to B_Q^min by FPS, so the beacon
// set keeps evolving while memory stays bounded. One warp per query head.
#include "fps_warp.cuh"
#include "kvc_internal.cuh"

namespace kvc {

template <typename T, int D>
__global__ void fps_update_kernel(T* __restrict__ qbuf, int nheads, int qmax, int32_t* __restrict__ count,
                                  int32_t* __restrict__ picks_out, int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int npad = (qmax + 15) & ~15;
  const size_t per = (fps_scratch_bytes<T, D>(npad) + 15) & ~(size_t)15;
  void* scratch = smem_raw + warp * per;
  const int qh = blockIdx.x * wpb + warp;
  if (qh >= nheads) return;  // the whole warp leaves together
  const int m = qmax / 2;
  const int c = count[qh];
  T* x = qbuf + (size_t)qh * qmax * D;
  if (c != qmax) {
    if (lane == 0 && (c < 0 || c > qmax)) status_or(status, KVC_STATUS_COUNT_RANGE);
    if (picks_out)
      for (int k = lane; k < m; k += kWarp) picks_out[(size_t)qh * m + k] = -1;
    return;
  }
  int* pk;
  const T* xs = fps_buffer<T, D>(x, qmax, m, npad, scratch, &pk);
  // Survivors to the front in time order, written back from the staged copy (same bytes).
  constexpr int LD = Staging<T, D>::LD;
  for (int k = 0; k < m; ++k) {
    const int src = pk[k];
    if (src != k)
      for (int d = lane; d < D; d += kWarp) x[(size_t)k * D + d] = xs[src * LD + d];
  }
  __syncwarp();
  if (lane == 0) count[qh] = m;
  if (picks_out)
    for (int k = lane; k < m; k += kWarp) picks_out[(size_t)qh * m + k] = pk[k];
}

int launch_fps_update(int dtype, int nheads_q, int D, void* qbuf, int qmax, int32_t* count, int32_t* picks,
                      int32_t* status, cudaStream_t s) {
  if (nheads_q == 0) return KVC_OK;
  const int npad = (qmax + 15) & ~15;
  auto go = [&](auto kernel, auto* typed, size_t per_warp) -> int {
    per_warp = (per_warp + 15) & ~(size_t)15;
    int wpb = (int)((200u * 1024u) / per_warp);
    wpb = wpb < 1 ? 1 : (wpb > 4 ? 4 : wpb);
    const size_t smem = per_warp * wpb;
    const int grid = (nheads_q + wpb - 1) / wpb;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    kernel<<<grid, 32 * wpb, smem, s>>>(typed, nheads_q, qmax, count, picks, status);
    return KVC_OK;
  };
  int rc;
  if (dtype == KVC_BF16)
    rc = D == 128 ? go(fps_update_kernel<__nv_bfloat16, 128>, static_cast<__nv_bfloat16*>(qbuf),
                       fps_scratch_bytes<__nv_bfloat16, 128>(npad))
                  : go(fps_update_kernel<__nv_bfloat16, 64>, static_cast<__nv_bfloat16*>(qbuf),
                       fps_scratch_bytes<__nv_bfloat16, 64>(npad));
  else
    rc = D == 128 ? go(fps_update_kernel<float, 128>, static_cast<float*>(qbuf), fps_scratch_bytes<float, 128>(npad))
                  : go(fps_update_kernel<float, 64>, static_cast<float*>(qbuf), fps_scratch_bytes<float, 64>(npad));
  if (rc) return rc;
  return launch_ok();
}

}  // namespace kvc
