// compact.cu -- kvc_compact: the kept tokens' K and V rows move to the head's front, in order.
// The move itself (and why a forward sweep is safe in place) is compact_warp in compact.cuh.
#include "compact.cuh"

namespace kvc {

// one warp per (head, K or V)
__global__ void __launch_bounds__(32) compact_bulk_kernel(CompactArgs a) {
  extern __shared__ __align__(128) uint8_t sm[];
  griddep_wait();  // the kept lists come from the previous kernel
  compact_warp(a, blockIdx.x, blockIdx.y, sm);
}

int launch_compact(const CacheGeom& g, int dtype, const LayerPtrs& K, const LayerPtrs& V, const int32_t* kept_idx,
                   const int32_t* kept_len, int32_t* status, bool validate, cudaStream_t s, bool list_per_seq) {
  const int heads = g.L * g.B * g.Hkv;
  if (heads == 0) return KVC_OK;
  CompactArgs a;
  a.g = g;
  a.K = K;
  a.V = V;
  a.kept_idx = kept_idx;
  a.kept_len = kept_len;
  a.status = status;
  a.rowbytes = g.D * (dtype == KVC_BF16 ? 2 : 4);
  a.validate = validate ? 1 : 0;
  a.list_seq = list_per_seq ? 1 : 0;
  const size_t smem = (size_t)kCompactWarpSmem;
  if (cudaFuncSetAttribute(compact_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (launch_pdl(compact_bulk_kernel, dim3(heads, 2), dim3(32), smem, s, false, a) != cudaSuccess) return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
