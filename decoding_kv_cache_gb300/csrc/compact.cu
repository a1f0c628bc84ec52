// compact.cu -- kvc_compact: the kept tokens' K and V rows move to the head's front, in order.
//
// The BeaconKV write-up's policy decides which tokens stay (keep / evict, "打分时的 RoPE 对齐");
// the slots of evicted tokens are reused by sliding the survivors forward in place.
//
// Why a forward sweep is safe in place: the kept list src[] is strictly increasing with
// src[k] >= k. Process destinations in tiles [t0, t0+T). Tile i writes rows [t0, t0+T);
// the original contents of those rows are sources only of kept entries k <= t0+T-1, i.e.
// of this tile or earlier ones, and every later tile reads rows >= its own first index.
// So each tile may write as soon as its own loads (and all earlier tiles' loads) are done,
// and the loads of tile i+1 may be issued before tile i is written. The leading run with
// src[k] == k needs no move and is skipped (found by binary search: src[k] - k is
// non-decreasing).
//
// One CTA per (head, K-or-V). 16-byte vectors, register double buffering across tiles.
#include "kvc_internal.cuh"

namespace kvc {

constexpr int kCpThreads = 256;
constexpr int kCpVec = 4;  // 16-byte vectors per thread per tile

struct CompactArgs {
  CacheGeom g;
  LayerPtrs K, V;
  const int32_t* kept_idx;
  const int32_t* kept_len;
  int32_t* status;
  int rowbytes;
  int validate;
};

__global__ void __launch_bounds__(kCpThreads) compact_kernel(CompactArgs a) {
  const int head = blockIdx.x;
  const int l = head / (a.g.B * a.g.Hkv), bh = head % (a.g.B * a.g.Hkv);
  char* base = static_cast<char*>(blockIdx.y ? a.V.p[l] : a.K.p[l]) + (size_t)bh * a.g.ncap * a.rowbytes;
  const int32_t* src = a.kept_idx + (size_t)head * a.g.N;
  const int len = a.kept_len[head];
  const int N = a.g.N;
  if (a.validate) {
    bool bad = len < 0 || len > N;
    if (!bad)
      for (int k = threadIdx.x; k < len; k += blockDim.x) {
        const int v = src[k];
        bad |= v < k || v >= N || (k > 0 && v <= src[k - 1]);
      }
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0 && blockIdx.y == 0) status_or(a.status, KVC_STATUS_BAD_INDEX);
      return;
    }
  }
  // first index that moves: smallest k with src[k] != k
  int lo = 0, hi = len;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (src[mid] == mid) lo = mid + 1; else hi = mid;
  }
  const int first = lo;
  if (first >= len) return;
  const int vpr = a.rowbytes / 16;
  const int tile_rows = kCpThreads * kCpVec / vpr;
  uint4 cur[kCpVec], nxt[kCpVec];

  auto load = [&](int t0, uint4 (&v)[kCpVec]) {
#pragma unroll
    for (int q = 0; q < kCpVec; ++q) {
      const int e = threadIdx.x + q * kCpThreads;
      const int k = t0 + e / vpr;
      if (k < len) v[q] = reinterpret_cast<const uint4*>(base + (size_t)src[k] * a.rowbytes)[e % vpr];
    }
  };
  load(first, cur);
  for (int t0 = first; t0 < len; t0 += tile_rows) {
    if (t0 + tile_rows < len) load(t0 + tile_rows, nxt);
    __syncthreads();  // every load of this tile (and all earlier ones) has been performed
#pragma unroll
    for (int q = 0; q < kCpVec; ++q) {
      const int e = threadIdx.x + q * kCpThreads;
      const int k = t0 + e / vpr;
      if (k < len) reinterpret_cast<uint4*>(base + (size_t)k * a.rowbytes)[e % vpr] = cur[q];
    }
#pragma unroll
    for (int q = 0; q < kCpVec; ++q) cur[q] = nxt[q];
  }
}

int launch_compact(const CacheGeom& g, int dtype, const LayerPtrs& K, const LayerPtrs& V, const int32_t* kept_idx,
                   const int32_t* kept_len, int32_t* status, bool validate, cudaStream_t s) {
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
  compact_kernel<<<dim3(heads, 2), kCpThreads, 0, s>>>(a);
  return launch_ok();
}

}  // namespace kvc
