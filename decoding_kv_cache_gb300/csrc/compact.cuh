// compact.cuh -- the in-place move of one head's kept K or V rows by one warp (compact.cu's kernel
// and the fused selection-and-compaction kernel in select.cu).
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
// One warp per (head, K-or-V). Each tile of kept rows is fetched with one bulk copy per run of
// consecutive sources into a 4-stage shared-memory ring and written back with one bulk store.
// Three tiles' loads and one tile's store are in flight at a time (the stage reloaded next is the
// one stored in the previous step), and each tile's source indices are read one step ahead, so
// no global read of the kept list sits between a tile's arrival and the next loads.
#pragma once

#include "kvc_internal.cuh"

namespace kvc {

struct CompactArgs {
  CacheGeom g;
  LayerPtrs K, V;
  const int32_t* kept_idx;
  const int32_t* kept_len;
  int32_t* status;
  int rowbytes;
  int validate;
  int list_seq;  // one kept list per sequence, shared by every layer and KV head (else one per head)
};

constexpr int kRing = 4;
constexpr int kTileBytes = 12288;  // 48 rows of 256 bytes (96, 24 or 48 for the other row sizes)
constexpr int kSrcRegs = (kTileBytes / 128 + 31) / 32;  // source indices per lane for one tile
constexpr int kCompactWarpSmem = kRing * kTileBytes + 64;  // one warp's ring and barriers

__device__ __forceinline__ uint32_t sm_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// The move of one head's K (kv = 0) or V (kv = 1) rows by one warp; sm: the warp's ring of kRing
// tiles followed by kRing mbarriers (kCompactWarpSmem bytes, 128-byte aligned). The kept list must
// be visible to the warp when it starts.
__device__ __forceinline__ void compact_warp(const CompactArgs& a, int head, int kv, uint8_t* sm) {
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kRing * kTileBytes);
  const int lane = threadIdx.x & 31;
  const int l = head / (a.g.B * a.g.Hkv), bh = head % (a.g.B * a.g.Hkv);
  const int rb = a.rowbytes;
  const int T = kTileBytes / rb;  // rows per tile: 32, 64 or 128
  char* base = static_cast<char*>(kv ? a.V.p[l] : a.K.p[l]) + (size_t)bh * a.g.ncap * rb;
  const int lst = a.list_seq ? (head / a.g.Hkv) % a.g.B : head;
  const int32_t* src = a.kept_idx + (size_t)lst * a.g.N;
  const int len = a.kept_len[lst];
  const int N = a.g.N;
  if (a.validate) {
    bool bad = len < 0 || len > N;
    if (!bad)
      for (int k = lane; k < len; k += 32) {
        const int v = src[k];
        bad |= v < k || v >= N || (k > 0 && v <= src[k - 1]);
      }
    if (__any_sync(kFull, bad)) {
      if (lane == 0 && kv == 0) status_or(a.status, KVC_STATUS_BAD_INDEX);
      return;
    }
  }
  // first index that moves: smallest k with src[k] != k (src[k] - k never decreases, so the
  // test is monotone). A 32-way search: each step the lanes probe 32 points of [lo, hi) at once
  // and a ballot narrows it 33-fold, so 2048 entries take 3 dependent loads instead of 11.
  int lo = 0, hi = len;  // first lies in [lo, hi]
  while (lo < hi) {
    const int span = hi - lo;
    const int pt = lo + (int)(((long long)span * (lane + 1)) / 33);  // < hi, non-decreasing in lane
    const bool moved = pt < hi && src[pt] != pt;
    const unsigned m = __ballot_sync(kFull, moved);
    if (m) {
      const int l = __ffs(m) - 1;  // first probe that moved: first <= its point
      const int prev = l ? lo + (int)(((long long)span * l) / 33) : lo - 1;
      hi = lo + (int)(((long long)span * (l + 1)) / 33);
      lo = prev + 1;
    } else {
      lo = lo + (int)(((long long)span * 32) / 33) + 1;  // every probe kept its place
    }
  }
  const int first = lo;
  if (first >= len) return;
  const int ntiles = (len - first + T - 1) / T;
  if (lane == 0) {
    for (int i = 0; i < kRing; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(sm_u32(&bar[i])));
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncwarp();

  // source indices of tile i: row r0 + lane of each 32-row block (-1 past the tile's rows)
  auto fetch_src = [&](int i, int (&v)[kSrcRegs]) {
    const int k0 = first + i * T;
    const int nrows = i < ntiles ? min(T, len - k0) : 0;
#pragma unroll
    for (int b = 0; b < kSrcRegs; ++b) {
      const int r = b * 32 + lane;
      v[b] = (r < nrows) ? src[k0 + r] : -1;
    }
  };
  auto issue_loads = [&](int i, const int (&v)[kSrcRegs]) {
    const int s = i % kRing;
    const int k0 = first + i * T;
    const int nrows = min(T, len - k0);
    uint8_t* dst = sm + s * kTileBytes;
    if (lane == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(sm_u32(&bar[s])),
                   "r"(nrows * rb)
                   : "memory");
    __syncwarp();
#pragma unroll
    for (int b = 0; b < kSrcRegs; ++b) {
      const int r0 = b * 32;
      if (r0 >= nrows) break;
      const int r = r0 + lane;
      const bool live = r < nrows;
      const int sk = v[b];
      const int prev = __shfl_up_sync(kFull, sk, 1);
      const bool start = live && (lane == 0 || prev + 1 != sk);
      const unsigned starts = __ballot_sync(kFull, start);
      if (start) {
        const unsigned later = (lane < 31) ? (starts >> (lane + 1)) : 0u;
        const int blk_end = min(r0 + 32, nrows);
        const int end = later ? (r + 1 + __ffs(later) - 1) : blk_end;
        const uint32_t bytes = (uint32_t)((end - r) * rb);
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                sm_u32(dst + r * rb)),
            "l"(base + (size_t)sk * rb), "r"(bytes), "r"(sm_u32(&bar[s]))
            : "memory");
      }
    }
  };

  // prologue: loads of the first kRing - 1 tiles, and the indices of the next one
  int nxt[kSrcRegs];
  const int pro = ntiles < kRing - 1 ? ntiles : kRing - 1;
  for (int i = 0; i < pro; ++i) {
    fetch_src(i, nxt);
    issue_loads(i, nxt);
  }
  fetch_src(kRing - 1, nxt);
  bool ok = true;
  for (int i = 0; i < ntiles && ok; ++i) {
    const int s = i % kRing;
    const int k0 = first + i * T;
    const int nrows = min(T, len - k0);
    if (lane == 0) {
      const uint32_t a0 = sm_u32(&bar[s]), par = (uint32_t)((i / kRing) & 1);
      bool done = false;
      for (uint32_t it = 0; it < (1u << 24) && !done; ++it) {
        uint32_t d;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(d)
                     : "r"(a0), "r"(par)
                     : "memory");
        done = d != 0;
      }
      if (!done) {
        status_or(a.status, KVC_STATUS_TIMEOUT);
        ok = false;
      } else {
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(base + (size_t)k0 * rb),
                     "r"(sm_u32(sm + s * kTileBytes)), "r"(nrows * rb)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
        // the stage reloaded next is the one stored in the previous step: its store must have read it
        asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory");
      }
    }
    ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
    if (ok && i + kRing - 1 < ntiles) {
      issue_loads(i + kRing - 1, nxt);
      fetch_src(i + kRing, nxt);
    }
  }
  if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
  __syncwarp();
}

}  // namespace kvc
