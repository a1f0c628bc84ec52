// score_split.cu -- bf16 scoring in two streaming passes with no waits between CTAs.
//
// What it computes is kvc_score's definition (BeaconKV write-up, "打分时的 RoPE 对齐": a key's
// importance is the max over the observation rows of its softmax weight over all cached keys).
// For long caches and 256-row observation tiles the single-read kernel (score_resident.cu) has to
// spread a head over many CTAs that meet every round (32 per head at 8k keys, 128 at 32k), and
// those meetings, not the memory system, set its pace. Here the keys of a head are cut into
// ranges of 1024 or 4096 keys and every (head, range) is an independent work item:
//   pass 1      per item: S = Q K^T on the tensor cores (all observation rows of the head, one or
//               two 128-row tiles against each 128-key chunk), each row's running (max, sum of
//               exp2) over the range; the row's log2-sum-exp2 over the range is stored
//   combine     per head and row: the ranges' partials merged into lse2
//   pass 2      per item: S again, and per key the max over rows of s*c2 - lse2, then exp2
// Keys cross HBM twice, but no CTA ever waits for another, so both passes run at streaming rate.
//
// Roles in a CTA (persistent, one per SM; items b, b + grid, b + 2 grid, ... for CTA b):
//   warp 0      TMA producer: the item's observation tile(s) and its key chunks into a ring
//   warp 1      tcgen05.mma issuer (one thread): per chunk one 128x128 MMA chain per row tile into
//               a TMEM slot of NT x 128 columns (4 / NT slots)
//   warps 2-9   epilogue, two warps per TMEM lane quarter (one 64-column half each)
// Every wait is bounded; a wait that gives up sets KVC_STATUS_TIMEOUT and a CTA-wide abort flag,
// after which every role skips its work but still passes every named barrier.
#include "score_tc.cuh"

namespace kvc {

constexpr int kSplitEpi = 8;
constexpr int kSplitThreads = 64 + 32 * kSplitEpi;
constexpr int kSplitRows = 128;  // rows of one MMA tile

__device__ __forceinline__ void split_epi_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kSplitEpi) : "memory"); }

// Max-reduce-scatter over lane bits 4, 3, 2 (as in the single-read kernel): on exit w[0] holds the
// max, over the 8 lanes that differ only in those bits, of slot (lane >> 2) & 7.
__device__ __forceinline__ void split_rs_max8(float (&w)[8], int lane) {
#pragma unroll
  for (int h = 4, bit = 16; h; h >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? w[i] : w[i + h];
      const float keep = up ? w[i + h] : w[i];
      w[i] = fmaxf(keep, __shfl_xor_sync(kFull, send, bit));
    }
  }
}

template <int D, int NT, int kPass>
__global__ void __launch_bounds__(kSplitThreads, 1)
    score_split_kernel(const __grid_constant__ FusedMaps maps, ScoreArgs a, ScoreWs ws, SplitPlan p, float c2) {
  constexpr int HALVES = D / 64;
  constexpr int kStage = kChunk * D * 2;
  constexpr int kQTile = kSplitRows * D * 2;
  constexpr int kQBuf = NT == 1 ? 2 : 1;
  constexpr int NSLOT = 4 / NT;
  constexpr uint32_t kSlotCols = NT * 128u;
  extern __shared__ uint8_t smraw[];
  uint8_t* Qs = align1024(smraw);
  uint8_t* Ks = Qs + kQBuf * NT * kQTile;
  const int S = p.stages;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(Ks + S * kStage);
  uint64_t* kempty = kfull + S;
  uint64_t* qfull = kempty + S;
  uint64_t* qempty = qfull + kQBuf;
  uint64_t* tfull = qempty + kQBuf;
  uint64_t* tempty = tfull + NSLOT;
  uint64_t* mdone = tempty + NSLOT;
  uint32_t* slot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  float2* merge = reinterpret_cast<float2*>(Ks + S * kStage + 512);  // pass 1: [2][NT * 128]
  float* pbest = reinterpret_cast<float*>(merge + 2 * NT * kSplitRows);  // pass 2: [2][4][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // As the wide kernel's exact fallback the items are listed by the previous kernel, usually none: a
  // CTA without a listed item leaves before it takes tensor memory or sets anything up.
  if (p.list) {
    griddep_wait();
    const int n = *reinterpret_cast<const volatile int32_t*>(p.list);
    if ((int)blockIdx.x >= n * fallback_sub(n, (int)gridDim.x, p.rk)) return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < kQBuf; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
    }
    for (int i = 0; i < NSLOT; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], kSplitEpi);
    }
    tc::mbar_init(mdone, 1);
    *abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  const int bhkv = a.g.B * a.g.Hkv;
  // Work items: all of them, or (pass 1 as the wide kernel's exact fallback) sub-ranges of the listed
  // ones, whose count and ids the previous kernel wrote: then every role waits for it first.
  int nitems = p.items, sub = 1;
  if (p.list) {
    griddep_wait();
    const int n = *reinterpret_cast<const volatile int32_t*>(p.list);
    sub = fallback_sub(n, (int)gridDim.x, p.rk);
    nitems = n * sub;
  }
  auto item_at = [&](int v) { return p.list ? p.list[1 + v / sub] : v; };
  // work unit v: its item and key chunks [cb, cb + nc) (the whole range unless the item is split)
  auto range_of = [&](int v, int item, int& cb, int& nc) {
    const int c0 = (item % p.R) * p.rk, c1 = min(c0 + p.rk, a.nchunk);
    const int cs = (p.rk + sub - 1) / sub;
    cb = min(c0 + (v % sub) * cs, c1);
    nc = min(cb + cs, c1) - cb;
  };

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t kc = 0;
      bool waited = false, stop = false;
      int it = 0;
      for (int idx = blockIdx.x; idx < nitems && !stop && !*abort_flag; idx += gridDim.x, ++it) {
        const int item = item_at(idx);
        const int head = item / p.R;
        const int l = head / bhkv, bh = head % bhkv;
        int cb, nc;
        range_of(idx, item, cb, nc);
        if (idx + (int)gridDim.x < nitems) tc::prefetch_tensormap(&maps.k[item_at(idx + gridDim.x) / p.R / bhkv]);
        auto load_k = [&](int j) -> bool {
          const int s = kc % S;
          if (kc >= (uint32_t)S && !wait_or_abort(&kempty[s], ((kc / S) - 1) & 1, abort_flag, a.status)) return false;
          tc::mbar_expect_tx(&kfull[s], (uint32_t)kStage);
          for (int h = 0; h < HALVES; ++h)
            tc::tma_load_3d(Ks + s * kStage + h * 16384, &maps.k[l], &kfull[s], h * 64, (cb + j) * kChunk, bh);
          ++kc;
          return true;
        };
        // Up to a ring's worth of the item's keys goes out before its observation tile: those loads
        // wait only for the previous item's MMAs, while the tile buffer may still be in use by them.
        // The keys are the caller's cache, so the first ones also go out before waiting for the
        // kernel that produced this launch's other inputs.
        int j0 = 0;
        for (; j0 < nc && j0 < S; ++j0)
          if (!load_k(j0)) {
            stop = true;
            break;
          }
        if (stop) break;
        if (!waited) {
          griddep_wait();
          waited = true;
        }
        const int qb = it % kQBuf, use = it / kQBuf;
        if (use >= 1 && !wait_or_abort(&qempty[qb], (use - 1) & 1, abort_flag, a.status)) break;
        tc::mbar_expect_tx(&qfull[qb], (uint32_t)(NT * kQTile));
        for (int t = 0; t < NT; ++t)
          for (int h = 0; h < HALVES; ++h)
            tc::tma_load_2d(Qs + (qb * NT + t) * kQTile + h * (kSplitRows * 128), &maps.q, &qfull[qb], h * 64,
                            head * a.M_pad + t * kSplitRows);
        for (int j = j0; j < nc; ++j)
          if (!load_k(j)) {
            stop = true;
            break;
          }
      }
      if (!waited) griddep_wait();
      // every issued load has landed before the CTA exits (immediate on the normal path)
      const uint32_t tail = kc < (uint32_t)S ? kc : (uint32_t)S;
      for (uint32_t k = kc - tail; k < kc; ++k)
        if (!tc::mbar_wait(&kfull[k % S], (k / S) & 1)) status_or(a.status, KVC_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t kc = 0, tcount = 0;
      const uint32_t id = tc::idesc_bf16(128, kChunk);
      bool ok = true, issued = false;
      int it = 0;
      for (int idx = blockIdx.x; idx < nitems && ok && !*abort_flag; idx += gridDim.x, ++it) {
        const int item = item_at(idx);
        int cb, nc;
        range_of(idx, item, cb, nc);
        const int qb = it % kQBuf;
        if (!wait_or_abort(&qfull[qb], (it / kQBuf) & 1, abort_flag, a.status)) break;
        tc::fence_after_sync();
        for (int j = 0; j < nc; ++j) {
          const int s = kc % S;
          const uint32_t sl = tcount % NSLOT;
          if (!spin_or_abort(&kfull[s], (kc / S) & 1, abort_flag, a.status) ||
              (tcount >= (uint32_t)NSLOT && !spin_or_abort(&tempty[sl], ((tcount / NSLOT) - 1) & 1, abort_flag, a.status))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t kaddr = tc::smem_u32(Ks + s * kStage);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint32_t qaddr = tc::smem_u32(Qs + (qb * NT + t) * kQTile);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              tc::umma_bf16(tmem + sl * kSlotCols + t * 128u,
                            tc::desc_k_sw128(qaddr + (ks >> 2) * (kSplitRows * 128) + (ks & 3) * 32),
                            tc::desc_k_sw128(kaddr + (ks >> 2) * 16384 + (ks & 3) * 32), id, ks > 0);
          }
          tc::umma_commit(&kempty[s]);
          tc::umma_commit(&tfull[sl]);
          issued = true;
          ++kc;
          ++tcount;
        }
        if (ok) tc::umma_commit(&qempty[qb]);
      }
      if (issued) {  // every MMA has completed before TMEM is released
        tc::umma_commit(mdone);
        if (!tc::mbar_wait(mdone, 0)) status_or(a.status, KVC_STATUS_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (2-9) ----------------
    griddep_wait();  // pass 2 reads lse2 from the combine kernel
    const int e = warp - 2;
    const int q = warp & 3;  // the TMEM lane quarter this warp may read
    const int hf = e >> 2;   // which 64 of a chunk's 128 columns
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int gt = e * 32 + lane;  // 0..255
    uint32_t tcount = 0;
    int it = 0;
    for (int idx = blockIdx.x; idx < nitems; idx += gridDim.x, ++it) {
      const int item = item_at(idx);
      const int head = item / p.R;
      int cb, nc;
      range_of(idx, item, cb, nc);
      if constexpr (kPass == 1) {
        float2 st[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) st[t] = make_float2(-INFINITY, 0.f);
        for (int j = 0; j < nc; ++j, ++tcount) {
          const uint32_t sl = tcount % NSLOT;
          const bool go = !*abort_flag && wait_or_abort(&tfull[sl], (tcount / NSLOT) & 1, abort_flag, a.status);
          if (__all_sync(kFull, go)) {
            tc::fence_after_sync();
            const int nvalid = min(kChunk, a.g.N - (cb + j) * kChunk);
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int h32 = 0; h32 < 2; ++h32) {
                uint32_t r0[32];
                const int cbase = hf * 64 + h32 * 32;
                tc::tmem_ld32_async(tmem + sl * kSlotCols + t * 128u + lane_off + (uint32_t)cbase, r0);
                tc::tmem_wait();
                tc::tmem_regs_ready(r0);
                float v0[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r0[i]);
                if (nvalid < kChunk)  // ragged last chunk only
#pragma unroll
                  for (int i = 0; i < 32; ++i)
                    if (cbase + i >= nvalid) v0[i] = -INFINITY;
                const float mraw = tree_max32_3(v0);  // c2 > 0: scale the max once
                if (mraw > -INFINITY) {
                  const float mn = fmaxf(st[t].x, mraw * c2);
                  const float2 c2v = make_float2(c2, c2), nmv = make_float2(-mn, -mn);
                  float2 sum2[8];
#pragma unroll
                  for (int i = 0; i < 16; ++i) {
                    const float2 x = __ffma2_rn(make_float2(v0[2 * i], v0[2 * i + 1]), c2v, nmv);
                    const float2 e2 = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    sum2[i & 7] = i < 8 ? e2 : __fadd2_rn(sum2[i & 7], e2);
                  }
#pragma unroll
                  for (int w = 4; w; w >>= 1)
#pragma unroll
                    for (int i = 0; i < w; ++i) sum2[i] = __fadd2_rn(sum2[i], sum2[i + w]);
                  st[t] = make_float2(mn, st[t].y * ex2_approx(st[t].x - mn) + (sum2[0].x + sum2[0].y));
                }
              }
          }
          // the slot is free once this warp's values are in registers
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
        }
        // the two warps of a lane quarter merge their column halves; the hf == 0 warp stores the
        // row's log2-sum-exp2 over the range (merge is double-buffered by item parity)
        float2* mg = merge + (it & 1) * (NT * kSplitRows);
        if (hf == 1)
#pragma unroll
          for (int t = 0; t < NT; ++t) mg[t * kSplitRows + row] = st[t];
        asm volatile("bar.sync %0, 64;\n" ::"r"(2 + q) : "memory");
        // the item's partial, or a later sub-range's in the exchange area (merged by the combine kernel)
        float* dst = (idx % sub == 0) ? ws.lse2p + (size_t)item * a.M_pad
                                      : reinterpret_cast<float*>(ws.part) + (size_t)idx * a.M_pad;
        if (hf == 0 && !*abort_flag)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float2 m = lse_merge(st[t], mg[t * kSplitRows + row]);
            dst[t * kSplitRows + row] = m.y > 0.f ? m.x + log2f(m.y) : -INFINITY;
          }
      } else {
        // lse2 of this thread's rows (q*32 + lane/4 + 8k of each tile) from the combine kernel;
        // rows without observations hold +inf, so their terms drop out of the max
        float2 nl[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float l2 = ws.lse2[(size_t)head * a.M_pad + t * kSplitRows + q * 32 + (lane >> 2) + 8 * k];
            nl[t][k] = make_float2(-l2, -l2);
          }
        const float2 c2v = make_float2(c2, c2);
        const int slot8 = (lane >> 2) & 7;
        const int col_in = 8 * (slot8 >> 1) + 2 * (lane & 3) + (slot8 & 1);
        for (int j = 0; j < nc; ++j, ++tcount) {
          const uint32_t sl = tcount % NSLOT;
          const bool go = !*abort_flag && wait_or_abort(&tfull[sl], (tcount / NSLOT) & 1, abort_flag, a.status);
          float best[2] = {-INFINITY, -INFINITY};
          if (__all_sync(kFull, go)) {
            tc::fence_after_sync();
            const uint32_t base = tmem + sl * kSlotCols + lane_off + (uint32_t)(hf * 64);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              // slot 2i + cc: column 8i + 2*(lane%4) + cc of the block, max over this thread's rows
              float w[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) w[i] = -INFINITY;
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                uint32_t ra[16], rb[16];  // rows (t/4, t/4+8) and (t/4+16, t/4+24) of 32 columns
                tc::tmem_ld16x256_x4_async(base + t * 128u + (uint32_t)(c * 32), ra);
                tc::tmem_ld16x256_x4_async(base + t * 128u + (16u << 16) + (uint32_t)(c * 32), rb);
                tc::tmem_wait();
                tc::tmem_regs_ready(ra);
                tc::tmem_regs_ready(rb);
                if (c == 1 && t == NT - 1) {  // the slot is free once its last values are in registers
                  tc::fence_before_sync();
                  __syncwarp();
                  if (lane == 0)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(ra[4 * i]), __uint_as_float(ra[4 * i + 1])), c2v,
                                               nl[t][0]);
                  const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(ra[4 * i + 2]), __uint_as_float(ra[4 * i + 3])),
                                               c2v, nl[t][1]);
                  const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(rb[4 * i]), __uint_as_float(rb[4 * i + 1])), c2v,
                                               nl[t][2]);
                  const float2 x3 = __ffma2_rn(make_float2(__uint_as_float(rb[4 * i + 2]), __uint_as_float(rb[4 * i + 3])),
                                               c2v, nl[t][3]);
                  w[2 * i] = fmaxf(w[2 * i], fmaxf(max3f(x0.x, x1.x, x2.x), x3.x));
                  w[2 * i + 1] = fmaxf(w[2 * i + 1], fmaxf(max3f(x0.y, x1.y, x2.y), x3.y));
                }
              }
              split_rs_max8(w, lane);
              best[c] = w[0];
            }
          } else {
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
          }
          // pbest[chunk parity][quarter][column]: the barrier of chunk n + 1 lies between two uses
          float* pb = pbest + (tcount & 1) * (4 * kChunk);
#pragma unroll
          for (int c = 0; c < 2; ++c) pb[q * kChunk + hf * 64 + c * 32 + col_in] = best[c];
          split_epi_bar();
          if (gt < kChunk && !*abort_flag) {
            const int key = (cb + j) * kChunk + gt;
            if (key < a.g.N) {
              const float m = fmaxf(fmaxf(pb[gt], pb[kChunk + gt]), fmaxf(pb[2 * kChunk + gt], pb[3 * kChunk + gt]));
              a.scores[(size_t)head * a.g.N + key] = exp2f(m);
            }
          }
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// per (head, row): the ranges' log2-sum-exp2 partials merged into lse2; rows without
// observations get +inf
__global__ void split_combine_kernel(ScoreArgs a, ScoreWs ws, SplitPlan p) {
  griddep_wait();
  const int head = blockIdx.x, r = threadIdx.x;
  if (r >= a.M_pad) return;
  const float* src = ws.lse2p + (size_t)head * p.R * a.M_pad + r;
  float m = -INFINITY, s = 0.f;
  auto add = [&](float v) {
    if (v == -INFINITY) return;
    if (v > m) {
      s = s * exp2f(m - v) + 1.f;
      m = v;
    } else {
      s += exp2f(v - m);
    }
  };
  for (int ri = 0; ri < p.R; ++ri) add(src[(size_t)ri * a.M_pad]);
  // the wide kernel's fallback: the later sub-ranges of this head's listed items (split only when
  // there are at most grid / 2 of them: their ids go to shared memory first, one read each)
  __shared__ int s_items[kMaxSMs / 2];
  if (p.list) {
    const int n = p.list[0];
    const int sub = fallback_sub(n, p.grid, p.rk);
    if (sub > 1) {
      if (r < n) s_items[r] = p.list[1 + r];
      __syncthreads();
    }
    if (sub > 1)
      for (int i = 0; i < n; ++i)
        if (s_items[i] / p.R == head) {
          // every sub-range's partial in flight at once, then merged
          const float* sp = reinterpret_cast<const float*>(ws.part) + (size_t)i * sub * a.M_pad + r;
          float v[kFallbackSub];
#pragma unroll
          for (int u = 1; u < kFallbackSub; ++u) v[u] = u < sub ? sp[(size_t)u * a.M_pad] : -INFINITY;
#pragma unroll
          for (int u = 1; u < kFallbackSub; ++u) add(v[u]);
        }
  }
  const bool ok = ws.valid[(size_t)head * a.M_pad + r] != 0 && s > 0.f;
  ws.lse2[(size_t)head * a.M_pad + r] = ok ? m + log2f(s) : INFINITY;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int split_tail_bytes(int NT) { return 1024 + 512 + 2 * NT * kSplitRows * 8 + 2 * 4 * kChunk * 4; }

// Chunks per range: 8 (1024 keys) for one row tile, 32 (4096 keys) for two (whose single tile
// buffer is reloaded between items with the tensor pipe idle), so that the item's
// observation tile(s) are loaded once per 256 KB or 1 MB of keys.
int split_ranges(int nchunk, int M_pad) {
  const int rk = M_pad > 128 ? 32 : 8;
  return (nchunk + rk - 1) / rk;
}

bool score_split_plan(const ScoreArgs& a, SplitPlan* p, size_t* smem) {
  if (a.dtype != KVC_BF16 || a.ext || (a.M_pad != 128 && a.M_pad != 256)) return false;
  int dev = 0, nsm = 0, smem_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  const int NT = a.M_pad / kSplitRows, D = a.g.D;
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  p->rk = NT == 1 ? 8 : 32;
  p->R = split_ranges(a.nchunk, a.M_pad);
  p->items = heads * p->R;
  p->grid = p->items < nsm ? p->items : nsm;
  const int qbytes = (NT == 1 ? 2 : 1) * NT * kSplitRows * D * 2;
  const int stage = kChunk * D * 2;
  int stages = (smem_optin - split_tail_bytes(NT) - qbytes) / stage;
  if (stages > 6) stages = 6;
  if (stages < 2) return false;
  p->stages = stages;
  p->list = nullptr;
  *smem = (size_t)split_tail_bytes(NT) + qbytes + (size_t)stages * stage;
  return true;
}

int launch_score_split(const ScoreArgs& a, const ScoreWs& ws, const SplitPlan& p, size_t smem, cudaStream_t s) {
  const int D = a.g.D, NT = a.M_pad / kSplitRows;
  FusedMaps maps;
  if (!fused_maps(&maps, a, ws)) return KVC_ERR_LAUNCH;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  using Kern = void (*)(const FusedMaps, ScoreArgs, ScoreWs, SplitPlan, float);
  // [D == 128][two row tiles][pass 2]
  static const Kern table[2][2][2] = {
      {{score_split_kernel<64, 1, 1>, score_split_kernel<64, 1, 2>}, {score_split_kernel<64, 2, 1>, score_split_kernel<64, 2, 2>}},
      {{score_split_kernel<128, 1, 1>, score_split_kernel<128, 1, 2>},
       {score_split_kernel<128, 2, 1>, score_split_kernel<128, 2, 2>}}};
  ScoreArgs aa = a;
  ScoreWs wss = ws;
  SplitPlan pp = p;
  float cc = c2;
  for (int pass = 1; pass <= 2; ++pass) {
    Kern kern = table[D == 128][NT == 2][pass - 1];
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    if (launch_pdl(kern, dim3(p.grid), dim3(kSplitThreads), smem, s, false, maps, aa, wss, pp, cc) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    if (pass == 1 && launch_pdl(split_combine_kernel, dim3(a.g.L * a.g.B * a.g.Hkv), dim3(a.M_pad), 0, s, false, aa,
                                wss, pp) != cudaSuccess)
      return KVC_ERR_LAUNCH;
  }
  return KVC_OK;
}

int launch_score_split_pass1_list(const ScoreArgs& a, const ScoreWs& ws, const int32_t* list, int rk, int R,
                                  int grid, cudaStream_t s) {
  SplitPlan p;
  size_t smem = 0;
  if (!score_split_plan(a, &p, &smem)) return KVC_ERR_LAUNCH;
  p.list = list;
  p.rk = rk;  // the listing kernel's ranges
  p.R = R;
  p.items = a.g.L * a.g.B * a.g.Hkv * R;
  p.grid = grid;  // the combine kernel splits the listed items by the same count
  // the wide kernel's footprint (three key stages), so that the SMs keep their shared-memory split
  // between the launches around this one
  const size_t per_stage = (size_t)kChunk * a.g.D * 2;
  if (p.stages > 3) {
    smem -= (size_t)(p.stages - 3) * per_stage;
    p.stages = 3;
  }
  const int D = a.g.D, NT = a.M_pad / kSplitRows;
  FusedMaps maps;
  if (!fused_maps(&maps, a, ws)) return KVC_ERR_LAUNCH;
  using Kern = void (*)(const FusedMaps, ScoreArgs, ScoreWs, SplitPlan, float);
  static const Kern table[2][2] = {{score_split_kernel<64, 1, 1>, score_split_kernel<64, 2, 1>},
                                   {score_split_kernel<128, 1, 1>, score_split_kernel<128, 2, 1>}};
  Kern kern = table[D == 128][NT == 2];
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  ScoreArgs aa = a;
  ScoreWs wss = ws;
  if (launch_pdl(kern, dim3(p.grid), dim3(kSplitThreads), smem, s, false, maps, aa, wss, p, c2) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
