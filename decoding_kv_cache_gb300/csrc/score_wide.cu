// score_wide.cu -- bf16 scoring for observation tiles of more than 128 rows, in two streaming passes
// with the keys on the tensor-memory lanes.
//
// What it computes is kvc_score's definition (BeaconKV write-up, "打分时的 RoPE 对齐": a key's
// importance is the max over the observation rows of its softmax weight over all cached keys).
// The tile of a GQA group with many query heads (224 rows at G = 7, 240 at G = 5 with 32 beacons)
// does not fit one 128-row MMA tile. Here each 128-key chunk is one MMA chain S^T = K Q^T with
// the keys as M (128 TMEM lanes) and every observation row as N (up to 256 TMEM columns): one
// chain of D/16 instructions per chunk, which the tensor pipe runs near its peak (two 128-row
// tiles as 128x128 chains took ~1.4x as long per chunk). As in score_split.cu, the keys of a head
// are cut into ranges and every (head, range) is an independent work item of both passes:
//   pass 1      per item: every epilogue thread owns one key lane and up to 128 rows (TMEM
//               columns). It keeps, per row, the sum of exp2(s c2 - ref) over its lane's keys of
//               the item, with one reference per thread: ref = the largest s c2 of its first key.
//               At the item's end the 128 lanes' sums are brought to their largest reference R,
//               reduce-scattered over the warp and summed over the four lane quarters in shared
//               memory: the row's log2-sum-exp2 over the range is R + log2(sum).
//               The sums are exact to fp32 rounding while the item's references (base 2) stay
//               within 96 of each other, no sum overflows and every valid row's sum stays above
//               2^-80 of the common reference; an item outside that is listed and recomputed with
//               a running max per row by the two-pass kernel's pass 1 (score_split.cu) over the
//               list (keys far out in a heavy tail reach it; the tests force it).
//   fallback    score_split_kernel's pass 1 over the listed items, each split into sub-ranges over
//               the launch's CTAs (usually none or a few: with none it exits at once)
//   combine     split_combine_kernel: per head and row, the ranges' partials (and the listed items'
//               sub-ranges) merged into lse2
//   pass 2      per item: the same MMA; per key the max over its rows of s c2 - lse2 (lse2 from
//               shared memory), the two column halves merged in shared memory, exp2 per key.
//
// Roles (persistent, one CTA per SM; items b, b + grid, ... for CTA b):
//   warp 0      TMA producer: the item's observation tile (one buffer) and its key chunks (a ring of
//               three 32 KB stages: a stage stays held until its MMA completes; a deeper ring
//               measured slower, and this footprint leaves shared memory for the L1 cache)
//   warp 1      tcgen05.mma issuer (one thread): per chunk one chain into one of two TMEM slots of
//               256 columns
//   warps 2-17  epilogue, two groups of eight: group g takes the chunks in TMEM slot g, so that one
//               group's TMEM loads are in flight while the other computes; in a group, warp w reads
//               lane quarter w % 4 (its 32 keys of each chunk) and one column half (128 rows); pass 1
//               reads with the 16x256b shape, so a thread holds 32 columns of 4 keys per chunk and
//               keeps 32 sums
// Every wait is bounded; a wait that gives up sets KVC_STATUS_TIMEOUT and a CTA-wide abort flag,
// after which every role skips its work but still passes every named barrier.
#include "score_tc.cuh"

namespace kvc {

constexpr int kWideEpi = 16;
constexpr int kWideThreads = 64 + 32 * kWideEpi;
constexpr int kWideSlotCols = 256;  // TMEM columns per chunk slot (two slots)
// An item whose references spread by more than this (base 2) is recomputed by the fallback.
constexpr float kWideSpread = 96.f;
// A valid row whose range sum falls below 2^-80 of the common reference likewise.
constexpr float kWideTiny = 8.271806125530277e-25f;  // 2^-80

__device__ __forceinline__ void wide_epi_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kWideEpi) : "memory"); }

// 16 consecutive 32-bit columns of this thread's TMEM lane, without waiting (see tmem_ld32_async).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// 16x256b loads (see tmem_ld16x256_x4_async) of 16 columns: thread t receives r[4i + j] = (lane
// t/4 + 8*(j/2), column 8i + 2*(t%4) + j%2) for i < 2.
__device__ __forceinline__ void tmem_ld16x256_x2_async(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}

// Pass 1 on the values of one 16x256b load (n column groups of 8): for each group i, the two keys'
// pairs of columns (8i + 2(t%4), +1): acc[i] += 2^(v * c2 - ref) for both keys.
template <int n>
__device__ __forceinline__ void wide_acc(float2* acc, const uint32_t* r, float2 c2v, float2 nA, float2 nB) {
#pragma unroll
  for (int i = 0; i < n; ++i) {
    const float2 xa = __ffma2_rn(make_float2(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1])), c2v, nA);
    const float2 xb = __ffma2_rn(make_float2(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3])), c2v, nB);
    const float2 ea = make_float2(ex2_approx(xa.x), ex2_approx(xa.y));
    const float2 eb = make_float2(ex2_approx(xb.x), ex2_approx(xb.y));
    acc[i] = __fadd2_rn(acc[i], __fadd2_rn(ea, eb));
  }
}
// max over the values of one 16x256b load of n column groups, only the keys flagged valid
template <int n>
__device__ __forceinline__ float wide_max(const uint32_t* r, bool okA, bool okB) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    const float a = fmaxf(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]));
    const float b = fmaxf(__uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    m = max3f(m, okA ? a : -INFINITY, okB ? b : -INFINITY);
  }
  return m;
}

template <int D, int kPass>
__global__ void __launch_bounds__(kWideThreads, 1)
    score_wide_kernel(const __grid_constant__ FusedMaps maps, ScoreArgs a, ScoreWs ws, WidePlan p, float c2) {
  constexpr int HALVES = D / 64;
  constexpr int kStage = kChunk * D * 2;
  extern __shared__ uint8_t smraw[];
  uint8_t* Qs = align1024(smraw);
  const int ncols = a.M_n;                // observation rows in the MMA (a multiple of 16, 144..256)
  const int qhalf = ncols * 128;          // one 64-column half of a tile: ncols rows of 128 bytes
  const int qbytes = HALVES * qhalf;
  uint8_t* Ks = Qs + qbytes;  // one tile buffer: a deeper key ring pays more than a second tile
  const int S = p.stages;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(Ks + S * kStage);
  uint64_t* kempty = kfull + S;
  uint64_t* qfull = kempty + S;
  uint64_t* qempty = qfull + 1;
  uint64_t* tfull = qempty + 1;   // [2]
  uint64_t* tempty = tfull + 2;   // [2]
  uint64_t* mdone = tempty + 2;
  uint32_t* slot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  volatile int* bad = reinterpret_cast<volatile int*>(slot + 2);     // [2] by item parity (pass 1)
  float* wref = reinterpret_cast<float*>(Ks + S * kStage + 256);      // pass 1: [2 half][2 group][4 quarter][2]
  float* part = wref + 32;                                            // pass 1: [2 half][4 quarter][128]
  float* nl2 = wref;                                                  // pass 2: [256] -lse2
  float* pbest = nl2 + 256;                                           // pass 2: [2 ring][2 group][4 quarter][2 half][32]
  unsigned* pcount = reinterpret_cast<unsigned*>(pbest + 1024);      // pass 2: [2 ring][2 group][4 quarter] arrivals

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
    }
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qempty, 1);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], kWideEpi / 2);  // the eight warps of the slot's group
    }
    tc::mbar_init(mdone, 1);
    *abort_flag = 0;
    bad[0] = bad[1] = 0;
    for (int i = 0; i < 16; ++i) pcount[i] = 0u;
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;
  const int bhkv = a.g.B * a.g.Hkv;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t kc = 0;
      bool waited = false, stop = false;
      int it = 0;
      for (int item = blockIdx.x; item < p.items && !stop && !*abort_flag; item += gridDim.x, ++it) {
        const int head = item / p.R, ri = item % p.R;
        const int l = head / bhkv, bh = head % bhkv;
        const int cb = ri * p.rk, nc = min(cb + p.rk, a.nchunk) - cb;
        if (item + (int)gridDim.x < p.items) tc::prefetch_tensormap(&maps.k[(item + gridDim.x) / p.R / bhkv]);
        auto load_k = [&](int j) -> bool {
          const int s = kc % S;
          if (kc >= (uint32_t)S && !wait_or_abort(&kempty[s], ((kc / S) - 1) & 1, abort_flag, a.status)) return false;
          tc::mbar_expect_tx(&kfull[s], (uint32_t)kStage);
          for (int h = 0; h < HALVES; ++h)
            tc::tma_load_3d(Ks + s * kStage + h * 16384, &maps.k[l], &kfull[s], h * 64, (cb + j) * kChunk, bh);
          ++kc;
          return true;
        };
        // the first keys go out before the tile (they wait only for ring slots); the keys are the
        // caller's cache, so they also go out before waiting for the kernel that made the tiles
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
        // the tile buffer is free once the previous item's last MMA has completed
        if (it >= 1 && !wait_or_abort(qempty, (it - 1) & 1, abort_flag, a.status)) break;
        tc::mbar_expect_tx(qfull, (uint32_t)qbytes);
        for (int h = 0; h < HALVES; ++h)
          tc::tma_load_2d(Qs + h * qhalf, &maps.q, qfull, h * 64, head * a.M_pad);
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
      const uint32_t id = tc::idesc_bf16(128, ncols);
      bool ok = true, issued = false;
      int it = 0;
      for (int item = blockIdx.x; item < p.items && ok && !*abort_flag; item += gridDim.x, ++it) {
        const int ri = item % p.R;
        const int cb = ri * p.rk, nc = min(cb + p.rk, a.nchunk) - cb;
        if (!wait_or_abort(qfull, it & 1, abort_flag, a.status)) break;
        tc::fence_after_sync();
        const uint32_t qaddr = tc::smem_u32(Qs);
        for (int j = 0; j < nc; ++j) {
          const int s = kc % S;
          const uint32_t sl = tcount & 1;
          if (!spin_or_abort(&kfull[s], (kc / S) & 1, abort_flag, a.status) ||
              (tcount >= 2 && !spin_or_abort(&tempty[sl], ((tcount >> 1) - 1) & 1, abort_flag, a.status))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t kaddr = tc::smem_u32(Ks + s * kStage);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc::umma_bf16(tmem + sl * kWideSlotCols, tc::desc_k_sw128(kaddr + (ks >> 2) * 16384 + (ks & 3) * 32),
                          tc::desc_k_sw128(qaddr + (ks >> 2) * qhalf + (ks & 3) * 32), id, ks > 0);
          tc::umma_commit(&kempty[s]);
          tc::umma_commit(&tfull[sl]);
          issued = true;
          ++kc;
          ++tcount;
        }
        if (ok) tc::umma_commit(qempty);
      }
      if (issued) {  // every MMA has completed before TMEM is released
        tc::umma_commit(mdone);
        if (!tc::mbar_wait(mdone, 0)) status_or(a.status, KVC_STATUS_TIMEOUT);
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (2-17): two groups of eight ----------------
    // Group g takes the chunks the MMA writes into TMEM slot g (every other chunk), so that one
    // group's TMEM loads are in flight while the other group computes. Within a group, warp w reads
    // lane quarter w % 4 (its 32 keys of a chunk) and column half hf (rows 128 hf .. 128 hf + 127).
    griddep_wait();  // pass 2 reads lse2 from the combine kernel
    const int e = warp - 2;
    const int grp = e >> 3;
    const int q = warp & 3;
    const int hf = (e & 7) >> 2;
    const int col0 = hf * 128;
    const int ncol = max(0, min(128, ncols - col0));  // a multiple of 16 (ncols > 128: both halves hold rows)
    const int n32 = ncol >> 5;                        // pass 1: whole 32-column loads, and a 16-column tail
    const bool tail16 = (ncol & 16) != 0;
    const int ng = ncol >> 4;                         // pass 2: 16-column loads
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int gt = e * 32 + lane;  // 0..511
    const float2 c2v = make_float2(c2, c2);
    uint32_t tcount = 0;  // chunks of this CTA so far; chunk n is in TMEM slot n & 1
    int it = 0;
    for (int item = blockIdx.x; item < p.items; item += gridDim.x, ++it) {
      const int head = item / p.R, ri = item % p.R;
      const int cb = ri * p.rk, nc = min(cb + p.rk, a.nchunk) - cb;
      const int par = it & 1;
      if constexpr (kPass == 1) {
        // acc[4k + i]: this thread's columns col0 + 32k + 8i + 2(t%4) + {0, 1} (x, y), summed over its keys
        float2 acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = make_float2(0.f, 0.f);
        float ref = -INFINITY;
        bool first = true;
        for (int j = 0; j < nc; ++j, ++tcount) {
          if ((int)(tcount & 1) != grp) continue;  // the other group's chunk
          const uint32_t sl = tcount & 1;
          const bool go = !*abort_flag && wait_or_abort(&tfull[sl], (tcount >> 1) & 1, abort_flag, a.status);
          if (__all_sync(kFull, go)) {
            tc::fence_after_sync();
            const int kbase = (cb + j) * kChunk + q * 32 + (lane >> 2);  // this thread's first key
            // two 16-lane blocks (keys kbase + 16 blk and kbase + 16 blk + 8), two batches of two
            // 32-column loads each, one wait per batch
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
              const uint32_t base = tmem + sl * kWideSlotCols + lane_off + ((uint32_t)(16 * blk) << 16) + (uint32_t)col0;
              const bool okA = kbase + 16 * blk < a.g.N, okB = kbase + 16 * blk + 8 < a.g.N;
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                uint32_t r[2][16];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int k = 2 * kk + u;
                  if (k < n32)
                    tc::tmem_ld16x256_x4_async(base + (uint32_t)(32 * k), r[u]);
                  else if (k == n32 && tail16)
                    tmem_ld16x256_x2_async(base + (uint32_t)(32 * k), *reinterpret_cast<uint32_t(*)[8]>(r[u]));
                }
                if (2 * kk < n32 + (tail16 ? 1 : 0)) {
                  tc::tmem_wait();
                  tc::tmem_regs_ready(r[0]);
                  tc::tmem_regs_ready(r[1]);
                }
                if (blk == 1 && kk == 1) {  // the slot is free once its last values are in registers
                  tc::fence_before_sync();
                  __syncwarp();
                  if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
                }
                if (first && blk == 0 && kk == 0) {
                  // this thread's reference: the largest logit of the first 64 columns of its first keys
                  // (a thread whose first block lies past N has no key in the item: it stays -inf)
                  float m = -INFINITY;
#pragma unroll
                  for (int u = 0; u < 2; ++u) {
                    if (u < n32) m = fmaxf(m, wide_max<4>(r[u], okA, okB));
                    else if (u == n32 && tail16) m = fmaxf(m, wide_max<2>(r[u], okA, okB));
                  }
                  ref = m > -INFINITY ? m * c2 : -INFINITY;
                }
                // a key past N gets the offset -inf: its exp2 is exactly 0
                const float2 nA = okA ? make_float2(-ref, -ref) : make_float2(-INFINITY, -INFINITY);
                const float2 nB = okB ? make_float2(-ref, -ref) : make_float2(-INFINITY, -INFINITY);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                  const int k = 2 * kk + u;
                  if (k < n32) wide_acc<4>(acc + 4 * k, r[u], c2v, nA, nB);
                  else if (k == n32 && tail16) wide_acc<2>(acc + 4 * k, r[u], c2v, nA, nB);
                }
              }
            }
            first = false;
          } else {
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
          }
        }
        // ---- the item's end: one reference per column half (both groups), sums over the item's keys ----
        float* wh = wref + hf * 16;  // [2 half][2 group][4 quarter][2] (max, min)
        {
          float mx = ref, mn = ref > -INFINITY ? ref : INFINITY;
#pragma unroll
          for (int o = 16; o; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
            mn = fminf(mn, __shfl_xor_sync(kFull, mn, o));
          }
          if (lane == 0) {
            wh[(grp * 4 + q) * 2] = mx;
            wh[(grp * 4 + q) * 2 + 1] = mn;
          }
        }
        wide_epi_bar();
        // the next item's flag: every reader of its previous use (two items ago) has passed this barrier,
        // and its next writers come after the next item's first barrier
        if (gt == 0) bad[par ^ 1] = 0;
        float R = -INFINITY, Rmin = INFINITY;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          R = fmaxf(R, wh[2 * u]);
          Rmin = fminf(Rmin, wh[2 * u + 1]);
        }
        const float scale = ref > -INFINITY ? ex2_approx(ref - R) : 0.f;
        bool overflow = false;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc[i] = __fmul2_rn(acc[i], make_float2(scale, scale));
          overflow |= !(fabsf(acc[i].x) < INFINITY) || !(fabsf(acc[i].y) < INFINITY);
        }
        if (ncol > 0 && (__any_sync(kFull, overflow) || (R - Rmin > kWideSpread))) {
          if (lane == 0) bad[par] = 1;
        }
        // reduce-scatter over the 8 lanes that hold the same columns (lane bits 4, 3, 2): lane l ends
        // with acc index a = 8 b4 + 4 b3 + 2 b2 + {0, 1}, i.e. k = a / 4, i = a % 4
#pragma unroll
        for (int h = 8, bit = 16; h >= 2; h >>= 1, bit >>= 1) {
          const bool up = (lane & bit) != 0;
#pragma unroll
          for (int i = 0; i < h; ++i) {
            const float2 send = up ? acc[i] : acc[i + h];
            const float2 keep = up ? acc[i + h] : acc[i];
            acc[i] = make_float2(keep.x + __shfl_xor_sync(kFull, send.x, bit), keep.y + __shfl_xor_sync(kFull, send.y, bit));
          }
        }
        // part[half][quarter][column]: group 1 stores its sums, then group 0 adds its own
        {
          float* pt = part + (hf * 4 + q) * 128;
          int cc[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int a_ = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + u;
            cc[u] = 32 * (a_ >> 2) + 8 * (a_ & 3) + 2 * (lane & 3);
          }
          if (grp == 1)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              pt[cc[u]] = acc[u].x;
              pt[cc[u] + 1] = acc[u].y;
            }
          wide_epi_bar();
          if (grp == 0)
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              pt[cc[u]] += acc[u].x;
              pt[cc[u] + 1] += acc[u].y;
            }
        }
        wide_epi_bar();
        // thread gt < 256: row gt's range sum over the four lane quarters
        float tot = 0.f, R2 = -INFINITY;
        if (gt < 256) {
          const int h2 = gt >> 7, c = gt & 127;
          const float* pp = part + h2 * 512 + c;
          tot = (pp[0] + pp[128]) + (pp[256] + pp[384]);
          const float* w2 = wref + h2 * 16;
#pragma unroll
          for (int u = 0; u < 8; ++u) R2 = fmaxf(R2, w2[2 * u]);
          const bool row_valid = gt < a.M && ws.valid[(size_t)head * a.M_pad + gt] != 0;
          if (row_valid && !(tot >= kWideTiny)) bad[par] = 1;
        }
        // every flag write is ordered before the readers, and every read of part and wref before the
        // next item's writes, by these two barriers
        wide_epi_bar();
        if (gt < 256 && !*abort_flag) {
          if (bad[par]) {
            if (gt == 0) {
              const int slot_i = atomicAdd(ws.fb, 1);
              ws.fb[1 + slot_i] = item;
            }
          } else {
            ws.lse2p[(size_t)item * a.M_pad + gt] = tot > 0.f ? R2 + log2f(tot) : -INFINITY;
          }
        }
        wide_epi_bar();
      } else {
        // -lse2 of the head's rows for this item (rows without observations: -inf); the barrier orders it
        // before every group's first read
        float* nl = nl2;
        if (gt < 256) nl[gt] = -(gt < ncols ? ws.lse2[(size_t)head * a.M_pad + gt] : INFINITY);
        wide_epi_bar();
        const float4* nl4 = reinterpret_cast<const float4*>(nl + col0);
        for (int j = 0; j < nc; ++j, ++tcount) {
          if ((int)(tcount & 1) != grp) continue;  // the other group's chunk
          const uint32_t sl = tcount & 1;
          const bool go = !*abort_flag && wait_or_abort(&tfull[sl], (tcount >> 1) & 1, abort_flag, a.status);
          float m = -INFINITY;
          if (__all_sync(kFull, go)) {
            tc::fence_after_sync();
            const uint32_t base = tmem + sl * kWideSlotCols + lane_off + (uint32_t)col0;
            // two batches of four 16-column loads, one wait each
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              uint32_t r[4][16];
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (4 * bb + u < ng) tmem_ld16_async(base + (uint32_t)(16 * (4 * bb + u)), r[u]);
              if (4 * bb < ng) {
                tc::tmem_wait();
#pragma unroll
                for (int u = 0; u < 4; ++u) tc::tmem_regs_ready(r[u]);
              }
              if (bb == 1) {
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
              }
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (4 * bb + u < ng) {
                  const int g = 4 * bb + u;
#pragma unroll
                  for (int i = 0; i < 4; ++i) {
                    const float4 o = nl4[g * 4 + i];
                    const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(r[u][4 * i]), __uint_as_float(r[u][4 * i + 1])),
                                                 c2v, make_float2(o.x, o.y));
                    const float2 x1 = __ffma2_rn(make_float2(__uint_as_float(r[u][4 * i + 2]), __uint_as_float(r[u][4 * i + 3])),
                                                 c2v, make_float2(o.z, o.w));
                    m = fmaxf(m, fmaxf(max3f(x0.x, x0.y, x1.x), x1.y));
                  }
                }
            }
          } else {
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[sl])) : "memory");
          }
          // The two warps of a lane quarter in a group (one per column half) hold the same 32 keys:
          // each leaves its maxima in pbest[ring][group][quarter][half][key] and counts itself in; the
          // second to arrive takes the max and stores the scores. No warp waits for another. A ring of
          // two per group is enough: a warp of group g reaches its chunk n + 4 only after its group has
          // released the TMEM slot of chunk n + 2, which the second warp of chunk n does after its combine.
          const int rs = ((int)((tcount >> 1) & 1) * 2 + grp) * 4 + q;
          float* pb = pbest + rs * 64;
          pb[hf * 32 + lane] = m;
          __threadfence_block();
          __syncwarp();
          unsigned last = 0;
          if (lane == 0) last = atomicAdd(&pcount[rs], 1u) == 1u;
          if (__shfl_sync(kFull, last, 0)) {
            __threadfence_block();
            const float v = fmaxf(pb[lane], pb[32 + lane]);
            const int key = (cb + j) * kChunk + q * 32 + lane;
            if (key < a.g.N && !*abort_flag) a.scores[(size_t)head * a.g.N + key] = exp2f(v);
            __syncwarp();
            if (lane == 0) pcount[rs] = 0u;
          }
        }
        wide_epi_bar();  // every read of nl is done before the next item writes it
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// alignment slack, barriers and flags, then pass 1's wref and part (32 + 1024 floats) or, in the same
// place, pass 2's nl2, pbest and pcount (256 + 1024 + 16 words)
static int wide_tail_bytes() { return 1024 + 256 + (256 + 1024 + 16) * 4 + 64; }

bool score_wide_plan(const ScoreArgs& a, WidePlan* p, size_t* smem) {
  if (a.dtype != KVC_BF16 || a.ext || a.M_pad != 256 || a.M_n <= 128) return false;
  int dev = 0, nsm = 0, smem_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  const int D = a.g.D;
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  // ranges of 32 key chunks (the two-pass kernel's for 256-row tiles, split_ranges), or of 64 for heads
  // of 8192 keys and more: half the items' ends (a few us each, when the epilogue's reductions and
  // barriers leave the tensor pipe idle) while every SM still gets several items
  p->rk = a.nchunk >= 64 ? 64 : 32;
  p->R = (a.nchunk + p->rk - 1) / p->rk;
  p->items = heads * p->R;
  p->grid = p->items < nsm ? p->items : nsm;
  const int qbytes = a.M_n * D * 2;
  const int stage = kChunk * D * 2;
  int stages = (smem_optin - wide_tail_bytes() - qbytes) / stage;
  if (stages > 3) stages = 3;  // three chunks in flight per SM keep HBM busy; a deeper ring measured no faster
  if (stages < 2) return false;
  p->stages = stages;
  *smem = (size_t)wide_tail_bytes() + qbytes + (size_t)stages * stage;
  return true;
}

int launch_score_wide(const ScoreArgs& a, const ScoreWs& ws, const WidePlan& p, size_t smem, cudaStream_t s) {
  const int D = a.g.D;
  FusedMaps maps;  // the observation map's box covers the tile's ncols rows: one load per 64-column half
  if (!fused_maps(&maps, a, ws, a.M_n)) return KVC_ERR_LAUNCH;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  using Kern = void (*)(const FusedMaps, ScoreArgs, ScoreWs, WidePlan, float);
  static const Kern table[2][2] = {{score_wide_kernel<64, 1>, score_wide_kernel<64, 2>},
                                   {score_wide_kernel<128, 1>, score_wide_kernel<128, 2>}};
  ScoreArgs aa = a;
  ScoreWs wss = ws;
  WidePlan pp = p;
  float cc = c2;
  for (int pass = 1; pass <= 2; ++pass) {
    Kern kern = table[D == 128][pass - 1];
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    if (launch_pdl(kern, dim3(p.grid), dim3(kWideThreads), smem, s, false, maps, aa, wss, pp, cc) != cudaSuccess)
      return KVC_ERR_LAUNCH;
    if (pass == 1) {
      // the listed items again, with a running max per row (the two-pass kernel's pass 1)
      if (launch_score_split_pass1_list(a, ws, ws.fb, p.rk, p.R, p.grid, s) != KVC_OK) return KVC_ERR_LAUNCH;
      const SplitPlan sp{p.rk, p.R, p.items, p.grid, p.stages, ws.fb};
      if (launch_pdl(split_combine_kernel, dim3(a.g.L * a.g.B * a.g.Hkv), dim3(a.M_pad), 0, s, false, aa, wss, sp) !=
          cudaSuccess)
        return KVC_ERR_LAUNCH;
    }
  }
  return KVC_OK;
}

}  // namespace kvc
