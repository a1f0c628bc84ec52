// score_resident.cu -- bf16 scoring that reads every key once: pass-1 logits stay in tensor memory.
//
// What it computes is kvc_score's definition (BeaconKV write-up, "打分时的 RoPE 对齐": a key's
// importance is the max over the observation rows of its softmax weight over all cached keys).
// The softmax needs each row's log-sum-exp over ALL keys of the head before any score exists.
// The two-pass kernel (score_fused.cu) loads every key twice for that; here the logits
// S = Q K^T of pass 1 are kept in TMEM until the head's log-sum-exp is known, and pass 2
// reads them back from TMEM. K crosses the memory system once.
//
// Capacity sets the shape. With an observation tile of 128 rows (one MMA tile: lane = row), a
// 128-key chunk of logits is 128 TMEM columns, so an SM holds four chunks. Each CTA takes two
// chunks of a head per round and double-buffers rounds: round r+1's MMAs and pass 1 run while
// the group exchanges round r's partials. A head of N keys is spread over ceil(N / 256) CTAs
// (a "group"); the grid is #groups x group size CTAs, at most one per SM, launched cooperatively
// because group partners wait on one another.
//
// Roles (all derive the same chunk sequence from blockIdx; no queue):
//   warp 0      TMA producer of key chunks: each round's chunks into a ring of K stages.
//   warp 1      tcgen05.mma issuer (one thread): S = Q K^T per chunk into TMEM accumulator
//               (round & 1) * 2 + j.
//   warp 18     TMA producer of observation tiles: each round's tile into one of two Q buffers
//               (a separate warp, so key loads never wait behind a tile buffer).
//   warps 2-9   pass 1, two warps per TMEM lane quarter (one column half each): each thread owns
//               one row and folds its columns into the row's running (max, sum of exp2); the
//               quarter's two warps merge and publish the row's partial. Two warps per SM
//               sub-partition keep the MUFU (exp2) pipe busy while one waits on it.
//   warps 10-17 pass 2, laid out the same way and running concurrently with pass 1 of the next
//               round. First the exchange: the 256 threads poll the group's partials of the
//               round (sixteen words each in flight at once) and merge them into lse2. Then a
//               chunk's TMEM values are read in the 16x256b fragment shape (each thread: 4 of
//               the warp's 32 rows x 2 columns per 8-column group) and its accumulator freed;
//               s*c2 - lse2 and the max over the 4 rows in registers, then a 3-step
//               reduce-scatter over the 8 lanes sharing a column pair leaves each lane one
//               column's max over 32 rows (7 shuffles per 32 columns); the eight warps' maxima
//               meet in shared memory and one thread per key writes exp2 of the max.
// Exchange protocol: a partial is one 64-bit word, the row's log2-sum-exp2 over the CTA's keys
// in the low half and round + 1 in the high half, written with one relaxed store; a reader
// accepts a word once its tag matches, so data and "published" travel together and nobody
// waits for a store to be acknowledged. The observation kernel that runs just before zeroes them.
// Launched with programmatic stream serialisation: the key producer and the MMA thread may start
// before the observation kernel has finished; every role that reads its output waits for it.
// Every wait is bounded; a wait that gives up sets KVC_STATUS_TIMEOUT and a CTA-wide abort flag,
// after which every role skips its work but still passes every named barrier. Before exiting,
// the producer waits (bounded) for its own loads in flight and the MMA thread for its MMAs.
#include "score_tc.cuh"

namespace kvc {

constexpr int kResChunks = 2;    // key chunks per CTA per round
constexpr int kResRows = 128;    // observation rows per head this kernel handles (one MMA tile)
constexpr int kResAcc = 2 * kResChunks;
constexpr unsigned long long kExchangeTimeoutNs = 50ull * 1000 * 1000;  // a partner's word: ~1 us normally
// Partner words each exchange thread keeps in flight (the kernel's kXB): a head spread over g CTAs
// needs g/2 words per thread, so with 32 or 128 CTAs per head (8k or 32k keys) narrow batches
// serialise round trips, while with 8 (2k keys) a wide batch only costs registers.
constexpr int kXchNarrow = 4, kXchWide = 16;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;\n" : "=l"(t));
  return t;
}
constexpr int kP1Warps = 8;  // warps 2-9: pass 1, two per TMEM lane quarter (one column half each)
constexpr int kP2Warps = 8;  // warps 10-17: pass 2, likewise
constexpr int kQWarp = 2 + kP1Warps + kP2Warps;              // warp 18: observation-tile producer
constexpr int kResThreads = 32 * (kQWarp + 1);
// Observation-tile buffers: two, so that the tile of round r + 1 is in place before round r's
// MMAs have completed (one buffer put the tile's load latency on the MMA's path).
constexpr int kQBuf = 2;

// named barrier among the pass-2 warps only
__device__ __forceinline__ void p2_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kP2Warps) : "memory"); }

__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;\n" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];\n" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Max-reduce-scatter over lane bits 4, 3, 2: on entry w[k] is this lane's value for slot k; on
// exit w[0] holds the max, over the 8 lanes that differ only in those bits, of slot (lane >> 2) & 7.
__device__ __forceinline__ void reduce_scatter_max8(float (&w)[8], int lane) {
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

// Reduce-scatter like reduce_scatter_max8, with a sum (kSum) or a max.
template <bool kSum>
__device__ __forceinline__ void reduce_scatter8(float (&w)[8], int lane) {
#pragma unroll
  for (int h = 4, bit = 16; h; h >>= 1, bit >>= 1) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? w[i] : w[i + h];
      const float keep = up ? w[i + h] : w[i];
      const float other = __shfl_xor_sync(kFull, send, bit);
      w[i] = kSum ? keep + other : fmaxf(keep, other);
    }
  }
}

// kExt: the extended epilogue (the aggregation variants); otherwise max/max. kEnt: the rows'
// attention entropy is accumulated too (pass 1 keeps each row's mean logit; pass 2 merges).
template <int D, bool kExt, bool kEnt, int kXchBatch>
__global__ void __launch_bounds__(kResThreads, 1)
    score_resident_kernel(const __grid_constant__ FusedMaps maps, ScoreArgs a, ScoreWs ws, FusedPlan p, FusedXch xch,
                          float c2) {
  constexpr int HALVES = D / 64;
  constexpr int kStage = kChunk * D * 2;
  constexpr int kQBytes = kResRows * D * 2;
  extern __shared__ uint8_t smraw[];
  uint8_t* Qs = align1024(smraw);
  uint8_t* Ks = Qs + kQBuf * kQBytes;
  const int S = p.stages;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(Ks + S * kStage);
  uint64_t* kempty = kfull + S;
  uint64_t* qfull = kempty + S;
  uint64_t* qempty = qfull + kQBuf;
  uint64_t* tfull = qempty + kQBuf;
  uint64_t* tempty = tfull + kResAcc;
  uint64_t* mdone = tempty + kResAcc;
  uint32_t* slot = reinterpret_cast<uint32_t*>(mdone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  float* lse2s = reinterpret_cast<float*>(Ks + S * kStage + 512);  // [2][128]
  float2* merge = reinterpret_cast<float2*>(lse2s + 2 * kResRows);  // [2][128]
  float* mtau = reinterpret_cast<float*>(merge + 2 * kResRows);     // [2][128] (kEnt)
  float* pbest = mtau + 2 * kResRows;                                // [2][2 chunks][4 quarters, or 8 halves][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < kResAcc; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], kP2Warps);
    }
    for (int i = 0; i < kQBuf; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
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

  // A unit is one 128-row observation tile of a head (a.tiles of them per head: the rows of a
  // head are independent in the softmax, so its tiles are scored apart and their per-key
  // values combined with atomics into the zeroed scores).
  const int units = a.g.L * a.g.B * a.g.Hkv * a.tiles;
  const int group = blockIdx.x / p.group_size, rank = blockIdx.x % p.group_size;
  const int rounds = group < units ? (units - group + p.ngroups - 1) / p.ngroups : 0;
  const int c0 = rank * p.chunks_per_cta;
  const int n = max(0, min(c0 + p.chunks_per_cta, a.nchunk) - c0);  // chunks per round, the same every round

  if (warp == 0) {
    // ---------------- TMA producer: key chunks ----------------
    if (lane == 0) {
      uint32_t kc = 0;
      const int bhkv = a.g.B * a.g.Hkv;
      // a round usually moves to another layer's tensor map: fetch the next rounds' maps early
      for (int r = 0; r < 2 && r < rounds; ++r) tc::prefetch_tensormap(&maps.k[(group + r * p.ngroups) / a.tiles / bhkv]);
      for (int r = 0; r < rounds && !*abort_flag; ++r) {
        const int head = (group + r * p.ngroups) / a.tiles;
        const int l = head / bhkv, bh = head % bhkv;
        if (r + 2 < rounds) tc::prefetch_tensormap(&maps.k[(group + (r + 2) * p.ngroups) / a.tiles / bhkv]);
        bool stop = false;
        for (int j = 0; j < n; ++j) {
          const int s = kc % S;
          if (kc >= (uint32_t)S && !wait_or_abort(&kempty[s], ((kc / S) - 1) & 1, abort_flag, a.status)) {
            stop = true;
            break;
          }
          tc::mbar_expect_tx(&kfull[s], (uint32_t)kStage);
          for (int h = 0; h < HALVES; ++h)
            tc::tma_load_3d(Ks + s * kStage + h * 16384, &maps.k[l], &kfull[s], h * 64, (c0 + j) * kChunk, bh);
          ++kc;
        }
        if (stop) break;
      }
      // Drain: every issued load has landed before the CTA exits (immediate on the normal path).
      const uint32_t tail = kc < (uint32_t)S ? kc : (uint32_t)S;
      for (uint32_t k = kc - tail; k < kc; ++k)
        if (!tc::mbar_wait(&kfull[k % S], (k / S) & 1)) status_or(a.status, KVC_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t kc = 0;
      const uint32_t id = tc::idesc_bf16(128, kChunk);
      bool ok = true, issued = false;
      for (int r = 0; r < rounds && ok && !*abort_flag; ++r) {
        const int qb = r % kQBuf;
        if (!wait_or_abort(&qfull[qb], (r / kQBuf) & 1, abort_flag, a.status)) break;
        tc::fence_after_sync();
        const uint32_t qaddr = tc::smem_u32(Qs + qb * kQBytes);
        for (int j = 0; j < n; ++j) {
          const int s = kc % S;
          const uint32_t acc = (uint32_t)((r & 1) * kResChunks + j);
          if (!spin_or_abort(&kfull[s], (kc / S) & 1, abort_flag, a.status) ||
              (r >= 2 && !spin_or_abort(&tempty[acc], ((r >> 1) - 1) & 1, abort_flag, a.status))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t kaddr = tc::smem_u32(Ks + s * kStage);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            tc::umma_bf16(tmem + acc * kChunk,
                          tc::desc_k_sw128(qaddr + (ks >> 2) * (kResRows * 128) + (ks & 3) * 32),
                          tc::desc_k_sw128(kaddr + (ks >> 2) * 16384 + (ks & 3) * 32), id, ks > 0);
          tc::umma_commit(&kempty[s]);
          tc::umma_commit(&tfull[acc]);
          issued = true;
          ++kc;
        }
        if (ok) tc::umma_commit(&qempty[qb]);
      }
      // every MMA has completed before TMEM is released
      if (issued) {
        tc::umma_commit(mdone);
        if (!tc::mbar_wait(mdone, 0)) status_or(a.status, KVC_STATUS_TIMEOUT);
      }
    }
    __syncwarp();
  } else if (warp == kQWarp) {
    // ---------------- TMA producer: observation tiles ----------------
    if (lane == 0) {
      griddep_wait();  // the tiles come from the observation kernel
      int qloads = 0;
      for (int r = 0; r < rounds && !*abort_flag; ++r) {
        const int unit = group + r * p.ngroups;
        const int qb = r % kQBuf, use = r / kQBuf;
        if (use >= 1 && !wait_or_abort(&qempty[qb], (use - 1) & 1, abort_flag, a.status)) break;
        tc::mbar_expect_tx(&qfull[qb], (uint32_t)kQBytes);
        for (int h = 0; h < HALVES; ++h)
          tc::tma_load_2d(Qs + qb * kQBytes + h * (kResRows * 128), &maps.q, &qfull[qb], h * 64, unit * kResRows);
        qloads = r + 1;
      }
      for (int r = qloads - kQBuf < 0 ? 0 : qloads - kQBuf; r < qloads; ++r)
        if (!tc::mbar_wait(&qfull[r % kQBuf], (r / kQBuf) & 1)) status_or(a.status, KVC_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------- pass-1 warps (2-9) and pass-2 warps (10-17) ----------------
    // the exchange words and row flags come from the observation kernel (the key producer and
    // the MMA thread start without waiting: the keys are the caller's cache)
    griddep_wait();
    const bool is_p1 = warp < 2 + kP1Warps;
    const int e = is_p1 ? warp - 2 : warp - 2 - kP1Warps;  // 0..7 within the group
    const int q = warp & 3;  // TMEM lane quarter this warp may read: rows q*32 .. q*32+31
    const int hf = e >> 2;   // which 64 of a chunk's 128 columns
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint64_t* words = reinterpret_cast<uint64_t*>(xch.part);
    // with kEnt a second set of words (the rows' mean logits) follows the first
    const size_t words_per_set = (size_t)4 * p.ngroups * p.group_size * kResRows;
    // after the pass-2 reduce-scatter a lane holds slot (lane >> 2) & 7 of each 32-column block
    const int slot8 = (lane >> 2) & 7;
    const int col_in = 8 * (slot8 >> 1) + 2 * (lane & 3) + (slot8 & 1);

    // pass 1 of a round: fold this thread's row over its column half of every chunk into the
    // running (max, sum of exp2); the accumulators stay allocated for pass 2. With kEnt also
    // tau = sum of exp2(x - max) * (x - max), x = s*c2, which gives the row's mean logit under
    // this CTA's softmax (for the entropy) without a second exponential.
    auto pass1 = [&](int round) {
      float2 st = make_float2(-INFINITY, 0.f);
      float tau = 0.f;
      for (int j = 0; j < n; ++j) {
        const uint32_t acc = (uint32_t)((round & 1) * kResChunks + j);
        const int c = c0 + j;
        const bool go = !*abort_flag && wait_or_abort(&tfull[acc], (round >> 1) & 1, abort_flag, a.status);
        if (!__all_sync(kFull, go)) continue;  // tcgen05.ld is warp-collective: decide per warp
        tc::fence_after_sync();
        const int nvalid = min(kChunk, a.g.N - c * kChunk);
#pragma unroll
        for (int h32 = 0; h32 < 2; ++h32) {  // 32 columns at a time
          uint32_t r0[32];
          const int cbase = hf * 64 + h32 * 32;
          tc::tmem_ld32_async(tmem + acc * kChunk + lane_off + (uint32_t)cbase, r0);
          tc::tmem_wait();
          tc::tmem_regs_ready(r0);
          float v0[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r0[i]);
          if (nvalid < kChunk) {  // ragged last chunk only
            if (kEnt && cbase >= nvalid) continue;
            // with kEnt a finite stand-in, so that exp2 gives 0 and 0 * x stays 0
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (cbase + i >= nvalid) v0[i] = kEnt ? -3.0e38f : -INFINITY;
          }
          const float mraw = tree_max32_3(v0);  // c2 > 0: scale the max once
          if (mraw > -INFINITY) {
            const float mn = fmaxf(st.x, mraw * c2);
            // s*c2 - mn two lanes at a time (packed fp32 FMA), exp2 on the MUFU, packed sum tree
            const float2 c2v = make_float2(c2, c2), nmv = make_float2(-mn, -mn);
            float2 sum2[8], t2[2];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = __ffma2_rn(make_float2(v0[2 * i], v0[2 * i + 1]), c2v, nmv);
              const float2 e2 = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              sum2[i & 7] = i < 8 ? e2 : __fadd2_rn(sum2[i & 7], e2);
              if constexpr (kEnt) t2[i & 1] = i < 2 ? __fmul2_rn(e2, x) : __ffma2_rn(e2, x, t2[i & 1]);
            }
#pragma unroll
            for (int w = 4; w; w >>= 1)
#pragma unroll
              for (int i = 0; i < w; ++i) sum2[i] = __fadd2_rn(sum2[i], sum2[i + w]);
            const float alpha = ex2_approx(st.x - mn);
            if constexpr (kEnt) {
              const float tb = (t2[0].x + t2[0].y) + (t2[1].x + t2[1].y);
              tau = (st.y > 0.f ? alpha * fmaf(st.x - mn, st.y, tau) : 0.f) + tb;
            }
            st = make_float2(mn, st.y * alpha + (sum2[0].x + sum2[0].y));
          }
        }
      }
      // The two warps of a lane quarter merge their column halves; the hf == 0 warp publishes
      // the row's log2-sum-exp2 over this CTA's keys as one tagged word (no fence), and with
      // kEnt the row's mean logit in a second one. merge is double-buffered by round parity:
      // the pair passes round r + 1's barrier before hf == 1 writes the buffer of round r again.
      float2* mg = merge + (round & 1) * kResRows;
      float* mt = mtau + (round & 1) * kResRows;
      if (hf == 1) {
        mg[row] = st;
        if constexpr (kEnt) mt[row] = tau;
      }
      asm volatile("bar.sync %0, 64;\n" ::"r"(2 + q) : "memory");
      // test-only fault (kvc_debug_fault 1): the first CTA never publishes, so its group's
      // bounded exchange waits run out
      if (hf == 0 && !(a.debug_fault == 1 && blockIdx.x == 0)) {
        const float2 o = mg[row];
        const float2 m = lse_merge(st, o);
        const float part = m.y > 0.f ? m.x + log2f(m.y) : -INFINITY;
        const size_t widx = ((size_t)((round & 3) * p.ngroups + group) * p.group_size + rank) * kResRows + row;
        const uint64_t tag = (uint64_t)((uint32_t)round + 1u) << 32;
        st_relaxed_u64(words + widx, tag | __float_as_uint(part));
        if constexpr (kEnt) {
          // both halves' tau relative to the merged max, then mean logit = max + tau / sum
          float tt = 0.f;
          if (st.y > 0.f) tt += exp2f(st.x - m.x) * fmaf(st.x - m.x, st.y, tau);
          if (o.y > 0.f) tt += exp2f(o.x - m.x) * fmaf(o.x - m.x, o.y, mt[row]);
          const float mu = m.y > 0.f ? m.x + tt / m.y : 0.f;
          st_relaxed_u64(words + words_per_set + widx, tag | __float_as_uint(mu));
        }
      }
    };

    // pass 2 of a round: per key, the max over rows of s*c2 - lse2, from the logits still in TMEM;
    // each chunk's accumulator is freed as soon as its values are in registers.
    auto pass2 = [&](int round) {
      const int unit = group + round * p.ngroups;
      const int head = unit / a.tiles, tile = unit % a.tiles;
      // ---- exchange: lse2 of every row from the group's tagged partials. Thread t of the group
      // polls row t/2 of partners t%2, t%2 + 2, ... (four words in flight at a time) and merges
      // them; the two threads of a row combine with one shuffle.
      const int gt = e * 32 + lane;  // 0..255
      const int xrow = gt >> 1, xpar = gt & 1;
      const bool xvalid = ws.valid[(size_t)unit * kResRows + xrow] != 0;
      // extended epilogue: the weights of this thread's rows in a mean, fetched before the exchange
      float wr[4];
      if constexpr (kExt) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          wr[k] = a.row_agg == KVC_AGG_MEAN ? ws.rw[(size_t)unit * kResRows + q * 32 + (lane >> 2) + 8 * k] : 0.f;
      }
      // Slot round % 4 last held round - 4. A partner overwrites it (round + 4) only after its
      // pass 1 of round + 4, which needs its TMEM buffer back from its pass 2 of round + 2, which
      // follows the whole group's partials of round + 2, which this CTA publishes only after its
      // pass 2 of round has freed the TMEM buffer, i.e. after this read.
      const uint32_t tag = (uint32_t)round + 1u;
      const uint64_t* grp = words + ((size_t)((round & 3) * p.ngroups + group) * p.group_size) * kResRows + xrow;
      float mx = -INFINITY, sm = 0.f;
      bool ok = !*abort_flag;
      for (int u0 = 0; ok && xpar + 2 * u0 < p.group_size; u0 += kXchBatch) {
        uint64_t w[kXchBatch];
#pragma unroll
        for (int u = 0; u < kXchBatch; ++u) {
          const int k = xpar + 2 * (u0 + u);
          w[u] = k < p.group_size ? ld_relaxed_u64(grp + (size_t)k * kResRows)
                                  : ((uint64_t)tag << 32) | __float_as_uint(-INFINITY);
        }
        unsigned long long t_start = 0;
        for (uint32_t it = 0;; ++it) {
          unsigned need = 0u;
#pragma unroll
          for (int u = 0; u < kXchBatch; ++u)
            if ((uint32_t)(w[u] >> 32) != tag) need |= 1u << u;
          if (need == 0u) break;
          if (it == 0) t_start = global_ns();
          if (it >= (1u << 22) || *abort_flag || global_ns() - t_start > kExchangeTimeoutNs) {
            ok = false;
            if (!*abort_flag) {
              *abort_flag = 1;
              status_or(a.status, KVC_STATUS_TIMEOUT);
            }
            break;
          }
          __nanosleep(32);
#pragma unroll
          for (int u = 0; u < kXchBatch; ++u)
            if (need & (1u << u)) w[u] = ld_relaxed_u64(grp + (size_t)(xpar + 2 * (u0 + u)) * kResRows);
        }
        float bm = -INFINITY;
#pragma unroll
        for (int u = 0; u < kXchBatch; ++u) bm = fmaxf(bm, __uint_as_float((uint32_t)w[u]));
        const float nm = fmaxf(mx, bm);
        if (nm > -INFINITY) {
          float accs = mx > -INFINITY ? sm * exp2f(mx - nm) : 0.f;
#pragma unroll
          for (int u = 0; u < kXchBatch; ++u) accs += exp2f(__uint_as_float((uint32_t)w[u]) - nm);  // -inf adds 0
          mx = nm;
          sm = accs;
        }
      }
      {
        const float om = __shfl_xor_sync(kFull, mx, 1), os = __shfl_xor_sync(kFull, sm, 1);
        const float2 m2 = lse_merge(make_float2(mx, sm), make_float2(om, os));
        const float l2 = (xvalid && m2.y > 0.f) ? m2.x + log2f(m2.y) : INFINITY;
        if (xpar == 0) lse2s[(round & 1) * kResRows + xrow] = l2;
        if constexpr (kEnt) {
          // Entropy in bits of a row: lse2 - sum_j p_j x_j, and sum_j p_j x_j = sum over the group's
          // CTAs of exp2(part - lse2) * (that CTA's mean logit). This CTA adds its term for each
          // valid row (the group's first CTA adds lse2 too), from its own two published words.
          float d = 0.f;
          if (xpar == 0 && xvalid && ok && l2 < INFINITY) {
            const size_t widx = ((size_t)((round & 3) * p.ngroups + group) * p.group_size + rank) * kResRows + xrow;
            uint64_t wp = ld_relaxed_u64(words + widx), wm = ld_relaxed_u64(words + words_per_set + widx);
            for (uint32_t it = 0; ((uint32_t)(wp >> 32) != tag || (uint32_t)(wm >> 32) != tag) && it < (1u << 20); ++it) {
              __nanosleep(32);
              wp = ld_relaxed_u64(words + widx);
              wm = ld_relaxed_u64(words + words_per_set + widx);
            }
            if ((uint32_t)(wp >> 32) == tag && (uint32_t)(wm >> 32) == tag) {
              d = (rank == 0 ? l2 : 0.f) - exp2f(__uint_as_float((uint32_t)wp) - l2) * __uint_as_float((uint32_t)wm);
            } else if (!*abort_flag) {
              *abort_flag = 1;
              status_or(a.status, KVC_STATUS_TIMEOUT);
            }
          }
          d = warp_sum(d);
          if (lane == 0 && d != 0.f && !*abort_flag) atomicAdd(&a.entropy[head], d * ws.escale[head]);
        }
      }
      p2_bar();
      const bool have = !*abort_flag;
      if constexpr (kExt) {
        // ---- extended epilogue: p = exp2(s*c2 - lse2) per logit; per 16-row half of each lane
        // quarter the max (or the row-weighted sum) over its rows, per key; the halves meet in
        // shared memory, where one thread per key folds them by query head (rows of head g start
        // at g * qstride, a multiple of 16) into the max or sum over the group.
        const bool mean = a.row_agg == KVC_AGG_MEAN;
        float2 nl[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = q * 32 + (lane >> 2) + 8 * k;
          const float l2 = lse2s[(round & 1) * kResRows + r];  // unused rows: +inf, so p = 0
          nl[k] = make_float2(-l2, -l2);
        }
        const float2 c2v = make_float2(c2, c2);
        float bestA[kResChunks][2], bestB[kResChunks][2];
#pragma unroll
        for (int j = 0; j < kResChunks; ++j) bestA[j][0] = bestA[j][1] = bestB[j][0] = bestB[j][1] = 0.f;
        if (__all_sync(kFull, have)) {
          for (int j = 0; j < n; ++j) wait_or_abort(&tfull[(round & 1) * kResChunks + j], (round >> 1) & 1, abort_flag, a.status);
          tc::fence_after_sync();
#pragma unroll
          for (int j = 0; j < kResChunks; ++j) {
            if (j >= n) break;
            const uint32_t acc = (uint32_t)((round & 1) * kResChunks + j);
            const uint32_t base = tmem + acc * kChunk + lane_off + (uint32_t)(hf * 64);
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
              uint32_t ra[16], rb[16];  // rows (t/4, t/4+8) and (t/4+16, t/4+24) of 32 columns
              tc::tmem_ld16x256_x4_async(base + (uint32_t)(cb * 32), ra);
              tc::tmem_ld16x256_x4_async(base + (16u << 16) + (uint32_t)(cb * 32), rb);
              tc::tmem_wait();
              tc::tmem_regs_ready(ra);
              tc::tmem_regs_ready(rb);
              if (cb == 1) {  // the accumulator is free once its last values are in registers
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0)
                  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[acc])) : "memory");
              }
              float wA[8], wB[8];  // slot 2i + cc: column 8i + 2*(lane%4) + cc; A rows k0,k1, B rows k2,k3
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float2 y[4], e[4];
                y[0] = __ffma2_rn(make_float2(__uint_as_float(ra[4 * i]), __uint_as_float(ra[4 * i + 1])), c2v, nl[0]);
                y[1] = __ffma2_rn(make_float2(__uint_as_float(ra[4 * i + 2]), __uint_as_float(ra[4 * i + 3])), c2v, nl[1]);
                y[2] = __ffma2_rn(make_float2(__uint_as_float(rb[4 * i]), __uint_as_float(rb[4 * i + 1])), c2v, nl[2]);
                y[3] = __ffma2_rn(make_float2(__uint_as_float(rb[4 * i + 2]), __uint_as_float(rb[4 * i + 3])), c2v, nl[3]);
#pragma unroll
                for (int k = 0; k < 4; ++k) e[k] = make_float2(ex2_approx(y[k].x), ex2_approx(y[k].y));
                if (mean) {
                  wA[2 * i] = fmaf(wr[1], e[1].x, wr[0] * e[0].x);
                  wA[2 * i + 1] = fmaf(wr[1], e[1].y, wr[0] * e[0].y);
                  wB[2 * i] = fmaf(wr[3], e[3].x, wr[2] * e[2].x);
                  wB[2 * i + 1] = fmaf(wr[3], e[3].y, wr[2] * e[2].y);
                } else {
                  wA[2 * i] = fmaxf(e[0].x, e[1].x);
                  wA[2 * i + 1] = fmaxf(e[0].y, e[1].y);
                  wB[2 * i] = fmaxf(e[2].x, e[3].x);
                  wB[2 * i + 1] = fmaxf(e[2].y, e[3].y);
                }
              }
              if (mean) {
                reduce_scatter8<true>(wA, lane);
                reduce_scatter8<true>(wB, lane);
              } else {
                reduce_scatter8<false>(wA, lane);
                reduce_scatter8<false>(wB, lane);
              }
              bestA[j][cb] = wA[0];
              bestB[j][cb] = wB[0];
            }
          }
        } else {
          __syncwarp();
          if (lane == 0)
            for (int j = 0; j < n; ++j)
              asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(
                               tc::smem_u32(&tempty[(round & 1) * kResChunks + j]))
                           : "memory");
        }
        // pbest[buffer][chunk][half h = 2 * quarter + (0: rows +0..15, 1: rows +16..31)][column]
        float* pb = pbest + (round & 1) * (kResChunks * 8 * kChunk);
#pragma unroll
        for (int j = 0; j < kResChunks; ++j)
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) {
            pb[(j * 8 + 2 * q) * kChunk + hf * 64 + cb * 32 + col_in] = bestA[j][cb];
            pb[(j * 8 + 2 * q + 1) * kChunk + hf * 64 + cb * 32 + col_in] = bestB[j][cb];
          }
        p2_bar();
        const int j = gt >> 7, col = gt & (kChunk - 1);  // 256 threads: one key each
        if (j < n && !*abort_flag) {
          const float* pj = pb + j * 8 * kChunk;
          const bool gsum = a.group_agg == KVC_AGG_SUM;
          float gacc = 0.f, cur = 0.f;  // every value is >= 0: 0 is the identity of max and sum
          int cs = -1;
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const int sg = (tile * kResRows + 16 * h) / a.qstride;
            const float v = pj[h * kChunk + col];
            if (sg != cs) {
              if (cs >= 0) gacc = gsum ? gacc + cur : fmaxf(gacc, cur);
              cs = sg;
              cur = v;
            } else {
              cur = mean ? cur + v : fmaxf(cur, v);
            }
          }
          gacc = gsum ? gacc + cur : fmaxf(gacc, cur);
          const int key = (c0 + j) * kChunk + col;
          if (key < a.g.N) {
            float* dst = a.scores + (size_t)head * a.g.N + key;
            if (a.tiles == 1)
              *dst = gacc;
            else if (gsum)  // two tiles: a + b either way round, so the sum is deterministic
              atomicAdd(dst, gacc);
            else  // non-negative floats order like their bit patterns
              atomicMax(reinterpret_cast<unsigned*>(dst), __float_as_uint(gacc));
          }
        }
      } else {
        float2 nl[4];  // -lse2 of rows q*32 + lane/4 + 8k, twice (packed operands)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float l2 = lse2s[(round & 1) * kResRows + q * 32 + (lane >> 2) + 8 * k];
          nl[k] = make_float2(-l2, -l2);
        }
        const float2 c2v = make_float2(c2, c2);
        // ---- per key, the max over rows of s*c2 - lse2, from the logits still in TMEM
        float best[kResChunks][2];
#pragma unroll
        for (int j = 0; j < kResChunks; ++j) best[j][0] = best[j][1] = -INFINITY;
        if (__all_sync(kFull, have)) {
          // lse2 exists only after this CTA's pass 1 published, so the round's MMAs are complete;
          // waiting on their (completed) phases orders this warp's TMEM reads after them
          for (int j = 0; j < n; ++j) wait_or_abort(&tfull[(round & 1) * kResChunks + j], (round >> 1) & 1, abort_flag, a.status);
          tc::fence_after_sync();
#pragma unroll
          for (int j = 0; j < kResChunks; ++j) {
            if (j >= n) break;
            const uint32_t acc = (uint32_t)((round & 1) * kResChunks + j);
            const uint32_t base = tmem + acc * kChunk + lane_off + (uint32_t)(hf * 64);
            uint32_t ra[2][16], rb[2][16];  // [block] x rows (t/4, t/4+8) and (t/4+16, t/4+24)
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
              tc::tmem_ld16x256_x4_async(base + (uint32_t)(cb * 32), ra[cb]);
              tc::tmem_ld16x256_x4_async(base + (16u << 16) + (uint32_t)(cb * 32), rb[cb]);
            }
            tc::tmem_wait();
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
              tc::tmem_regs_ready(ra[cb]);
              tc::tmem_regs_ready(rb[cb]);
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0)  // the accumulator is free as soon as its values are in registers
              asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[acc])) : "memory");
#pragma unroll
            for (int cb = 0; cb < 2; ++cb) {
              // a row without observations has lse2 = +inf, so its terms are -inf and drop out of the max
              // slot 2i + cc: column 8i + 2*(lane%4) + cc of the block, max over 4 rows; the two
              // columns of a pair share each row's lse2, so s*c2 - lse2 is one packed FMA per row
              float w[8];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 x0 = __ffma2_rn(make_float2(__uint_as_float(ra[cb][4 * i]), __uint_as_float(ra[cb][4 * i + 1])),
                                             c2v, nl[0]);
                const float2 x1 = __ffma2_rn(
                    make_float2(__uint_as_float(ra[cb][4 * i + 2]), __uint_as_float(ra[cb][4 * i + 3])), c2v, nl[1]);
                const float2 x2 = __ffma2_rn(make_float2(__uint_as_float(rb[cb][4 * i]), __uint_as_float(rb[cb][4 * i + 1])),
                                             c2v, nl[2]);
                const float2 x3 = __ffma2_rn(
                    make_float2(__uint_as_float(rb[cb][4 * i + 2]), __uint_as_float(rb[cb][4 * i + 3])), c2v, nl[3]);
                w[2 * i] = fmaxf(max3f(x0.x, x1.x, x2.x), x3.x);
                w[2 * i + 1] = fmaxf(max3f(x0.y, x1.y, x2.y), x3.y);
              }
              reduce_scatter_max8(w, lane);
              best[j][cb] = w[0];
            }
          }
        } else {
          __syncwarp();
          if (lane == 0)
            for (int j = 0; j < n; ++j)
              asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(
                               tc::smem_u32(&tempty[(round & 1) * kResChunks + j]))
                           : "memory");
        }
        // pbest[buffer][chunk][quarter][column]; buffer = round parity (the group's barriers of
        // round r + 1 lie between two uses)
        float* pb = pbest + (round & 1) * (kResChunks * 4 * kChunk);
#pragma unroll
        for (int j = 0; j < kResChunks; ++j)
#pragma unroll
          for (int cb = 0; cb < 2; ++cb) pb[(j * 4 + q) * kChunk + hf * 64 + cb * 32 + col_in] = best[j][cb];
        p2_bar();
        const int j = gt >> 7, col = gt & (kChunk - 1);  // 256 threads: one key each
        if (j < n && !*abort_flag) {
          const float* pj = pb + j * 4 * kChunk;
          const float m = fmaxf(fmaxf(pj[col], pj[kChunk + col]), fmaxf(pj[2 * kChunk + col], pj[3 * kChunk + col]));
          const int key = (c0 + j) * kChunk + col;
          if (key < a.g.N) {
            float* dst = a.scores + (size_t)head * a.g.N + key;
            if (a.tiles == 1)
              *dst = exp2f(m);
            else  // non-negative floats order like their bit patterns
              atomicMax(reinterpret_cast<unsigned*>(dst), __float_as_uint(exp2f(m)));
          }
        }
      }
    };

    // The two groups run concurrently: pass 1 of round r + 1 overlaps pass 2 of round r.
    if (is_p1)
      for (int round = 0; round < rounds; ++round) pass1(round);
    else
      for (int round = 0; round < rounds; ++round) pass2(round);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Shared memory: align slack, barriers, lse2 x2, merge x2, tau x2, pbest x2; then the Q tile(s) and the ring.
static int resident_tail_bytes(bool ext) {
  return 1024 + 512 + 2 * kResRows * 4 + 2 * kResRows * 8 + 2 * kResRows * 4 + 2 * kResChunks * (ext ? 8 : 4) * kChunk * 4;
}

bool score_resident_plan(const ScoreArgs& a, FusedPlan* p, size_t* smem) {
  if (a.dtype != KVC_BF16 || a.M_pad != kResRows * a.tiles) return false;
  int dev = 0, nsm = 0, smem_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return false;
  if (nsm > kMaxSMs) nsm = kMaxSMs;
  const int D = a.g.D;
  const int heads = a.g.L * a.g.B * a.g.Hkv * a.tiles;  // units
  p->chunks_per_cta = a.nchunk >= kResChunks ? kResChunks : 1;
  p->group_size = (a.nchunk + p->chunks_per_cta - 1) / p->chunks_per_cta;
  if (p->group_size > nsm) return false;
  p->ngroups = nsm / p->group_size;
  if (p->ngroups > heads) p->ngroups = heads;
  p->qbytes = kResRows * D * 2;
  const int stage_bytes = kChunk * D * 2;
  int stages = (smem_optin - resident_tail_bytes(a.ext != 0) - kQBuf * p->qbytes) / stage_bytes;
  if (stages > 6) stages = 6;
  if (stages < 2) return false;
  p->stages = stages;
  *smem = (size_t)resident_tail_bytes(a.ext != 0) + kQBuf * (size_t)p->qbytes + (size_t)stages * stage_bytes;
  return true;
}

// tagged partial words [4][ngroups][group_size][128], and as many again for the rows' mean
// logits when the entropy is wanted; zero, so no tag of an earlier launch matches
long long score_resident_words(const FusedPlan& p, bool entropy) {
  return (entropy ? 2LL : 1LL) * 4LL * p.ngroups * p.group_size * kResRows;
}

int launch_score_resident(const ScoreArgs& a, const ScoreWs& ws, const FusedPlan& p, size_t smem, cudaStream_t s) {
  const int D = a.g.D;
  FusedXch xch;
  xch.part = ws.part;
  xch.arrive = nullptr;
  FusedMaps maps;
  if (!fused_maps(&maps, a, ws)) return KVC_ERR_LAUNCH;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  using Kern = void (*)(const FusedMaps, ScoreArgs, ScoreWs, FusedPlan, FusedXch, float);
  // [D == 128][extended epilogue][entropy][wide exchange batch]
#define KVC_RES_K(d, x, e) {score_resident_kernel<d, x, e, kXchNarrow>, score_resident_kernel<d, x, e, kXchWide>}
  static const Kern table[2][2][2][2] = {
      {{KVC_RES_K(64, false, false), KVC_RES_K(64, false, true)}, {KVC_RES_K(64, true, false), KVC_RES_K(64, true, true)}},
      {{KVC_RES_K(128, false, false), KVC_RES_K(128, false, true)},
       {KVC_RES_K(128, true, false), KVC_RES_K(128, true, true)}}};
#undef KVC_RES_K
  const bool variant = a.row_agg != KVC_AGG_MAX || a.group_agg != KVC_AGG_MAX;
  // wide batches once a thread would need more than two narrow ones (group_size / 2 partners each)
  const bool wide = p.group_size / 2 > 2 * kXchNarrow;
  Kern kern = table[D == 128][variant][a.entropy != nullptr][wide];
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kResThreads, smem) != cudaSuccess ||
      per_sm < 1)
    return KVC_ERR_LAUNCH;
  ScoreArgs aa = a;
  ScoreWs wss = ws;
  FusedPlan pp = p;
  float cc = c2;
  if (launch_pdl(kern, dim3(p.ngroups * p.group_size), dim3(kResThreads), smem, s, true, maps, aa, wss, pp, xch, cc) !=
      cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
