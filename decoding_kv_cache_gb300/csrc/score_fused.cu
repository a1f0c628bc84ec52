// score_fused.cu -- the bf16 scoring passes as one persistent, warp-specialised kernel.
//
// What it computes is kvc_score's definition (BeaconKV write-up, "打分时的 RoPE 对齐": a key's
// importance is the max over the observation rows of its softmax weight over all cached keys).
// The softmax needs each row's log-sum-exp over ALL keys before any score can be formed, so
// the keys are visited twice: pass 1 folds (max, sum of exp2) per row, pass 2 recomputes the
// logits and takes the max over rows of exp2(s*c2 - lse2).
//
// Work split. A head's keys are cut into G_s contiguous ranges of whole 128-key chunks, one
// per CTA of a "group"; the grid is (#groups x G_s) CTAs, one per SM, launched cooperatively so
// every CTA is resident. Group g handles heads g, g + #groups, ... in rounds. In a round a CTA
// runs pass 1 over its range and publishes its per-row partials; once the whole group has
// published, the partials merge into lse2 and the CTA runs pass 2 over the same range. Pass 1
// of the next round is interleaved before pass 2 of the current one, so nobody waits for the
// group. Pass 2's TMA reads find the range in L2: at most two ranges per SM (~512 KB) are live.
//
// Roles inside a CTA (all derive the same chunk sequence from blockIdx, so no queue is needed):
//   warp 0      TMA producer: the round's observation tile Q into one of two Q buffers, then
//               each key chunk of pass 1 and again of pass 2 into a ring of K stages.
//   warp 1      tcgen05.mma issuer (one thread) with two 256-column TMEM accumulators: pass 1
//               S = Q K^T (lane = row), pass 2 S^T = K Q^T (lane = key).
//   warps 2-9   epilogue: pass 1 keeps each row's running (max, sum) in registers (two warps
//               per TMEM lane quarter split the columns); pass 2 keeps each key's running max.
//   warp 10     exchange: waits until the group has published a round's partials and merges
//               them into lse2 per row (double-buffered in shared memory), off the critical path.
// Barriers: kfull/kempty per K stage, qfull/qempty per Q buffer, tfull/tempty per TMEM
// accumulator (four of 128 columns when both passes fit, else two of 256), lfull/lempty per
// lse2 buffer. Partials are published with one release add after a CTA-local barrier.
// Every wait is bounded; a wait that gives up sets KVC_STATUS_TIMEOUT and a CTA-wide abort
// flag, after which every role skips its work but still passes every named barrier.
#include "score_tc.cuh"

namespace kvc {

// kExt: the extended epilogue (aggregation variants and the entropy); otherwise max/max only.
template <int D, int MT, int NACC, bool kExt>
__global__ void __launch_bounds__(kFusedThreads, 1)
    score_fused_kernel(const __grid_constant__ FusedMaps maps, ScoreArgs a, ScoreWs ws, FusedPlan p, FusedXch xch,
                       float c2) {
  constexpr int HALVES = D / 64;
  constexpr int kStage = kChunk * D * 2;
  constexpr uint32_t kAcc = 512u / NACC;  // TMEM columns per accumulator
  extern __shared__ uint8_t smraw[];
  uint8_t* Qs = align1024(smraw);
  uint8_t* Ks = Qs + 2 * p.qbytes;
  const int S = p.stages;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(Ks + S * kStage);
  uint64_t* kempty = kfull + S;
  uint64_t* qfull = kempty + S;
  uint64_t* qempty = qfull + 2;
  uint64_t* tfull = qempty + 2;
  uint64_t* tempty = tfull + NACC;
  uint64_t* lfull = tempty + NACC;
  uint64_t* lempty = lfull + 2;
  uint32_t* slot = reinterpret_cast<uint32_t*>(lempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(slot + 1);
  float* lse2s = reinterpret_cast<float*>(Ks + S * kStage + 512);  // [2][kMaxRows], 16-byte aligned
  float2* merge = reinterpret_cast<float2*>(lse2s + 2 * kMaxRows);   // [kMaxRows]
  float* pbest = reinterpret_cast<float*>(merge + kMaxRows);         // [2][kChunk]
  float* rws = pbest + 2 * kChunk;                                    // kExt: [2][kMaxRows] row weights
  float* pext = rws + 2 * kMaxRows;                                   // kExt: [2][5][kChunk] half partials

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      tc::mbar_init(&tfull[i], 1);
      tc::mbar_init(&tempty[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
      tc::mbar_init(&lfull[i], 1);
      tc::mbar_init(&lempty[i], kEpiWarps);
    }
    *abort_flag = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) tc::tmem_alloc(slot, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *slot;

  const int heads = a.g.L * a.g.B * a.g.Hkv;
  const int group = blockIdx.x / p.group_size, rank = blockIdx.x % p.group_size;
  const int rounds = group < heads ? (heads - group + p.ngroups - 1) / p.ngroups : 0;
  const int c0 = rank * p.chunks_per_cta;
  const int c1 = min(c0 + p.chunks_per_cta, a.nchunk);
  const int qrow_bytes = a.M_pad * 128;  // one 64-column half of an observation tile

  // Chunk order, identical in every role: segment seg = pass 1 of round seg (if any), then
  // pass 2 of round seg - 1 (if any). Pass 1 of the next round thus runs while the group's
  // partials for the previous round are gathered.
  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      uint32_t kc = 0;
      const int n = c1 > c0 ? c1 - c0 : 0;
      for (int seg = 0; seg <= rounds && !*abort_flag; ++seg) {
        if (seg < rounds) {  // this round's observation tile, into the buffer its round parity names
          const int round = seg, head = group + round * p.ngroups;
          const int qb = round & 1;
          if (round >= 2 && !wait_or_abort(&qempty[qb], ((round - 2) >> 1) & 1, abort_flag, a.status)) break;
          uint8_t* qdst = Qs + qb * p.qbytes;
          tc::mbar_expect_tx(&qfull[qb], (uint32_t)p.qbytes);
          for (int h = 0; h < HALVES; ++h)
            for (int mt = 0; mt < MT; ++mt)
              tc::tma_load_2d(qdst + h * qrow_bytes + mt * 16384, &maps.q, &qfull[qb], h * 64,
                              head * a.M_pad + mt * 128);
        }
        bool stop = false;
        for (int j = 0; j < n + 2 && !stop; ++j)
          for (int pass = 0; pass < 2; ++pass) {
            const int round = seg - pass;
            const int c = c0 + j - 2 * pass;
            if (round < 0 || round >= rounds || c < c0 || c >= c1) continue;
            const int head = group + round * p.ngroups;
            const int l = head / (a.g.B * a.g.Hkv), bh = head % (a.g.B * a.g.Hkv);
            const int s = kc % S;
            if (kc >= (uint32_t)S && !wait_or_abort(&kempty[s], ((kc / S) - 1) & 1, abort_flag, a.status)) {
              stop = true;
              break;
            }
            tc::mbar_expect_tx(&kfull[s], (uint32_t)kStage);
            for (int h = 0; h < HALVES; ++h)
              tc::tma_load_3d(Ks + s * kStage + h * 16384, &maps.k[l], &kfull[s], h * 64, c * kChunk, bh);
            ++kc;
          }
        if (stop) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t kc = 0;
      const uint32_t id1 = tc::idesc_bf16(128, kChunk);
      const uint32_t id2 = tc::idesc_bf16(128, a.M_n);
      const int n = c1 > c0 ? c1 - c0 : 0;
      bool ok = true;
      for (int seg = 0; seg <= rounds && ok && !*abort_flag; ++seg) {
        if (seg < rounds) {
          if (!wait_or_abort(&qfull[seg & 1], (seg >> 1) & 1, abort_flag, a.status)) break;
          tc::fence_after_sync();
        }
        for (int j = 0; j < n + 2 && ok; ++j)
          for (int pass = 0; pass < 2; ++pass) {
            const int round = seg - pass;
            const int c = c0 + j - 2 * pass;
            if (round < 0 || round >= rounds || c < c0 || c >= c1) continue;
            const uint32_t qaddr = tc::smem_u32(Qs + (round & 1) * p.qbytes);
            const int s = kc % S;
            const uint32_t acc = kc % NACC;
            if (!wait_or_abort(&kfull[s], (kc / S) & 1, abort_flag, a.status) ||
                (kc >= (uint32_t)NACC &&
                 !wait_or_abort(&tempty[acc], ((kc / NACC) - 1) & 1, abort_flag, a.status))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t kaddr = tc::smem_u32(Ks + s * kStage);
            const uint32_t d = tmem + acc * kAcc;
            if (pass == 0) {
#pragma unroll
              for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                  tc::umma_bf16(d + mt * kChunk,
                                tc::desc_k_sw128(qaddr + (ks >> 2) * qrow_bytes + mt * 16384 + (ks & 3) * 32),
                                tc::desc_k_sw128(kaddr + (ks >> 2) * 16384 + (ks & 3) * 32), id1, ks > 0);
            } else {
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks)
                tc::umma_bf16(d, tc::desc_k_sw128(kaddr + (ks >> 2) * 16384 + (ks & 3) * 32),
                              tc::desc_k_sw128(qaddr + (ks >> 2) * qrow_bytes + (ks & 3) * 32), id2, ks > 0);
            }
            tc::umma_commit(&kempty[s]);
            tc::umma_commit(&tfull[acc]);
            ++kc;
          }
        // the previous round's tile is done once its pass 2 has been issued (n == 0 issues none)
        if (ok && seg >= 1) tc::umma_commit(&qempty[(seg - 1) & 1]);
      }
    }
    __syncwarp();
  } else if (warp == 2 + kEpiWarps) {
    // ---------------- exchange warp: lse2 of every row once the group has published ----------------
    for (int round = 0; round < rounds && !*abort_flag; ++round) {
      const int b = round & 1;
      if (round >= 2 && !wait_or_abort(&lempty[b], ((round - 2) >> 1) & 1, abort_flag, a.status)) break;
      const int head = group + round * p.ngroups;
      // Slot round % 4 has been published by the group (round >> 2) times before; a partner can
      // only publish round + 4 into it after the whole group published round + 2, so reaching
      // this count means every partner has published `round`.
      if (lane == 0) {
        const unsigned target = (unsigned)((round >> 2) + 1) * (unsigned)p.group_size;
        const unsigned* ctr = &xch.arrive[(round & 3) * p.ngroups + group];
        bool done = false;
        for (uint32_t it = 0; it < (1u << 22) && !*abort_flag; ++it) {
          if (ld_acquire(ctr) >= target) {
            done = true;
            break;
          }
          __nanosleep(32);
        }
        if (!done && !*abort_flag) {
          *abort_flag = 1;
          status_or(a.status, KVC_STATUS_TIMEOUT);
        }
      }
      __syncwarp();
      const float2* grp = xch.part + ((size_t)((round & 3) * p.ngroups + group) * p.group_size) * a.M_pad;
      float* dst = lse2s + b * kMaxRows;
      // unused rows: +inf drops them from a max; the extended epilogue takes a large finite value
      // instead, so that p = 0 and p * log2 p = 0 there (no inf * 0)
      const float none = kExt ? 1e30f : INFINITY;
      const bool mean_w = kExt && a.row_agg == KVC_AGG_MEAN;
      for (int r = lane; r < a.M_pad; r += kWarp) {
        float2 acc2 = make_float2(-INFINITY, 0.f);
        for (int k = 0; k < p.group_size; ++k) acc2 = lse_merge(acc2, grp[(size_t)k * a.M_pad + r]);
        const bool valid = ws.valid[(size_t)head * a.M_pad + r] != 0;
        dst[r] = (valid && acc2.y > 0.f) ? acc2.x + log2f(acc2.y) : none;
        if (mean_w) rws[b * kMaxRows + r] = ws.rw[(size_t)head * a.M_pad + r];
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&lfull[b])) : "memory");
    }
  } else {
    // ---------------- epilogue ----------------
    const int e = warp - 2;      // 0..7
    const int q = warp & 3;      // TMEM lane quarter this warp may read
    const int hf = e >> 2;       // which half of the columns
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int key = q * 32 + lane;
    const int nslice = (a.M_n + 31) >> 5;
    const int half_s = (nslice + 1) >> 1;
    const int s_lo = hf == 0 ? 0 : half_s, s_hi = hf == 0 ? half_s : nslice;
    const int n = c1 > c0 ? c1 - c0 : 0;
    uint32_t kc = 0;
    float2 st[MT];
    bool have = false;  // lse2 of the round whose pass 2 is running is in shared memory

    // publish this CTA's partials of round `round` (slot = round % 4)
    auto publish = [&](int round) {
      if (hf == 1)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) merge[mt * 128 + q * 32 + lane] = st[mt];
      epi_bar();
      float2* mine = xch.part + ((size_t)((round & 3) * p.ngroups + group) * p.group_size + rank) * a.M_pad;
      if (hf == 0)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int r = mt * 128 + q * 32 + lane;
          mine[r] = lse_merge(st[mt], merge[r]);
        }
      epi_bar();
      // one release add after the CTA-local barrier publishes every epilogue thread's writes
      if (e == 0 && lane == 0)
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;\n" ::"l"(&xch.arrive[(round & 3) * p.ngroups + group])
                     : "memory");
    };
    auto lse_wait = [&](int round) {
      have = !*abort_flag && wait_or_abort(&lfull[round & 1], (round >> 1) & 1, abort_flag, a.status);
    };
    auto lse_release = [&](int round) {
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&lempty[round & 1])) : "memory");
    };
    auto free_acc = [&](uint32_t acc) {
      __syncwarp();
      if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tc::smem_u32(&tempty[acc])) : "memory");
    };

    // pass 1 chunk: fold this thread's row(s) into the running (max, sum of exp2)
    auto pass1_chunk = [&](int c) {
      const uint32_t acc = kc % NACC;
      const bool go = !*abort_flag && wait_or_abort(&tfull[acc], (kc / NACC) & 1, abort_flag, a.status);
      if (__all_sync(kFull, go)) {  // tcgen05.ld is warp-collective: decide per warp
        tc::fence_after_sync();
        const int nvalid = min(kChunk, a.g.N - c * kChunk);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t r0[32], r1[32];
          const uint32_t col0 = (uint32_t)(mt * kChunk + hf * 64);
          tc::tmem_ld32_async(tmem + acc * kAcc + lane_off + col0, r0);
          tc::tmem_ld32_async(tmem + acc * kAcc + lane_off + col0 + 32, r1);
          tc::tmem_wait();
          tc::tmem_regs_ready(r0);
          tc::tmem_regs_ready(r1);
          if (mt == MT - 1) {  // the accumulator is free as soon as its last values are in registers
            tc::fence_before_sync();
            free_acc(acc);
          }
          float v0[32], v1[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v0[i] = __uint_as_float(r0[i]);
            v1[i] = __uint_as_float(r1[i]);
          }
          if (nvalid < kChunk) {  // ragged last chunk only
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (hf * 64 + i >= nvalid) v0[i] = -INFINITY;
              if (hf * 64 + 32 + i >= nvalid) v1[i] = -INFINITY;
            }
          }
          const float mraw = fmaxf(tree_max32(v0), tree_max32(v1));  // c2 > 0: scale the max once
          if (mraw > -INFINITY) {
            const float mn = fmaxf(st[mt].x, mraw * c2);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              v0[i] = ex2_approx(fmaf(v0[i], c2, -mn));
              v1[i] = ex2_approx(fmaf(v1[i], c2, -mn));
            }
            st[mt] = make_float2(mn, st[mt].y * ex2_approx(st[mt].x - mn) + (tree_sum32(v0) + tree_sum32(v1)));
          }
        }
      } else {
        free_acc(acc);
      }
      ++kc;
    };

    // pass 2 chunk: each key's max over rows of s*c2 - lse2, then exp2
    auto pass2_chunk = [&](int round, int c) {
      const uint32_t acc = kc % NACC;
      const int head = group + round * p.ngroups;
      const float* L2 = lse2s + (round & 1) * kMaxRows;
      if constexpr (kExt) {
        // Extended epilogue: p = exp2(s*c2 - lse2) per logit; per 16-row half-slice the max
        // (or the row-weighted sum) of p; the half-slices fold by query head (rows of head g
        // start at g * qstride, a multiple of 16) into the max or sum over the group. A thread
        // sees its column half's rows in order, so it keeps its first and last head's partial
        // apart; the two halves' partials meet in shared memory. -sum p log2 p is summed too.
        const float* RW = rws + (round & 1) * kMaxRows;
        const bool mean = a.row_agg == KVC_AGG_MEAN, gsum = a.group_agg == KVC_AGG_SUM;
        const bool kvalid = c * kChunk + key < a.g.N;
        int fseg = -1, cur = -1;  // first head (if a later one followed) and current head
        float fval = 0.f, cv = 0.f, gacc = 0.f, hacc = 0.f;  // values >= 0: 0 is the identity
        const bool go = have && !*abort_flag && wait_or_abort(&tfull[acc], (kc / NACC) & 1, abort_flag, a.status);
        if (__all_sync(kFull, go)) {
          tc::fence_after_sync();
#pragma unroll 1
          for (int cs = s_lo; cs < s_hi; ++cs) {
            uint32_t ra[32];
            tc::tmem_ld32_async(tmem + acc * kAcc + lane_off + (uint32_t)(cs * 32), ra);
            tc::tmem_wait();
            tc::tmem_regs_ready(ra);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int r0 = cs * 32 + hh * 16;
              if (r0 >= a.M_n) break;  // columns the MMA did not write (M_n is a multiple of 16)
              float v = 0.f;
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const float y = fmaf(__uint_as_float(ra[hh * 16 + i]), c2, -L2[r0 + i]);
                const float e = ex2_approx(y);
                hacc = fmaf(e, y, hacc);
                v = mean ? fmaf(RW[r0 + i], e, v) : fmaxf(v, e);
              }
              const int sg = r0 / a.qstride;
              if (sg != cur) {
                if (cur >= 0) {
                  if (fseg < 0) {
                    fseg = cur;
                    fval = cv;
                  } else {
                    gacc = gsum ? gacc + cv : fmaxf(gacc, cv);
                  }
                }
                cur = sg;
                cv = v;
              } else {
                cv = mean ? cv + v : fmaxf(cv, v);
              }
            }
          }
          tc::fence_before_sync();
          if (a.entropy) {
            const float h = warp_sum(kvalid ? hacc : 0.f);
            if (lane == 0) atomicAdd(&a.entropy[head], -h * ws.escale[head]);
          }
        }
        free_acc(acc);
        float* px = pext + (kc & 1) * 5 * kChunk;
        if (hf == 1) {
          px[key] = __int_as_float(fseg);
          px[kChunk + key] = fval;
          px[2 * kChunk + key] = gacc;
          px[3 * kChunk + key] = __int_as_float(cur);
          px[4 * kChunk + key] = cv;
        }
        epi_bar();
        if (hf == 0 && !*abort_flag) {
          const int fsegB = __float_as_int(px[key]), curB = __float_as_int(px[3 * kChunk + key]);
          const float fvalB = px[kChunk + key], gaccB = px[2 * kChunk + key], cvB = px[4 * kChunk + key];
          auto gop = [&](float x, float y) { return gsum ? x + y : fmaxf(x, y); };
          float tot = gacc;
          if (fseg >= 0) tot = gop(tot, fval);
          const int bfs = fsegB >= 0 ? fsegB : curB;  // the other half's first head
          const float bfv = fsegB >= 0 ? fvalB : cvB;
          if (cur >= 0 && cur == bfs) {
            tot = gop(tot, mean ? cv + bfv : fmaxf(cv, bfv));
          } else {
            if (cur >= 0) tot = gop(tot, cv);
            if (bfs >= 0) tot = gop(tot, bfv);
          }
          if (fsegB >= 0) {
            tot = gop(tot, gaccB);
            tot = gop(tot, cvB);
          }
          const int j = c * kChunk + key;
          if (j < a.g.N) a.scores[(size_t)head * a.g.N + j] = tot;
        }
        ++kc;
        return;
      }
      float best = -INFINITY;
      const bool go = have && !*abort_flag && wait_or_abort(&tfull[acc], (kc / NACC) & 1, abort_flag, a.status);
      if (__all_sync(kFull, go)) {  // tcgen05.ld is warp-collective: decide per warp
        tc::fence_after_sync();
        // rows past M_n read TMEM columns the MMA did not write; their lse2 is +inf, so the term
        // is -inf or NaN, which fmaxf drops
#pragma unroll 1
        for (int cs = s_lo; cs < s_hi; cs += 2) {
          uint32_t ra[32], rb[32];
          const bool two = cs + 1 < s_hi;
          tc::tmem_ld32_async(tmem + acc * kAcc + lane_off + (uint32_t)(cs * 32), ra);
          if (two) tc::tmem_ld32_async(tmem + acc * kAcc + lane_off + (uint32_t)(cs * 32 + 32), rb);
          tc::tmem_wait();
          tc::tmem_regs_ready(ra);
          tc::tmem_regs_ready(rb);
          float v[32];
          const float4* l4 = reinterpret_cast<const float4*>(L2 + cs * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 lb = l4[i];
            v[4 * i + 0] = fmaf(__uint_as_float(ra[4 * i + 0]), c2, -lb.x);
            v[4 * i + 1] = fmaf(__uint_as_float(ra[4 * i + 1]), c2, -lb.y);
            v[4 * i + 2] = fmaf(__uint_as_float(ra[4 * i + 2]), c2, -lb.z);
            v[4 * i + 3] = fmaf(__uint_as_float(ra[4 * i + 3]), c2, -lb.w);
          }
          best = fmaxf(best, tree_max32(v));
          if (two) {
            const float4* m4 = reinterpret_cast<const float4*>(L2 + cs * 32 + 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 lb = m4[i];
              v[4 * i + 0] = fmaf(__uint_as_float(rb[4 * i + 0]), c2, -lb.x);
              v[4 * i + 1] = fmaf(__uint_as_float(rb[4 * i + 1]), c2, -lb.y);
              v[4 * i + 2] = fmaf(__uint_as_float(rb[4 * i + 2]), c2, -lb.z);
              v[4 * i + 3] = fmaf(__uint_as_float(rb[4 * i + 3]), c2, -lb.w);
            }
            best = fmaxf(best, tree_max32(v));
          }
        }
        tc::fence_before_sync();
      }
      free_acc(acc);
      float* pb = pbest + (kc & 1) * kChunk;
      if (hf == 1) pb[key] = best;
      epi_bar();
      if (hf == 0 && !*abort_flag) {
        best = fmaxf(best, pb[key]);
        const int j = c * kChunk + key;
        if (j < a.g.N) a.scores[(size_t)head * a.g.N + j] = exp2f(best);
      }
      ++kc;
    };

    // Same chunk order as the producer and MMA warps: in segment seg, pass-1 chunk j of round
    // seg is followed by pass-2 chunk j - 2 of round seg - 1.
    for (int seg = 0; seg <= rounds; ++seg) {
      if (seg < rounds)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) st[mt] = make_float2(-INFINITY, 0.f);
      if (n == 0) {  // no keys here: still take part in the group's exchange
        if (seg < rounds) publish(seg);
        if (seg >= 1) {
          lse_wait(seg - 1);
          lse_release(seg - 1);
        }
        continue;
      }
      for (int j = 0; j < n + 2; ++j) {
        if (seg < rounds && j < n) {
          pass1_chunk(c0 + j);
          if (j == n - 1) publish(seg);
        }
        if (seg >= 1 && j >= 2) {
          if (j == 2) lse_wait(seg - 1);
          pass2_chunk(seg - 1, c0 + j - 2);
          if (j == n + 1) lse_release(seg - 1);
        }
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
static PFN_cuTensorMapEncodeTiled_v12000 fused_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;  // resolved once from the driver
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool fused_maps(FusedMaps* m, const ScoreArgs& a, const ScoreWs& ws, int qrows) {
  auto enc = fused_encoder();
  if (!enc) return false;
  const int D = a.g.D;
  const cuuint32_t es[3] = {1, 1, 1};
  for (int l = 0; l < a.g.L; ++l) {
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.g.ncap, (cuuint64_t)a.g.B * a.g.Hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.g.ncap * D * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)kChunk, 1};
    if (enc(&m->k[l], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.K.p[l], dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const int heads = a.g.L * a.g.B * a.g.Hkv;
  const cuuint64_t qdims[2] = {(cuuint64_t)D, (cuuint64_t)heads * a.M_pad};
  const cuuint64_t qstrides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t qbox[2] = {64, (cuuint32_t)qrows};
  return enc(&m->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws.obs, qdims, qstrides, qbox, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t fused_xch_bytes(int M_pad) {
  return (size_t)4 * kMaxSMs * (size_t)M_pad * sizeof(float2) + (size_t)4 * kMaxSMs * sizeof(unsigned) + 256;
}

int launch_score_fused(const ScoreArgs& a, const ScoreWs& ws, void* xch_base, cudaStream_t s) {
  int dev = 0, nsm = 0, smem_optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  if (nsm > kMaxSMs) nsm = kMaxSMs;
  const int D = a.g.D;
  FusedPlan p;
  // about eight 128-key chunks (1024 keys) per CTA, with the group size a divisor of the SM count
  const int want = (a.nchunk + 7) / 8;
  int gs = nsm;
  for (int d = 1; d <= nsm; ++d)
    if (nsm % d == 0 && d >= want) {
      gs = d;
      break;
    }
  p.group_size = gs;
  p.ngroups = nsm / gs;
  p.chunks_per_cta = (a.nchunk + gs - 1) / gs;
  p.qbytes = a.M_pad * D * 2;
  const int stage_bytes = kChunk * D * 2;
  // align slack, barriers, lse2 x2, merge, pbest; with the extended epilogue row weights x2 and
  // the half partials x2
  const int tail = 1024 + 512 + kMaxRows * 16 + 2 * kChunk * 4 + 256 + (a.ext ? 2 * kMaxRows * 4 + 10 * kChunk * 4 : 0);
  int stages = (smem_optin - 2 * p.qbytes - tail) / stage_bytes;
  if (stages > 6) stages = 6;
  if (stages < 2) return KVC_ERR_TOO_LARGE;
  p.stages = stages;
  const size_t smem = (size_t)tail + 2 * (size_t)p.qbytes + (size_t)stages * stage_bytes;

  FusedXch xch;
  xch.part = reinterpret_cast<float2*>(xch_base);
  xch.arrive = reinterpret_cast<unsigned*>(static_cast<char*>(xch_base) +
                                           (size_t)4 * kMaxSMs * (size_t)a.M_pad * sizeof(float2));
  if (cudaMemsetAsync(xch.arrive, 0, sizeof(unsigned) * 4 * (size_t)p.ngroups, s) != cudaSuccess)
    return KVC_ERR_LAUNCH;

  FusedMaps maps;
  if (!fused_maps(&maps, a, ws)) return KVC_ERR_LAUNCH;
  const float c2 = (float)(1.4426950408889634074 / sqrt((double)D));
  // four 128-column accumulators when both passes fit in 128 columns, else two of 256
  void (*kern)(const FusedMaps, ScoreArgs, ScoreWs, FusedPlan, FusedXch, float);
  if (a.ext)
    kern = D == 128 ? (a.M_pad > 128 ? score_fused_kernel<128, 2, 2, true> : score_fused_kernel<128, 1, 4, true>)
                    : (a.M_pad > 128 ? score_fused_kernel<64, 2, 2, true> : score_fused_kernel<64, 1, 4, true>);
  else
    kern = D == 128 ? (a.M_pad > 128 ? score_fused_kernel<128, 2, 2, false> : score_fused_kernel<128, 1, 4, false>)
                    : (a.M_pad > 128 ? score_fused_kernel<64, 2, 2, false> : score_fused_kernel<64, 1, 4, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFusedThreads, smem) != cudaSuccess ||
      per_sm < 1)
    return KVC_ERR_LAUNCH;
  ScoreArgs aa = a;
  ScoreWs wss = ws;
  float cc = c2;
  void* args[] = {(void*)&maps, (void*)&aa, (void*)&wss, (void*)&p, (void*)&xch, (void*)&cc};
  if (cudaLaunchCooperativeKernel((const void*)kern, dim3(p.ngroups * p.group_size), dim3(kFusedThreads), args, smem,
                                  s) != cudaSuccess)
    return KVC_ERR_LAUNCH;
  return KVC_OK;
}

}  // namespace kvc
