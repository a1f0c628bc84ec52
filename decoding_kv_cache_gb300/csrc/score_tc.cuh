// score_tc.cuh -- pieces shared by the two tensor-core scoring kernels (score_fused.cu and
// score_resident.cu): the role layout, tensor maps, the cross-CTA exchange of per-row
// (max, sum of exp2) partials, bounded waits and small reductions.
#pragma once

#include <cudaTypedefs.h>

#include "kvc_internal.cuh"
#include "tc_ptx.cuh"

namespace kvc {

constexpr int kEpiWarps = 8;
constexpr int kFusedThreads = 64 + 32 * kEpiWarps + 32;  // producer, MMA, epilogue warps, exchange warp

struct FusedMaps {
  CUtensorMap k[KVC_MAX_LAYERS];  // per layer: dims {D, ncap, B*Hkv}, box {64, 128, 1}
  CUtensorMap q;                  // observation rows: dims {D, heads*M_pad}, box {64, 128}
};

struct FusedXch {
  float2* part;      // [4][ngroups][group_size][M_pad] per-row (max, sum) of each range, slot = round % 4
  unsigned* arrive;  // [4][ngroups] publications per exchange slot, zero at launch
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~(uintptr_t)1023);
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kEpiWarps) : "memory"); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// mbarrier wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  for (int round = 0; round < 64; ++round) {
    if (*abort_flag) return false;
    if (tc::mbar_wait(bar, parity, 1u << 18)) return true;
  }
  *abort_flag = 1;
  status_or(status, KVC_STATUS_TIMEOUT);
  return false;
}

// The same wait by polling without suspension, for the MMA issuer's waits on the critical path
// (a key stage landing, a TMEM slot coming free): a suspended try_wait resumed too late there and
// left the tensor pipe idle between chunks. Bounded: gives up (abort flag, KVC_STATUS_TIMEOUT)
// after 2^26 polls (about 2 s with the 32 ns pauses), and as soon as another role has aborted.
__device__ __forceinline__ bool spin_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              int32_t* status) {
  const uint32_t a = tc::smem_u32(bar);
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(a), "r"(parity)
        : "memory");
    if (done) return true;
    if ((it & 1023u) == 1023u && *abort_flag) return false;
    __nanosleep(32);  // a short pause keeps the poll from taking issue slots from the SMSP's other warps
  }
  *abort_flag = 1;
  status_or(status, KVC_STATUS_TIMEOUT);
  return false;
}

// Tree reductions over a 32-value slice: five dependent steps instead of 32.
__device__ __forceinline__ float tree_max32(const float (&x)[32]) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = fmaxf(x[i], x[i + 16]);
#pragma unroll
  for (int w = 8; w; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] = fmaxf(a[i], a[i + w]);
  return a[0];
}
__device__ __forceinline__ float tree_sum32(const float (&x)[32]) {
  float a[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = x[i] + x[i + 16];
#pragma unroll
  for (int w = 8; w; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) a[i] += a[i + w];
  return a[0];
}

// max of three (a NaN operand is ignored, as with fmaxf)
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// max of 32 values with three-input max steps: 17 instructions instead of 31
__device__ __forceinline__ float tree_max32_3(const float (&x)[32]) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3f(x[3 * i], x[3 * i + 1], x[3 * i + 2]);
  a[10] = fmaxf(x[30], x[31]);
  const float b0 = max3f(a[0], a[1], a[2]), b1 = max3f(a[3], a[4], a[5]), b2 = max3f(a[6], a[7], a[8]);
  return fmaxf(max3f(b0, b1, b2), fmaxf(a[9], a[10]));
}

__device__ __forceinline__ float ex2_approx(float x) {  // MUFU.EX2; relative error about 2^-22
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// merge two (max, sum-of-exp2) states
__device__ __forceinline__ float2 lse_merge(float2 x, float2 y) {
  if (y.y <= 0.f) return x;
  if (x.y <= 0.f) return y;
  const float m = fmaxf(x.x, y.x);
  return make_float2(m, x.y * exp2f(x.x - m) + y.y * exp2f(y.x - m));
}

// Tensor maps over the K cache (per layer) and the observation rows (a box of qrows rows); false
// if encoding fails.
bool fused_maps(FusedMaps* m, const ScoreArgs& a, const ScoreWs& ws, int qrows = 128);

}  // namespace kvc
