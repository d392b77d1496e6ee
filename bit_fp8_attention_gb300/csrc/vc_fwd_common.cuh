// vc_fwd_common.cuh -- pieces shared by the forward kernels: launch arguments, the visit order, the
// ExpCast code paths, bounded waits and the mean operand ("VC-Attention" Sec. 3.2 Eq. 6, Sec. 3.3
// Eq. 7; "Open-VC Attention", "Scheduling around ExpCast").
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "vc_device.cuh"

namespace vc {

constexpr uint32_t kWaitLimit = 1u << 20;
constexpr float kB0 = 119.65f;             // 8*8 + 56 + beta, beta = -0.35
// Below 2^22 code units, |M| keeps y = fma(s, a, 119.65 - M) under 120.5: the rounding of s * a to the
// running max and of b each add at most half an ulp of M (<= 0.25), so no code needs the clip at 120.
constexpr float kClampFreeMaxAbsM = 4194304.f;

struct FwdArgs {
  const float* qscales;
  const float* kscales;
  const float* vscales;
  const float* vscales_ch;  // [BH, D] per-channel residual scales, or null (one scale per head)
  uint16_t* out;
  int* status;
  const float* krep_scales;  // [BH, nrt] scales of the repair key tiles
  int S, S_pad, nkb;
  int nrt, R_pad;            // repair tiles after the nkb regular ones (0: none), rows per head
  unsigned flags;
  float code_scale;
  int use_mean;
};

// Position p of the visit order -> key tile index.
__device__ __forceinline__ int tile_at(int p, int start) { return p <= start ? start - p : p; }
// Does position p open a new run of tiles from one 16-tile block?
__device__ __forceinline__ bool seg_start(int p, int start) {
  return p == 0 || (tile_at(p, start) >> 4) != (tile_at(p - 1, start) >> 4);
}

__device__ __forceinline__ uint64_t pack2f(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}

// ExpCast-FP8 codes of four scores, one code per byte (byte i from score i).
//   y = fmaf(s, a, b) two at a time (FFMA2);
//   y * 2^-149 lands in the subnormal range, where the product is rounded to a multiple of 2^-149,
//   i.e. y to the nearest integer with ties to even, and the float's bit pattern is that integer
//   with y's sign (FMUL2);
//   cvt.pack.sat.u8 reads the patterns as s32, so negative codes clamp to 0, and packs them.
// Equals clip[0,120](rne(fmaf(s, a, b))) whenever y < 120.5. Above that the code bytes only need a
// byte-wise min with 120 (y >= 2^23 leaves the subnormal range and saturates to 255 first), which
// the forward applies when |M| >= 2^22 and the single-score export always applies.
__device__ __forceinline__ uint32_t expcast4(float s0, float s1, float s2, float s3, uint64_t a01, uint64_t a23,
                                             uint64_t b01, uint64_t b23) {
  const uint64_t tiny2 = (1ull << 32) | 1ull;  // (2^-149, 2^-149)
  uint64_t y01, y23;
  asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%1, %2};\n\tfma.rn.f32x2 %0, x, %3, %4;\n\t}"
      : "=l"(y01)
      : "f"(s0), "f"(s1), "l"(a01), "l"(b01));
  asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%1, %2};\n\tfma.rn.f32x2 %0, x, %3, %4;\n\t}"
      : "=l"(y23)
      : "f"(s2), "f"(s3), "l"(a23), "l"(b23));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(y01) : "l"(tiny2));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(y23) : "l"(tiny2));
  uint32_t h, d;
  asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(h) : "r"((uint32_t)(y23 >> 32)), "r"((uint32_t)y23), "r"(0u));
  asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(d) : "r"((uint32_t)(y01 >> 32)), "r"((uint32_t)y01), "r"(h));
  return d;
}

// The conventional path: exponentiate in fp32, then a rounding E4M3 cast.
__device__ __forceinline__ uint32_t expcast_off_code(float s, float a, float b) {
  float y = __fmaf_rn(s, a, b);
  float ze = __fadd_rn(__fmul_rn(__fsub_rn(y, kB0), 0.125f), 8.f);
  return cvt_e4m3x2(exp2f(ze), 0.f) & 0xFFu;
}
__device__ __forceinline__ uint32_t pack4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3) {
  return c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
}

__device__ __forceinline__ void record_failure(int* status, volatile int* abort_flag, int bit) {
  atomicOr(status, bit);
  *abort_flag = 1;
}
// Bounded wait that also gives up as soon as another role of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, uint32_t limit,
                                              volatile int* abort_flag) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  return false;
}
// The same wait taken by a whole warp: the outcome is voted so that the warp stays converged
// before the .sync.aligned TMEM instructions that follow.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t limit, volatile int* abort_flag) {
  const bool ok = wait_or_abort(bar, parity, limit, abort_flag);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) {
  return __any_sync(0xffffffffu, *abort_flag != 0);
}

// Row sums of a 16-tile block, scaled, as the bf16 hi + lo A operand of the mean MMA.
__device__ __forceinline__ void store_flush_operand(uint32_t tF, const float (&w)[16], float scale) {
  uint32_t f[16];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const float x0 = w[2 * c] * scale, x1 = w[2 * c + 1] * scale;
    const __nv_bfloat162 hi = __floats2bfloat162_rn(x0, x1);
    const __nv_bfloat162 lo = __floats2bfloat162_rn(x0 - __low2float(hi), x1 - __high2float(hi));
    f[c] = *reinterpret_cast<const uint32_t*>(&hi);
    f[8 + c] = *reinterpret_cast<const uint32_t*>(&lo);
  }
  tmem_st16(tF, f);
}

}  // namespace vc
