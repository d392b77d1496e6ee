// vc_fwd.cu -- the fused ExpCast-FP8 + V-Smooth attention forward for sm_103a.
//
// "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention": Sec. 3.1 Eq. 1
// (online softmax), Sec. 3.2 Eq. 6 (online mean restoration A <- alpha A + P~ R_q + r mu^T),
// Sec. 3.3 Eq. 7 (ExpCast-FP8); "Open-VC Attention" (MachGen blog), "Scheduling around ExpCast":
// one FMA per score with all scales and the running max folded in, running max on the true
// score with every increase applied, row sum of the decoded FP8 probabilities that feed PV,
// mid-window key order, packed transposed V.
//
// GB300 design (not the pages' kernel): one CTA per 128-row query tile and batch-head.
//   warp 4      TMA producer: Q once; K' and V^T tiles of 128 keys into 3-stage rings; with
//               V-Smooth, the transposed bf16 means of each 16-tile block run into a 2-stage ring.
//   warp 5      MMA issuer (one thread): S = Q K'^T (kind::f8f6f4, SS) into one of two TMEM score
//               buffers; O += P V and W += P E_{j mod 16} (TS: the codes P are read from TMEM),
//               where E_s is a one-hot 16 x 128 block, so column j mod 16 of W receives the exact
//               row sum of tile j; at the end of each run of tiles from one 16-tile block, the
//               mean term O += F M^T (kind::f16, F = W / sV split into bf16 hi + lo, M the block's
//               16 means) -- Eq. 6's r mu^T for 16 tiles at once, in the same accumulator.
//   warps 0-3   softmax, one thread per query row: tile max on the raw scores, true-score max in
//               code units, O/W rescale on every increase, E4M3 codes written into TMEM.
// TMEM columns: O [0, D), W [D, D+16), F [D+16, D+32), P [160, 192) and [192, 224), score
// buffers S [256, 384) and [384, 512).  P has its own columns so that the commit of S(p+2), which
// tracks every earlier MMA, also proves that PV(p) has finished reading P(p).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {

constexpr uint32_t kWaitLimit = 1u << 20;
constexpr float kB0 = 119.65f;             // 8*8 + 56 + beta, beta = -0.35
constexpr float kFastMaxAbsM = 1048576.f;  // |M| below 2^20 code units: the one-FMA code is <= 120

template <int D>
struct FwdCfg {
  static constexpr int NK = 3, NV = 3, NMU = 2;
  static constexpr int QB = 128 * D;  // bytes of a Q or K tile (128 rows x D codes)
  static constexpr int VB = D * 128;  // bytes of a V^T tile (D rows x 128 keys)
  static constexpr int MUB = D * 32;  // bytes of a mean block (D rows x 16 bf16)
  static constexpr uint32_t QK_LAYOUT = D == 128 ? kSw128 : kSw64;
  static constexpr uint32_t QK_SBO = 8 * D;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + NK * QB;
  static constexpr int OFF_ONE = OFF_V + NV * VB;
  static constexpr int OFF_MU = OFF_ONE + 16 * 2048;
  static constexpr int OFF_BAR = OFF_MU + NMU * MUB;
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 * NMU + 2 + 2 + 2 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + slack for aligning the base to 1024
  static constexpr uint32_t T_O = 0, T_W = D, T_F = D + 16, T_P0 = 160, T_P1 = 192, T_S0 = 256, T_S1 = 384;
};

struct FwdArgs {
  const float* qscales;
  const float* kscales;
  const float* vscales;
  uint16_t* out;
  int* status;
  int S, S_pad, nkb;
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
// Equals clip[0,120](rne(fmaf(s, a, b))) whenever y < 120.5; the forward only calls it when the
// running max keeps y below that (|M| < 2^20), and the single-score export clamps at 120 after it.
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

// Reference form of one code, used when |M| is too large for the fast path.
__device__ __forceinline__ uint32_t expcast_code(float s, float a, float b) {
  float r = rintf(__fmaf_rn(s, a, b));
  r = fminf(fmaxf(r, 0.f), 120.f);
  return (uint32_t)r;
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

// Single-score export: the forward's four-score code path, clamped at 120 afterwards so that it
// matches the clip of Eq. 7 for every input (the forward never needs the clamp).
__global__ void expcast_kernel(const float* __restrict__ s, const float* __restrict__ a, const float* __restrict__ b,
                               int64_t n, uint8_t* __restrict__ out) {
  int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i0 >= n) return;
  float sv[4], av[4], bv[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    int64_t i = i0 + q < n ? i0 + q : i0;
    sv[q] = s[i];
    av[q] = a[i];
    bv[q] = b[i];
  }
  uint32_t d = expcast4(sv[0], sv[1], sv[2], sv[3], pack2f(av[0], av[1]), pack2f(av[2], av[3]), pack2f(bv[0], bv[1]),
                        pack2f(bv[2], bv[3]));
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (i0 + q < n) out[i0 + q] = (uint8_t)min((d >> (8 * q)) & 0xFFu, 120u);
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

template <int D>
__global__ void __launch_bounds__(192, 1) vc_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base + C::OFF_Q;
  uint8_t* sK = base + C::OFF_K;
  uint8_t* sV = base + C::OFF_V;
  uint8_t* sOne = base + C::OFF_ONE;
  uint8_t* sMu = base + C::OFF_MU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* mu_full = v_empty + C::NV;
  uint64_t* mu_empty = mu_full + C::NMU;
  uint64_t* s_full = mu_empty + C::NMU;
  uint64_t* p_full = s_full + 2;
  // o_done[t & 1] completes when PV(t) and every earlier MMA are done. Two barriers alternating by
  // tile: when the softmax waits for tile t, the same barrier's previous tile t-2 is known to be
  // complete, so the barrier is never two phases away from the one waited for (parity waits only
  // tell the current phase from the previous one).
  uint64_t* o_done = p_full + 2;
  uint64_t* f_full = o_done + 2;
  uint64_t* drain = f_full + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + C::OFF_MISC + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int nkb = args.nkb;
  const int start = (args.flags & VC_MIDWINDOW) ? min(nkb - 1, qt + 2) : -1;
  const bool use_mean = args.use_mean != 0;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < C::NV; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int s = 0; s < C::NMU; ++s) { mbar_init(&mu_full[s], 1); mbar_init(&mu_empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&s_full[b], 1); mbar_init(&p_full[b], 128); }
    mbar_init(&o_done[0], 1);
    mbar_init(&o_done[1], 1);
    mbar_init(f_full, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // One-hot blocks E_s (16 rows x 128 keys, 128-byte swizzled rows): row s holds E4M3 1.0.
  // A constant row is invariant under the 16-byte chunk swizzle, so it is written in place.
  for (int i = tid; i < 16 * 128; i += blockDim.x) {
    int blk = i >> 7, row = (i & 127) >> 3;
    uint32_t v = (row == blk) ? 0x38383838u : 0u;
    reinterpret_cast<uint4*>(sOne)[i] = make_uint4(v, v, v, v);
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      prefetch_tmap(&maps.v);
      if (use_mean) prefetch_tmap(&maps.mu);
      const int row0 = bh * args.S_pad;
      mbar_arrive_expect_tx(q_full, C::QB);
      tma_load_2d(sQ, &maps.q, 0, row0 + qt * 128, q_full);
      int issued_k = 0, issued_v = 0, issued_mu = 0;
      // The means of a block run are loaded when the run ends, just before the next run's first K
      // tile: the ring stage they reuse was released by the mean MMA of the run two back, which the
      // MMA thread issues before it can ever wait for that K tile.
      auto load_mean_block = [&](int block) -> bool {
        const int q = issued_mu, sm = q % C::NMU;
        if (!wait_or_abort(&mu_empty[sm], ((q / C::NMU) & 1) ^ 1, kWaitLimit, abort_flag)) return false;
        mbar_arrive_expect_tx(&mu_full[sm], C::MUB);
        tma_load_2d(sMu + sm * C::MUB, &maps.mu, block * 16, bh * D, &mu_full[sm]);
        issued_mu = q + 1;
        return true;
      };
      bool loads_ok = true;
      for (int p = 0; p < nkb; ++p) {
        if (*abort_flag) { loads_ok = false; break; }
        const int j = tile_at(p, start);
        if (use_mean && p > 0 && seg_start(p, start) && !load_mean_block(tile_at(p - 1, start) >> 4)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          loads_ok = false;
          break;
        }
        const int s = p % C::NK;
        if (!wait_or_abort(&k_empty[s], ((p / C::NK) & 1) ^ 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          loads_ok = false;
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], C::QB);
        tma_load_2d(sK + s * C::QB, &maps.k, 0, row0 + j * 128, &k_full[s]);
        issued_k = p + 1;
        const int sv = p % C::NV;
        if (!wait_or_abort(&v_empty[sv], ((p / C::NV) & 1) ^ 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          loads_ok = false;
          break;
        }
        mbar_arrive_expect_tx(&v_full[sv], C::VB);
        tma_load_2d(sV + sv * C::VB, &maps.v, j * 128, bh * D, &v_full[sv]);
        issued_v = p + 1;
      }
      if (use_mean && loads_ok && !load_mean_block(tile_at(nkb - 1, start) >> 4))  // the last run
        record_failure(args.status, abort_flag, kStatusTimeoutLoad);
      // Teardown: confirm that every load issued into this CTA's shared memory has landed.
      bool ok = mbar_wait(q_full, 0, kWaitLimit);
      for (int p = max(0, issued_k - C::NK); p < issued_k; ++p)
        ok &= mbar_wait(&k_full[p % C::NK], (p / C::NK) & 1, kWaitLimit);
      for (int p = max(0, issued_v - C::NV); p < issued_v; ++p)
        ok &= mbar_wait(&v_full[p % C::NV], (p / C::NV) & 1, kWaitLimit);
      for (int q = max(0, issued_mu - C::NMU); q < issued_mu; ++q)
        ok &= mbar_wait(&mu_full[q % C::NMU], (q / C::NMU) & 1, kWaitLimit);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tO = tmem + C::T_O, tW = tmem + C::T_W, tF = tmem + C::T_F;
      const uint32_t tS0 = tmem + C::T_S0, tS1 = tmem + C::T_S1, tP0 = tmem + C::T_P0, tP1 = tmem + C::T_P1;
      constexpr uint32_t id_qk = idesc_e4m3(128, 128), id_pv = idesc_e4m3(128, D), id_w = idesc_e4m3(128, 16);
      constexpr uint32_t id_mu = idesc_bf16(128, D);
      auto issue_qk = [&](int p) -> bool {
        const int s = p % C::NK;
        if (!wait_or_abort(&k_full[s], (p / C::NK) & 1, kWaitLimit, abort_flag)) return false;
        tc_fence_after();
        const uint32_t dst = (p & 1) ? tS1 : tS0;
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          mma_e4m3_ss(dst, smem_desc(sQ + 32 * kk, C::QK_SBO, C::QK_LAYOUT),
                      smem_desc(sK + s * C::QB + 32 * kk, C::QK_SBO, C::QK_LAYOUT), id_qk, kk > 0);
        mma_commit(&s_full[p & 1]);
        mma_commit(&k_empty[s]);
        return true;
      };
      // O += F M^T for the block run with ordinal q: two K=16 bf16 MMAs, hi then lo.
      auto issue_mean = [&](int q) -> bool {
        const int sm = q % C::NMU;
        if (!wait_or_abort(&mu_full[sm], (q / C::NMU) & 1, kWaitLimit, abort_flag)) return false;
        tc_fence_after();
        const uint64_t bdesc = smem_desc(sMu + sm * C::MUB, 256, kSw32);
        mma_bf16_ts(tO, tF, bdesc, id_mu, 1);
        mma_bf16_ts(tO, tF + 8, bdesc, id_mu, 1);
        mma_commit(&mu_empty[sm]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, kWaitLimit);
      if (ok) ok = issue_qk(0);
      if (ok && nkb > 1) ok = issue_qk(1);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutLoad);
      int seg = -1;  // ordinal of the current block run
      for (int p = 0; ok && p < nkb; ++p) {
        if (*abort_flag) { ok = false; break; }
        const int b = p & 1;
        if (!wait_or_abort(&p_full[b], (p >> 1) & 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutP);
          ok = false;
          break;
        }
        const bool fresh = seg_start(p, start);
        if (fresh) {
          if (use_mean && seg >= 0 && !issue_mean(seg)) {
            record_failure(args.status, abort_flag, kStatusTimeoutLoad);
            ok = false;
            break;
          }
          ++seg;
        }
        const int sv = p % C::NV;
        if (!wait_or_abort(&v_full[sv], (p / C::NV) & 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tP = b ? tP1 : tP0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_e4m3_ts(tO, tP + 8 * kk, smem_desc(sV + sv * C::VB + 32 * kk, 1024, kSw128), id_pv,
                      (p > 0 || kk > 0));
        const uint8_t* one = sOne + (tile_at(p, start) & 15) * 2048;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_e4m3_ts(tW, tP + 8 * kk, smem_desc(one + 32 * kk, 1024, kSw128), id_w, (!fresh || kk > 0));
        mma_commit(&o_done[p & 1]);
        mma_commit(&v_empty[sv]);
        if (p + 2 < nkb && !issue_qk(p + 2)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          ok = false;
          break;
        }
      }
      if (ok && use_mean && !*abort_flag) {  // the last block run: its F arrives after the loop
        if (!wait_or_abort(f_full, 0, kWaitLimit, abort_flag) || !issue_mean(seg))
          record_failure(args.status, abort_flag, kStatusTimeoutP);
        else
          mma_commit(&o_done[nkb & 1]);  // as if it were tile nkb
      }
      // Teardown: every MMA this thread issued has completed before TMEM is released.
      mma_commit(drain);
      if (!mbar_wait(drain, 0, kWaitLimit)) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps 0-3
    const int row = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + C::T_O, tW = tmem + lane_base + C::T_W, tF = tmem + lane_base + C::T_F;
    const uint32_t tS0 = tmem + lane_base + C::T_S0, tS1 = tmem + lane_base + C::T_S1;
    const uint32_t tP0 = tmem + lane_base + C::T_P0, tP1 = tmem + lane_base + C::T_P1;
    const float* skh = args.kscales + (int64_t)bh * nkb;
    const float aq = args.code_scale * args.qscales[(int64_t)bh * nkb + qt];
    const float sv = args.vscales[bh];
    const float inv_sv = 1.f / sv;
    const bool expcast = (args.flags & VC_EXPCAST) != 0;
    const int tail_valid = args.S - (nkb - 1) * 128;
    float M = -INFINITY, l = 0.f;
    bool ok = true;
    float sk_next = skh[tile_at(0, start)];

    // PV(t) and everything before it done. Only called for t = p-1 at tile p (or t = nkb-1, nkb at
    // the end), when tile t-2 is already known to be complete.
    auto wait_o = [&](int t) -> bool {
      if (!warp_wait(&o_done[t & 1], (t >> 1) & 1, kWaitLimit, abort_flag)) {
        record_failure(args.status, abort_flag, kStatusTimeoutO);
        return false;
      }
      tc_fence_after();
      return true;
    };
    auto read_w = [&](float(&w)[16]) {
      uint32_t wr[16];
      tmem_ld16(tW, wr);
      tmem_wait_ld();
#pragma unroll
      for (int s = 0; s < 16; ++s) w[s] = __uint_as_float(wr[s]);
    };

    for (int p = 0; p < nkb; ++p) {
      if (warp_aborted(abort_flag)) { ok = false; break; }
      const int j = tile_at(p, start);
      const int b = p & 1;
      const uint32_t tS = b ? tS1 : tS0, tP = b ? tP1 : tP0;
      const float sk = sk_next;
      if (p + 1 < nkb) sk_next = skh[tile_at(p + 1, start)];
      // A new block run: the previous run's row sums (complete once PV(p-1) is done) leave W.
      const bool flush = p > 0 && seg_start(p, start);
      bool o_ready = false;
      float w[16];
      if (flush) {
        if (!wait_o(p - 1)) { ok = false; break; }
        o_ready = true;
        read_w(w);
        float ws = 0.f;
#pragma unroll
        for (int s = 0; s < 16; ++s) ws += w[s];
        l += ws;
      }
      const uint32_t lim = (p == 0 && (args.flags & VC_DEBUG_TIMEOUT)) ? 0u : kWaitLimit;
      if (!warp_wait(&s_full[b], (p >> 1) & 1, lim, abort_flag)) {
        record_failure(args.status, abort_flag, kStatusTimeoutS);
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tmem_wait_ld();
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      if (j == nkb - 1 && tail_valid < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= tail_valid) s[c] = -INFINITY;
      }
      // Row max of the raw scores: eight independent chains, then a short tree.
      float m8[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        float x = max3f(s[16 * g], s[16 * g + 1], s[16 * g + 2]);
#pragma unroll
        for (int c = 3; c < 15; c += 2) x = max3f(x, s[16 * g + c], s[16 * g + c + 1]);
        m8[g] = fmaxf(x, s[16 * g + 15]);
      }
      const float mx = fmaxf(max3f(m8[0], m8[1], m8[2]), max3f(max3f(m8[3], m8[4], m8[5]), m8[6], m8[7]));
      const float aj = aq * sk;
      const float t = mx * aj;  // = max_c fl(s_c * a_j): rounding is monotone and a_j > 0
      const float Mn = fmaxf(M, t);
      const bool inc = (Mn > M) && (M > -INFINITY);
      float alpha = 1.f;
      if (__any_sync(0xffffffffu, inc)) {
        if (p > 0 && !o_ready) {
          if (!wait_o(p - 1)) { ok = false; break; }
          o_ready = true;
        }
        alpha = inc ? ex2_approx(__fmul_rn(__fsub_rn(M, Mn), 0.125f)) : 1.f;
        l *= alpha;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + c0, o);
        }
        if (!flush) {  // a flushed W is about to be overwritten by this tile's row sums
          uint32_t wr[16];
          tmem_ld16(tW, wr);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) wr[i] = __float_as_uint(__uint_as_float(wr[i]) * alpha);
          tmem_st16(tW, wr);
        }
      }
      if (flush && use_mean) store_flush_operand(tF, w, inv_sv * alpha);
      M = Mn;
      const float bb = __fsub_rn(kB0, M);
      uint32_t pk[32];
      if (expcast && __all_sync(0xffffffffu, fabsf(M) < kFastMaxAbsM)) {
        const uint64_t a2 = pack2f(aj, aj), b2 = pack2f(bb, bb);
#pragma unroll
        for (int g = 0; g < 32; ++g)
          pk[g] = expcast4(s[4 * g], s[4 * g + 1], s[4 * g + 2], s[4 * g + 3], a2, a2, b2, b2);
      } else if (expcast) {
#pragma unroll
        for (int g = 0; g < 32; ++g)
          pk[g] = pack4(expcast_code(s[4 * g], aj, bb), expcast_code(s[4 * g + 1], aj, bb),
                        expcast_code(s[4 * g + 2], aj, bb), expcast_code(s[4 * g + 3], aj, bb));
      } else {
#pragma unroll
        for (int g = 0; g < 32; ++g)
          pk[g] = pack4(expcast_off_code(s[4 * g], aj, bb), expcast_off_code(s[4 * g + 1], aj, bb),
                        expcast_off_code(s[4 * g + 2], aj, bb), expcast_off_code(s[4 * g + 3], aj, bb));
      }
      tmem_st32(tP, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }

    if (ok && !warp_aborted(abort_flag) && wait_o(nkb - 1)) {
      float w[16];
      read_w(w);
      float ws = 0.f;
#pragma unroll
      for (int s = 0; s < 16; ++s) ws += w[s];
      l += ws;
      bool ready = true;
      if (use_mean) {  // the last block run's mean term, then the accumulator is final
        store_flush_operand(tF, w, inv_sv);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(f_full);
        ready = wait_o(nkb);
      }
      if (ready) {
        const float scale = sv / l;
        const int64_t qrow = (int64_t)qt * 128 + row;
        uint16_t* orow = args.out + ((int64_t)bh * args.S + qrow) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h2 =
                __floats2bfloat162_rn(__uint_as_float(o[2 * i]) * scale, __uint_as_float(o[2 * i + 1]) * scale);
            packed[i] = *reinterpret_cast<uint32_t*>(&h2);
          }
          if (qrow < args.S) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

static int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows,
                     uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return VC_ERR_CUDA;
  cuuint64_t gd[2] = {inner, rows};
  cuuint64_t gs[1] = {pitch_bytes};
  cuuint32_t bd[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, base, gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VC_OK : VC_ERR_CUDA;
}

int encode_fwd_maps(const PlanBuffers& p, FwdMaps* maps) {
  const uint64_t BH = (uint64_t)p.B * p.H;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle qsw = p.D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  int rc = encode_2d(&maps->q, u8, p.qcodes, p.D, BH * p.S_pad, p.D, p.D, 128, qsw);
  if (rc == VC_OK) rc = encode_2d(&maps->k, u8, p.kcodes, p.D, BH * p.S_pad, p.D, p.D, 128, qsw);
  if (rc == VC_OK)
    rc = encode_2d(&maps->v, u8, p.vcodes, p.S_pad, BH * p.D, p.S_pad, 128, p.D, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == VC_OK)
    rc = encode_2d(&maps->mu, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.meansT, p.nkb16, BH * p.D, (uint64_t)p.nkb16 * 2,
                   16, p.D, CU_TENSOR_MAP_SWIZZLE_32B);
  return rc;
}

template <int D>
static int launch_fwd(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  using C = FwdCfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(vc_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
      return VC_ERR_CUDA;
    attr_set = true;
  }
  FwdArgs a;
  a.qscales = p.qscales;
  a.kscales = p.kscales;
  a.vscales = p.vscales;
  a.out = O;
  a.status = p.status;
  a.S = p.S;
  a.S_pad = p.S_pad;
  a.nkb = p.nkb;
  a.flags = flags;
  a.code_scale = (float)(8.0 * 1.4426950408889634 / __builtin_sqrt((double)D));
  a.use_mean = (p.has_means && (flags & VC_VSMOOTH)) ? 1 : 0;
  dim3 grid(p.nkb, p.B * p.H);
  vc_fwd_kernel<D><<<grid, 192, C::SMEM, st>>>(maps, a);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

int forward_launch(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  return p.D == 128 ? launch_fwd<128>(p, maps, O, flags, st) : launch_fwd<64>(p, maps, O, flags, st);
}

int expcast_launch(const float* s, const float* a, const float* b, int64_t n, uint8_t* out, cudaStream_t st) {
  if (n <= 0) return VC_OK;
  const int64_t threads = (n + 3) / 4;
  expcast_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(s, a, b, n, out);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace vc
