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
//   warp 4      TMA producer: Q once, then K' and V^T tiles of 128 keys into 3-stage rings.
//   warp 5      MMA issuer (one thread): S = Q K'^T (kind::f8f6f4, SS) into one of two TMEM
//               score buffers, then O += P V (TS: P read from TMEM where the softmax wrote it) and
//               W += P E_s, where E_s is a one-hot 16 x 128 block: column s = p mod 16 of the TMEM
//               block W receives the exact row sum r_j of tile p on the tensor core.
//   warps 0-3   softmax, one thread per query row: tile max on the raw scores, true-score max in
//               code units, O/W rescale on every increase, E4M3 codes written back into TMEM.
//               Every 16 tiles the 16 row sums in W are folded into l and, with V-Smooth, the
//               rank-16 mean term sum_s W_s mu_{j_s}^T / sV is added to O.
// TMEM columns: O [0, D), W [D, D+16), score buffers [256, 384) and [384, 512); the codes of P
// overwrite the first 32 columns of their score buffer (four E4M3 per 32-bit column).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {

constexpr uint32_t kWaitLimit = 1u << 20;
constexpr float kB0 = 119.65f;  // 8*8 + 56 + beta, beta = -0.35

template <int D>
struct FwdCfg {
  static constexpr int NK = 3, NV = 3;
  static constexpr int QB = 128 * D;  // bytes of a Q or K tile (128 rows x D codes)
  static constexpr int VB = D * 128;  // bytes of a V^T tile (D rows x 128 keys)
  static constexpr uint32_t QK_LAYOUT = D == 128 ? kSw128 : kSw64;
  static constexpr uint32_t QK_SBO = 8 * D;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + NK * QB;
  static constexpr int OFF_ONE = OFF_V + NV * VB;
  static constexpr int OFF_BAR = OFF_ONE + 16 * 2048;
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 2 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + slack for aligning the base to 1024
  static constexpr uint32_t T_O = 0, T_W = D, T_S0 = 256, T_S1 = 384;
};

struct FwdArgs {
  const float* qscales;
  const float* kscales;
  const float* vscales;
  const uint16_t* means;
  uint16_t* out;
  int* status;
  int S, S_pad, nkb;
  unsigned flags;
  float code_scale;
  int use_mean;
};

// Position p of the visit order -> key tile index.
__device__ __forceinline__ int tile_at(int p, int start) { return p <= start ? start - p : p; }

// ExpCast-FP8 code of one score: clip[0,120](rne(fmaf(s, a, b))).
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

__global__ void expcast_kernel(const float* __restrict__ s, const float* __restrict__ a, const float* __restrict__ b,
                               int64_t n, uint8_t* __restrict__ out) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = (uint8_t)expcast_code(s[i], a[i], b[i]);
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
__device__ __forceinline__ bool warp_aborted(volatile int* abort_flag) { return __any_sync(0xffffffffu, *abort_flag != 0); }

template <int D>
__global__ void __launch_bounds__(192, 1) vc_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base + C::OFF_Q;
  uint8_t* sK = base + C::OFF_K;
  uint8_t* sV = base + C::OFF_V;
  uint8_t* sOne = base + C::OFF_ONE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* s_full = v_empty + C::NV;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* drain = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + C::OFF_MISC + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int nkb = args.nkb;
  const int start = (args.flags & VC_MIDWINDOW) ? min(nkb - 1, qt + 2) : -1;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < C::NV; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&s_full[b], 1); mbar_init(&p_full[b], 128); }
    mbar_init(o_done, 1);
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
      const int row0 = bh * args.S_pad;
      mbar_arrive_expect_tx(q_full, C::QB);
      tma_load_2d(sQ, &maps.q, 0, row0 + qt * 128, q_full);
      int issued_k = 0, issued_v = 0;
      for (int p = 0; p < nkb; ++p) {
        if (*abort_flag) break;
        const int j = tile_at(p, start);
        const int s = p % C::NK;
        if (!wait_or_abort(&k_empty[s], ((p / C::NK) & 1) ^ 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          break;
        }
        mbar_arrive_expect_tx(&k_full[s], C::QB);
        tma_load_2d(sK + s * C::QB, &maps.k, 0, row0 + j * 128, &k_full[s]);
        issued_k = p + 1;
        const int sv = p % C::NV;
        if (!wait_or_abort(&v_empty[sv], ((p / C::NV) & 1) ^ 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          break;
        }
        mbar_arrive_expect_tx(&v_full[sv], C::VB);
        tma_load_2d(sV + sv * C::VB, &maps.v, j * 128, bh * D, &v_full[sv]);
        issued_v = p + 1;
      }
      // Teardown: confirm that every load issued into this CTA's shared memory has landed.
      bool ok = mbar_wait(q_full, 0, kWaitLimit);
      for (int p = max(0, issued_k - C::NK); p < issued_k; ++p)
        ok &= mbar_wait(&k_full[p % C::NK], (p / C::NK) & 1, kWaitLimit);
      for (int p = max(0, issued_v - C::NV); p < issued_v; ++p)
        ok &= mbar_wait(&v_full[p % C::NV], (p / C::NV) & 1, kWaitLimit);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tO = tmem + C::T_O, tW = tmem + C::T_W;
      const uint32_t tS0 = tmem + C::T_S0, tS1 = tmem + C::T_S1;
      constexpr uint32_t id_qk = idesc_e4m3(128, 128), id_pv = idesc_e4m3(128, D), id_w = idesc_e4m3(128, 16);
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
      bool ok = mbar_wait(q_full, 0, kWaitLimit);
      if (ok) ok = issue_qk(0);
      if (ok && nkb > 1) ok = issue_qk(1);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutLoad);
      for (int p = 0; ok && p < nkb; ++p) {
        if (*abort_flag) break;
        const int b = p & 1;
        if (!wait_or_abort(&p_full[b], (p >> 1) & 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutP);
          break;
        }
        const int sv = p % C::NV;
        if (!wait_or_abort(&v_full[sv], (p / C::NV) & 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          break;
        }
        tc_fence_after();
        const uint32_t tP = b ? tS1 : tS0;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_e4m3_ts(tO, tP + 8 * kk, smem_desc(sV + sv * C::VB + 32 * kk, 1024, kSw128), id_pv, (p > 0 || kk > 0));
        const uint8_t* one = sOne + (p & 15) * 2048;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_e4m3_ts(tW, tP + 8 * kk, smem_desc(one + 32 * kk, 1024, kSw128), id_w, ((p & 15) != 0 || kk > 0));
        mma_commit(o_done);
        mma_commit(&v_empty[sv]);
        if (p + 2 < nkb && !issue_qk(p + 2)) {
          record_failure(args.status, abort_flag, kStatusTimeoutLoad);
          break;
        }
      }
      // Teardown: every MMA this thread issued has completed before TMEM is released.
      mma_commit(drain);
      if (!mbar_wait(drain, 0, kWaitLimit)) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------------ softmax warps 0-3
    const int row = tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + C::T_O, tW = tmem + lane_base + C::T_W;
    const uint32_t tS0 = tmem + lane_base + C::T_S0, tS1 = tmem + lane_base + C::T_S1;
    const float* skh = args.kscales + (int64_t)bh * nkb;
    const float aq = args.code_scale * args.qscales[(int64_t)bh * nkb + qt];
    const float sv = args.vscales[bh];
    const float inv_sv = 1.f / sv;
    const uint16_t* mu_h = args.means + (int64_t)bh * nkb * D;
    const bool expcast = (args.flags & VC_EXPCAST) != 0;
    const int tail_valid = args.S - (nkb - 1) * 128;
    float M = -INFINITY, l = 0.f;
    bool ok = true;

    auto wait_o = [&](int p) -> bool {
      if (!warp_wait(o_done, p & 1, kWaitLimit, abort_flag)) {
        record_failure(args.status, abort_flag, kStatusTimeoutO);
        return false;
      }
      tc_fence_after();
      return true;
    };
    // Fold the row sums of tiles at positions q0 .. q0+cnt-1 (held in W) into l and, with
    // V-Smooth, add sum_s W_s mu_{j_s} / sV to the accumulator (rank-cnt update on CUDA cores).
    auto flush = [&](int q0, int cnt) {
      uint32_t wr[16];
      tmem_ld16(tW, wr);
      tmem_wait_ld();
      float wsum = 0.f;
#pragma unroll
      for (int s = 0; s < 16; ++s) wsum += __uint_as_float(wr[s]);
      l += wsum;
      if (args.use_mean) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c0, o);
          tmem_wait_ld();
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(o[i]);
#pragma unroll
          for (int s = 0; s < 16; ++s) {
            if (s >= cnt) break;
            const float ws = __uint_as_float(wr[s]) * inv_sv;
            const uint4* m4 = reinterpret_cast<const uint4*>(mu_h + (int64_t)tile_at(q0 + s, start) * D + c0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 mv = __ldg(m4 + q);
              const uint32_t* mw = reinterpret_cast<const uint32_t*>(&mv);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                acc[8 * q + 2 * h] = fmaf(ws, __uint_as_float(mw[h] << 16), acc[8 * q + 2 * h]);
                acc[8 * q + 2 * h + 1] = fmaf(ws, __uint_as_float(mw[h] & 0xFFFF0000u), acc[8 * q + 2 * h + 1]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(acc[i]);
          tmem_st32(tO + c0, o);
        }
        tmem_wait_st();
      }
    };

    for (int p = 0; p < nkb; ++p) {
      if (warp_aborted(abort_flag)) { ok = false; break; }
      const int j = tile_at(p, start);
      const int b = p & 1;
      const uint32_t tS = b ? tS1 : tS0;
      bool o_ready = false;
      if (p > 0 && (p & 15) == 0) {  // chunk p-16 .. p-1 complete once PV(p-1) is done
        if (!wait_o(p - 1)) { ok = false; break; }
        o_ready = true;
        flush(p - 16, 16);
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
      float mx = s[0];
#pragma unroll
      for (int c = 1; c + 1 < 128; c += 2) mx = max3f(mx, s[c], s[c + 1]);
      mx = fmaxf(mx, s[127]);
      const float aj = aq * skh[j];
      const float t = mx * aj;  // = max_c fl(s_c * a_j): rounding is monotone and a_j > 0
      const float Mn = fmaxf(M, t);
      const bool inc = (Mn > M) && (M > -INFINITY);
      if (__any_sync(0xffffffffu, inc)) {
        if (p > 0 && !o_ready) {
          if (!wait_o(p - 1)) { ok = false; break; }
          o_ready = true;
        }
        const float alpha = inc ? ex2_approx(__fmul_rn(__fsub_rn(M, Mn), 0.125f)) : 1.f;
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
        uint32_t w[16];
        tmem_ld16(tW, w);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
        tmem_st16(tW, w);
        tmem_wait_st();
      }
      M = Mn;
      const float bb = __fsub_rn(kB0, M);
      uint32_t pk[32];
      if (expcast) {
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
      tmem_st32(tS, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[b]);
    }

    if (ok && !warp_aborted(abort_flag) && wait_o(nkb - 1)) {
      const int q0 = ((nkb - 1) / 16) * 16;
      flush(q0, nkb - q0);
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
          __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[2 * i]) * scale,
                                                    __uint_as_float(o[2 * i + 1]) * scale);
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

static int encode_2d(CUtensorMap* m, void* base, uint64_t inner, uint64_t rows, uint64_t pitch, uint32_t box_inner,
                     uint32_t box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return VC_ERR_CUDA;
  cuuint64_t gd[2] = {inner, rows};
  cuuint64_t gs[1] = {pitch};
  cuuint32_t bd[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? VC_OK : VC_ERR_CUDA;
}

int encode_fwd_maps(const PlanBuffers& p, FwdMaps* maps) {
  const uint64_t BH = (uint64_t)p.B * p.H;
  const CUtensorMapSwizzle qsw = p.D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  int rc = encode_2d(&maps->q, p.qcodes, p.D, BH * p.S_pad, p.D, p.D, 128, qsw);
  if (rc == VC_OK) rc = encode_2d(&maps->k, p.kcodes, p.D, BH * p.S_pad, p.D, p.D, 128, qsw);
  if (rc == VC_OK)
    rc = encode_2d(&maps->v, p.vcodes, p.S_pad, BH * p.D, p.S_pad, 128, p.D, CU_TENSOR_MAP_SWIZZLE_128B);
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
  a.means = p.means;
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
  expcast_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(s, a, b, n, out);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace vc
