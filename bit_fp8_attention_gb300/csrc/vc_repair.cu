// vc_repair.cu -- V residual repair rows ("Open-VC Attention", "Why V residual repair").
//
// Without V-Smooth every value token j leaves a rounding residual r_j = s * (x_j - dec(E4M3(x_j))),
// x_j = fl32(v_j * inv) with the residual scale of the head (or of each channel). The n_rep tokens of
// largest energy sum_c r_j,c^2 become extra key rows: a copy of the token's key, quantised as extra
// 128-row key blocks, and the E4M3 code of x_j - dec(E4M3(x_j)) in the main residual codes' units.
// The forward visits these tiles after all regular ones and adds them to the numerator only.
//
// Kernels, in stream order after the residual maxima are known:
//   repair_energy_kernel  one thread per token: the energy, accumulated as fp32 fmaf in channel order
//   repair_select_kernel  one CTA per head: radix select of the n_rep largest energies (ties to the
//                         lower index), written in ascending token order
//   quant_blocks_kernel   the copied keys (gathered through the selection), as any key block
//   repair_vpack_kernel   the selected residuals' codes, transposed [D, R_pad] like the main codes
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

// The residual quantiser's reciprocal and scale for channel d: from the head maximum, or from the
// channel's own maximum when per-channel maxima are given. An all-zero range gives 1 and 1.
__device__ __forceinline__ void residual_inv_scale(const unsigned int* amax_head, const unsigned int* amax_ch, int bh,
                                                   int d, int D, float& inv, float& sc) {
  const float a = __uint_as_float(amax_ch ? amax_ch[(int64_t)bh * D + d] : amax_head[bh]);
  const bool zero = !(a > 0.f);
  inv = zero ? 1.f : __fdiv_rn(448.f, a);
  sc = zero ? 1.f : __fdiv_rn(a, 448.f);
}

// Two values in code units -> their E4M3 rounding residuals (exact: the subtraction of the nearest
// E4M3 value from x loses no bits).
__device__ __forceinline__ float2 rounding_residual2(float x0, float x1) {
  const float2 q = e4m3x2_to_f2(cvt_e4m3x2(x0, x1));
  return make_float2(__fsub_rn(x0, q.x), __fsub_rn(x1, q.y));
}

// energy[bh][t] = sum_c (s_c * (x - dec(E4M3(x))))^2, x = fl32(v[t][c] * inv_c), c = 0..D-1 in order.
template <int D>
__global__ void __launch_bounds__(128) repair_energy_kernel(const uint16_t* __restrict__ v, int S,
                                                            const unsigned int* __restrict__ amax_head,
                                                            const unsigned int* __restrict__ amax_ch,
                                                            float* __restrict__ energy) {
  const int bh = blockIdx.y, t = blockIdx.x * 128 + threadIdx.x;
  __shared__ float invs[D], scs[D];
  for (int d = threadIdx.x; d < D; d += 128) residual_inv_scale(amax_head, amax_ch, bh, d, D, invs[d], scs[d]);
  __syncthreads();
  if (t >= S) return;
  const uint4* row = reinterpret_cast<const uint4*>(v + ((int64_t)bh * S + t) * D);
  constexpr int BATCH = 8;  // 16-byte chunks loaded before any is used
  float e = 0.f;
#pragma unroll
  for (int c0 = 0; c0 < D / 8; c0 += BATCH) {
    uint4 w[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) w[b] = __ldg(row + c0 + b);
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const uint32_t* wv = reinterpret_cast<const uint32_t*>(&w[b]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int d = 8 * (c0 + b) + 2 * q;
        const float x0 = __fmul_rn(bf16_bits_to_f32(wv[q] & 0xFFFFu), invs[d]);
        const float x1 = __fmul_rn(bf16_bits_to_f32(wv[q] >> 16), invs[d + 1]);
        const float2 r = rounding_residual2(x0, x1);
        const float t0 = __fmul_rn(scs[d], r.x), t1 = __fmul_rn(scs[d + 1], r.y);
        e = __fmaf_rn(t0, t0, e);
        e = __fmaf_rn(t1, t1, e);
      }
    }
  }
  energy[(int64_t)bh * S + t] = e;
}

// Exclusive prefix count of a per-thread flag over a 1024-thread block, and the block total.
// Uses cnt[32] and base[32] in shared memory; ends with a barrier, so it can be called back to back.
__device__ __forceinline__ int block_excl_count(bool f, int* cnt, int* base, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xffffffffu, f);
  if (lane == 0) cnt[warp] = __popc(b);
  __syncthreads();
  if (warp == 0) {
    const int c = cnt[lane];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    base[lane] = incl - c;
    if (lane == 31) cnt[0] = incl;  // every warp has read its count above
  }
  __syncthreads();
  const int r = base[warp] + __popc(b & ((1u << lane) - 1u));
  total = cnt[0];
  __syncthreads();
  return r;
}

// The n largest energies of head bh (n >= 1), ties to the lower index, listed in ascending index order.
// Energies are non-negative floats, so their bit patterns order like the values: a radix select over
// four 8-bit digits from the top finds the n-th largest key T and how many keys equal to T to keep;
// one ordered pass then keeps every key above T and the first such keys equal to T.
__global__ void __launch_bounds__(1024) repair_select_kernel(const float* __restrict__ energy, int S, int n,
                                                             int32_t* __restrict__ idx) {
  const int bh = blockIdx.x, tid = threadIdx.x;
  const uint32_t* key = reinterpret_cast<const uint32_t*>(energy + (int64_t)bh * S);
  __shared__ int hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ int s_left;
  __shared__ int cnt[32], base[32];
  uint32_t prefix = 0, mask = 0;
  int left = n;  // keys still to take among those matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int t = tid; t < S; t += 1024) {
      const uint32_t k = key[t];
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int above = 0, d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= left) break;
        above += hist[d];
      }
      s_prefix = prefix | ((uint32_t)d << shift);
      s_left = left - above;
    }
    __syncthreads();
    prefix = s_prefix;
    left = s_left;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;
  int32_t* out = idx + (int64_t)bh * n;
  int taken = 0, eq_seen = 0;
  for (int c0 = 0; c0 < S; c0 += 1024) {
    const int t = c0 + tid;
    const uint32_t k = t < S ? key[t] : 0u;
    const bool eq = t < S && k == T;
    int eq_total, sel_total;
    const int eq_before = block_excl_count(eq, cnt, base, eq_total);
    const bool sel = (t < S && k > T) || (eq && eq_seen + eq_before < left);
    const int sel_before = block_excl_count(sel, cnt, base, sel_total);
    if (sel) out[taken + sel_before] = t;
    taken += sel_total;
    eq_seen += eq_total;
  }
}

// Codes of the selected tokens' rounding residuals, transposed: vrep[bh][d][i] for repair row i of
// repair tile blockIdx.x; rows past n are 0. Same thread layout as the main residual pack.
template <int D>
__global__ void __launch_bounds__(256) repair_vpack_kernel(const uint16_t* __restrict__ v,
                                                           const int32_t* __restrict__ rep_idx, int S, int n,
                                                           int R_pad, const unsigned int* __restrict__ amax_head,
                                                           const unsigned int* __restrict__ amax_ch,
                                                           uint8_t* __restrict__ vrep) {
  const int jr = blockIdx.x, bh = blockIdx.y;
  const int t0 = jr * 128, nv = min(128, n - t0);
  __shared__ __align__(16) uint16_t blk[128][D];
  __shared__ float invs[D];
  for (int d = threadIdx.x; d < D; d += 256) {
    float sc;
    residual_inv_scale(amax_head, amax_ch, bh, d, D, invs[d], sc);
  }
  gather_block<D>(blk, v + (int64_t)bh * S * D, rep_idx + (int64_t)bh * n, t0, nv);
  __syncthreads();
  uint8_t* out = vrep + (int64_t)bh * D * R_pad + t0;
  for (int task = threadIdx.x; task < D * 4; task += 256) {
    const int d = task % D, seg = task / D;  // rows [32 seg, 32 seg + 32) of channel d
    const float inv = invs[d];
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = seg * 32 + 4 * q + 2 * h;
        const float x0 = r < nv ? __fmul_rn(bf16_bits_to_f32(blk[r][d]), inv) : 0.f;
        const float x1 = r + 1 < nv ? __fmul_rn(bf16_bits_to_f32(blk[r + 1][d]), inv) : 0.f;
        const float2 res = rounding_residual2(x0, x1);
        word |= cvt_e4m3x2(res.x, res.y) << (16 * h);
      }
      w[q] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)d * R_pad + seg * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

}  // namespace

int repair_launch(const PlanBuffers& p, const uint16_t* K, const uint16_t* V, const uint16_t* kcen, cudaStream_t st) {
  if (p.nrep <= 0) return VC_OK;
  const int BH = p.B * p.H, S = p.S, D = p.D;
  const unsigned int* ach = p.has_vchannel ? p.vamax_ch : nullptr;
  const dim3 ge((S + 127) / 128, BH), gv(p.nrt, BH);
  if (D == 128) repair_energy_kernel<128><<<ge, 128, 0, st>>>(V, S, p.vamax, ach, p.energy);
  else repair_energy_kernel<64><<<ge, 128, 0, st>>>(V, S, p.vamax, ach, p.energy);
  repair_select_kernel<<<BH, 1024, 0, st>>>(p.energy, S, p.nrep, p.rep_idx);
  quant_blocks_launch(K, p.rep_idx, kcen, D, p.nrep, p.R_pad, S, BH, p.krep, p.krep_scales, st, p.has_hadamard);
  if (D == 128) repair_vpack_kernel<128><<<gv, 256, 0, st>>>(V, p.rep_idx, S, p.nrep, p.R_pad, p.vamax, ach, p.vrep);
  else repair_vpack_kernel<64><<<gv, 256, 0, st>>>(V, p.rep_idx, S, p.nrep, p.R_pad, p.vamax, ach, p.vrep);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace vc
