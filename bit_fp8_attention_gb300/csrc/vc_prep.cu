// vc_prep.cu -- the prepare step on the GPU: per-128-token block quantisation of Q and K',
// k-means over V rows with a stable counting-sort argsort, gather of K and V by the permutation,
// bf16 block means, and the per-head residual quantisation packed transposed for the PV operand.
//
// "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention", Sec. 3.2
// ("Value-guided permutation" Eq. 3, "Block demeaning" Eq. 4, "Unbalanced clusters cost little"),
// Sec. 3.4 "Fused preprocessing"; "Open-VC Attention" (MachGen blog), "Scheduling around ExpCast"
// (one scale per 128-token Q/K block, one V scale per head) and "Packed V" ([H, D, S_pad], key
// dimension contiguous).  All of these passes are memory-bound except the k-means assignment.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {


// Round a double to bf16, to nearest even, in one step (no intermediate fp32 rounding).
static __device__ uint16_t f64_to_bf16_rne(double x) {
  uint64_t u = (uint64_t)__double_as_longlong(x);
  uint16_t sign = (uint16_t)((u >> 48) & 0x8000u);
  uint64_t mag = u & 0x7FFFFFFFFFFFFFFFull;
  if (mag == 0) return sign;
  if (mag >= 0x7FF0000000000000ull) return sign | (mag > 0x7FF0000000000000ull ? 0x7FC0 : 0x7F80);
  int e = (int)(mag >> 52) - 1023;  // unbiased exponent (normal doubles only in practice)
  uint64_t m = (mag & 0xFFFFFFFFFFFFFull) | (1ull << 52);
  if (e < -126) {
    // bf16 subnormal: value = q * 2^-133 with q = rne(x * 2^133)
    int shift = 52 - (e + 133);  // bits of m below the 2^-133 position
    if (shift > 63) return sign;
    uint64_t q = m >> shift;
    uint64_t rem = m & ((1ull << shift) - 1), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
    return sign | (uint16_t)q;  // q <= 128 (128 is the smallest normal)
  }
  uint64_t q = m >> 45;  // 8 significant bits
  uint64_t rem = m & ((1ull << 45) - 1), half = 1ull << 44;
  if (rem > half || (rem == half && (q & 1))) ++q;
  if (q == 256) { q = 128; ++e; }
  if (e > 127) return sign | 0x7F80;
  return sign | (uint16_t)(((uint32_t)(e + 127) << 7) | ((uint32_t)q - 128u));
}

// ---------------------------------------------------------------------------------------------
// Block quantiser.  One CTA per (128-token block j, batch-head bh).  Rows are read through `perm`
// when it is given (the K' = K[pi] gather), otherwise in order.  amax over the whole 128 x D
// block, scale = amax/448, code = E4M3_rne_satfinite(x * (448/amax)); pad rows get code 0.
// ---------------------------------------------------------------------------------------------
// One element of a 16-byte chunk of 8 bf16, as fp32, minus the matching centre element when centred.
template <bool kCentred>
__device__ __forceinline__ float chunk_elem(const uint4& w, const uint4& c, int i) {
  const uint32_t* wv = reinterpret_cast<const uint32_t*>(&w);
  const uint32_t* cv = reinterpret_cast<const uint32_t*>(&c);
  const int sh = (i & 1) * 16;
  float f = bf16_bits_to_f32((wv[i >> 1] >> sh) & 0xFFFFu);
  if (kCentred) f = __fsub_rn(f, bf16_bits_to_f32((cv[i >> 1] >> sh) & 0xFFFFu));
  return f;
}

// Per-128-token block E4M3 quantisation of Q (token order) or K (gathered through pi, optionally minus
// the head's channel centre): one CTA per (block, bh), amax over the valid rows, scale = amax/448,
// code = E4M3_RNE_sat(x * (448/amax)); pad rows are code 0.  Every thread issues all of its row loads
// before it uses any of them.  S rows per head are coded (perm: [BH, S] source rows); the source
// tensor holds S_src rows per head.
template <int D, bool kCentred>
__global__ void __launch_bounds__(256) quant_blocks_kernel(const uint16_t* __restrict__ x,
                                                           const int32_t* __restrict__ perm,
                                                           const uint16_t* __restrict__ center, int S, int S_pad,
                                                           int S_src, uint8_t* __restrict__ codes,
                                                           float* __restrict__ scales) {
  constexpr int CPR = D / 8;                 // 16-byte chunks per row
  constexpr int NCH = 128 * CPR / 256;       // chunks per thread
  const int j = blockIdx.x, bh = blockIdx.y;
  const int nkb = S_pad / 128;
  const uint16_t* xh = x + (int64_t)bh * S_src * D;
  const int32_t* ph = perm ? perm + (int64_t)bh * S : nullptr;
  __shared__ uint4 cen_s[CPR];
  __shared__ float red[8];
  if (kCentred && threadIdx.x < CPR)
    cen_s[threadIdx.x] = __ldg(reinterpret_cast<const uint4*>(center + (int64_t)bh * D) + threadIdx.x);
  uint4 v[NCH];
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    const int c = threadIdx.x + 256 * m;
    const int t = j * 128 + c / CPR;
    v[m] = make_uint4(0, 0, 0, 0);
    if (t < S) v[m] = *reinterpret_cast<const uint4*>(xh + (int64_t)(ph ? ph[t] : t) * D + (c % CPR) * 8);
  }
  if (kCentred) __syncthreads();
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    const int c = threadIdx.x + 256 * m;
    const uint4 cm = kCentred ? cen_s[c % CPR] : make_uint4(0, 0, 0, 0);
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(chunk_elem<kCentred>(v[m], cm, i)));
    if (j * 128 + c / CPR < S) amax = fmaxf(amax, a);  // pad rows do not count
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const bool zero = !(amax > 0.f);
  const float inv = zero ? 0.f : __fdiv_rn(448.f, amax);
  if (threadIdx.x == 0) scales[(int64_t)bh * nkb + j] = zero ? 1.f : __fdiv_rn(amax, 448.f);
  uint8_t* ch = codes + ((int64_t)bh * S_pad + (int64_t)j * 128) * D;
#pragma unroll
  for (int m = 0; m < NCH; ++m) {
    const int c = threadIdx.x + 256 * m;
    const int r = c / CPR, cc = c % CPR;
    const uint4 cm = kCentred ? cen_s[cc] : make_uint4(0, 0, 0, 0);
    uint32_t lo = 0, hi = 0;
    if (!zero && j * 128 + r < S) {
      uint32_t w[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        w[q] = cvt_e4m3x2(__fmul_rn(chunk_elem<kCentred>(v[m], cm, 2 * q), inv),
                          __fmul_rn(chunk_elem<kCentred>(v[m], cm, 2 * q + 1), inv));
      lo = w[0] | (w[1] << 16);
      hi = w[2] | (w[3] << 16);
    }
    *reinterpret_cast<uint2*>(ch + (int64_t)r * D + cc * 8) = make_uint2(lo, hi);
  }
}

// The same quantiser with each row rotated first ("VC-Attention", Sec. 3.4 "Fused preprocessing", App. B:
// the Q and K passes fuse a Hadamard rotation): the unnormalised Walsh-Hadamard transform in fp32, as
// the butterfly with stages s = 1, 2, ..., D/2 in that order, pair (x[i], x[i+s]) -> (x[i] + x[i+s],
// x[i] - x[i+s]). A thread holds 32 consecutive channels of a row, so stages 1-16 stay in its registers
// and stages 32 and up pair it with the lane holding the partner channels (lane ^ s/32, same row).
template <int D, bool kCentred>
__global__ void __launch_bounds__(256) quant_blocks_rot_kernel(const uint16_t* __restrict__ x,
                                                               const int32_t* __restrict__ perm,
                                                               const uint16_t* __restrict__ center, int S,
                                                               int S_pad, int S_src, uint8_t* __restrict__ codes,
                                                               float* __restrict__ scales) {
  constexpr int G = 4;                       // 16-byte chunks per thread and row: 32 channels
  constexpr int W = 8 * G;
  constexpr int TPR = D / W;                 // threads per row
  constexpr int RSTEP = 256 / TPR;           // rows between a thread's rows
  constexpr int RPT = 128 / RSTEP;           // rows per thread
  static_assert(32 % TPR == 0 && RPT >= 1, "a row's threads sit in consecutive lanes of one warp");
  const int j = blockIdx.x, bh = blockIdx.y;
  const int nkb = S_pad / 128;
  const uint16_t* xh = x + (int64_t)bh * S_src * D;
  const int32_t* ph = perm ? perm + (int64_t)bh * S : nullptr;
  const int sub = threadIdx.x % TPR;         // channels [W sub, W sub + W) of rows r0 + RSTEP m
  const int r0 = threadIdx.x / TPR;
  __shared__ uint4 cen_s[D / 8];
  __shared__ float red[8];
  if (kCentred && threadIdx.x < D / 8)
    cen_s[threadIdx.x] = __ldg(reinterpret_cast<const uint4*>(center + (int64_t)bh * D) + threadIdx.x);
  uint4 v[RPT][G];
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const int t = j * 128 + r0 + RSTEP * m;
    const uint4* src = t < S ? reinterpret_cast<const uint4*>(xh + (int64_t)(ph ? ph[t] : t) * D + sub * W) : nullptr;
#pragma unroll
    for (int g = 0; g < G; ++g) v[m][g] = src ? src[g] : make_uint4(0, 0, 0, 0);
  }
  if (kCentred) __syncthreads();
  float y[RPT][W];
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint4 cm = kCentred ? cen_s[sub * G + g] : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < 8; ++i) y[m][8 * g + i] = chunk_elem<kCentred>(v[m][g], cm, i);
    }
#pragma unroll
    for (int s = 1; s < W; s <<= 1)
#pragma unroll
      for (int i = 0; i < W; ++i)
        if (!(i & s)) {
          const float a = y[m][i], b = y[m][i + s];
          y[m][i] = __fadd_rn(a, b);
          y[m][i + s] = __fsub_rn(a, b);
        }
  }
#pragma unroll
  for (int s = W; s < D; s <<= 1) {
    const int lm = s / W;                     // partner lane offset
    const bool lower = (sub & lm) == 0;       // this thread holds x[i], the partner x[i + s]
#pragma unroll
    for (int m = 0; m < RPT; ++m)
#pragma unroll
      for (int i = 0; i < W; ++i) {
        const float p = __shfl_xor_sync(0xffffffffu, y[m][i], lm);
        y[m][i] = lower ? __fadd_rn(y[m][i], p) : __fsub_rn(p, y[m][i]);
      }
  }
  float amax = 0.f;
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < W; ++i) a = fmaxf(a, fabsf(y[m][i]));
    if (j * 128 + r0 + RSTEP * m < S) amax = fmaxf(amax, a);  // pad rows do not count
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const bool zero = !(amax > 0.f);
  const float inv = zero ? 0.f : __fdiv_rn(448.f, amax);
  if (threadIdx.x == 0) scales[(int64_t)bh * nkb + j] = zero ? 1.f : __fdiv_rn(amax, 448.f);
  uint8_t* ch = codes + ((int64_t)bh * S_pad + (int64_t)j * 128) * D;
#pragma unroll
  for (int m = 0; m < RPT; ++m) {
    const int r = r0 + RSTEP * m;
    const bool live = !zero && j * 128 + r < S;
    uint32_t w[W / 4];
#pragma unroll
    for (int q = 0; q < W / 4; ++q) {
      const uint32_t lo = cvt_e4m3x2(__fmul_rn(y[m][4 * q], inv), __fmul_rn(y[m][4 * q + 1], inv));
      const uint32_t hi = cvt_e4m3x2(__fmul_rn(y[m][4 * q + 2], inv), __fmul_rn(y[m][4 * q + 3], inv));
      w[q] = live ? (lo | (hi << 16)) : 0u;
    }
    uint4* dst = reinterpret_cast<uint4*>(ch + (int64_t)r * D + sub * W);
#pragma unroll
    for (int q = 0; q < W / 16; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// Launch of the block quantiser for D in {64, 128}, centred or not (grid: S_pad/128 x BH).
void quant_blocks_launch(const uint16_t* x, const int32_t* perm, const uint16_t* center, int D, int S, int S_pad,
                         int S_src, int BH, uint8_t* codes, float* scales, cudaStream_t st, bool rotate) {
  const dim3 grid(S_pad / 128, BH);
  if (rotate) {
    const uint16_t* c = center;
    if (D == 128) {
      if (c) quant_blocks_rot_kernel<128, true><<<grid, 256, 0, st>>>(x, perm, c, S, S_pad, S_src, codes, scales);
      else quant_blocks_rot_kernel<128, false><<<grid, 256, 0, st>>>(x, perm, c, S, S_pad, S_src, codes, scales);
    } else {
      if (c) quant_blocks_rot_kernel<64, true><<<grid, 256, 0, st>>>(x, perm, c, S, S_pad, S_src, codes, scales);
      else quant_blocks_rot_kernel<64, false><<<grid, 256, 0, st>>>(x, perm, c, S, S_pad, S_src, codes, scales);
    }
    return;
  }
  if (D == 128) {
    if (center) quant_blocks_kernel<128, true><<<grid, 256, 0, st>>>(x, perm, center, S, S_pad, S_src, codes, scales);
    else quant_blocks_kernel<128, false><<<grid, 256, 0, st>>>(x, perm, nullptr, S, S_pad, S_src, codes, scales);
  } else {
    if (center) quant_blocks_kernel<64, true><<<grid, 256, 0, st>>>(x, perm, center, S, S_pad, S_src, codes, scales);
    else quant_blocks_kernel<64, false><<<grid, 256, 0, st>>>(x, perm, nullptr, S, S_pad, S_src, codes, scales);
  }
}

// ---------------------------------------------------------------------------------------------
// K channel centre ("VC-Attention", Sec. 3.4 "Fused preprocessing" and App. B: the K pass gathers
// centering statistics and subtracts the mean): mu[bh][d] = bf16_RNE(sum_t K[t][d] / S). The sum is
// taken exactly in int64: each bf16 is M * 2^(E - 134) with an 8-bit significand M; relative to the
// column's largest exponent E_max it is M * 2^(E - E_max + 28) (|sum| < 2^56 for S <= 2^20), so only
// values more than 28 binades below the column maximum lose low bits.
// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) kstat_exp_kernel(const uint16_t* __restrict__ x, int S, int* __restrict__ kexp) {
  constexpr int SPLIT = 256 / D;
  const int j = blockIdx.x, bh = blockIdx.y;
  const int d = threadIdx.x % D, part = threadIdx.x / D;
  const int t0 = j * 128, n = min(128, S - t0);
  const uint16_t* xh = x + ((int64_t)bh * S + t0) * D;
  __shared__ int ep[SPLIT][D];
  int em = 1;
  for (int r = part; r < n; r += SPLIT) em = max(em, max((xh[(int64_t)r * D + d] >> 7) & 0xFF, 1));
  ep[part][d] = em;
  __syncthreads();
  if (part == 0) {
#pragma unroll
    for (int q = 1; q < SPLIT; ++q) em = max(em, ep[q][d]);
    atomicMax(kexp + (int64_t)bh * D + d, em);
  }
}

template <int D>
__global__ void __launch_bounds__(256) kstat_sum_kernel(const uint16_t* __restrict__ x, int S,
                                                        const int* __restrict__ kexp,
                                                        unsigned long long* __restrict__ ksum) {
  constexpr int SPLIT = 256 / D;
  const int j = blockIdx.x, bh = blockIdx.y;
  const int d = threadIdx.x % D, part = threadIdx.x / D;
  const int t0 = j * 128, n = min(128, S - t0);
  const uint16_t* xh = x + ((int64_t)bh * S + t0) * D;
  const int em = kexp[(int64_t)bh * D + d];
  __shared__ long long sp[SPLIT][D];
  long long acc = 0;
  for (int r = part; r < n; r += SPLIT) {
    const uint32_t b = xh[(int64_t)r * D + d];
    const int e = (b >> 7) & 0xFF;
    const long long m = (long long)((b & 0x7Fu) | (e ? 0x80u : 0u));
    const int sh = max(e, 1) - em + 28;
    const long long xv = sh >= 0 ? (m << sh) : (m >> min(-sh, 63));
    acc += (b & 0x8000u) ? -xv : xv;
  }
  sp[part][d] = acc;
  __syncthreads();
  if (part == 0) {
#pragma unroll
    for (int q = 1; q < SPLIT; ++q) acc += sp[q][d];
    atomicAdd(ksum + (int64_t)bh * D + d, (unsigned long long)acc);  // two's complement: order-free
  }
}

__global__ void kstat_mean_kernel(const int* __restrict__ kexp, const unsigned long long* __restrict__ ksum, int S,
                                  int n, uint16_t* __restrict__ kmu) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const double total = ldexp((double)(long long)ksum[i], kexp[i] - 162);  // 2^(E - 134) * 2^-28
  kmu[i] = f64_to_bf16_rne(total / (double)S);
}

__global__ void iota_kernel(int32_t* __restrict__ perm, int S, int64_t total) {
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < total) perm[i] = (int32_t)(i % S);
}

// ---------------------------------------------------------------------------------------------
// Block means of V' = V[pi] and the per-head residual maximum.  One CTA per (block, bh); the block's
// rows are gathered into shared memory once, and each thread then holds one channel pair of
// 128/PARTS rows in registers for all three passes (largest exponent, exact sum, residual maximum).
// mu_j = (sum of the valid rows) / n_j, rounded once to bf16. The sum is exact: every bf16 value is an
// 8-bit significand M times 2^(E-134); relative to the column's largest exponent E_max it becomes the
// integer M * 2^(E - E_max + 45) (|sum| < 2^60 in int64), exact whenever the column spans at most 45
// binades. Whenever an fp64 running sum would be exact too (a span of at most 38 binades), the double
// (sum * 2^(E_max - 179)) / n_j is then the same double, and so is the bf16 mean. R = V' - mu_b in
// fp32; amax_h = max |R| over the head (atomicMax on the bit pattern of a non-negative float) and,
// when amax_ch is given, amax_d = max |R[:, d]| of every channel over the head the same way.
__device__ __forceinline__ long long exact_term(uint32_t b, int em) {
  const int e = (b >> 7) & 0xFF;
  const long long m = (long long)((b & 0x7Fu) | (e ? 0x80u : 0u));
  const int sh = max(e, 1) - em + 45;  // in [.., 45]; below 0 only past a 45-binade span
  const long long x = sh >= 0 ? (m << sh) : (m >> min(-sh, 63));
  return (b & 0x8000u) ? -x : x;
}

template <int D>
__global__ void __launch_bounds__(256) vmeans_kernel(const uint16_t* __restrict__ v, const int32_t* __restrict__ perm,
                                                     int S, int demean, uint16_t* __restrict__ mub,
                                                     unsigned int* __restrict__ amax_bits,
                                                     uint16_t* __restrict__ mubT = nullptr, int nkb16 = 0,
                                                     unsigned int* __restrict__ amax_ch = nullptr) {
  constexpr int NP = D / 2;          // channel pairs
  constexpr int PARTS = 256 / NP;    // threads per pair
  constexpr int RPT = 128 / PARTS;   // rows per thread: part, part + PARTS, ...
  const int j = blockIdx.x, bh = blockIdx.y;
  const int nkb = (S + 127) / 128;
  const int c = threadIdx.x % NP, part = threadIdx.x / NP;
  const int t0 = j * 128, n = min(128, S - t0);
  const uint16_t* vh = v + (int64_t)bh * S * D;
  const int32_t* ph = perm ? perm + (int64_t)bh * S : nullptr;
  __shared__ __align__(16) uint16_t blk[128][D];
  __shared__ uint32_t emax_part[PARTS][NP];
  __shared__ long long sums[PARTS][D];
  __shared__ int emc[D];
  __shared__ float mus[D];
  __shared__ float red[8];
  __shared__ float cmax[PARTS][D];
  gather_block<D>(blk, vh, ph, t0, n);  // rows n..127 read as +0: no exponent, no sum term
  __syncthreads();
  uint32_t w[RPT];  // (channel 2c) | (channel 2c + 1) << 16 of row part + PARTS * i
  const uint32_t* bw = reinterpret_cast<const uint32_t*>(&blk[0][0]);
#pragma unroll
  for (int i = 0; i < RPT; ++i) w[i] = bw[(part + PARTS * i) * NP + c];
  // exponent fields of both channels in place, with subnormals and zero read as 1 below
  uint32_t ex = 0;
#pragma unroll
  for (int i = 0; i < RPT; ++i) ex = __vmaxu2(ex, w[i] & 0x7F807F80u);
  emax_part[part][c] = ex;
  __syncthreads();
#pragma unroll
  for (int q = 0; q < PARTS; ++q) ex = __vmaxu2(ex, emax_part[q][c]);
  const int em0 = max((int)((ex >> 7) & 0xFFu), 1), em1 = max((int)((ex >> 23) & 0xFFu), 1);
  long long a0 = 0, a1 = 0;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    a0 += exact_term(w[i] & 0xFFFFu, em0);
    a1 += exact_term(w[i] >> 16, em1);
  }
  sums[part][2 * c] = a0;
  sums[part][2 * c + 1] = a1;
  if (part == 0) {
    emc[2 * c] = em0;
    emc[2 * c + 1] = em1;
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int d = threadIdx.x;
    long long tot = 0;
#pragma unroll
    for (int q = 0; q < PARTS; ++q) tot += sums[q][d];
    const double total = ldexp((double)tot, emc[d] - 179);  // 2^(E - 134) * 2^-45
    uint16_t b = demean ? f64_to_bf16_rne(total / (double)n) : (uint16_t)0;
    mub[((int64_t)bh * nkb + j) * D + d] = b;
    if (mubT) mubT[((int64_t)bh * D + d) * nkb16 + j] = b;  // [BH, D, nkb16]: the forward's flush operand
    mus[d] = bf16_bits_to_f32(b);
  }
  __syncthreads();
  const float mu0 = mus[2 * c], mu1 = mus[2 * c + 1];
  float am0 = 0.f, am1 = 0.f;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    if (part + PARTS * i < n) {
      am0 = fmaxf(am0, fabsf(__fsub_rn(bf16_bits_to_f32(w[i] & 0xFFFFu), mu0)));
      am1 = fmaxf(am1, fabsf(__fsub_rn(__uint_as_float(w[i] & 0xFFFF0000u), mu1)));
    }
  }
  if (amax_ch) {  // per channel: combine the column's parts, one atomic per channel
    cmax[part][2 * c] = am0;
    cmax[part][2 * c + 1] = am1;
    __syncthreads();
    if (threadIdx.x < D) {
      const int d = threadIdx.x;
      float m = cmax[0][d];
#pragma unroll
      for (int q = 1; q < PARTS; ++q) m = fmaxf(m, cmax[q][d]);
      atomicMax(amax_ch + (int64_t)bh * D + d, __float_as_uint(m));
    }
  }
  float amax = fmaxf(am0, am1);
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
    for (int w8 = 1; w8 < 8; ++w8) m = fmaxf(m, red[w8]);
    atomicMax(amax_bits + bh, __float_as_uint(m));
  }
}

// Residual codes, transposed: Vt[bh][d][t] = E4M3(R[t][d] * 448/amax), t < S_pad (pad = 0), with
// amax the head's (amax_h) or, when amax_ch is given, the channel's (amax_d).
// One CTA per (block, bh): the block's rows are gathered into shared memory with 16-byte loads, then
// each thread codes 32 rows of one channel (reads along the channels are conflict-free) and writes
// them as one 32-byte sector of the transposed output.  The first block's CTA writes the scales
// (svc: the scale of every channel, equal to the head's without amax_ch).  With amax_ch the
// transposed means the forward reads become bf16(mu / s_d), one correctly rounded fp32 division.
template <int D>
__global__ void __launch_bounds__(256) vpack_kernel(const uint16_t* __restrict__ v, const int32_t* __restrict__ perm,
                                                    int S, int S_pad, const uint16_t* __restrict__ mub,
                                                    const unsigned int* __restrict__ amax_bits,
                                                    uint8_t* __restrict__ vt, float* __restrict__ sv,
                                                    const unsigned int* __restrict__ amax_ch = nullptr,
                                                    float* __restrict__ svc = nullptr,
                                                    uint16_t* __restrict__ mubT = nullptr, int nkb16 = 0) {
  const int j = blockIdx.x, bh = blockIdx.y;
  const int nkb = S_pad / 128;
  const int t0 = j * 128, n = min(128, S - t0);
  const uint16_t* vh = v + (int64_t)bh * S * D;
  const int32_t* ph = perm ? perm + (int64_t)bh * S : nullptr;
  __shared__ __align__(16) uint16_t blk[128][D];
  __shared__ float mus[D];
  __shared__ float invs[D];
  const float amax = __uint_as_float(amax_bits[bh]);
  const bool zero = !(amax > 0.f);
  const float inv_h = zero ? 1.f : __fdiv_rn(448.f, amax);
  const float sv_h = zero ? 1.f : __fdiv_rn(amax, 448.f);
  if (j == 0 && threadIdx.x == 0) sv[bh] = sv_h;
  for (int d = threadIdx.x; d < D; d += 256) {
    const float mu = bf16_bits_to_f32(mub[((int64_t)bh * nkb + j) * D + d]);
    mus[d] = mu;
    if (amax_ch) {
      const float a = __uint_as_float(amax_ch[(int64_t)bh * D + d]);
      const bool z = !(a > 0.f);
      const float s_d = z ? 1.f : __fdiv_rn(a, 448.f);
      invs[d] = z ? 1.f : __fdiv_rn(448.f, a);
      if (j == 0) svc[(int64_t)bh * D + d] = s_d;
      mubT[((int64_t)bh * D + d) * nkb16 + j] = f64_to_bf16_rne((double)__fdiv_rn(mu, s_d));
    } else {
      invs[d] = inv_h;
      if (j == 0 && svc) svc[(int64_t)bh * D + d] = sv_h;
    }
  }
  gather_block<D>(blk, vh, ph, t0, n);
  __syncthreads();
  uint8_t* out = vt + (int64_t)bh * D * S_pad + (int64_t)t0;
  for (int task = threadIdx.x; task < D * 4; task += 256) {
    const int d = task % D, seg = task / D;  // rows [32 seg, 32 seg + 32) of channel d
    const float mu = mus[d], inv = invs[d];
    uint32_t w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int r = seg * 32 + 4 * q + 2 * h;
        const float r0 = r < n ? __fmul_rn(__fsub_rn(bf16_bits_to_f32(blk[r][d]), mu), inv) : 0.f;
        const float r1 = r + 1 < n ? __fmul_rn(__fsub_rn(bf16_bits_to_f32(blk[r + 1][d]), mu), inv) : 0.f;
        word |= cvt_e4m3x2(r0, r1) << (16 * h);
      }
      w[q] = word;
    }
    uint4* dst = reinterpret_cast<uint4*>(out + (int64_t)d * S_pad + seg * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// ---------------------------------------------------------------------------------------------
// Host-side launch sequence of the prepare step (all on one stream, no host synchronisation).
// ---------------------------------------------------------------------------------------------
static int check_launch() { return cudaPeekAtLastError() == cudaSuccess ? 0 : VC_ERR_CUDA; }

int prepare_launch(const PlanBuffers& p, const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                   const int32_t* perm_in, bool vsmooth, bool kcenter, bool reuse_perm, bool warm, bool vchannel,
                   int iters, cudaStream_t st) {
  const int BH = p.B * p.H, S = p.S, D = p.D, nkb = p.nkb, S_pad = p.S_pad;
  dim3 gblk(nkb, BH);
  // Q: per-block quantisation in token order
  quant_blocks_launch(Q, nullptr, nullptr, D, S, S_pad, S, BH, p.qcodes, p.qscales, st, p.has_hadamard);
  if (check_launch()) return VC_ERR_CUDA;
  const int32_t* perm = nullptr;
  if (reuse_perm) {  // the permutation of an earlier prepare stays (grouping schedule)
    perm = p.perm;
  } else if (vsmooth) {
    if (perm_in) {
      if (cudaMemcpyAsync(p.perm, perm_in, sizeof(int32_t) * (size_t)BH * S, cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess)
        return VC_ERR_CUDA;
    } else {
      int rc = kmeans_launch(p, V, iters, warm, st);
      if (rc != VC_OK) return rc;
    }
    perm = p.perm;
  } else {
    int64_t total = (int64_t)BH * S;
    iota_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(p.perm, S, total);
  }
  if (check_launch()) return VC_ERR_CUDA;
  // K' = K[pi], per-block quantisation
  const uint16_t* kcen = nullptr;
  if (kcenter) {  // the head's channel centre of K, in token order
    if (cudaMemsetAsync(p.kexp, 0, sizeof(int) * (size_t)BH * D, st) != cudaSuccess ||
        cudaMemsetAsync(p.ksum, 0, sizeof(unsigned long long) * (size_t)BH * D, st) != cudaSuccess)
      return VC_ERR_CUDA;
    if (D == 128) {
      kstat_exp_kernel<128><<<gblk, 256, 0, st>>>(K, S, p.kexp);
      kstat_sum_kernel<128><<<gblk, 256, 0, st>>>(K, S, p.kexp, p.ksum);
    } else {
      kstat_exp_kernel<64><<<gblk, 256, 0, st>>>(K, S, p.kexp);
      kstat_sum_kernel<64><<<gblk, 256, 0, st>>>(K, S, p.kexp, p.ksum);
    }
    kstat_mean_kernel<<<(BH * D + 255) / 256, 256, 0, st>>>(p.kexp, p.ksum, S, BH * D, p.kmu);
    kcen = p.kmu;
  }
  quant_blocks_launch(K, perm, kcen, D, S, S_pad, S, BH, p.kcodes, p.kscales, st, p.has_hadamard);
  // V' = V[pi]: block means, residual maximum per head, residual codes transposed
  if (cudaMemsetAsync(p.vamax, 0, sizeof(unsigned int) * BH, st) != cudaSuccess) return VC_ERR_CUDA;
  unsigned int* ach = vchannel ? p.vamax_ch : nullptr;
  if (vchannel && cudaMemsetAsync(p.vamax_ch, 0, sizeof(unsigned int) * (size_t)BH * D, st) != cudaSuccess)
    return VC_ERR_CUDA;
  if (D == 128) {
    vmeans_kernel<128><<<gblk, 256, 0, st>>>(V, perm, S, vsmooth ? 1 : 0, p.means, p.vamax, p.meansT, p.nkb16, ach);
    vpack_kernel<128><<<gblk, 256, 0, st>>>(V, perm, S, S_pad, p.means, p.vamax, p.vcodes, p.vscales, ach,
                                            p.vscales_ch, p.meansT, p.nkb16);
  } else {
    vmeans_kernel<64><<<gblk, 256, 0, st>>>(V, perm, S, vsmooth ? 1 : 0, p.means, p.vamax, p.meansT, p.nkb16, ach);
    vpack_kernel<64><<<gblk, 256, 0, st>>>(V, perm, S, S_pad, p.means, p.vamax, p.vcodes, p.vscales, ach,
                                           p.vscales_ch, p.meansT, p.nkb16);
  }
  if (check_launch()) return VC_ERR_CUDA;
  return repair_launch(p, K, V, kcen, st);  // nothing without repair rows
}

}  // namespace vc

namespace vc {

// Block means and packed residual codes of V' = V[pi] with a caller-provided per-head scratch
// word (the residual maximum). Used by the allocation-free entry point; the prepare step above
// keeps using the plan's own scratch.
int residual_pack_launch(const uint16_t* V, const int32_t* perm, int BH, int S, int D, uint16_t* means,
                         uint8_t* vcodes, float* vscales, unsigned int* amax_scratch, cudaStream_t st) {
  const int nkb = (S + 127) / 128, S_pad = nkb * 128;
  dim3 gblk(nkb, BH);
  if (cudaMemsetAsync(amax_scratch, 0, sizeof(unsigned int) * BH, st) != cudaSuccess) return VC_ERR_CUDA;
  if (D == 128) {
    vmeans_kernel<128><<<gblk, 256, 0, st>>>(V, perm, S, 1, means, amax_scratch);
    vpack_kernel<128><<<gblk, 256, 0, st>>>(V, perm, S, S_pad, means, amax_scratch, vcodes, vscales);
  } else {
    vmeans_kernel<64><<<gblk, 256, 0, st>>>(V, perm, S, 1, means, amax_scratch);
    vpack_kernel<64><<<gblk, 256, 0, st>>>(V, perm, S, S_pad, means, amax_scratch, vcodes, vscales);
  }
  return check_launch();
}

}  // namespace vc
