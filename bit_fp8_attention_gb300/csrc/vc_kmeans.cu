// vc_kmeans.cu -- the grouping step of V-Smooth: online k-means over the V rows of every head,
// then the stable argsort of the labels ("VC-Attention", Sec. 3.2 "Value-guided permutation").
//
// Reading of the pages' k-means: Lloyd rounds at inference time; centroid i starts as row
// floor(i*S/k); a token goes to the nearest centroid in squared Euclidean distance, the lowest
// index on a tie; a centroid becomes the mean of its members, an empty cluster keeps its centroid.
//
// GB300 design:
//   assignment  tcgen05 (kind::f16), persistent (one CTA per SM): per work item two 128-token
//               tiles of V (bf16, exact) against the centroids in chunks of 128, each centroid split
//               into bf16 hi + lo (about 16 significant bits) streamed as separate stages; fp32 dot
//               products accumulate in TMEM (two tiles x two chunk buffers = 512 columns), eight
//               epilogue warps scan the columns in ascending order for argmin ||c||^2 - 2 x.c. One
//               warp loads the token tiles by TMA (double-buffered, so the next item's tiles land
//               while this one computes), one the centroid chunks, and one elected thread issues the
//               MMAs. A cold start's first round skips the lo halves, which are zero for data rows.
//   argsort     stable counting sort in three launches: per-chunk label histograms, a scan over
//               chunks and bins, then a scatter in token order within each chunk.
//   update      one warp per cluster, compensated fp32 sums (TwoSum) of the member rows read
//               through the permutation: within about one fp32 ulp of the exact mean.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_internal.h"

namespace vc {
namespace {

constexpr uint32_t kWaitLimit = 1u << 20;
constexpr int kStatusTimeoutKmeans = 32;  // a wait in the assignment kernel ran out
constexpr int kChunk = 2048;              // tokens per argsort chunk

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// The bf16 hi + lo split of a centroid row and its squared norm, as the assignment reads them.
__device__ __forceinline__ void store_split(uint16_t* hi, uint16_t* lo, int d, float c) {
  const uint16_t h = f32_to_bf16_bits(c);
  hi[d] = h;
  lo[d] = f32_to_bf16_bits(__fsub_rn(c, bf16_to_f32(h)));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------------------------------------
// Initial centroids: c_i = x_floor(i*S/k); pad centroids (i >= k) get ||c||^2 = +inf so that no
// token ever selects them.  One warp per centroid.
// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) kmeans_init_kernel(const uint16_t* __restrict__ v, int S, int k, int kpad,
                                                          float* __restrict__ cent, float* __restrict__ cnorm,
                                                          uint16_t* __restrict__ cent16, float* __restrict__ cnormp) {
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5), bh = blockIdx.y;
  if (i >= kpad) return;
  uint16_t* hi = cent16 + ((int64_t)bh * 2 * kpad + i) * D;
  uint16_t* lo = hi + (int64_t)kpad * D;
  if (i >= k) {
    for (int d = lane; d < D; d += 32) hi[d] = lo[d] = 0;
    if (lane == 0) cnormp[(int64_t)bh * kpad + i] = INFINITY;
    return;
  }
  const int64_t src = (int64_t)i * S / k;
  const uint16_t* row = v + ((int64_t)bh * S + src) * D;
  float* c = cent + ((int64_t)bh * k + i) * D;
  float acc = 0.f;
  for (int d = lane; d < D; d += 32) {
    const float x = bf16_to_f32(row[d]);
    c[d] = x;
    store_split(hi, lo, d, x);
    acc = fmaf(x, x, acc);
  }
  acc = warp_sum(acc);
  if (lane == 0) {
    cnorm[(int64_t)bh * k + i] = acc;
    cnormp[(int64_t)bh * kpad + i] = acc;
  }
}

// ---------------------------------------------------------------------------------------------
// Assignment on the tensor cores.
// ---------------------------------------------------------------------------------------------
template <int D>
struct AsgCfg {
  static constexpr int TPC = 2;                 // 128-token tiles per work item
  static constexpr int CH = 128;                // centroids per chunk (MMA N)
  static constexpr int NST = 3;                 // stages, each one part (hi or lo) of a chunk
  static constexpr int NXB = 2;                 // token-tile buffers: the next item's tiles load during this one
  static constexpr int ATOM = 128 * 128;        // one 128-byte-swizzled K half of a 128-row operand
  static constexpr int HALVES = D / 64;         // K halves of 64 bf16
  static constexpr int XT = HALVES * ATOM;      // bytes of a token tile
  static constexpr int CB = HALVES * CH * 128;  // bytes of one part (hi or lo) of a chunk
  static constexpr int OFF_X = 0;
  static constexpr int OFF_C = OFF_X + NXB * TPC * XT;
  static constexpr int OFF_BAR = OFF_C + NST * CB;
  static constexpr int NBAR = 2 * NXB + 2 * NST + 2 + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack for aligning the base to 1024
  static constexpr int TMEM_COLS = TPC * 2 * CH;     // two accumulator buffers per tile
  static_assert(SMEM <= 227 * 1024, "fits one SM's shared memory");
};

__device__ __forceinline__ void mma_bf16_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 15u && *abort_flag) return false;
  }
  return false;
}

__device__ __forceinline__ void fail(int* status, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(status, kStatusTimeoutKmeans);
}

// xmap: V as [B*H*S rows, D] bf16, box 64 x 128, 128-byte swizzle.
// cmap: centroid splits as [B*H*2*kpad rows, D] bf16 (per head: kpad hi rows, then kpad lo rows),
//       box 64 x CH.
// Persistent: CTA b takes work items b, b + gridDim.x, ... (item w = head w / ntp, tokens
// [256 (w % ntp), 256 (w % ntp) + 256)), so that one item's token tiles load while the previous item
// computes. Local item i uses token buffer i % 2; the c-th chunk this CTA consumes, counted over all
// its items, uses accumulator buffer c % 2, and its nparts parts (hi, then lo when nparts = 2) are the
// stage loads u = nparts c, ..., nparts c + nparts - 1 (stage u % NST).
template <int D>
__global__ void __launch_bounds__(352, 1)
    kmeans_assign_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap cmap,
                         const float* __restrict__ cnormp, int S, int kpad, int nwork, int nparts,
                         int32_t* __restrict__ labels, int* __restrict__ status) {
  using C = AsgCfg<D>;
  extern __shared__ uint8_t asg_smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(asg_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sX = base + C::OFF_X;
  uint8_t* sC = base + C::OFF_C;
  uint64_t* x_full = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* x_empty = x_full + C::NXB;
  uint64_t* c_full = x_empty + C::NXB;
  uint64_t* c_empty = c_full + C::NST;
  uint64_t* acc_full = c_empty + C::NST;  // per TMEM buffer: both tiles' dot products of a chunk
  uint64_t* acc_empty = acc_full + 2;     // per TMEM buffer: read by all eight epilogue warps
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + C::OFF_MISC + 8);

  // The warp index read back from lane 0 is one the compiler knows to be warp-uniform: each role's
  // loop state and the MMA descriptors then live in uniform registers.
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  const int ntp = (S + C::TPC * 128 - 1) / (C::TPC * 128);  // work items per head
  const int nch = kpad / C::CH;
  const int nitems = nwork > (int)blockIdx.x ? (nwork - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (tid == 0) {
    for (int x = 0; x < C::NXB; ++x) { mbar_init(&x_full[x], 1); mbar_init(&x_empty[x], 1); }
    for (int s = 0; s < C::NST; ++s) { mbar_init(&c_full[s], 1); mbar_init(&c_empty[s], 1); }
    for (int b = 0; b < 2; ++b) { mbar_init(&acc_full[b], 1); mbar_init(&acc_empty[b], 256); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 10) {
    // ---------------------------------------------------------------- TMA producer: token tiles
    if (lane == 0) {
      prefetch_tmap(&xmap);
      int issued = 0;
      for (int i = 0; i < nitems; ++i) {
        const int xb = i % C::NXB;
        if (i >= C::NXB && !wait_or_abort(&x_empty[xb], ((i / C::NXB) & 1) ^ 1, abort_flag)) {
          fail(status, abort_flag);
          break;
        }
        const int w = blockIdx.x + i * gridDim.x;
        const int bh = w / ntp, t0 = (w % ntp) * C::TPC * 128;
        mbar_arrive_expect_tx(&x_full[xb], C::TPC * C::XT);
        for (int g = 0; g < C::TPC; ++g)
          for (int h = 0; h < C::HALVES; ++h)
            tma_load_2d(sX + (xb * C::TPC + g) * C::XT + h * C::ATOM, &xmap, h * 64, bh * S + t0 + g * 128,
                        &x_full[xb]);
        issued = i + 1;
      }
      // Teardown: every load issued into this CTA's shared memory has landed.
      bool done = true;
      for (int i = issued > C::NXB ? issued - C::NXB : 0; i < issued; ++i)
        done &= mbar_wait(&x_full[i % C::NXB], (i / C::NXB) & 1, kWaitLimit);
      if (!done) fail(status, abort_flag);
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- TMA producer: centroid chunks
    if (lane == 0) {
      prefetch_tmap(&cmap);
      int issued = 0;
      bool ok = true;
      for (int i = 0; ok && i < nitems; ++i) {
        const int bh = (blockIdx.x + i * gridDim.x) / ntp;
        for (int ch = 0; ok && ch < nch; ++ch)
          for (int part = 0; part < nparts; ++part) {
            const int u = nparts * (i * nch + ch) + part, s = u % C::NST;
            if (!wait_or_abort(&c_empty[s], ((u / C::NST) & 1) ^ 1, abort_flag)) { ok = false; break; }
            mbar_arrive_expect_tx(&c_full[s], C::CB);
            for (int h = 0; h < C::HALVES; ++h)
              tma_load_2d(sC + s * C::CB + h * (C::CH * 128), &cmap, h * 64, (bh * 2 + part) * kpad + ch * C::CH,
                          &c_full[s]);
            issued = u + 1;
          }
      }
      if (!ok) fail(status, abort_flag);
      bool done = true;
      for (int u = issued > C::NST ? issued - C::NST : 0; u < issued; ++u)
        done &= mbar_wait(&c_full[u % C::NST], (u / C::NST) & 1, kWaitLimit);
      if (!done) fail(status, abort_flag);
    }
  } else if (warp == 9) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the schedule (waits voted, so it stays converged); one elected lane issues.
    const bool leader = elect_one();
    constexpr uint32_t idesc = idesc_bf16(128, C::CH);
    const uint64_t dx0 = smem_desc(sX, 1024, kSw128);
    const uint64_t dc0 = smem_desc(sC, 1024, kSw128);
    auto wwait = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_or_abort(bar, parity, abort_flag));
    };
    bool ok = true;
    for (int i = 0; ok && i < nitems; ++i) {
      const int xb = i % C::NXB;
      if (!wwait(&x_full[xb], (i / C::NXB) & 1)) { ok = false; break; }
      for (int ch = 0; ok && ch < nch; ++ch) {
        const int c = i * nch + ch, b = c & 1;
        if (!wwait(&acc_empty[b], ((c >> 1) & 1) ^ 1)) { ok = false; break; }
        for (int part = 0; part < nparts; ++part) {
          const int u = nparts * c + part, s = u % C::NST;
          if (!wwait(&c_full[s], (u / C::NST) & 1)) { ok = false; break; }
          tc_fence_after();
          if (leader) {
#pragma unroll
            for (int g = 0; g < C::TPC; ++g) {
              const uint32_t d = tmem + (uint32_t)((g * 2 + b) * C::CH);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                // K step of 16 bf16 = 32 bytes inside a 128-byte swizzle atom; a new atom every 4
                const uint64_t kx = (uint64_t)((kk >> 2) * (C::ATOM >> 4) + 2 * (kk & 3));
                const uint64_t kc = (uint64_t)((kk >> 2) * ((C::CH * 128) >> 4) + 2 * (kk & 3));
                const uint64_t a = dx0 + (uint64_t)((xb * C::TPC + g) * (C::XT >> 4)) + kx;
                const uint64_t bd = dc0 + (uint64_t)(s * (C::CB >> 4)) + kc;
                mma_bf16_ss(d, a, bd, idesc, (part | kk) ? 1u : 0u);  // hi, then lo onto it
              }
            }
            mma_commit(&c_empty[s]);
            if (part == nparts - 1) {
              mma_commit(&acc_full[b]);
              if (ch == nch - 1) mma_commit(&x_empty[xb]);  // the item's token tiles are no longer read
            }
          }
          __syncwarp();
        }
      }
    }
    if (!ok && lane == 0) fail(status, abort_flag);
    if (leader) mma_commit(drain);
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(drain, 0, kWaitLimit)) && lane == 0) fail(status, abort_flag);
  } else {
    // ---------------------------------------------------------------- argmin epilogue, warps 0-7
    const int g = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t tbase = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(g * 2 * C::CH);
    bool ok = true;
    for (int i = 0; ok && i < nitems; ++i) {
      const int w = blockIdx.x + i * gridDim.x;
      const int bh = w / ntp, tok = (w % ntp) * C::TPC * 128 + g * 128 + row;
      const float* cn = cnormp + (int64_t)bh * kpad;
      float best = INFINITY;
      int bi = 0;
      for (int ch = 0; ch < nch; ++ch) {
        const int c = i * nch + ch, b = c & 1;
        const bool got = wait_or_abort(&acc_full[b], (c >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) fail(status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        // All dot products of the chunk in one round trip; the buffer is released before the scan.
        uint32_t r[C::CH];
#pragma unroll
        for (int c0 = 0; c0 < C::CH; c0 += 32)
          tmem_ld32(tbase + (uint32_t)(b * C::CH + c0), *reinterpret_cast<uint32_t(*)[32]>(&r[c0]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&acc_empty[b]);
        const float4* cn4 = reinterpret_cast<const float4*>(cn + ch * C::CH);
#pragma unroll
        for (int q = 0; q < C::CH / 4; ++q) {
          const float4 n4 = __ldg(cn4 + q);
          const float nn[4] = {n4.x, n4.y, n4.z, n4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float dist = fmaf(-2.f, __uint_as_float(r[4 * q + e]), nn[e]);
            if (dist < best) {  // ascending scan: a tie keeps the lower index
              best = dist;
              bi = ch * C::CH + 4 * q + e;
            }
          }
        }
      }
      if (ok && tok < S) labels[(int64_t)bh * S + tok] = bi;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------------------------
// Stable argsort of the labels (counting sort), three launches.
// ---------------------------------------------------------------------------------------------
// (1) hist[bh][c][i] = number of tokens with label i in chunk c.
__global__ void __launch_bounds__(256) label_hist_kernel(const int32_t* __restrict__ labels, int S, int k,
                                                         int nchunk, int32_t* __restrict__ hist) {
  __shared__ int h[1024];
  const int c = blockIdx.x, bh = blockIdx.y;
  for (int i = threadIdx.x; i < k; i += 256) h[i] = 0;
  __syncthreads();
  const int32_t* z = labels + (int64_t)bh * S;
  const int end = min(S, (c + 1) * kChunk);
  for (int t = c * kChunk + threadIdx.x; t < end; t += 256) atomicAdd(&h[z[t]], 1);
  __syncthreads();
  int32_t* out = hist + ((int64_t)bh * nchunk + c) * k;
  for (int i = threadIdx.x; i < k; i += 256) out[i] = h[i];
}

// (2) counts, exclusive offsets over clusters, and hist[bh][c][i] replaced by the position of the
// first token of cluster i in chunk c.  One CTA of 1024 threads per batch-head.
__global__ void __launch_bounds__(1024) label_scan_kernel(int k, int nchunk, int32_t* __restrict__ hist,
                                                          int32_t* __restrict__ counts,
                                                          int32_t* __restrict__ offsets) {
  __shared__ int warp_tot[32];
  const int bh = blockIdx.x, i = threadIdx.x, lane = i & 31, w = i >> 5;
  int32_t* hh = hist + (int64_t)bh * nchunk * k;
  // Eight chunks' counts are loaded before any of them is overwritten, so each group of eight costs one
  // memory latency instead of eight.
  constexpr int G = 8;
  int run = 0;
  if (i < k)
    for (int c0 = 0; c0 < nchunk; c0 += G) {
      int n[G];
#pragma unroll
      for (int u = 0; u < G; ++u) n[u] = c0 + u < nchunk ? hh[(int64_t)(c0 + u) * k + i] : 0;
#pragma unroll
      for (int u = 0; u < G; ++u) {
        if (c0 + u < nchunk) hh[(int64_t)(c0 + u) * k + i] = run;
        run += n[u];
      }
    }
  // exclusive scan of the totals over the clusters
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = warp_tot[lane], xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += n;
    }
    warp_tot[lane] = xi - x;
  }
  __syncthreads();
  const int off = warp_tot[w] + incl - run;
  if (i < k) {
    counts[(int64_t)bh * k + i] = run;
    offsets[(int64_t)bh * k + i] = off;
    for (int c0 = 0; c0 < nchunk; c0 += G) {
      int n[G];
#pragma unroll
      for (int u = 0; u < G; ++u) n[u] = c0 + u < nchunk ? hh[(int64_t)(c0 + u) * k + i] : 0;
#pragma unroll
      for (int u = 0; u < G; ++u)
        if (c0 + u < nchunk) hh[(int64_t)(c0 + u) * k + i] = n[u] + off;
    }
  }
}

// (3) scatter: eight warps per chunk, warp w owning tokens [w*256, w*256+256) of the chunk; each
// warp's starting positions are the chunk's plus the counts of the warps before it, and within a
// warp the tokens go out 32 at a time in token order.
__global__ void __launch_bounds__(256) label_scatter_kernel(const int32_t* __restrict__ labels, int S, int k,
                                                            int nchunk, const int32_t* __restrict__ hist,
                                                            int32_t* __restrict__ perm) {
  __shared__ int pos[8][1024];
  const int c = blockIdx.x, bh = blockIdx.y;
  const int w = threadIdx.x >> 5;
  const unsigned lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 8 * 1024; i += 256) (&pos[0][0])[i] = 0;
  __syncthreads();
  const int32_t* z = labels + (int64_t)bh * S;
  const int t_begin = c * kChunk + w * (kChunk / 8);
  const int t_end = min(S, t_begin + kChunk / 8);
  for (int t = t_begin + (int)lane; t < t_end; t += 32) atomicAdd(&pos[w][z[t]], 1);
  __syncthreads();
  const int32_t* hc = hist + ((int64_t)bh * nchunk + c) * k;
  for (int i = threadIdx.x; i < k; i += 256) {
    int run = hc[i];
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {
      const int n = pos[ww][i];
      pos[ww][i] = run;
      run += n;
    }
  }
  __syncthreads();
  int32_t* p = perm + (int64_t)bh * S;
  for (int tb = t_begin; tb < t_end; tb += 32) {
    const int t = tb + (int)lane;
    const bool act = t < t_end;
    const int zz = act ? z[t] : -1 - (int)lane;  // inactive lanes get unique keys
    const unsigned peers = __match_any_sync(0xffffffffu, zz);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    if (act) p[pos[w][zz] + rank] = t;
    __syncwarp();
    if (act && rank == 0) pos[w][zz] += __popc(peers);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------------------------
// Update: one warp per cluster; lane l sums dims [l*D/32, (l+1)*D/32) of the member rows.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void two_sum_add(float& s, float& e, float x) {
  const float t = __fadd_rn(s, x);
  const float bp = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(x, bp));
  e = __fadd_rn(e, err);
  s = t;
}

template <int D>
__global__ void __launch_bounds__(256) kmeans_update_kernel(const uint16_t* __restrict__ v, int S, int k, int kpad,
                                                            const int32_t* __restrict__ perm,
                                                            const int32_t* __restrict__ counts,
                                                            const int32_t* __restrict__ offsets,
                                                            float* __restrict__ cent, float* __restrict__ cnorm,
                                                            uint16_t* __restrict__ cent16,
                                                            float* __restrict__ cnormp) {
  constexpr int E = D / 32;  // dims per lane: 4 (D = 128) or 2 (D = 64)
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + (threadIdx.x >> 5), bh = blockIdx.y;
  if (i >= k) return;
  const int n = counts[(int64_t)bh * k + i];
  const int o = offsets[(int64_t)bh * k + i];
  const uint16_t* vh = v + (int64_t)bh * S * D + lane * E;
  const int32_t* ph = perm + (int64_t)bh * S + o;
  float* c = cent + ((int64_t)bh * k + i) * D + lane * E;
  float cv[E];
  if (n > 0) {
    float s[E], e[E];
#pragma unroll
    for (int q = 0; q < E; ++q) s[q] = e[q] = 0.f;
    // Eight independent row loads in flight; the row indices of the next eight are fetched (one per
    // lane, handed out by shuffles) while this batch's rows load, so a batch waits for one memory
    // latency, not two. The rows are added in order, one after another, as in the plain loop.
    constexpr int R = 8;
    int m = 0;
    int idx = (lane < R && lane < n) ? __ldg(ph + lane) : 0;
    for (; m + R <= n; m += R) {
      uint32_t w[R][E / 2];
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const uint16_t* r = vh + (int64_t)__shfl_sync(0xffffffffu, idx, u) * D;
        if constexpr (E == 4) {
          const uint2 x = __ldg(reinterpret_cast<const uint2*>(r));
          w[u][0] = x.x;
          w[u][1] = x.y;
        } else {
          w[u][0] = __ldg(reinterpret_cast<const uint32_t*>(r));
        }
      }
      idx = (lane < R && m + R + lane < n) ? __ldg(ph + m + R + lane) : 0;
#pragma unroll
      for (int u = 0; u < R; ++u)
#pragma unroll
        for (int q = 0; q < E / 2; ++q) {
          two_sum_add(s[2 * q], e[2 * q], bf16_to_f32(w[u][q] & 0xFFFFu));
          two_sum_add(s[2 * q + 1], e[2 * q + 1], bf16_to_f32(w[u][q] >> 16));
        }
    }
    for (; m < n; ++m) {
      const uint16_t* r = vh + (int64_t)__ldg(ph + m) * D;
#pragma unroll
      for (int q = 0; q < E; ++q) two_sum_add(s[q], e[q], bf16_to_f32(r[q]));
    }
#pragma unroll
    for (int q = 0; q < E; ++q) {
      cv[q] = __fdiv_rn(__fadd_rn(s[q], e[q]), (float)n);
      c[q] = cv[q];
    }
  } else {
#pragma unroll
    for (int q = 0; q < E; ++q) cv[q] = c[q];
  }
  float nrm = 0.f;
#pragma unroll
  for (int q = 0; q < E; ++q) nrm = fmaf(cv[q], cv[q], nrm);
  nrm = warp_sum(nrm);
  uint16_t* hi = cent16 + ((int64_t)bh * 2 * kpad + i) * D;
  uint16_t* lo = hi + (int64_t)kpad * D;
#pragma unroll
  for (int q = 0; q < E; ++q) store_split(hi, lo, lane * E + q, cv[q]);
  if (lane == 0) {
    cnorm[(int64_t)bh * k + i] = nrm;
    cnormp[(int64_t)bh * kpad + i] = nrm;
  }
}

template <int D>
int launch_kmeans(const PlanBuffers& p, const uint16_t* V, int iters, bool warm, cudaStream_t st) {
  using C = AsgCfg<D>;
  const int BH = p.B * p.H, S = p.S, k = p.k, kpad = p.kpad;
  static std::atomic<uint64_t> attr_done{0};
  if (ensure_smem_attr(kmeans_assign_kernel<D>, C::SMEM, attr_done) != VC_OK) return VC_ERR_CUDA;
  CUtensorMap xmap, cmap;
  int rc = encode_2d(&xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<uint16_t*>(V), D, (uint64_t)BH * S,
                     (uint64_t)D * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc == VC_OK)
    rc = encode_2d(&cmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.cent16, D, (uint64_t)BH * 2 * kpad, (uint64_t)D * 2,
                   64, C::CH, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != VC_OK) return rc;
  const dim3 gc((kpad + 7) / 8, BH), gu((k + 7) / 8, BH);
  // Persistent assignment: one CTA per SM (all of an SM's shared memory), items spread round-robin.
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    return VC_ERR_CUDA;
  const int nwork = (S + C::TPC * 128 - 1) / (C::TPC * 128) * BH;
  const int ga = nwork < nsm ? nwork : nsm;
  const dim3 gh(p.nchunk, BH);
  // Warm start: the centroids of the plan's previous grouping (and their splits and norms) stay.
  if (!warm) kmeans_init_kernel<D><<<gc, 256, 0, st>>>(V, S, k, kpad, p.cent, p.cnorm, p.cent16, p.cnormp);
  for (int it = 0; it < iters; ++it) {
    // The first round of a cold start compares with data rows, whose lo halves are exactly zero: the
    // hi halves alone give the same dot products, so that round reads and multiplies only those.
    const int nparts = (it == 0 && !warm) ? 1 : 2;
    kmeans_assign_kernel<D><<<ga, 352, C::SMEM, st>>>(xmap, cmap, p.cnormp, S, kpad, nwork, nparts, p.labels,
                                                      p.status);
    label_hist_kernel<<<gh, 256, 0, st>>>(p.labels, S, k, p.nchunk, p.chist);
    label_scan_kernel<<<BH, 1024, 0, st>>>(k, p.nchunk, p.chist, p.counts, p.offsets);
    label_scatter_kernel<<<gh, 256, 0, st>>>(p.labels, S, k, p.nchunk, p.chist, p.perm);
    kmeans_update_kernel<D><<<gu, 256, 0, st>>>(V, S, k, kpad, p.perm, p.counts, p.offsets, p.cent, p.cnorm,
                                                p.cent16, p.cnormp);
  }
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace

int kmeans_launch(const PlanBuffers& p, const uint16_t* V, int iters, bool warm, cudaStream_t st) {
  return p.D == 128 ? launch_kmeans<128>(p, V, iters, warm, st) : launch_kmeans<64>(p, V, iters, warm, st);
}

int kmeans_chunks(int S) { return (S + kChunk - 1) / kChunk; }

}  // namespace vc
