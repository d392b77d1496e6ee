// vc_fwd.cu -- the fused ExpCast-FP8 + V-Smooth attention forward for sm_103a.
//
// "VC-Attention: Value Smoothing and Softmax Casting for Low-bit Attention": Sec. 3.1 Eq. 1
// (online softmax), Sec. 3.2 Eq. 6 (online mean restoration A <- alpha A + P~ R_q + r mu^T),
// Sec. 3.3 Eq. 7 (ExpCast-FP8); "Open-VC Attention" (MachGen blog), "Scheduling around ExpCast":
// one FMA per score with all scales and the running max folded in, running max on the true
// score with every increase applied, row sum of the decoded FP8 probabilities that feed PV,
// mid-window key order, packed transposed V.
//
// GB300 design (not the pages' kernel): one CTA per 128-row query tile and batch-head. This kernel serves
// D = 128; D = 64 runs the two-query-tile kernel of vc_fwd2.cu.
//   producers   TMA: Q once; K' tiles of 128 keys two at a time into a 2-stage ring, V^T tiles into
//               4 stages; with V-Smooth, the transposed bf16 means of each 16-tile block run into a
//               2-stage ring. The K' block scales of the head sit in shared memory in visiting order.
//   MMA issuer  one warp, one elected lane issuing: S = Q K'^T for two key tiles at once
//               (kind::f8f6f4, SS, N = 256) into the two TMEM score buffers; O += P V and
//               W += P E_{j mod 16} (TS: the codes P are read from TMEM),
//               where E_s is a one-hot 16 x 128 block, so column j mod 16 of W receives the exact
//               row sum of tile j; at the end of each run of tiles from one 16-tile block, the
//               mean term O += F M^T (kind::f16, F = W / sV split into bf16 hi + lo, M the block's
//               16 means) -- Eq. 6's r mu^T for 16 tiles at once, in the same accumulator.
//   warps 0-7   softmax, two warpgroups on alternate key tiles, one thread per query row: tile max
//               on the raw scores, handed to the other group as soon as it is known; each group
//               keeps the running max (code units) by folding in the other group's tile maxima;
//               O/W/l rescale on every increase, E4M3 codes written into TMEM.
//   warp 8      TMA producer of Q and the K pairs; warp 10 TMA producer of V (with the one-hot rows)
//               and the mean blocks; warp 9 MMA issuer.
// V residual repair ("Open-VC Attention", "Why V residual repair"): after the regular tiles the CTA
// visits the plan's repair tiles (copied keys, residual codes) through the same pipeline, with zero
// one-hot rows (nothing enters W or l) and the running max kept (codes clipped at 120).
// TMEM columns: O [0, D), W [D, D+16), F [D+16, D+32), l [D+32], P [176, 208) and [208, 240),
// score buffers S [256, 384) and [384, 512). P has its own columns, so the commit of score pair k, which
// tracks every earlier MMA of the issuing thread, also proves that PV(2k-3) has finished reading its P.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_fwd_common.cuh"
#include "vc_internal.h"

namespace vc {

template <int D>
struct FwdCfg {
  static constexpr int NKP = 2, NV = 4, NMU = 2;
  static constexpr int QB = 128 * D;             // bytes of a Q or K tile (128 rows x D codes)
  static constexpr int KPB = 2 * QB;             // a K stage: the two key tiles of one S pair
  static constexpr int VB = D * 128;             // bytes of a V^T tile (D rows x 128 keys)
  static constexpr int VSTAGE = (D + 16) * 128;  // V^T tile + 16 one-hot rows: the B operand of O|W += P [V; E]
  static constexpr int MUB = D * 32;             // bytes of a mean block (D rows x 16 bf16)
  static constexpr uint32_t QK_LAYOUT = D == 128 ? kSw128 : kSw64;
  static constexpr uint32_t QK_SBO = 8 * D;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB;
  static constexpr int OFF_V = OFF_K + NKP * KPB;
  static constexpr int OFF_MU = OFF_V + NV * VSTAGE;
  static constexpr int OFF_BAR = OFF_MU + NMU * MUB;
  static constexpr int NBAR = 1 + NKP + NV + 2 * NMU + 1 + 1 + 2 + 4 + 1 + 1 + 32;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_MBUF = OFF_MISC + 64;       // tile maxima hand-off, 8 slots x 128 floats
  static constexpr int OFF_SKS = OFF_MBUF + 4096;      // the K' block scales in visiting order, nkb floats
  static constexpr int SMEM = OFF_SKS + 1024;          // + the scale table; + slack for aligning the base to 1024
  static constexpr int MAX_NKB = 8192;                 // S <= 2^20
  static_assert(SMEM + 4 * MAX_NKB <= 227 * 1024, "shared memory per CTA");
  static_assert(OFF_V % 1024 == 0 && VSTAGE % 1024 == 0 && OFF_K % 1024 == 0, "128-byte swizzle atoms");
  // A V stage is refilled once PV of its previous tile is complete (o_done): with at most four
  // stages PV(t + 4) needs the tile being loaded, so that barrier cannot run two phases ahead.
  static_assert(NV <= 4, "V stages are released through o_done[t & 3]");
  // TMEM columns: O|W [0, D+16), F [D+16, D+32), l [D+32], P0 [176, 208), P1 [208, 240),
  // S pair [256, 512): the scores of tile 2k in [256, 384), of tile 2k+1 in [384, 512).
  static constexpr uint32_t T_O = 0, T_W = D, T_F = D + 16, T_L = D + 32, T_P0 = 176, T_P1 = 208, T_S = 256;
};

// Single-score export of the forward's four-score code path. kClamp: clamped at 120 afterwards, so
// that it matches the clip of Eq. 7 for every input. Without the clamp it writes exactly the bytes the
// forward's fast path writes (the forward skips the clamp while |M| < 2^22, where no code needs it).
template <bool kClamp>
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
  if (kClamp) d = __vminu4(d, 0x78787878u);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (i0 + q < n) out[i0 + q] = (uint8_t)((d >> (8 * q)) & 0xFFu);
}

template <int D, bool kExpCast, bool kRepair>
__global__ void __launch_bounds__(352, 1) vc_fwd_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base + C::OFF_Q;
  uint8_t* sK = base + C::OFF_K;
  uint8_t* sV = base + C::OFF_V;
  uint8_t* sMu = base + C::OFF_MU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;          // per K pair stage (a stage is free again once S of its pair is)
  uint64_t* v_full = k_full + C::NKP;     // per V pair slot (the first two of NV barriers): both tiles landed
  uint64_t* mu_full = v_full + C::NV;
  uint64_t* mu_empty = mu_full + C::NMU;
  uint64_t* s_full = mu_empty + C::NMU;   // S pair k landed (one phase per pair)
  // s_free phase k: both groups hold S pair k in registers (256 arrivals) and the K tiles of pair k+1
  // have landed (one arrival by the K producer), so the MMA thread learns both from one wait.
  uint64_t* s_free = s_full + 1;
  // p_full[g]: P of group g's tile written, O/W/l up to date (128 arrivals); p_full[0] also counts one
  // arrival by the V producer once both V^T tiles of the pair have landed, so that one wait of the MMA
  // thread covers the values of the pair as well.
  uint64_t* p_full = s_free + 1;
  // o_done[t & 3] completes when PV(t) and every earlier MMA are done. Parity waits only tell the
  // current phase from the previous one, so a wait for PV(v) must never find PV(v+4) complete too.
  // A group at tile t waits only for v > t-5 (every PV up to t-4 is known complete from S, see
  // below), and nothing past PV(t-1) can complete before this group's P(t) is published.
  uint64_t* o_done = p_full + 2;
  uint64_t* f_full = o_done + 4;
  uint64_t* drain = f_full + 1;
  // mx_full[slot][quarter]: the 32 raw-score tile maxima (code units) of one row quarter for
  // position t, slot t & 7, published by the group that owns t (32 arrivals, each after its own
  // mbuf store). Slot t & 7 is rewritten at t+8, whose scores exist only after the other group has
  // loaded position t+5 or later, i.e. after it has finished t+1, where it read the slot.
  uint64_t* mx_full = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + C::OFF_MISC + 8);
  float* mbuf = reinterpret_cast<float*>(base + C::OFF_MBUF);
  float* sks = reinterpret_cast<float*>(base + C::OFF_SKS);

  // The warp index read back from lane 0 is one the compiler knows to be warp-uniform: each role's
  // loop state and the MMA descriptors then live in uniform registers.
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int nkb = args.nkb;
  // Positions 0..nkb-1 visit the regular key tiles in the chosen order, positions nkb..ntiles-1 the
  // repair tiles (V residual repair) in order.
  const int ntiles = kRepair ? nkb + args.nrt : nkb;
  const int npairs = (ntiles + 1) / 2;
  // Mid-window order shared by the query tiles 2m and 2m+1: start at key tile 2m+2.
  const int start = (args.flags & VC_MIDWINDOW) ? min(nkb - 1, (qt & ~1) + 2) : -1;
  const bool use_mean = args.use_mean != 0;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NKP; ++s) mbar_init(&k_full[s], 1);
    for (int s = 0; s < C::NV; ++s) mbar_init(&v_full[s], 1);
    for (int s = 0; s < C::NMU; ++s) { mbar_init(&mu_full[s], 1); mbar_init(&mu_empty[s], 1); }
    mbar_init(s_full, 1);
    mbar_init(s_free, 257);
    mbar_init(&p_full[0], 129);
    mbar_init(&p_full[1], 128);
    for (int i = 0; i < 4; ++i) mbar_init(&o_done[i], 1);
    mbar_init(f_full, 128);
    mbar_init(drain, 1);
    *abort_flag = 0;
    for (int i = 0; i < 32; ++i) mbar_init(&mx_full[i], 32);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 512);
  // The K' block scales of this batch-head, in visiting order: the softmax loop then issues no global
  // load, so none is in flight when its barrier arrivals (releases) execute.
  for (int p = tid; p < nkb; p += blockDim.x) sks[p] = args.kscales[(int64_t)bh * nkb + tile_at(p, start)];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == 8) {
    // ------------------------------------------------------------------ K producer
    // Q once, then the two key tiles of every S pair into a 2-stage ring; independent of the V
    // ring, so the next pair is always in flight well before the MMA issuer needs it. The stage of
    // pair k-2 is free once S pair k-2 has landed (s_full), which the MMA thread committed after
    // its last read of the stage. Once pair k has landed, the producer adds its arrival to s_free's
    // phase k-1 (after which the MMA thread issues S pair k).
    if (lane == 0) {
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      if (kRepair) prefetch_tmap(&maps.krep);
      mbar_arrive_expect_tx(q_full, C::QB);
      tma_load_2d(sQ, &maps.q, 0, bh * args.S_pad + qt * 128, q_full);
      const int row0 = bh * args.S_pad, rrow0 = bh * args.R_pad;
      auto load_k = [&](uint8_t* dst, int t, uint64_t* bar) {
        if (!kRepair || t < nkb) tma_load_2d(dst, &maps.k, 0, row0 + tile_at(t, start) * 128, bar);
        else tma_load_2d(dst, &maps.krep, 0, rrow0 + (t - nkb) * 128, bar);
      };
      int issued_kp = 0;
      bool loads_ok = true;
      for (int k = 0; k < npairs; ++k) {
        if (*abort_flag) { loads_ok = false; break; }
        const int s = k % C::NKP;
        const int t0 = 2 * k, t1 = 2 * k + 1;
        if (k >= C::NKP && !wait_or_abort(s_full, (k - C::NKP) & 1, kWaitLimit, abort_flag)) { loads_ok = false; break; }
        mbar_arrive_expect_tx(&k_full[s], t1 < ntiles ? 2 * C::QB : C::QB);
        load_k(sK + s * C::KPB, t0, &k_full[s]);
        if (t1 < ntiles) load_k(sK + s * C::KPB + C::QB, t1, &k_full[s]);
        issued_kp = k + 1;
        if (k >= 1) {  // after phase k-2 of s_free, so that this arrival counts for phase k-1
          if (k >= 2 && !wait_or_abort(s_free, (k - 2) & 1, kWaitLimit, abort_flag)) { loads_ok = false; break; }
          if (!wait_or_abort(&k_full[s], (k / C::NKP) & 1, kWaitLimit, abort_flag)) { loads_ok = false; break; }
          mbar_arrive(s_free);
        }
      }
      if (!loads_ok) record_failure(args.status, abort_flag, kStatusTimeoutLoad);
      // Teardown: confirm that every load issued into this CTA's shared memory has landed.
      bool ok = mbar_wait(q_full, 0, kWaitLimit);
      for (int k = max(0, issued_kp - C::NKP); k < issued_kp; ++k)
        ok &= mbar_wait(&k_full[k % C::NKP], (k / C::NKP) & 1, kWaitLimit);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ V producer
    // Lane 0 waits and issues the copies; the whole warp writes the 16 one-hot rows under each V^T
    // tile (row j mod 16 holds E4M3 1.0), so that one MMA computes O += P V and W += P E at once.
    // The means of a block run are loaded just before the V tile of the next run's first position:
    // their ring stage was released by the mean MMA of the run two back, issued by the MMA thread
    // before it needs any V tile from that position on.
    const bool leader = lane == 0;
    if (leader) {
      prefetch_tmap(&maps.v);
      if (use_mean) prefetch_tmap(&maps.mu);
      if (kRepair) prefetch_tmap(&maps.vrep);
    }
    int issued_v = 0, issued_mu = 0;
    auto leader_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      bool ok = true;
      if (leader) ok = wait_or_abort(bar, parity, kWaitLimit, abort_flag);
      return __shfl_sync(0xffffffffu, ok, 0);
    };
    auto load_mean_block = [&](int block) -> bool {
      const int q = issued_mu, sm = q % C::NMU;
      if (!leader_wait(&mu_empty[sm], ((q / C::NMU) & 1) ^ 1)) return false;
      if (leader) {
        mbar_arrive_expect_tx(&mu_full[sm], C::MUB);
        tma_load_2d(sMu + sm * C::MUB, &maps.mu, block * 16, bh * D, &mu_full[sm]);
      }
      issued_mu = q + 1;
      return true;
    };
    // The two V^T tiles of a pair land on one barrier (v_full[pair % 2]); once they have, the producer
    // adds one arrival to the pair's p_full[0] phase, so the MMA thread learns of both from one wait.
    // A pair's slots are refilled once PV of the pair two back has completed.
    auto signal_v = [&](int kp) -> bool {
      if (kp >= 1 && !leader_wait(&p_full[0], (kp - 1) & 1)) return false;  // phase kp-1 done: this counts for kp
      if (!leader_wait(&v_full[kp & 1], (kp >> 1) & 1)) return false;
      if (leader) mbar_arrive(&p_full[0]);
      return true;
    };
    bool loads_ok = true;
    for (int t0 = 0; t0 < ntiles && loads_ok; t0 += 2) {
      if (warp_aborted(abort_flag)) { loads_ok = false; break; }
      if (t0 >= 2 && !signal_v(t0 / 2 - 1)) { loads_ok = false; break; }
      const int np = t0 + 1 < ntiles ? 2 : 1;
      for (int t = t0; t < t0 + np; ++t)
        if (use_mean && t > 0 && seg_start(t, start) && !load_mean_block(tile_at(t - 1, start) >> 4)) {
          loads_ok = false;
          break;
        }
      if (!loads_ok) break;
      if (t0 >= C::NV && !leader_wait(&o_done[(t0 - 3) & 3], ((t0 - 3) >> 2) & 1)) { loads_ok = false; break; }
      for (int t = t0; t < t0 + np; ++t) {  // one-hot rows (all zero under a repair tile: it adds nothing to
                                            // the row sums); a constant row is invariant under the swizzle
        const bool regular = !kRepair || t < nkb;
        const int j = regular ? tile_at(t, start) : t - nkb;
        uint4* onehot = reinterpret_cast<uint4*>(sV + (t % C::NV) * C::VSTAGE + C::VB);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = lane + 32 * q;
          const uint32_t v = (regular && (i >> 3) == (j & 15)) ? 0x38383838u : 0u;
          onehot[i] = make_uint4(v, v, v, v);
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (leader) {
        uint64_t* bar = &v_full[(t0 >> 1) & 1];
        mbar_arrive_expect_tx(bar, np * C::VB);
        for (int t = t0; t < t0 + np; ++t) {
          const bool regular = !kRepair || t < nkb;
          const int j = regular ? tile_at(t, start) : t - nkb;
          tma_load_2d(sV + (t % C::NV) * C::VSTAGE, regular ? &maps.v : &maps.vrep, j * 128, bh * D, bar);
        }
      }
      issued_v = t0 + np;
    }
    if (loads_ok && issued_v > 0 && !signal_v((issued_v - 1) / 2)) loads_ok = false;
    if (loads_ok && use_mean && !load_mean_block(tile_at(nkb - 1, start) >> 4)) loads_ok = false;  // the last run
    if (!loads_ok && leader) record_failure(args.status, abort_flag, kStatusTimeoutLoad);
    if (leader) {
      bool ok = true;
      const int issued_pairs = (issued_v + 1) / 2;
      for (int k = max(0, issued_pairs - 2); k < issued_pairs; ++k)
        ok &= mbar_wait(&v_full[k & 1], (k >> 1) & 1, kWaitLimit);
      for (int q = max(0, issued_mu - C::NMU); q < issued_mu; ++q)
        ok &= mbar_wait(&mu_full[q % C::NMU], (q / C::NMU) & 1, kWaitLimit);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule, so its loop state stays warp-uniform; one elected lane
    // issues every MMA group and commit (a commit tracks the MMAs of the thread that issues it).
    // Per pair k: once both groups hold S pair k in registers, S pair k+1 = Q K'(2k+2, 2k+3)^T as
    // one N = 256 MMA group; then per tile t of the pair, the mean term of a finished block run and
    // O|W += P(t) [V(t); E_{j mod 16}] as one N = D+16 MMA group.
    const bool leader = elect_one();
    const uint32_t tO = tmem + C::T_O, tF = tmem + C::T_F, tS = tmem + C::T_S;
    const uint32_t tP0 = tmem + C::T_P0, tP1 = tmem + C::T_P1;
    constexpr uint32_t id_qk = idesc_e4m3(128, 256), id_pv = idesc_e4m3(128, D + 16);
    constexpr uint32_t id_mu = idesc_bf16(128, D);
    // Descriptors are built once; a stage or K step only adds to the start-address field
    // (addresses are below 2^18, so the 14-bit field never carries).
    const uint64_t dq = smem_desc(sQ, C::QK_SBO, C::QK_LAYOUT);
    const uint64_t dk0 = smem_desc(sK, C::QK_SBO, C::QK_LAYOUT);
    const uint64_t dv0 = smem_desc(sV, 1024, kSw128);
    const uint64_t dmu0 = smem_desc(sMu, 256, kSw32);
    auto fail = [&](int bit) {
      if (lane == 0) record_failure(args.status, abort_flag, bit);
    };
    // S pair k; for k >= 1 the caller's s_free wait covers the K tiles (see s_free).
    auto issue_qk = [&](int k) -> bool {
      const int s = k % C::NKP;
      if (k == 0 && !warp_wait(&k_full[s], 0, kWaitLimit, abort_flag)) return false;
      tc_fence_after();
      if (leader) {
        const uint64_t dk = dk0 + (uint64_t)(s * (C::KPB >> 4));
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) mma_e4m3_ss(tS, dq + 2 * kk, dk + 2 * kk, id_qk, kk > 0);
        mma_commit(s_full);
      }
      __syncwarp();
      return true;
    };
    // O += F M^T for the block run with ordinal q: two K=16 bf16 MMAs, hi then lo.
    auto issue_mean = [&](int q) -> bool {
      const int sm = q % C::NMU;
      if (!warp_wait(&mu_full[sm], (q / C::NMU) & 1, kWaitLimit, abort_flag)) return false;
      tc_fence_after();
      if (leader) {
        const uint64_t bdesc = dmu0 + (uint64_t)(sm * (C::MUB >> 4));
        mma_bf16_ts(tO, tF, bdesc, id_mu, 1);
        mma_bf16_ts(tO, tF + 8, bdesc, id_mu, 1);
        mma_commit(&mu_empty[sm]);
      }
      __syncwarp();
      return true;
    };
    bool ok = warp_wait(q_full, 0, kWaitLimit, abort_flag) && issue_qk(0);
    if (!ok) fail(kStatusTimeoutLoad);
    int seg = -1;  // ordinal of the current block run
    for (int k = 0; ok && k < npairs; ++k) {
      if (k + 1 < npairs) {
        if (!warp_wait(s_free, k & 1, kWaitLimit, abort_flag)) {
          fail(kStatusTimeoutP);
          ok = false;
          break;
        }
        tc_fence_after();
        if (!issue_qk(k + 1)) {
          fail(kStatusTimeoutLoad);
          ok = false;
          break;
        }
      }
      for (int t = 2 * k; t <= 2 * k + 1 && t < ntiles; ++t) {
        const int g = t & 1;
        if (!warp_wait(&p_full[g], k & 1, kWaitLimit, abort_flag)) {
          fail(kStatusTimeoutP);
          ok = false;
          break;
        }
        tc_fence_after();
        if (seg_start(t, start)) {
          if (use_mean && seg >= 0 && !issue_mean(seg)) {
            fail(kStatusTimeoutLoad);
            ok = false;
            break;
          }
          ++seg;
        }
        const int sv = t % C::NV;
        if (leader) {
          const uint32_t tP = g ? tP1 : tP0;
          const uint64_t dv = dv0 + (uint64_t)(sv * (C::VSTAGE >> 4));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_e4m3_ts(tO, tP + 8 * kk, dv + 2 * kk, id_pv, (t > 0 || kk > 0));
          mma_commit(&o_done[t & 3]);  // also releases V stage t % NV to the V producer
        }
        __syncwarp();
      }
    }
    if (ok && use_mean && !warp_aborted(abort_flag)) {  // the last block run: its F arrives after the loop
      if (!warp_wait(f_full, 0, kWaitLimit, abort_flag) || !issue_mean(seg)) {
        fail(kStatusTimeoutP);
      } else {
        if (leader) mma_commit(&o_done[nkb & 3]);  // as if it were tile nkb
        __syncwarp();
      }
    }
    // Teardown: every MMA this warp issued has completed before TMEM is released.
    if (leader) mma_commit(drain);
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(drain, 0, kWaitLimit))) fail(kStatusTimeoutDrain);
  } else if (warp < 8) {
    // ------------------------------------------------------------------ softmax warps 0-7
    // Group g takes tile t = 2k + g of every S pair k, one thread per query row, its 128 scores
    // held in registers. The running max passes from one group to the next through shared memory
    // (published with a release store of the position). O, W and the row sum l (one TMEM column)
    // are touched only after PV of the previous tile has completed, which orders both groups'
    // updates; the rescale is done after the codes, so the wait for PV(t-1) overlaps the coding.
    const int wg = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const uint32_t tO = tmem + lane_base + C::T_O, tW = tmem + lane_base + C::T_W, tF = tmem + lane_base + C::T_F;
    const uint32_t tL = tmem + lane_base + C::T_L;
    const uint32_t tS = tmem + lane_base + C::T_S + 128 * wg;
    const uint32_t tP = tmem + lane_base + (wg ? C::T_P1 : C::T_P0);
    const float* skr = args.krep_scales + (int64_t)bh * args.nrt;
    const float aq = args.code_scale * args.qscales[(int64_t)bh * nkb + qt];
    // One scale per head: the means are in true units and the flush operand carries 1/sV. Per
    // channel: the means are already divided by the channel scales, and the epilogue applies them.
    const float* svch = args.vscales_ch ? args.vscales_ch + (int64_t)bh * D : nullptr;
    const float sv = args.vscales[bh];
    const float inv_sv = svch ? 1.f : 1.f / sv;
    const int tail_valid = args.S - (nkb - 1) * 128;
    bool ok = true;
    int known = -1;  // every PV up to this tile is known complete

    auto wait_o = [&](int t) -> bool {
      if (!warp_wait(&o_done[t & 3], (t >> 2) & 1, kWaitLimit, abort_flag)) {
        record_failure(args.status, abort_flag, kStatusTimeoutO);
        return false;
      }
      return true;
    };
    // PV(u) and everything before it complete, waiting tile by tile from the last known one.
    auto ensure_pv = [&](int u) -> bool {
      for (int v = known + 1; v <= u; ++v) {
        if (!wait_o(v)) return false;
        known = v;
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
    // Wait (bounded) until the tile max of position t-1 has been published (see mx_full).
    auto wait_tmax = [&](int t) -> bool {
      return warp_wait(&mx_full[((t - 1) & 7) * 4 + wq], ((t - 1) >> 3) & 1, kWaitLimit, abort_flag);
    };
    float Mrun = -INFINITY;  // this group's copy of the running max, after its previous tile

    if (wg == 0) {  // l starts at 0
      tmem_st1(tL, 0u);
      tmem_wait_st();
    }

    for (int k = 0; ok; ++k) {
      const int t = 2 * k + wg;
      if (t >= nkb) break;
      if (warp_aborted(abort_flag)) { ok = false; break; }
      const int j = tile_at(t, start);
      const float sk = sks[t];
      const uint32_t lim = (t == 0 && (args.flags & VC_DEBUG_TIMEOUT)) ? 0u : kWaitLimit;
      if (!warp_wait(s_full, k & 1, lim, abort_flag)) {
        record_failure(args.status, abort_flag, kStatusTimeoutS);
        ok = false;
        break;
      }
      tc_fence_after();
      known = max(known, 2 * k - 3);  // S pair k was issued after PV(2k-3)
      uint32_t sr[128];
      tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free);  // the next S pair may overwrite the score buffers
      float s[128];
#pragma unroll
      for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(sr[c]);
      if (j == nkb - 1 && tail_valid < 128) {  // keys past S: -inf for the max, code 0
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= tail_valid) s[c] = -INFINITY;
      }
      // Row max of the raw scores: eight independent max3 chains, then a short tree.
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
      const float tmax = mx * aj;  // = max_c fl(s_c * a_j): rounding is monotone and a_j > 0
      // The tile max goes to the other group at once; it depends on nothing else (with repair tiles the
      // last regular tile's max goes over too).
      if (t + 1 < ntiles) {
        mbuf[(t & 7) * 128 + row] = tmax;
        mbar_arrive(&mx_full[(t & 7) * 4 + wq]);  // release: orders this lane's store before the arrival
      }
      // M(t-1) = max(M(t-2), tmax(t-1)): this group's running max after its previous tile, with the
      // other group's tile in between folded in.
      float M = -INFINITY;
      if (t > 0) {
        if (!wait_tmax(t)) {
          record_failure(args.status, abort_flag, kStatusTimeoutS);
          ok = false;
          break;
        }
        M = fmaxf(Mrun, mbuf[((t - 1) & 7) * 128 + row]);
      }
      const float Mn = fmaxf(M, tmax);
      Mrun = Mn;
      // Codes. P(t) reuses the columns of P(t-2), which PV(t-2) must have read.
      if (!ensure_pv(t - 2)) { ok = false; break; }
      const float bb = __fsub_rn(kB0, Mn);
      const uint64_t a2 = pack2f(aj, aj), b2 = pack2f(bb, bb);
      if constexpr (kExpCast) {
        if (__all_sync(0xffffffffu, fabsf(Mn) < kClampFreeMaxAbsM)) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) {
              const int c = 64 * h + 4 * g;
              pk[g] = expcast4(s[c], s[c + 1], s[c + 2], s[c + 3], a2, a2, b2, b2);
            }
            tmem_st16(tP + 16 * h, pk);
          }
        } else {  // a running max beyond 2^22 code units: clip the codes at 120 byte by byte
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t pk[16];
#pragma unroll
            for (int g = 0; g < 16; ++g) {
              const int c = 64 * h + 4 * g;
              pk[g] = __vminu4(expcast4(s[c], s[c + 1], s[c + 2], s[c + 3], a2, a2, b2, b2), 0x78787878u);
            }
            tmem_st16(tP + 16 * h, pk);
          }
        }
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            const int c = 64 * h + 4 * g;
            pk[g] = pack4(expcast_off_code(s[c], aj, bb), expcast_off_code(s[c + 1], aj, bb),
                          expcast_off_code(s[c + 2], aj, bb), expcast_off_code(s[c + 3], aj, bb));
          }
          tmem_st16(tP + 16 * h, pk);
        }
      }
      // A new block run: the previous run's row sums (complete once PV(t-1) is done) leave W.
      // Every max increase rescales O, W and l by alpha = 2^((M - M')/8).
      const bool inc = (Mn > M) && (M > -INFINITY);
      const bool flush = t > 0 && seg_start(t, start);
      const bool any_inc = __any_sync(0xffffffffu, inc);
      if (flush || any_inc) {
        if (!ensure_pv(t - 1)) { ok = false; break; }
        const float alpha = inc ? ex2_approx(__fmul_rn(__fsub_rn(M, Mn), 0.125f)) : 1.f;
        float w[16];
        float ws = 0.f;
        if (flush) {  // take the run's row sums out of W and restart it at zero
          read_w(w);
#pragma unroll
          for (int i = 0; i < 16; ++i) ws += w[i];
          const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          tmem_st16(tW, zero);
        }
        const float lv = __uint_as_float(tmem_ld1(tL));
        tmem_wait_ld();
        if (any_inc) {
#pragma unroll 1
          for (int c0 = 0; c0 < (flush ? D : D + 16); c0 += 16) {
            uint32_t o[16];
            tmem_ld16(tO + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st16(tO + c0, o);
          }
        }
        tmem_st1(tL, __float_as_uint((lv + ws) * alpha));
        if (flush && use_mean) store_flush_operand(tF, w, inv_sv * alpha);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[wg]);
    }

    // Repair tiles (V residual repair): the running max is final after the regular tiles, so there is
    // no tile max, no rescale and no row-sum flush; the codes are clipped at 120 (a copied key's score
    // may sit slightly above M) and the zero one-hot rows keep them out of W and l.
    if constexpr (kRepair) {
      const int k0 = (nkb - wg + 1) / 2;  // this group's first repair position is 2 k0 + wg
      if (ok && 2 * k0 + wg - 1 == nkb - 1) {  // the other group had the last regular tile: fold in its max
        if (!wait_tmax(nkb)) {
          record_failure(args.status, abort_flag, kStatusTimeoutS);
          ok = false;
        } else {
          Mrun = fmaxf(Mrun, mbuf[((nkb - 1) & 7) * 128 + row]);
        }
      }
      const float bb = __fsub_rn(kB0, Mrun);
      const uint64_t b2 = pack2f(bb, bb);
      for (int k = k0; ok; ++k) {
        const int t = 2 * k + wg;
        if (t >= ntiles) break;
        if (warp_aborted(abort_flag)) { ok = false; break; }
        const float aj = aq * skr[t - nkb];
        if (!warp_wait(s_full, k & 1, kWaitLimit, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutS);
          ok = false;
          break;
        }
        tc_fence_after();
        known = max(known, 2 * k - 3);
        uint32_t sr[128];
        tmem_ld32(tS, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        tmem_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(s_free);
        if (!ensure_pv(t - 2)) { ok = false; break; }
        const uint64_t a2 = pack2f(aj, aj);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[16];
#pragma unroll
          for (int g = 0; g < 16; ++g) {
            const int c = 64 * h + 4 * g;
            const float s0 = __uint_as_float(sr[c]), s1 = __uint_as_float(sr[c + 1]);
            const float s2 = __uint_as_float(sr[c + 2]), s3 = __uint_as_float(sr[c + 3]);
            if constexpr (kExpCast) {
              pk[g] = __vminu4(expcast4(s0, s1, s2, s3, a2, a2, b2, b2), 0x78787878u);
            } else {
              pk[g] = pack4(expcast_off_code(s0, aj, bb), expcast_off_code(s1, aj, bb), expcast_off_code(s2, aj, bb),
                            expcast_off_code(s3, aj, bb));
            }
          }
          tmem_st16(tP + 16 * h, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[wg]);
      }
    }

    // Group 0 finishes: every PV done, the last run's row sums and means, then O = sV A / l (with
    // per-channel scales O[:, d] = s_d A[:, d] / l).
    if (wg == 0 && ok && !warp_aborted(abort_flag) && ensure_pv(ntiles - 1)) {
      float w[16];
      read_w(w);
      float ws = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ws += w[i];
      const float l = __uint_as_float(tmem_ld1(tL)) + ws;
      tmem_wait_ld();
      bool ready = true;
      if (use_mean) {  // the last block run's mean term, then the accumulator is final
        store_flush_operand(tF, w, inv_sv);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(f_full);
        ready = wait_o(nkb);
        tc_fence_after();
      }
      if (ready) {
        const float scale = svch ? 1.f / l : sv / l;
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
            float x0 = __uint_as_float(o[2 * i]), x1 = __uint_as_float(o[2 * i + 1]);
            if (svch) {
              x0 *= __ldg(svch + c0 + 2 * i);
              x1 *= __ldg(svch + c0 + 2 * i + 1);
            }
            __nv_bfloat162 h2 = __floats2bfloat162_rn(x0 * scale, x1 * scale);
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

int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows,
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
  if (rc == VC_OK && p.nrep > 0) {  // repair tiles: the copied keys and the residual codes, same boxes
    rc = encode_2d(&maps->krep, u8, p.krep, p.D, BH * p.R_pad, p.D, p.D, 128, qsw);
    if (rc == VC_OK)
      rc = encode_2d(&maps->vrep, u8, p.vrep, p.R_pad, BH * p.D, p.R_pad, 128, p.D, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  return rc;
}

template <int D, bool kExpCast, bool kRepair>
static int launch_fwd(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  using C = FwdCfg<D>;
  static std::atomic<uint64_t> attr_done{0};
  if (ensure_smem_attr(vc_fwd_kernel<D, kExpCast, kRepair>, C::SMEM + 4 * C::MAX_NKB, attr_done) != VC_OK)
    return VC_ERR_CUDA;
  FwdArgs a;
  a.qscales = p.qscales;
  a.kscales = p.kscales;
  a.vscales = p.vscales;
  a.vscales_ch = p.has_vchannel ? p.vscales_ch : nullptr;
  a.out = O;
  a.status = p.status;
  a.S = p.S;
  a.S_pad = p.S_pad;
  a.nkb = p.nkb;
  a.nrt = p.nrt;
  a.R_pad = p.R_pad;
  a.krep_scales = p.krep_scales;
  a.flags = flags;
  // 8 log2(e) / sqrt(D); rotated Q and K (Walsh-Hadamard, unnormalised) give D times the scores
  a.code_scale = (float)(p.has_hadamard ? 8.0 * 1.4426950408889634 / ((double)D * __builtin_sqrt((double)D))
                                        : 8.0 * 1.4426950408889634 / __builtin_sqrt((double)D));
  a.use_mean = (p.has_means && (flags & VC_VSMOOTH)) ? 1 : 0;
  if (a.use_mean && a.nrt > 0) return VC_ERR_INVALID_ARG;  // repair rows exist only without means
  dim3 grid(p.nkb, p.B * p.H);
  if (p.nkb > C::MAX_NKB) return VC_ERR_UNSUPPORTED;
  vc_fwd_kernel<D, kExpCast, kRepair><<<grid, 352, C::SMEM + 4 * ((p.nkb + 3) & ~3), st>>>(maps, a);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

template <int D>
static int launch_fwd_d(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  const bool ec = (flags & VC_EXPCAST) != 0, rp = p.nrt > 0;
  if (rp)
    return ec ? launch_fwd<D, true, true>(p, maps, O, flags, st) : launch_fwd<D, false, true>(p, maps, O, flags, st);
  return ec ? launch_fwd<D, true, false>(p, maps, O, flags, st) : launch_fwd<D, false, false>(p, maps, O, flags, st);
}

int forward_launch(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  // D = 64: the two-query-tile kernel (vc_fwd2.cu), faster there; at D = 128 its score buffers must be
  // split into halves to fit TMEM, and the one-query-tile kernel is faster.
  if (p.D == 64) return forward2_launch(p, maps, O, flags, st);
  // ExpCast on/off and repair tiles present/absent are separate instantiations, so the default kernel
  // carries only its own code.
  return launch_fwd_d<128>(p, maps, O, flags, st);
}

int expcast_launch(const float* s, const float* a, const float* b, int64_t n, uint8_t* out, cudaStream_t st,
                   bool clamp) {
  if (n <= 0) return VC_OK;
  const int64_t threads = (n + 3) / 4;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  if (clamp) expcast_kernel<true><<<blocks, 256, 0, st>>>(s, a, b, n, out);
  else expcast_kernel<false><<<blocks, 256, 0, st>>>(s, a, b, n, out);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

}  // namespace vc
