// vc_fwd2.cu -- the forward with two query tiles per CTA, one softmax warpgroup per query tile.
//
// Same arithmetic as vc_fwd.cu ("VC-Attention" Sec. 3.1 Eq. 1, Sec. 3.2 Eq. 6, Sec. 3.3 Eq. 7;
// "Open-VC Attention", "Scheduling around ExpCast": each CTA holds two 128-row query tiles that
// alternate, so one tile's softmax runs while the other's matrix multiplies execute). The query tiles
// 2m and 2m+1 share one mid-window order, so every K' and V^T tile is loaded once for both.
//
// Roles (11 warps):
//   warps 0-3   softmax of query tile 2m (group 0), warps 4-7 of query tile 2m+1 (group 1); one thread
//               per query row. Each group owns its rows outright: its running max and row sum stay in
//               registers, and nothing passes between the groups.
//   warp 8      TMA: both Q tiles, then the K' tiles into an NK-stage ring.
//   warp 10     TMA: the V^T tiles with their 16 one-hot rows into an NV-stage ring; the means.
//   warp 9      MMA issuer (one elected lane): per key tile, S_g = Q_g K'^T for both groups, in NH
//               sub-tiles of 128/NH keys (the score buffer of a group holds one sub-tile); then, once a
//               group's codes are written, its mean term and O_g|W_g += P_g [V; E_{j mod 16}].
// The K' block scales of the head sit in shared memory in visiting order, so the softmax loop issues no
// global load.
// TMEM, group g at column 256 g: O|W [0, D+16), P [D+16, D+48) (the 128 codes of a tile), F [D+48,
// D+64) (the mean operand), S [256 - 128/NH, 256).  D = 64 fits whole score tiles (NH = 1); D = 128
// would need NH = 2, measured slower than the one-query-tile kernel, so only D = 64 is launched.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_device.cuh"
#include "vc_fwd_common.cuh"
#include "vc_internal.h"

namespace vc {

template <int D>
struct Fwd2Cfg {
  static constexpr int NH = D == 128 ? 2 : 1;     // score sub-tiles per key tile
  static constexpr int SW = 128 / NH;             // keys (TMEM columns) per score sub-tile
  static constexpr int NK = 3, NV = 4, NMU = 2;
  static constexpr int QB = 128 * D;              // bytes of a Q or K tile
  static constexpr int VB = D * 128;              // bytes of a V^T tile
  static constexpr int VSTAGE = (D + 16) * 128;   // V^T tile + 16 one-hot rows
  static constexpr int MUB = D * 32;              // a mean block: D rows x 16 bf16
  static constexpr uint32_t QK_LAYOUT = D == 128 ? kSw128 : kSw64;
  static constexpr uint32_t QK_SBO = 8 * D;
  static constexpr int OFF_Q = 0;                 // Q of group 0, then of group 1
  static constexpr int OFF_K = OFF_Q + 2 * QB;
  static constexpr int OFF_V = OFF_K + NK * QB;
  static constexpr int OFF_MU = OFF_V + NV * VSTAGE;
  static constexpr int OFF_BAR = OFF_MU + NMU * MUB;
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 * NMU + 2 * 5 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int OFF_SKS = OFF_MISC + 64;      // the K' block scales in visiting order, nkb floats
  static constexpr int SMEM = OFF_SKS + 1024;         // + the scale table; + slack for aligning the base to 1024
  static constexpr int MAX_NKB = 8192;                // S <= 2^20
  static_assert(SMEM + 4 * MAX_NKB <= 227 * 1024, "shared memory per CTA");
  static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && VSTAGE % 1024 == 0 && QB % 1024 == 0,
                "swizzle atoms");
  static_assert((SW * D) % 1024 == 0, "a score sub-tile starts on a swizzle atom of the K tile");
  static constexpr uint32_t T_O = 0, T_W = D, T_P = D + 16, T_F = D + 48, T_S = 256 - SW;
  static_assert(T_F + 16 <= T_S, "TMEM columns of one group");
};

template <int D, bool kExpCast, bool kRepair>
__global__ void __launch_bounds__(352, 1) vc_fwd2_kernel(const __grid_constant__ FwdMaps maps, const FwdArgs args) {
  using C = Fwd2Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base + C::OFF_Q;
  uint8_t* sK = base + C::OFF_K;
  uint8_t* sV = base + C::OFF_V;
  uint8_t* sMu = base + C::OFF_MU;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;
  uint64_t* k_empty = k_full + C::NK;     // released by a commit after the last score MMA of the tile
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;     // released by a commit after group 1's PV of the tile
  uint64_t* mu_full = v_empty + C::NV;
  uint64_t* mu_empty = mu_full + C::NMU;
  // Per group g (two each): s_full[g] one phase per score sub-tile, s_free[g] the group holds that
  // sub-tile in registers (128 arrivals), p_full[g] one phase per tile (codes, O/W rescale and F
  // written; 128 arrivals), o_done[g] one phase per PV of the group (and one for its last mean term),
  // f_full[g] the last run's F (128 arrivals). s_free[0] phase t also counts one arrival by the K'
  // producer once tile t+1 has landed, and p_full[0] phase t one by the V producer once V^T tile t has
  // landed, so that the MMA thread waits for neither load separately. A phase can never run two ahead
  // of its waiter: each next phase needs an arrival or an MMA that the waiter's own progress gates.
  uint64_t* s_full = mu_empty + C::NMU;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* o_done = p_full + 2;
  uint64_t* f_full = o_done + 2;
  uint64_t* drain = f_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + C::OFF_MISC + 8);
  float* sks = reinterpret_cast<float*>(base + C::OFF_SKS);

  // The warp index read back from lane 0 is one the compiler knows to be warp-uniform: each role's
  // loop state and the MMA descriptors then live in uniform registers.
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  const int pair = blockIdx.x, bh = blockIdx.y;
  const int nkb = args.nkb;
  // Positions 0..nkb-1 visit the regular key tiles in the chosen order, nkb..ntiles-1 the repair tiles.
  const int ntiles = kRepair ? nkb + args.nrt : nkb;
  const int q0 = 2 * pair;  // query tiles q0 (group 0) and q0 + 1 (group 1; past the end when nkb is odd)
  const int start = (args.flags & VC_MIDWINDOW) ? min(nkb - 1, q0 + 2) : -1;
  const bool use_mean = args.use_mean != 0;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < C::NV; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int s = 0; s < C::NMU; ++s) { mbar_init(&mu_full[s], 1); mbar_init(&mu_empty[s], 1); }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&s_free[g], g == 0 ? 129 : 128);
      mbar_init(&p_full[g], g == 0 ? 129 : 128);  // group 0's two: + one producer arrival each
      mbar_init(&o_done[g], 1);
      mbar_init(&f_full[g], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
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
    // ------------------------------------------------------------------ Q and K' producer
    if (lane == 0) {
      prefetch_tmap(&maps.q);
      prefetch_tmap(&maps.k);
      if (kRepair) prefetch_tmap(&maps.krep);
      const int row0 = bh * args.S_pad;
      // The second Q tile of the last pair of an odd nkb starts past this head: the next head's
      // rows, or past the tensor (zero fill); its rows are never stored.
      mbar_arrive_expect_tx(q_full, 2 * C::QB);
      tma_load_2d(sQ, &maps.q, 0, row0 + q0 * 128, q_full);
      tma_load_2d(sQ + C::QB, &maps.q, 0, row0 + (q0 + 1) * 128, q_full);
      int issued = 0;
      bool loads_ok = true;
      for (int t = 0; t < ntiles; ++t) {
        if (*abort_flag) { loads_ok = false; break; }
        const int s = t % C::NK;
        if (!wait_or_abort(&k_empty[s], ((t / C::NK) & 1) ^ 1, kWaitLimit, abort_flag)) { loads_ok = false; break; }
        mbar_arrive_expect_tx(&k_full[s], C::QB);
        if (!kRepair || t < nkb) tma_load_2d(sK + s * C::QB, &maps.k, 0, row0 + tile_at(t, start) * 128, &k_full[s]);
        else tma_load_2d(sK + s * C::QB, &maps.krep, 0, bh * args.R_pad + (t - nkb) * 128, &k_full[s]);
        issued = t + 1;
        if (t >= 1) {  // tile t landed: one arrival on s_free[0]'s phase t-1 (after phase t-2)
          if (t >= 2 && !wait_or_abort(&s_free[0], (t - 2) & 1, kWaitLimit, abort_flag)) { loads_ok = false; break; }
          if (!wait_or_abort(&k_full[s], (t / C::NK) & 1, kWaitLimit, abort_flag)) { loads_ok = false; break; }
          mbar_arrive(&s_free[0]);
        }
      }
      if (!loads_ok) record_failure(args.status, abort_flag, kStatusTimeoutLoad);
      bool ok = mbar_wait(q_full, 0, kWaitLimit);
      for (int t = max(0, issued - C::NK); t < issued; ++t)
        ok &= mbar_wait(&k_full[t % C::NK], (t / C::NK) & 1, kWaitLimit);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ V^T and means producer
    // The whole warp writes the 16 one-hot rows under each V^T tile (row j mod 16 holds E4M3 1.0);
    // lane 0 waits and issues the copies. The means of a block run are loaded just before the V tile of
    // the next run's first position, as in the one-query-tile kernel.
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
    auto signal_v = [&](int u) -> bool {  // V(u) landed: one arrival on p_full[0]'s phase u
      if (u >= 1 && !leader_wait(&p_full[0], (u - 1) & 1)) return false;
      if (!leader_wait(&v_full[u % C::NV], (u / C::NV) & 1)) return false;
      if (leader) mbar_arrive(&p_full[0]);
      return true;
    };
    bool loads_ok = true;
    for (int t = 0; t < ntiles && loads_ok; ++t) {
      if (warp_aborted(abort_flag)) { loads_ok = false; break; }
      if (t >= 1 && !signal_v(t - 1)) { loads_ok = false; break; }
      const bool regular = !kRepair || t < nkb;  // a repair tile has zero one-hot rows: nothing enters W
      const int j = regular ? tile_at(t, start) : t - nkb;
      if (use_mean && t > 0 && seg_start(t, start) && !load_mean_block(tile_at(t - 1, start) >> 4)) {
        loads_ok = false;
        break;
      }
      const int sv = t % C::NV;
      if (!leader_wait(&v_empty[sv], ((t / C::NV) & 1) ^ 1)) { loads_ok = false; break; }
      {  // a constant row is invariant under the 16-byte chunk swizzle
        uint4* onehot = reinterpret_cast<uint4*>(sV + sv * C::VSTAGE + C::VB);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = lane + 32 * q;
          const uint32_t v = (regular && (i >> 3) == (j & 15)) ? 0x38383838u : 0u;
          onehot[i] = make_uint4(v, v, v, v);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }
      if (leader) {
        mbar_arrive_expect_tx(&v_full[sv], C::VB);
        tma_load_2d(sV + sv * C::VSTAGE, regular ? &maps.v : &maps.vrep, j * 128, bh * D, &v_full[sv]);
      }
      issued_v = t + 1;
    }
    if (loads_ok && issued_v > 0 && !signal_v(issued_v - 1)) loads_ok = false;
    if (loads_ok && use_mean && !load_mean_block(tile_at(nkb - 1, start) >> 4)) loads_ok = false;  // the last run
    if (!loads_ok && leader) record_failure(args.status, abort_flag, kStatusTimeoutLoad);
    if (leader) {
      bool ok = true;
      for (int t = max(0, issued_v - C::NV); t < issued_v; ++t)
        ok &= mbar_wait(&v_full[t % C::NV], (t / C::NV) & 1, kWaitLimit);
      for (int q = max(0, issued_mu - C::NMU); q < issued_mu; ++q)
        ok &= mbar_wait(&mu_full[q % C::NMU], (q / C::NMU) & 1, kWaitLimit);
      if (!ok) record_failure(args.status, abort_flag, kStatusTimeoutDrain);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------------ MMA issuer
    const bool leader = elect_one();
    uint32_t tS[2], tO[2], tP[2], tF[2];
    uint64_t dq[2];
    for (int g = 0; g < 2; ++g) {
      tS[g] = tmem + 256 * g + C::T_S;
      tO[g] = tmem + 256 * g + C::T_O;
      tP[g] = tmem + 256 * g + C::T_P;
      tF[g] = tmem + 256 * g + C::T_F;
      dq[g] = smem_desc(sQ + g * C::QB, C::QK_SBO, C::QK_LAYOUT);
    }
    constexpr uint32_t id_qk = idesc_e4m3(128, C::SW), id_pv = idesc_e4m3(128, D + 16);
    constexpr uint32_t id_mu = idesc_bf16(128, D);
    // Descriptors are built once; a stage, sub-tile or K step only adds to the start-address field
    // (addresses are below 2^18, so the 14-bit field never carries).
    const uint64_t dk0 = smem_desc(sK, C::QK_SBO, C::QK_LAYOUT);
    const uint64_t dv0 = smem_desc(sV, 1024, kSw128);
    const uint64_t dmu0 = smem_desc(sMu, 256, kSw32);
    auto fail = [&](int bit) {
      if (lane == 0) record_failure(args.status, abort_flag, bit);
    };
    // S_g = Q_g K'(t, sub-tile h)^T, once group g holds its previous sub-tile in registers.
    auto issue_qk = [&](int g, int t, int h) -> bool {
      const int u = t * C::NH + h;
      if (u > 0 && !warp_wait(&s_free[g], (u - 1) & 1, kWaitLimit, abort_flag)) return false;
      tc_fence_after();
      if (leader) {
        const uint64_t dk = dk0 + (uint64_t)(((t % C::NK) * C::QB + h * C::SW * D) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) mma_e4m3_ss(tS[g], dq[g] + 2 * kk, dk + 2 * kk, id_qk, kk > 0);
        mma_commit(&s_full[g]);
      }
      __syncwarp();
      return true;
    };
    // O_g += F_g M^T for the block run with ordinal q (hi then lo); the block is released after group 1.
    auto issue_mean = [&](int g, int q) -> bool {
      const int sm = q % C::NMU;
      if (g == 0) {
        if (!warp_wait(&mu_full[sm], (q / C::NMU) & 1, kWaitLimit, abort_flag)) return false;
        tc_fence_after();
      }
      if (leader) {
        const uint64_t bdesc = dmu0 + (uint64_t)(sm * (C::MUB >> 4));
        mma_bf16_ts(tO[g], tF[g], bdesc, id_mu, 1);
        mma_bf16_ts(tO[g], tF[g] + 8, bdesc, id_mu, 1);
        if (g == 1) mma_commit(&mu_empty[sm]);
      }
      __syncwarp();
      return true;
    };
    bool ok = warp_wait(q_full, 0, kWaitLimit, abort_flag) && warp_wait(&k_full[0], 0, kWaitLimit, abort_flag) &&
              issue_qk(0, 0, 0) && issue_qk(1, 0, 0);
    if (!ok) fail(kStatusTimeoutLoad);
    int seg = -1;  // ordinal of the current block run
    for (int t = 0; ok && t < ntiles; ++t) {
      for (int h = 1; ok && h < C::NH; ++h) {
        if (!issue_qk(0, t, h) || !issue_qk(1, t, h)) { fail(kStatusTimeoutP); ok = false; }
      }
      if (!ok) break;
      if (leader) mma_commit(&k_empty[t % C::NK]);  // every score MMA of tile t is issued
      __syncwarp();
      if (t + 1 < ntiles) {
        if (!issue_qk(0, t + 1, 0) || !issue_qk(1, t + 1, 0)) {
          fail(kStatusTimeoutP);
          break;
        }
      }
      const int sv = t % C::NV;
      const bool run = seg_start(t, start);
      for (int g = 0; ok && g < 2; ++g) {
        if (!warp_wait(&p_full[g], t & 1, kWaitLimit, abort_flag)) {
          fail(kStatusTimeoutP);
          ok = false;
          break;
        }
        tc_fence_after();
        if (run && use_mean && seg >= 0 && !issue_mean(g, seg)) {
          fail(kStatusTimeoutLoad);
          ok = false;
          break;
        }
        if (leader) {
          const uint64_t dv = dv0 + (uint64_t)(sv * (C::VSTAGE >> 4));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_e4m3_ts(tO[g], tP[g] + 8 * kk, dv + 2 * kk, id_pv, (t > 0 || kk > 0));
          mma_commit(&o_done[g]);
          if (g == 1) mma_commit(&v_empty[sv]);  // both PVs of this V tile are issued
        }
        __syncwarp();
      }
      if (run) ++seg;
    }
    if (ok && use_mean && !warp_aborted(abort_flag)) {  // the last block run: F arrives after the loops
      for (int g = 0; g < 2; ++g) {
        if (!warp_wait(&f_full[g], 0, kWaitLimit, abort_flag)) {
          fail(kStatusTimeoutP);
          break;
        }
        tc_fence_after();
        if (!issue_mean(g, seg)) {
          fail(kStatusTimeoutLoad);
          break;
        }
        if (leader) mma_commit(&o_done[g]);  // phase nkb of the group's o_done
        __syncwarp();
      }
    }
    // Teardown: every MMA issued here has completed before TMEM is released.
    if (leader) mma_commit(drain);
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(drain, 0, kWaitLimit))) fail(kStatusTimeoutDrain);
  } else if (warp < 8) {
    // ------------------------------------------------------------------ softmax, group g = query tile q0 + g
    const int g = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const int qt = q0 + g;
    const uint32_t tg = tmem + ((uint32_t)(wq * 32) << 16) + 256 * g;
    const uint32_t tO = tg + C::T_O, tW = tg + C::T_W, tP = tg + C::T_P, tF = tg + C::T_F, tS = tg + C::T_S;
    const float aq = args.code_scale * (qt < nkb ? args.qscales[(int64_t)bh * nkb + qt] : 1.f);
    // One scale per head: the means are in true units and the flush operand carries 1/sV. Per
    // channel: the means are already divided by the channel scales, and the epilogue applies them.
    const float* svch = args.vscales_ch ? args.vscales_ch + (int64_t)bh * D : nullptr;
    const float sv = args.vscales[bh];
    const float inv_sv = svch ? 1.f : 1.f / sv;
    const int tail_valid = args.S - (nkb - 1) * 128;
    bool ok = true;
    float Mrun = -INFINITY;  // running max of this group's rows (code units)
    float l = 0.f;           // row sum of every run flushed out of W so far
    auto wait_o = [&](int phase) -> bool {
      if (!warp_wait(&o_done[g], phase & 1, kWaitLimit, abort_flag)) {
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
    // The 128 raw scores of position t, sub-tile by sub-tile; each sub-tile's buffer is released as soon
    // as it is in registers.
    auto load_scores = [&](int t, float(&s)[128]) -> bool {
#pragma unroll
      for (int h = 0; h < C::NH; ++h) {
        const int u = t * C::NH + h;
        const uint32_t lim = (u == 0 && (args.flags & VC_DEBUG_TIMEOUT)) ? 0u : kWaitLimit;
        if (!warp_wait(&s_full[g], u & 1, lim, abort_flag)) {
          record_failure(args.status, abort_flag, kStatusTimeoutS);
          return false;
        }
        tc_fence_after();
        uint32_t sr[C::SW];
#pragma unroll
        for (int c0 = 0; c0 < C::SW; c0 += 32) tmem_ld32(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&s_free[g]);
#pragma unroll
        for (int c = 0; c < C::SW; ++c) s[h * C::SW + c] = __uint_as_float(sr[c]);
      }
      return true;
    };
    for (int t = 0; ok && t < nkb; ++t) {
      if (warp_aborted(abort_flag)) { ok = false; break; }
      const int j = tile_at(t, start);
      const float sk = sks[t];
      float s[128];
      if (!load_scores(t, s)) { ok = false; break; }
      if (j == nkb - 1 && tail_valid < 128) {  // keys past S: -inf for the max, code 0
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= tail_valid) s[c] = -INFINITY;
      }
      // Row max of the raw scores: eight independent max3 chains, then a short tree.
      float m8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float x = max3f(s[16 * q], s[16 * q + 1], s[16 * q + 2]);
#pragma unroll
        for (int c = 3; c < 15; c += 2) x = max3f(x, s[16 * q + c], s[16 * q + c + 1]);
        m8[q] = fmaxf(x, s[16 * q + 15]);
      }
      const float mx = fmaxf(max3f(m8[0], m8[1], m8[2]), max3f(max3f(m8[3], m8[4], m8[5]), m8[6], m8[7]));
      const float aj = aq * sk;
      const float M = Mrun;
      const float Mn = fmaxf(M, mx * aj);  // mx * aj = max_c fl(s_c * a_j): rounding is monotone, a_j > 0
      Mrun = Mn;
      const float bb = __fsub_rn(kB0, Mn);
      const uint64_t a2 = pack2f(aj, aj), b2 = pack2f(bb, bb);
      uint32_t pk[32];
      if constexpr (kExpCast) {
        if (__all_sync(0xffffffffu, fabsf(Mn) < kClampFreeMaxAbsM)) {
#pragma unroll
          for (int q = 0; q < 32; ++q)
            pk[q] = expcast4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3], a2, a2, b2, b2);
        } else {  // a running max beyond 2^22 code units: clip the codes at 120 byte by byte
#pragma unroll
          for (int q = 0; q < 32; ++q)
            pk[q] = __vminu4(expcast4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3], a2, a2, b2, b2), 0x78787878u);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 32; ++q)
          pk[q] = pack4(expcast_off_code(s[4 * q], aj, bb), expcast_off_code(s[4 * q + 1], aj, bb),
                        expcast_off_code(s[4 * q + 2], aj, bb), expcast_off_code(s[4 * q + 3], aj, bb));
      }
      // PV(t-1) has read P and updated O|W before either is touched again.
      if (t > 0 && !wait_o(t - 1)) { ok = false; break; }
      tmem_st16(tP, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
      tmem_st16(tP + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
      // A new block run: the previous run's row sums leave W. Every max increase rescales O, W and l
      // by alpha = 2^((M - M')/8).
      const bool inc = (Mn > M) && (M > -INFINITY);
      const bool flush = t > 0 && seg_start(t, start);
      const bool any_inc = __any_sync(0xffffffffu, inc);
      if (flush || any_inc) {
        const float alpha = inc ? ex2_approx(__fmul_rn(__fsub_rn(M, Mn), 0.125f)) : 1.f;
        float w[16];
        float ws = 0.f;
        if (flush) {
          read_w(w);
#pragma unroll
          for (int i = 0; i < 16; ++i) ws += w[i];
          const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          tmem_st16(tW, zero);
        }
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
        l = (l + ws) * alpha;
        if (flush && use_mean) store_flush_operand(tF, w, inv_sv * alpha);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[g]);
    }

    // Repair tiles (V residual repair): the running max is final, so there is no tile max, rescale or
    // flush; the codes are clipped at 120 (a copied key may score slightly above M), and the zero
    // one-hot rows keep them out of W and l.
    if constexpr (kRepair) {
      const float* skr = args.krep_scales + (int64_t)bh * args.nrt;
      const float bb = __fsub_rn(kB0, Mrun);
      const uint64_t b2 = pack2f(bb, bb);
      for (int t = nkb; ok && t < ntiles; ++t) {
        if (warp_aborted(abort_flag)) { ok = false; break; }
        const float aj = aq * skr[t - nkb];
        float s[128];
        if (!load_scores(t, s)) { ok = false; break; }
        const uint64_t a2 = pack2f(aj, aj);
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          if constexpr (kExpCast) {
            pk[q] = __vminu4(expcast4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3], a2, a2, b2, b2), 0x78787878u);
          } else {
            pk[q] = pack4(expcast_off_code(s[4 * q], aj, bb), expcast_off_code(s[4 * q + 1], aj, bb),
                          expcast_off_code(s[4 * q + 2], aj, bb), expcast_off_code(s[4 * q + 3], aj, bb));
          }
        }
        if (!wait_o(t - 1)) { ok = false; break; }
        tmem_st16(tP, *reinterpret_cast<const uint32_t(*)[16]>(&pk[0]));
        tmem_st16(tP + 16, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16]));
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_full[g]);
      }
    }

    // Every PV of this group done: the last run's row sums and means, then O = sV A / l (with
    // per-channel scales O[:, d] = s_d A[:, d] / l).
    if (ok && !warp_aborted(abort_flag) && wait_o(ntiles - 1)) {
      float w[16];
      read_w(w);
      float ws = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) ws += w[i];
      const float lf = l + ws;
      bool ready = true;
      if (use_mean) {  // the last run's mean term, then the accumulator is final
        store_flush_operand(tF, w, inv_sv);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&f_full[g]);
        ready = wait_o(ntiles);
      }
      if (ready && qt < nkb) {
        const float scale = svch ? 1.f / lf : sv / lf;
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

template <int D, bool kExpCast, bool kRepair>
static int launch_fwd2(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  using C = Fwd2Cfg<D>;
  static std::atomic<uint64_t> attr_done{0};
  if (ensure_smem_attr(vc_fwd2_kernel<D, kExpCast, kRepair>, C::SMEM + 4 * C::MAX_NKB, attr_done) != VC_OK)
    return VC_ERR_CUDA;
  FwdArgs a;
  a.qscales = p.qscales;
  a.kscales = p.kscales;
  a.vscales = p.vscales;
  a.vscales_ch = p.has_vchannel ? p.vscales_ch : nullptr;
  a.out = O;
  a.status = p.status;
  a.krep_scales = p.krep_scales;
  a.S = p.S;
  a.S_pad = p.S_pad;
  a.nkb = p.nkb;
  a.nrt = p.nrt;
  a.R_pad = p.R_pad;
  a.flags = flags;
  // 8 log2(e) / sqrt(D); rotated Q and K (Walsh-Hadamard, unnormalised) give D times the scores
  a.code_scale = (float)(p.has_hadamard ? 8.0 * 1.4426950408889634 / ((double)D * __builtin_sqrt((double)D))
                                        : 8.0 * 1.4426950408889634 / __builtin_sqrt((double)D));
  a.use_mean = (p.has_means && (flags & VC_VSMOOTH)) ? 1 : 0;
  if (a.use_mean && a.nrt > 0) return VC_ERR_INVALID_ARG;  // repair rows exist only without means
  dim3 grid((p.nkb + 1) / 2, p.B * p.H);
  if (p.nkb > C::MAX_NKB) return VC_ERR_UNSUPPORTED;
  vc_fwd2_kernel<D, kExpCast, kRepair><<<grid, 352, C::SMEM + 4 * ((p.nkb + 3) & ~3), st>>>(maps, a);
  return cudaPeekAtLastError() == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

// Used for D = 64. The kernel also builds for D = 128 with score half-tiles, but there the one-query-tile
// kernel is faster (59.1 against 71.8 ms on the 40-head, 75600-token case).
int forward2_launch(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st) {
  if (p.D != 64) return VC_ERR_UNSUPPORTED;
  const bool ec = (flags & VC_EXPCAST) != 0;
  if (p.nrt > 0)
    return ec ? launch_fwd2<64, true, true>(p, maps, O, flags, st)
              : launch_fwd2<64, false, true>(p, maps, O, flags, st);
  return ec ? launch_fwd2<64, true, false>(p, maps, O, flags, st)
            : launch_fwd2<64, false, false>(p, maps, O, flags, st);
}

}  // namespace vc
