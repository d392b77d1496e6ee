// vc_abi.cu -- the C ABI declared in include/vc_attn.h: argument checks, the plan object (one
// device allocation carved into the prepare/forward buffers), and stream-ordered dispatch.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "vc_internal.h"

struct vc_plan {
  vc::PlanBuffers b;
  vc::FwdMaps maps;
  void* block;
  size_t block_bytes;
  int device;
};

namespace {

constexpr int kMaxS = 1 << 20;
constexpr int kMaxK = 1024;
constexpr int kMaxIters = 64;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VC_ERR_NO_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return VC_ERR_NO_DEVICE;
  return (major == 10 && minor == 3) ? VC_OK : VC_ERR_NO_DEVICE;
}

// A plan's buffers and tensor maps live on the device that was current when it was created.
bool on_plan_device(const vc_plan* plan) {
  int cur = -1;
  return cudaGetDevice(&cur) == cudaSuccess && cur == plan->device;
}

int check_shape(int B, int H, int S, int D, int k) {
  if (B < 1 || H < 1 || S < 1 || k < 1) return VC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return VC_ERR_UNSUPPORTED;
  if (S > kMaxS || k > kMaxK || k > S) return VC_ERR_UNSUPPORTED;
  const int64_t BH = (int64_t)B * H;
  const int64_t S_pad = ((int64_t)S + 127) / 128 * 128;
  if (BH > 65535) return VC_ERR_UNSUPPORTED;             // grid.y
  if (BH * S_pad >= (int64_t)1 << 31) return VC_ERR_UNSUPPORTED;  // TMA row coordinate
  if (BH * S_pad * D >= (int64_t)1 << 40) return VC_ERR_UNSUPPORTED;
  return VC_OK;
}

size_t align_up(size_t x) { return (x + 255) & ~(size_t)255; }

int plan_create(int B, int H, int S, int D, int k, int nrep, vc_plan** out) {
  vc_plan* pl = (vc_plan*)calloc(1, sizeof(vc_plan));
  if (!pl) return VC_ERR_OOM;
  vc::PlanBuffers& b = pl->b;
  b.B = B; b.H = H; b.S = S; b.D = D; b.k = k;
  b.nkb = (S + 127) / 128;
  b.S_pad = b.nkb * 128;
  b.nkb16 = (b.nkb + 15) / 16 * 16;
  b.kpad = (k + 127) / 128 * 128;
  b.nchunk = vc::kmeans_chunks(S);
  b.nrep = nrep;
  b.nrt = (nrep + 127) / 128;
  b.R_pad = b.nrt * 128;
  const size_t BH = (size_t)B * H;
  const size_t codes = BH * b.S_pad * D;
  const size_t sizes[] = {
      codes,                          // qcodes
      BH * b.nkb * 4,                 // qscales
      codes,                          // kcodes
      BH * b.nkb * 4,                 // kscales
      codes,                          // vcodes
      BH * 4,                         // vscales
      BH * b.nkb * D * 2,             // means
      BH * b.nkb16 * D * 2,           // meansT
      BH * S * 4,                     // labels
      BH * S * 4,                     // perm
      BH * k * D * 4,                 // cent
      BH * k * 4,                     // cnorm
      BH * k * 4,                     // counts
      BH * k * 4,                     // offsets
      BH * 2 * b.kpad * D * 2,        // cent16
      BH * b.kpad * 4,                // cnormp
      BH * b.nchunk * k * 4,          // chist
      BH * D * 4,                     // kexp
      BH * D * 8,                     // ksum
      BH * D * 2,                     // kmu
      BH * 4,                         // vamax
      BH * D * 4,                     // vamax_ch
      BH * D * 4,                     // vscales_ch
      BH * nrep * 4,                  // rep_idx
      nrep ? BH * S * 4 : 0,          // energy
      BH * b.R_pad * D,               // krep
      BH * b.nrt * 4,                 // krep_scales
      BH * D * b.R_pad,               // vrep
      16,                             // status
  };
  size_t total = 0;
  for (size_t s : sizes) total += align_up(s);
  void* blk = nullptr;
  if (cudaMalloc(&blk, total) != cudaSuccess) {
    cudaGetLastError();
    free(pl);
    return VC_ERR_OOM;
  }
  uint8_t* p = (uint8_t*)blk;
  void** slots[] = {(void**)&b.qcodes, (void**)&b.qscales, (void**)&b.kcodes, (void**)&b.kscales,
                    (void**)&b.vcodes, (void**)&b.vscales, (void**)&b.means,   (void**)&b.meansT, (void**)&b.labels,
                    (void**)&b.perm,   (void**)&b.cent,    (void**)&b.cnorm,   (void**)&b.counts,
                    (void**)&b.offsets, (void**)&b.cent16, (void**)&b.cnormp,  (void**)&b.chist,
                    (void**)&b.kexp,   (void**)&b.ksum,    (void**)&b.kmu,
                    (void**)&b.vamax,  (void**)&b.vamax_ch, (void**)&b.vscales_ch, (void**)&b.rep_idx,
                    (void**)&b.energy, (void**)&b.krep,     (void**)&b.krep_scales, (void**)&b.vrep,
                    (void**)&b.status};
  for (size_t i = 0; i < sizeof(sizes) / sizeof(sizes[0]); ++i) {
    *slots[i] = p;
    p += align_up(sizes[i]);
  }
  if (cudaMemset(blk, 0, total) != cudaSuccess) {
    cudaFree(blk);
    free(pl);
    return VC_ERR_CUDA;
  }
  pl->block = blk;
  pl->block_bytes = total;
  cudaGetDevice(&pl->device);
  int rc = vc::encode_fwd_maps(b, &pl->maps);
  if (rc != VC_OK) {
    cudaFree(blk);
    free(pl);
    return rc;
  }
  *out = pl;
  return VC_OK;
}

int prepare_impl(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int k_clusters, int iters,
                 const int32_t* perm, unsigned flags, int n_repair, cudaStream_t stream, vc_plan** plan) {
  if (!Q || !K || !V || !plan) return VC_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V)) return VC_ERR_INVALID_ARG;
  int rc = check_shape(B, H, S, D, k_clusters);
  if (rc != VC_OK) return rc;
  const bool vsmooth = (flags & VC_VSMOOTH) != 0;
  const bool reuse_perm = (flags & VC_REUSE_PERM) != 0;
  const bool grouping = vsmooth && !perm && !reuse_perm;
  const bool warm = grouping && (flags & VC_WARM_START) != 0;
  if (grouping && (iters < 1 || iters > kMaxIters)) return VC_ERR_INVALID_ARG;
  if (reuse_perm && perm) return VC_ERR_INVALID_ARG;
  // Repair rows are defined on the plain per-head (or per-channel) quantisation only.
  if (n_repair < 0 || n_repair > S || (n_repair > 0 && (vsmooth || reuse_perm))) return VC_ERR_INVALID_ARG;
  // A warm start needs the centroids of an earlier grouping, a reuse the permutation of an earlier
  // prepare: both only on an existing plan.
  if ((warm && !(*plan && (*plan)->b.has_grouping)) || (reuse_perm && !(*plan && (*plan)->b.has_perm)))
    return VC_ERR_INVALID_ARG;
  rc = check_device();
  if (rc != VC_OK) return rc;
  if (*plan) {
    if (!on_plan_device(*plan)) return VC_ERR_INVALID_ARG;
    const vc::PlanBuffers& b = (*plan)->b;
    if (b.B != B || b.H != H || b.S != S || b.D != D || b.k != k_clusters || b.nrep != n_repair)
      return VC_ERR_PLAN_MISMATCH;
  } else {
    rc = plan_create(B, H, S, D, k_clusters, n_repair, plan);
    if (rc != VC_OK) return rc;
  }
  vc_plan* pl = *plan;
  pl->b.has_means = vsmooth;
  pl->b.has_kcenter = (flags & VC_KCENTER) != 0;
  pl->b.has_vchannel = (flags & VC_VSCALE_CHANNEL) != 0;
  pl->b.has_hadamard = (flags & VC_QK_HADAMARD) != 0;
  rc = vc::prepare_launch(pl->b, (const uint16_t*)Q, (const uint16_t*)K, (const uint16_t*)V,
                          vsmooth ? perm : nullptr, vsmooth, pl->b.has_kcenter, reuse_perm, warm,
                          pl->b.has_vchannel, iters, stream);
  if (rc == VC_OK) {
    if (grouping) pl->b.has_grouping = true;
    pl->b.has_perm = true;
  }
  return rc;
}

}  // namespace

extern "C" {

int vc_attn_prepare_ex(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int k_clusters,
                       int iters, const int32_t* perm, unsigned flags, cudaStream_t stream, vc_plan** plan) {
  return prepare_impl(Q, K, V, B, H, S, D, k_clusters, iters, perm, flags, 0, stream, plan);
}

int vc_attn_prepare_repair(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int n_repair,
                           unsigned flags, cudaStream_t stream, vc_plan** plan) {
  return prepare_impl(Q, K, V, B, H, S, D, 1, 1, nullptr, flags, n_repair, stream, plan);
}

int vc_attn_prepare(const void* Q, const void* K, const void* V, int B, int H, int S, int D, int k_clusters,
                    int iters, cudaStream_t stream, vc_plan** plan) {
  return vc_attn_prepare_ex(Q, K, V, B, H, S, D, k_clusters, iters, nullptr, VC_VSMOOTH, stream, plan);
}

int vc_attn_forward(const vc_plan* plan, void* O, unsigned flags, cudaStream_t stream) {
  if (!plan || !O || !aligned16(O)) return VC_ERR_INVALID_ARG;
  const unsigned known = VC_EXPCAST | VC_VSMOOTH | VC_MIDWINDOW | VC_DEBUG_TIMEOUT;
  if (flags & ~known) return VC_ERR_INVALID_ARG;
  if (!on_plan_device(plan)) return VC_ERR_INVALID_ARG;
  return vc::forward_launch(plan->b, plan->maps, (uint16_t*)O, flags, stream);
}

size_t vc_plan_size(const vc_plan* plan, int what) {
  if (!plan) return 0;
  const vc::PlanBuffers& b = plan->b;
  const size_t BH = (size_t)b.B * b.H;
  switch (what) {
    case VC_PLAN_LABELS:
    case VC_PLAN_PERM: return BH * b.S * 4;
    case VC_PLAN_QCODES:
    case VC_PLAN_KCODES:
    case VC_PLAN_VCODES: return BH * b.S_pad * b.D;
    case VC_PLAN_QSCALES:
    case VC_PLAN_KSCALES: return BH * b.nkb * 4;
    case VC_PLAN_VSCALES: return BH * 4;
    case VC_PLAN_MEANS: return BH * b.nkb * b.D * 2;
    case VC_PLAN_CENTROIDS: return BH * b.k * b.D * 4;
    case VC_PLAN_KCENTER: return BH * b.D * 2;
    case VC_PLAN_VCHSCALES: return BH * b.D * 4;
    case VC_PLAN_MEANS_T: return BH * b.D * b.nkb16 * 2;
    case VC_PLAN_REPAIR_IDX: return BH * b.nrep * 4;
    case VC_PLAN_REPAIR_ENERGY: return b.nrep ? BH * b.S * 4 : 0;
    case VC_PLAN_REPAIR_KCODES: return BH * b.R_pad * b.D;
    case VC_PLAN_REPAIR_KSCALES: return BH * b.nrt * 4;
    case VC_PLAN_REPAIR_VCODES: return BH * b.D * b.R_pad;
    default: return 0;
  }
}

int vc_plan_get(const vc_plan* plan, int what, void* dst, size_t bytes, cudaStream_t stream) {
  size_t n = vc_plan_size(plan, what);
  if (!n || !dst || bytes < n) return VC_ERR_INVALID_ARG;
  const vc::PlanBuffers& b = plan->b;
  const void* src = nullptr;
  switch (what) {
    case VC_PLAN_LABELS: src = b.labels; break;
    case VC_PLAN_PERM: src = b.perm; break;
    case VC_PLAN_QCODES: src = b.qcodes; break;
    case VC_PLAN_QSCALES: src = b.qscales; break;
    case VC_PLAN_KCODES: src = b.kcodes; break;
    case VC_PLAN_KSCALES: src = b.kscales; break;
    case VC_PLAN_VCODES: src = b.vcodes; break;
    case VC_PLAN_VSCALES: src = b.vscales; break;
    case VC_PLAN_MEANS: src = b.means; break;
    case VC_PLAN_CENTROIDS: src = b.cent; break;
    case VC_PLAN_KCENTER: src = b.kmu; break;
    case VC_PLAN_VCHSCALES: src = b.vscales_ch; break;
    case VC_PLAN_MEANS_T: src = b.meansT; break;
    case VC_PLAN_REPAIR_IDX: src = b.rep_idx; break;
    case VC_PLAN_REPAIR_ENERGY: src = b.energy; break;
    case VC_PLAN_REPAIR_KCODES: src = b.krep; break;
    case VC_PLAN_REPAIR_KSCALES: src = b.krep_scales; break;
    case VC_PLAN_REPAIR_VCODES: src = b.vrep; break;
  }
  return cudaMemcpyAsync(dst, src, n, cudaMemcpyDefault, stream) == cudaSuccess ? VC_OK : VC_ERR_CUDA;
}

int vc_plan_status(vc_plan* plan, cudaStream_t stream, int* bits) {
  if (!plan) return VC_ERR_INVALID_ARG;
  int h = 0;
  if (cudaMemcpyAsync(&h, plan->b.status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return VC_ERR_CUDA;
  if (h && cudaMemsetAsync(plan->b.status, 0, sizeof(int), stream) != cudaSuccess) return VC_ERR_CUDA;
  if (bits) *bits = h;
  return h ? VC_ERR_TIMEOUT : VC_OK;
}

int vc_plan_shape(const vc_plan* plan, int* B, int* H, int* S, int* D, int* k_clusters) {
  if (!plan) return VC_ERR_INVALID_ARG;
  if (B) *B = plan->b.B;
  if (H) *H = plan->b.H;
  if (S) *S = plan->b.S;
  if (D) *D = plan->b.D;
  if (k_clusters) *k_clusters = plan->b.k;
  return VC_OK;
}

void vc_plan_destroy(vc_plan* plan) {
  if (!plan) return;
  int cur = 0;
  cudaGetDevice(&cur);
  if (cur != plan->device) cudaSetDevice(plan->device);
  cudaDeviceSynchronize();
  cudaFree(plan->block);
  if (cur != plan->device) cudaSetDevice(cur);
  free(plan);
}

int vc_expcast_encode(const float* s, const float* a, const float* b, int64_t n, uint8_t* out, cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!s || !a || !b || !out))) return VC_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc != VC_OK) return rc;
  return vc::expcast_launch(s, a, b, n, out, stream, true);
}

int vc_expcast_encode_unclamped(const float* s, const float* a, const float* b, int64_t n, uint8_t* out,
                                cudaStream_t stream) {
  if (n < 0 || (n > 0 && (!s || !a || !b || !out))) return VC_ERR_INVALID_ARG;
  int rc = check_device();
  if (rc != VC_OK) return rc;
  return vc::expcast_launch(s, a, b, n, out, stream, false);
}

const char* vc_strerror(int status) {
  switch (status) {
    case VC_OK: return "ok";
    case VC_ERR_INVALID_ARG: return "invalid argument";
    case VC_ERR_UNSUPPORTED: return "unsupported shape";
    case VC_ERR_CUDA: return "CUDA runtime error";
    case VC_ERR_TIMEOUT: return "kernel wait timed out";
    case VC_ERR_PLAN_MISMATCH: return "plan shape mismatch";
    case VC_ERR_OOM: return "device allocation failed";
    case VC_ERR_NO_DEVICE: return "no sm_103 device";
    default: return "unknown status";
  }
}

int vc_schedule_action(int step, int n_steps, int reuse) {
  if (n_steps < 1 || reuse < 1 || step < 0 || step >= n_steps) return VC_ERR_INVALID_ARG;
  const int window = (n_steps + 3) / 4;  // the first 25% of the steps, rounded up
  if (step >= window) return VC_STEP_PLAIN;
  if (step % reuse != 0) return VC_STEP_REUSE;
  return step == 0 ? VC_STEP_GROUP : VC_STEP_GROUP_WARM;
}

const char* vc_version(void) { return "vc_attn 0.1.0 (sm_103a)"; }

}  // extern "C"
