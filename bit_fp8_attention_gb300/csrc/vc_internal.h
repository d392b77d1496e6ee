// vc_internal.h -- definitions shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "vc_attn.h"

namespace vc {

// Opt a kernel into its dynamic shared memory size once per device (the attribute is per device, and
// setting it again is harmless, so concurrent first calls need no lock).
template <typename Kernel>
int ensure_smem_attr(Kernel* fn, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return VC_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_relaxed) & bit) return VC_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return VC_ERR_CUDA;
  done.fetch_or(bit, std::memory_order_relaxed);
  return VC_OK;
}

// Device buffers of a plan (layouts as documented in vc_attn.h).
struct PlanBuffers {
  int B, H, S, D, k, nkb, S_pad;
  int nkb16;            // nkb rounded up to a multiple of 16
  uint8_t* qcodes;      // [BH, S_pad, D]
  float* qscales;       // [BH, nkb]
  uint8_t* kcodes;      // [BH, S_pad, D]
  float* kscales;       // [BH, nkb]
  uint8_t* vcodes;      // [BH, D, S_pad]
  float* vscales;       // [BH]
  uint16_t* means;      // [BH, nkb, D] bf16
  uint16_t* meansT;     // [BH, D, nkb16] bf16, the same means transposed (pad columns 0)
  int32_t* labels;      // [BH, S]
  int32_t* perm;        // [BH, S]
  float* cent;          // [BH, k, D]
  float* cnorm;         // [BH, k]
  int kpad;             // k rounded up to a multiple of 128
  int nchunk;           // argsort chunks per head
  uint16_t* cent16;     // [BH, 2, kpad, D] bf16 hi and lo parts of the centroids (pad rows 0)
  float* cnormp;        // [BH, kpad] squared centroid norms, +inf on the pad rows
  int32_t* chist;       // [BH, nchunk, k] per-chunk label counts, then chunk start positions
  int32_t* counts;      // [BH, k]
  int32_t* offsets;     // [BH, k]
  int* kexp;            // [BH, D] largest bf16 exponent of each K channel (centering statistic)
  unsigned long long* ksum;  // [BH, D] exact fixed-point channel sums of K
  uint16_t* kmu;        // [BH, D] bf16 channel centre of K
  bool has_kcenter;     // prepared with K centering
  bool has_grouping;    // the centroids hold a finished grouping (a warm start may begin from them)
  bool has_perm;        // pi holds a permutation from an earlier prepare
  unsigned int* vamax;  // [BH] residual |max| as float bits
  unsigned int* vamax_ch;  // [BH, D] residual |max| of each channel as float bits (per-channel scale)
  float* vscales_ch;    // [BH, D] residual scale of each channel
  bool has_vchannel;    // prepared with one residual scale per channel
  bool has_hadamard;    // Q and K rows rotated before their quantisation (scores carry a factor D)
  int* status;          // [1]
  bool has_means;       // prepared with V-Smooth
  // V residual repair: n_rep rows per head in nrt = ceil(n_rep/128) extra key tiles (R_pad rows)
  int nrep, nrt, R_pad;
  int32_t* rep_idx;     // [BH, nrep] selected tokens, ascending
  float* energy;        // [BH, S] residual energy of every token
  uint8_t* krep;        // [BH, R_pad, D] E4M3 codes of the copied keys (pad rows 0)
  float* krep_scales;   // [BH, nrt]
  uint8_t* vrep;        // [BH, D, R_pad] E4M3 codes of the selected residuals, transposed (pad 0)
};

// perm_in: a caller permutation to copy in; reuse_perm: keep the plan's pi (no k-means); otherwise
// with vsmooth, k-means (warm: from the plan's centroids).  Means only with vsmooth.
int prepare_launch(const PlanBuffers& p, const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                   const int32_t* perm_in, bool vsmooth, bool kcenter, bool reuse_perm, bool warm, bool vchannel,
                   int iters, cudaStream_t st);

int kmeans_launch(const PlanBuffers& p, const uint16_t* V, int iters, bool warm, cudaStream_t st);
int kmeans_chunks(int S);

// cuTensorMapEncodeTiled on a 2-D row-major tensor (rows x inner elements, row pitch in bytes).
int encode_2d(CUtensorMap* m, CUtensorMapDataType dt, void* base, uint64_t inner, uint64_t rows,
              uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw);

struct FwdMaps {
  CUtensorMap q, k, v, mu, krep, vrep;
};
int encode_fwd_maps(const PlanBuffers& p, FwdMaps* maps);
int forward_launch(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st);
int forward2_launch(const PlanBuffers& p, const FwdMaps& maps, uint16_t* O, unsigned flags, cudaStream_t st);
int residual_pack_launch(const uint16_t* V, const int32_t* perm, int BH, int S, int D, uint16_t* means,
                         uint8_t* vcodes, float* vscales, unsigned int* amax_scratch, cudaStream_t st);
// Block quantiser: S rows per head (through perm [BH, S] when given) of a source with S_src rows per head.
void quant_blocks_launch(const uint16_t* x, const int32_t* perm, const uint16_t* center, int D, int S, int S_pad,
                         int S_src, int BH, uint8_t* codes, float* scales, cudaStream_t st, bool rotate = false);
// V residual repair rows (no V-Smooth): energies, selection, copied keys, residual codes. kcen: the K
// centre or null. The residual maxima (vamax, or vamax_ch when has_vchannel) must be complete.
int repair_launch(const PlanBuffers& p, const uint16_t* K, const uint16_t* V, const uint16_t* kcen, cudaStream_t st);
int expcast_launch(const float* s, const float* a, const float* b, int64_t n, uint8_t* out, cudaStream_t st,
                   bool clamp);

}  // namespace vc
