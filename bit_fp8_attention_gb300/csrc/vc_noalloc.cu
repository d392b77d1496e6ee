// vc_noalloc.cu -- an entry point for callers that cannot allocate device memory.
//
// Some callers must not call cudaMalloc at all: a framework that has already reserved the whole
// device for its own memory pool (a stray allocation would fail or fragment it), or host code that
// runs under a rule that device memory is only allocated at start-up. vc_residual_pack_noalloc
// gives them the V-Smooth value preparation without any allocation: the only scratch it needs,
// one word per batch-head for the residual's absolute maximum, lives in a fixed array in the
// library's own device memory, sized for at most VC_NOALLOC_MAX_HEADS batch-heads (16 KiB, held by
// every GPU that loads the library until the process exits).
#include <cuda_runtime.h>
#include <stdint.h>

#include "vc_internal.h"

namespace {

// Per-head residual maxima (as float bit patterns) shared by every call on a device.
static __device__ __align__(256) unsigned int g_residual_amax[VC_NOALLOC_MAX_HEADS];

// Device address of the scratch array on the current device. In host code `g_residual_amax` only
// names a host-side stand-in, so the address must come from the runtime. It is looked up on every
// call (a table lookup once the module is loaded, and no allocation): a cached address would go
// stale if the caller reset the device (cudaDeviceReset) and the module were loaded again. The
// first call on a device also loads the library's module there.
int scratch_for_current_device(unsigned int** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_residual_amax) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return VC_ERR_CUDA;
  }
  *out = static_cast<unsigned int*>(p);
  return VC_OK;
}

}  // namespace

extern "C" int vc_residual_pack_noalloc(const void* V, const int32_t* perm, int B, int H, int S, int D, void* means,
                                        uint8_t* vcodes, float* vscales, cudaStream_t stream) {
  if (!V || !means || !vcodes || !vscales) return VC_ERR_INVALID_ARG;
  if (((uintptr_t)V & 15u) || ((uintptr_t)means & 15u) || ((uintptr_t)vcodes & 15u)) return VC_ERR_INVALID_ARG;
  if (((uintptr_t)perm & 3u) || ((uintptr_t)vscales & 3u)) return VC_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1) return VC_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return VC_ERR_UNSUPPORTED;
  if ((int64_t)B * H > VC_NOALLOC_MAX_HEADS) return VC_ERR_UNSUPPORTED;  // beyond the fixed scratch
  const int64_t S_pad = ((int64_t)S + 127) / 128 * 128;
  if (S > (1 << 20) || (int64_t)B * H * S_pad * D >= ((int64_t)1 << 40)) return VC_ERR_UNSUPPORTED;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3)
    return VC_ERR_NO_DEVICE;
  unsigned int* scratch = nullptr;
  int rc = scratch_for_current_device(&scratch);
  if (rc != VC_OK) return rc;
  return vc::residual_pack_launch(static_cast<const uint16_t*>(V), perm, B * H, S, D, static_cast<uint16_t*>(means),
                                  vcodes, vscales, scratch, stream);
}
