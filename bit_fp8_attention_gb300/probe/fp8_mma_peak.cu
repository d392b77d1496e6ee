// fp8_mma_peak.cu -- measures the dense FP8 (E4M3) tensor-core rate of this GPU with tcgen05.
//
// Measurement support for the forward's roofline, not part of the attention library: one CTA per
// SM issues a long chain of tcgen05.mma.cta_group::1.kind::f8f6f4 with M = 128, N = 256, K = 32
// (both operands E4M3 in 128-byte-swizzled shared memory, fp32 accumulator in TMEM, alternating
// between two accumulators), so the tensor pipe never waits for operands and the issuing thread
// never waits for results. FLOPs = 2 M N K per instruction. Exported as a plain C function:
//
//   int vc_probe_fp8_peak(int iters, float* ms, double* flops, int* status)
//     iters   MMA groups (4 instructions each, K = 128) per CTA; > 0
//     ms      [out] kernel time of the timed launch (CUDA events, after one warm-up launch)
//     flops   [out] FLOPs of the timed launch
//     status  [out] 0, or 1 if a bounded wait gave up (the result is then invalid)
//   returns 0, -1 on invalid arguments, -3 on a CUDA error.
//
// The same library counts the kernels of a captured stream section, so that the benchmark can report
// how many of the attention library's kernels one step launches (counted from the captured graph,
// not estimated):
//   int vc_probe_capture_begin(cudaStream_t s)          starts a relaxed-mode capture of s
//   int vc_probe_capture_end(cudaStream_t s, int* kernels, int* nodes)
//       ends it, counts the kernel nodes and all nodes of the captured graph, and discards it
//   both return 0 or -3 on a CUDA error.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../csrc/vc_device.cuh"

namespace {

using namespace vc;

constexpr int kA = 128 * 128;  // A tile: 128 rows x 128 K bytes
constexpr int kB = 256 * 128;  // B tile: 256 rows x 128 K bytes
constexpr int kSmem = kA + kB + 1024 + 64;

__global__ void __launch_bounds__(128, 1) fp8_peak_kernel(int iters, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + kA;
  uint64_t* done = reinterpret_cast<uint64_t*>(base + kA + kB);
  uint32_t* slot = reinterpret_cast<uint32_t*>(base + kA + kB + 8);
  // Operand bytes: finite E4M3 codes of both signs (0x7F / 0xFF, the NaN codes, never occur).
  for (int i = threadIdx.x; i < (kA + kB) / 4; i += blockDim.x) {
    const uint32_t x = (uint32_t)i * 2654435761u + blockIdx.x;
    reinterpret_cast<uint32_t*>(base)[i] = (x & 0xBEBEBEBEu) | 0x08080808u;
  }
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  const int warp = __shfl_sync(0xffffffffu, (int)threadIdx.x >> 5, 0);
  if (warp == 0) tmem_alloc(slot, 512);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (warp == 0) {
    const bool leader = elect_one();
    const uint64_t da = smem_desc(sA, 1024, kSw128), db = smem_desc(sB, 1024, kSw128);
    constexpr uint32_t id = idesc_e4m3(128, 256);
    for (int i = 0; i < iters; ++i) {
      if (leader) {
        const uint32_t d = tmem + 256u * (uint32_t)(i & 1);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_e4m3_ss(d, da + 2 * kk, db + 2 * kk, id, kk > 0);
      }
      __syncwarp();
    }
    if (leader) mma_commit(done);
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(done, 0, 1u << 26)) && (threadIdx.x & 31) == 0) atomicOr(status, 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

extern "C" int vc_probe_fp8_peak(int iters, float* ms, double* flops, int* status) {
  if (iters <= 0 || !ms || !flops || !status) return -1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -3;
  if (cudaFuncSetAttribute(fp8_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess)
    return -3;
  int* dstatus = nullptr;
  cudaEvent_t a = nullptr, b = nullptr;
  int rc = 0;
  if (cudaMalloc(&dstatus, sizeof(int)) != cudaSuccess) return -3;
  if (cudaMemset(dstatus, 0, sizeof(int)) != cudaSuccess || cudaEventCreate(&a) != cudaSuccess ||
      cudaEventCreate(&b) != cudaSuccess) {
    rc = -3;
  } else {
    fp8_peak_kernel<<<sms, 128, kSmem>>>(iters / 8 + 1, dstatus);  // warm-up
    cudaEventRecord(a);
    fp8_peak_kernel<<<sms, 128, kSmem>>>(iters, dstatus);
    cudaEventRecord(b);
    if (cudaEventSynchronize(b) != cudaSuccess || cudaGetLastError() != cudaSuccess) rc = -3;
    if (rc == 0) {
      cudaEventElapsedTime(ms, a, b);
      *flops = (double)sms * iters * 4.0 * (2.0 * 128 * 256 * 32);
      if (cudaMemcpy(status, dstatus, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) rc = -3;
    }
  }
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  cudaFree(dstatus);
  return rc;
}

extern "C" int vc_probe_capture_begin(cudaStream_t s) {
  return cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed) == cudaSuccess ? 0 : -3;
}

extern "C" int vc_probe_capture_end(cudaStream_t s, int* kernels, int* nodes) {
  cudaGraph_t g = nullptr;
  if (cudaStreamEndCapture(s, &g) != cudaSuccess || !g) return -3;
  size_t n = 0;
  int rc = cudaGraphGetNodes(g, nullptr, &n) == cudaSuccess ? 0 : -3;
  int nk = 0;
  if (rc == 0 && n > 0) {
    cudaGraphNode_t* list = new cudaGraphNode_t[n];
    if (cudaGraphGetNodes(g, list, &n) != cudaSuccess) rc = -3;
    for (size_t i = 0; rc == 0 && i < n; ++i) {
      cudaGraphNodeType t;
      if (cudaGraphNodeGetType(list[i], &t) != cudaSuccess) rc = -3;
      else if (t == cudaGraphNodeTypeKernel) ++nk;
    }
    delete[] list;
  }
  cudaGraphDestroy(g);
  if (rc == 0) {
    if (kernels) *kernels = nk;
    if (nodes) *nodes = (int)n;
  }
  return rc;
}
