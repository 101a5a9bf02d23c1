// Copies between page-locked host memory (through its device mapping) and
// device memory for splitk_gemm_bf16_hostio(), as kernels in the stream's
// programmatic-dependent-launch chain.  Each copy launches its dependents at
// once and waits for its predecessor's completion before touching memory,
// so the GEMM that follows a copy-in is already resident and streaming its
// weights (which do not depend on the activations) while the copy runs, and
// a copy-out that follows the GEMM is resident when the GEMM completes.
// Stream order is kept: no copy reads or writes before the kernel ahead of
// it in the stream has completed and its writes are visible.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "splitk_device.cuh"
#include "splitk_internal.h"

namespace splitk {

namespace {

constexpr int kCopyThreads = 256;

// dst[0, bytes) = src[0, bytes); both 16-byte aligned.
__global__ void __launch_bounds__(kCopyThreads) pdl_copy_kernel(const uint8_t* __restrict__ src,
                                                                uint8_t* __restrict__ dst, size_t bytes) {
  dev::griddep_launch_dependents();
  dev::griddep_wait();
  const size_t n16 = bytes / 16u;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4* d4 = reinterpret_cast<uint4*>(dst);
  for (size_t i = tid; i < n16; i += stride) d4[i] = s4[i];
  for (size_t i = n16 * 16u + tid; i < bytes; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_pdl_copy(const void* src, void* dst, size_t bytes, int num_sms, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  // One 16-byte word a thread where that fits 4 CTAs an SM: every load of
  // the copy in flight at once (a host-memory round trip is ~1 us).
  const size_t n16 = bytes / 16u + 1u;
  const size_t want = (n16 + kCopyThreads - 1) / kCopyThreads;
  const size_t cap = 4u * (size_t)num_sms;
  const unsigned blocks = (unsigned)(want < cap ? (want > 0 ? want : 1) : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kCopyThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pdl_copy_kernel, static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                            bytes);
}

}  // namespace splitk
