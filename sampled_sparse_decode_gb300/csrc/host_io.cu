// host_io.cu — the copies of santa_decode_host when its host buffers are page-locked and mapped
// into the device's address space: two small kernels that move the step's input slab from host
// memory into device memory and the output slab back, in place of two copy-engine transfers.
//
// A copy-engine transfer between two kernels adds its own scheduling round trip on each side.
// These kernels instead chain to the decode launch by programmatic dependent launch:
//   - stage-in lets the decode grid be scheduled as soon as it starts, and the decode kernel's
//     dependency wait (before its first global access) holds it until stage-in has completed
//     and its stores are visible;
//   - stage-out is launched as a programmatic dependent of the decode launch, so its blocks
//     are resident while the decode runs, and it waits for the decode grid before its first
//     load.
// Both move 16-byte words, every load of a thread issued before its stores.  Loads bypass L1
// (ld.global.cg): the source is written between launches, by the host or by the decode grid.
#include "kernels.h"

namespace santa {

namespace {

constexpr int kIoThreads = 256;
constexpr int kIoUnroll = 4;

__device__ __forceinline__ void copy_words(const uint4* src, uint4* dst, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kIoThreads * kIoUnroll;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * kIoThreads * kIoUnroll + threadIdx.x;
       base < n; base += stride) {
    uint4 w[kIoUnroll];
#pragma unroll
    for (int u = 0; u < kIoUnroll; ++u) {
      const int64_t i = base + static_cast<int64_t>(u) * kIoThreads;
      if (i < n) w[u] = __ldcg(src + i);
    }
#pragma unroll
    for (int u = 0; u < kIoUnroll; ++u) {
      const int64_t i = base + static_cast<int64_t>(u) * kIoThreads;
      if (i < n) dst[i] = w[u];
    }
  }
}

__global__ void __launch_bounds__(kIoThreads) stage_in_kernel(const uint4* src, uint4* dst,
                                                              int64_t n) {
  // the next launch (the decode) may be scheduled now: it waits for this grid to complete
  grid_launch_dependents();
  copy_words(src, dst, n);
}

__global__ void __launch_bounds__(kIoThreads) stage_out_kernel(const uint4* src, uint4* dst,
                                                               int64_t n) {
  // launched as a programmatic dependent: nothing is read before the previous grid completed
  grid_dependency_wait();
  copy_words(src, dst, n);
}

unsigned io_grid(int64_t words) {
  const int64_t per_block = static_cast<int64_t>(kIoThreads) * kIoUnroll;
  const int64_t blocks = (words + per_block - 1) / per_block;
  return static_cast<unsigned>(blocks < 1024 ? (blocks < 1 ? 1 : blocks) : 1024);
}

}  // namespace

cudaError_t launch_stage_in(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(bytes / 16);
  if (n == 0) return cudaSuccess;
  stage_in_kernel<<<io_grid(n), kIoThreads, 0, stream>>>(static_cast<const uint4*>(src),
                                                         static_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

cudaError_t launch_stage_out(const void* src, void* dst, size_t bytes, cudaStream_t stream) {
  const int64_t n = static_cast<int64_t>(bytes / 16);
  if (n == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(io_grid(n));
  cfg.blockDim = dim3(kIoThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, stage_out_kernel, static_cast<const uint4*>(src),
                            static_cast<uint4*>(dst), n);
}

}  // namespace santa
