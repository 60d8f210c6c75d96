// philox_check.cu — test-only kernel: the library's device Philox4x32-10 next to CUDA's own
// curand_Philox4x32_10 (a library routine) on the same counters and keys.
#include <curand_kernel.h>

#include "common.cuh"

__global__ void philox_pair_kernel(const uint4* ctr, const uint2* key, uint4* ours, uint4* ref,
                                   int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  ours[i] = santa::philox4x32_10(ctr[i], key[i]);
  ref[i] = curand_Philox4x32_10(ctr[i], key[i]);
}

extern "C" int philox_pair(const void* ctr, const void* key, void* ours, void* ref, int n) {
  philox_pair_kernel<<<(n + 127) / 128, 128>>>(static_cast<const uint4*>(ctr),
                                                static_cast<const uint2*>(key),
                                                static_cast<uint4*>(ours),
                                                static_cast<uint4*>(ref), n);
  if (cudaGetLastError() != cudaSuccess) return 1;
  return cudaDeviceSynchronize() == cudaSuccess ? 0 : 2;
}
