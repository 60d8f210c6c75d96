// decode_bf16_wide.cu — instantiations of the wide variant of the fused decode kernel for
// bf16 K/V (one CTA per SM, six stages, two warp groups on alternate chunks); used when the
// launch needs no more CTAs than the device has SMs.  The kernel is in decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace santa {

cudaError_t decode_launch_bf16_wide(const DecodeParams& p, int head_dim, int group, dim3 grid,
                              int cluster, cudaStream_t stream) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (decode_launch_t<true, 128, GG, true>(p, grid, cluster, stream)))
  }
  SANTA_DISPATCH_G(group, return (decode_launch_t<true, 64, GG, true>(p, grid, cluster, stream)))
}

int decode_resident_bf16_wide(int head_dim, int group) {
  if (head_dim == 128) { SANTA_DISPATCH_G(group, return (decode_resident_t<true, 128, GG, true>())) }
  SANTA_DISPATCH_G(group, return (decode_resident_t<true, 64, GG, true>()))
}

int decode_max_clusters_bf16_wide(int head_dim, int group, int cluster) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (decode_max_clusters_t<true, 128, GG, true>(cluster)))
  }
  SANTA_DISPATCH_G(group, return (decode_max_clusters_t<true, 64, GG, true>(cluster)))
}

}  // namespace santa
