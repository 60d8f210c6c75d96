// decode_f32.cu — instantiations of the fused decode kernel for f32 K/V (head_dim 64 and
// 128, 1 to 8 query heads per KV head).  The kernel is in decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace santa {

cudaError_t decode_launch_f32(const DecodeParams& p, int head_dim, int group, dim3 grid,
                              int cluster, cudaStream_t stream) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (decode_launch_t<false, 128, GG, false>(p, grid, cluster, stream)))
  }
  SANTA_DISPATCH_G(group, return (decode_launch_t<false, 64, GG, false>(p, grid, cluster, stream)))
}

int decode_resident_f32(int head_dim, int group) {
  if (head_dim == 128) { SANTA_DISPATCH_G(group, return (decode_resident_t<false, 128, GG, false>())) }
  SANTA_DISPATCH_G(group, return (decode_resident_t<false, 64, GG, false>()))
}

int decode_max_clusters_f32(int head_dim, int group, int cluster) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (decode_max_clusters_t<false, 128, GG, false>(cluster)))
  }
  SANTA_DISPATCH_G(group, return (decode_max_clusters_t<false, 64, GG, false>(cluster)))
}

}  // namespace santa
