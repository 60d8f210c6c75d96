// decode_bf16_wide_fast_var.cu — instantiations of the compact path of the fused decode kernel
// for bf16 K/V (wide variant: one CTA per SM, six stages) with the sampler variants compiled
// in: systematic draws, Hansen-Hurwitz weights and the defensive mixture.  The default
// sampler runs the instantiations of decode_bf16_wide_fast.cu.  The kernel is in
// decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace santa {

cudaError_t decode_launch_bf16_wide_fast_var(const DecodeParams& p, int head_dim, int group,
                                             dim3 grid, int cluster, cudaStream_t stream) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (decode_launch_t<true, 128, GG, true, 2>(p, grid, cluster, stream)))
  }
  SANTA_DISPATCH_G(group, return (decode_launch_t<true, 64, GG, true, 2>(p, grid, cluster, stream)))
}

int decode_resident_bf16_wide_fast_var(int head_dim, int group) {
  if (head_dim == 128) { SANTA_DISPATCH_G(group, return (decode_resident_t<true, 128, GG, true, 2>())) }
  SANTA_DISPATCH_G(group, return (decode_resident_t<true, 64, GG, true, 2>()))
}

}  // namespace santa
