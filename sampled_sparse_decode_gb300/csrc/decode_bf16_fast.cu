// decode_bf16_fast.cu — instantiations of the compact path of the fused decode kernel for
// bf16 K/V (two-CTA-per-SM variant): a decode step
// with i.i.d. Horvitz-Thompson draws, no mixture and one cluster per unit, whose sampling
// prologue is compiled without the general path's branches.  The kernel is in
// decode_kernel.cuh; DecodeTraits::fast_fits decides which shapes it serves.
#include "decode_kernel.cuh"

namespace santa {

cudaError_t decode_launch_bf16_fast(const DecodeParams& p, int head_dim, int group,
                                        dim3 grid, int cluster, cudaStream_t stream) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (decode_launch_t<true, 128, GG, false, true>(p, grid, cluster, stream)))
  }
  SANTA_DISPATCH_G(group, return (decode_launch_t<true, 64, GG, false, true>(p, grid, cluster, stream)))
}

bool decode_fast_fits_bf16(int head_dim, int group, int max_teams, int cluster,
                               int team_size, int num_draws) {
  if (head_dim == 128) {
    SANTA_DISPATCH_G(group, return (DecodeTraits<true, 128, GG, false>::fast_fits(
                                        max_teams, cluster, team_size, num_draws)))
  }
  SANTA_DISPATCH_G(group, return (DecodeTraits<true, 64, GG, false>::fast_fits(
                                      max_teams, cluster, team_size, num_draws)))
}

int decode_resident_bf16_fast(int head_dim, int group) {
  if (head_dim == 128) { SANTA_DISPATCH_G(group, return (decode_resident_t<true, 128, GG, false, true>())) }
  SANTA_DISPATCH_G(group, return (decode_resident_t<true, 64, GG, false, true>()))
}

}  // namespace santa
