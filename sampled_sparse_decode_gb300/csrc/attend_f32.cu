// attend_f32.cu — instantiations of the split-K attention kernel for f32 K/V (head_dim 64
// and 128, 1 to 8 query heads per KV head).  The kernel itself is in attend_kernel.cuh.
#include "attend_kernel.cuh"

namespace santa {

cudaError_t launch_attend_f32(const AttendParams& p, int head_dim, int group, dim3 grid,
                              bool programmatic, cudaStream_t stream) {
  return head_dim == 128 ? launch_attend_g<false, 128>(p, group, grid, programmatic, stream)
                         : launch_attend_g<false, 64>(p, group, grid, programmatic, stream);
}

size_t attend_smem_bytes_f32(int head_dim, int group) {
  return head_dim == 128 ? attend_smem_g<false, 128>(group) : attend_smem_g<false, 64>(group);
}

int attend_resident_ctas_f32(int head_dim, int group) {
  return head_dim == 128 ? attend_resident_g<false, 128>(group) : attend_resident_g<false, 64>(group);
}

}  // namespace santa
