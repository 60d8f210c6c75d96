// reps.cu — team representatives: the mean of the valid keys of each (page, KV head).
//
// "SANTA++: Sampling Attention through Representative Keys", abstract: the query scores one
// representative key per team instead of scanning the whole cache; the explainer
// ("SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%", section 三 step 2) lists the mean
// key as one choice of representative.  Teams are KV pages, so one representative per
// (page, head) kept in an fp32 side buffer serves every sequence that owns the page.
//
// One 256-thread block per (page, head).  A key row is read as 16-byte pieces: thread
// (col, group) owns piece col of the rows group, group + G, ... (G = 256 / pieces per row),
// issues all of its loads before adding, and sums them in fp32 in row order; the groups are
// then added in fixed order and divided by the valid-token count.  The pass reads the K
// pool once (HBM-bound) and runs once after prefill; santa_update_reps reruns it for the
// pages that grew during decode.
#include "kernels.h"

namespace santa {

namespace {

constexpr int kRepThreads = 256;

// The thread split shared by the build and the append (which must add in the same order).
template <bool BF16, int D>
struct RepSplit {
  static constexpr int kVec = BF16 ? 8 : 4;              // elements per 16-byte piece
  static constexpr int kCols = D / kVec;                 // pieces per key row
  static constexpr int kGroups = kRepThreads / kCols;    // row groups
  static constexpr int kMaxRows = 128 / kGroups;         // rows per group at T = 128
};

template <bool BF16>
__device__ __forceinline__ void add_piece(float (&acc)[BF16 ? 8 : 4], const uint4& w) {
  if constexpr (BF16) {
    acc[0] += bf16_lo(w.x); acc[1] += bf16_hi(w.x);
    acc[2] += bf16_lo(w.y); acc[3] += bf16_hi(w.y);
    acc[4] += bf16_lo(w.z); acc[5] += bf16_hi(w.z);
    acc[6] += bf16_lo(w.w); acc[7] += bf16_hi(w.w);
  } else {
    acc[0] += __uint_as_float(w.x); acc[1] += __uint_as_float(w.y);
    acc[2] += __uint_as_float(w.z); acc[3] += __uint_as_float(w.w);
  }
}

// Sum of rows group, group + kGroups, ... below `rows` of one (page, head) block, piece col,
// in row order; `extra` (if non-null) is added last.  All loads are in flight before the
// first addition.
template <bool BF16, int D>
__device__ __forceinline__ void sum_rows(const uint4* block, int col, int group, int rows,
                                         const uint4* extra, float (&acc)[BF16 ? 8 : 4]) {
  using Sp = RepSplit<BF16, D>;
#pragma unroll
  for (int e = 0; e < Sp::kVec; ++e) acc[e] = 0.f;
  uint4 v[Sp::kMaxRows];
#pragma unroll
  for (int u = 0; u < Sp::kMaxRows; ++u) {
    const int t = group + u * Sp::kGroups;
    v[u] = t < rows ? __ldg(block + static_cast<int64_t>(t) * Sp::kCols + col)
                    : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int u = 0; u < Sp::kMaxRows; ++u)
    if (group + u * Sp::kGroups < rows) add_piece<BF16>(acc, v[u]);
  if (extra) add_piece<BF16>(acc, __ldg(extra));
}

// The group partials [kGroups][D] in shared memory, added in group order by thread e < D.
template <bool BF16, int D>
__device__ __forceinline__ void store_partial(float* part, int col, int group,
                                              const float (&acc)[BF16 ? 8 : 4]) {
  using Sp = RepSplit<BF16, D>;
  float4* dst = reinterpret_cast<float4*>(part + group * D + col * Sp::kVec);
#pragma unroll
  for (int e = 0; e < Sp::kVec / 4; ++e)
    dst[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
}

template <bool BF16, int D>
__device__ __forceinline__ void write_mean(const float* part, int fill, float* rep) {
  using Sp = RepSplit<BF16, D>;
  for (int e = threadIdx.x; e < D; e += kRepThreads) {
    float s = part[e];
#pragma unroll
    for (int g = 1; g < Sp::kGroups; ++g) s += part[g * D + e];
    rep[e] = fill > 0 ? s / fill : 0.f;
  }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kRepThreads) reps_kernel(RepsParams p) {
  using Sp = RepSplit<BF16, D>;
  __shared__ __align__(16) float part[Sp::kGroups * D];
  const int col = threadIdx.x % Sp::kCols;
  const int group = threadIdx.x / Sp::kCols;
  const int64_t items = static_cast<int64_t>(p.num_items) * p.num_kv_heads;
  // launched as a programmatic dependent launch: global memory only after the previous
  // kernel of the stream has completed; the next one may be scheduled from here on (it is
  // launched once every block of this grid has passed this point, and waits in turn)
  grid_dependency_wait();
  grid_launch_dependents();
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int h = static_cast<int>(item % p.num_kv_heads);
    const int64_t listed = item / p.num_kv_heads;
    const int64_t page = p.pages ? static_cast<int64_t>(p.pages[listed]) : listed;
    if (page < 0 || page >= p.num_pages) {
      if (threadIdx.x == 0) set_status(p.status, SANTA_DEV_BAD_PAGE);
      continue;
    }
    int fill = p.page_fill ? p.page_fill[page] : p.team_size;
    if (fill < 0 || fill > p.team_size) {
      if (threadIdx.x == 0) set_status(p.status, SANTA_DEV_BAD_SEQLEN);
      fill = 0;
    }
    const int64_t blk = (page * p.num_kv_heads + h) * static_cast<int64_t>(p.team_size);
    const uint4* block = static_cast<const uint4*>(p.k_pool) + blk * Sp::kCols;
    float acc[Sp::kVec];
    sum_rows<BF16, D>(block, col, group, fill, nullptr, acc);
    store_partial<BF16, D>(part, col, group, acc);
    __syncthreads();
    write_mean<BF16, D>(part, fill, p.reps + (page * p.num_kv_heads + h) * D);
    __syncthreads();
  }
}

// One decode step's new token per (sequence, KV head): K and V go to slot L % T of page
// page_table[b][L / T] (L = seq_lens[b]), and the page's representative becomes the mean of
// its L % T + 1 valid keys.  The mean is summed exactly as reps_kernel sums it (same
// thread split, same order: the new key is the last term of its row group), from the pool
// rows already there plus the new key, so it equals santa_build_reps on the grown pool bit
// for bit while reading only this page.  It is launched plainly, not as a programmatic
// dependent launch: that would let the next decode grid become resident beside these few
// blocks, and at batch 8 its clusters then no longer fit the SMs in one wave (35-40% longer
// decode steps in a generation loop, where the step itself gained nothing at batch 1).
template <bool BF16, int D>
__global__ void __launch_bounds__(kRepThreads) append_kernel(AppendParams p) {
  using Sp = RepSplit<BF16, D>;
  __shared__ __align__(16) float part[Sp::kGroups * D];
  const int col = threadIdx.x % Sp::kCols;
  const int group = threadIdx.x / Sp::kCols;
  const int64_t items = static_cast<int64_t>(p.batch) * p.num_kv_heads;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = static_cast<int>(item / p.num_kv_heads);
    const int h = static_cast<int>(item % p.num_kv_heads);
    const int L = p.seq_lens[b];
    if (L < 0 || static_cast<int64_t>(L) >= static_cast<int64_t>(p.max_teams) * p.team_size) {
      if (threadIdx.x == 0) set_status(p.status, SANTA_DEV_BAD_SEQLEN);
      continue;
    }
    const int slot = L % p.team_size;
    const int64_t page = p.page_table[static_cast<int64_t>(b) * p.max_teams + L / p.team_size];
    if (page < 0 || page >= p.num_pages) {
      if (threadIdx.x == 0) set_status(p.status, SANTA_DEV_BAD_PAGE);
      continue;
    }
    const int64_t blk = (page * p.num_kv_heads + h) * static_cast<int64_t>(p.team_size);
    const uint4* knew = static_cast<const uint4*>(p.k_new) + item * Sp::kCols;
    const uint4* vnew = static_cast<const uint4*>(p.v_new) + item * Sp::kCols;
    // the new row: K by threads 0 .. kCols-1, V by the next kCols
    if (threadIdx.x < 2 * Sp::kCols) {
      const bool isk = threadIdx.x < Sp::kCols;
      const int c = isk ? threadIdx.x : threadIdx.x - Sp::kCols;
      uint4* dst = static_cast<uint4*>(isk ? p.k_pool : p.v_pool) +
                   (blk + slot) * Sp::kCols + c;
      *dst = __ldg((isk ? knew : vnew) + c);
    }
    // rows 0 .. slot-1 are not written by this launch (one writer per page and head)
    const uint4* block = static_cast<const uint4*>(p.k_pool) + blk * Sp::kCols;
    float acc[Sp::kVec];
    sum_rows<BF16, D>(block, col, group, slot,
                      slot % Sp::kGroups == group ? knew + col : nullptr, acc);
    store_partial<BF16, D>(part, col, group, acc);
    __syncthreads();
    write_mean<BF16, D>(part, slot + 1, p.reps + (page * p.num_kv_heads + h) * D);
    if (h == 0 && threadIdx.x == 0 && p.seq_lens_next) p.seq_lens_next[b] = L + 1;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.batch) * p.num_kv_heads;
  if (items == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(items < (1ll << 30) ? items : (1ll << 30));
  if (p.is_bf16) {
    if (head_dim == 128)
      append_kernel<true, 128><<<grid, kRepThreads, 0, stream>>>(p);
    else
      append_kernel<true, 64><<<grid, kRepThreads, 0, stream>>>(p);
  } else {
    if (head_dim == 128)
      append_kernel<false, 128><<<grid, kRepThreads, 0, stream>>>(p);
    else
      append_kernel<false, 64><<<grid, kRepThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_reps(const RepsParams& p, int head_dim, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.num_items) * p.num_kv_heads;
  if (items == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(items < (1ll << 30) ? items : (1ll << 30));
  // programmatic stream serialization: the blocks of this launch may be scheduled while the
  // previous kernel of the stream drains (they wait for it before touching memory)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kRepThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.is_bf16)
    return head_dim == 128 ? cudaLaunchKernelEx(&cfg, reps_kernel<true, 128>, p)
                           : cudaLaunchKernelEx(&cfg, reps_kernel<true, 64>, p);
  return head_dim == 128 ? cudaLaunchKernelEx(&cfg, reps_kernel<false, 128>, p)
                         : cudaLaunchKernelEx(&cfg, reps_kernel<false, 64>, p);
}

}  // namespace santa
