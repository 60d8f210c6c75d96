// reps.cu — team representatives: the mean of the valid keys of each (page, KV head).
//
// "SANTA++: Sampling Attention through Representative Keys", abstract: the query scores one
// representative key per team instead of scanning the whole cache; the explainer
// ("SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%", section 三 step 2) lists the mean
// key as one choice of representative.  Teams are KV pages, so one representative per
// (page, head) kept in an fp32 side buffer serves every sequence that owns the page.
//
// One 256-thread block per (page, head): thread (pair, group) sums key columns 2*pair and
// 2*pair+1 over tokens group, group+G, ... in fp32; the groups are added in fixed order and
// divided by the valid-token count.  The pass reads the K pool once (HBM-bound) and runs
// once after prefill; santa_update_reps reruns it for the pages that grew during decode.
#include "kernels.h"

namespace santa {

namespace {

constexpr int kRepThreads = 256;

template <int D>
__device__ __forceinline__ float2 load_pair(const void* pool, bool bf16, int64_t idx) {
  if (bf16) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(
        static_cast<const uint16_t*>(pool) + idx));
    return make_float2(bf16_lo(w), bf16_hi(w));
  }
  return __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(pool) + idx));
}

template <int D>
__global__ void __launch_bounds__(kRepThreads) reps_kernel(RepsParams p) {
  constexpr int kPairs = D / 2;
  constexpr int kGroups = kRepThreads / kPairs;
  __shared__ float2 part[kGroups][kPairs];

  const int pair = threadIdx.x % kPairs;
  const int group = threadIdx.x / kPairs;
  const int64_t items = static_cast<int64_t>(p.num_items) * p.num_kv_heads;
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
    const int64_t base = (page * p.num_kv_heads + h) * static_cast<int64_t>(p.team_size) * D;
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int t = group; t < fill; t += kGroups) {
      const float2 v = load_pair<D>(p.k_pool, p.is_bf16, base + static_cast<int64_t>(t) * D +
                                                              2 * pair);
      acc.x += v.x;
      acc.y += v.y;
    }
    part[group][pair] = acc;
    __syncthreads();
    if (group == 0) {
      float2 s = part[0][pair];
#pragma unroll
      for (int g = 1; g < kGroups; ++g) {
        s.x += part[g][pair].x;
        s.y += part[g][pair].y;
      }
      const float2 mean =
          fill > 0 ? make_float2(s.x / fill, s.y / fill) : make_float2(0.f, 0.f);
      reinterpret_cast<float2*>(p.reps + (page * p.num_kv_heads + h) * D)[pair] = mean;
    }
    __syncthreads();
  }
}

// One decode step's new token per (sequence, KV head): K and V go to slot L % T of page
// page_table[b][L / T] (L = seq_lens[b]), and the page's representative becomes the mean of
// its L % T + 1 valid keys.  The mean is summed exactly as reps_kernel sums it (same
// thread split, same order: the new key is the last term of its group), from the pool rows
// already there plus the new key, so it equals santa_build_reps on the grown pool bit for
// bit while reading only this page.
template <int D>
__global__ void __launch_bounds__(kRepThreads) append_kernel(AppendParams p) {
  constexpr int kPairs = D / 2;
  constexpr int kGroups = kRepThreads / kPairs;
  __shared__ float2 part[kGroups][kPairs];
  const int pair = threadIdx.x % kPairs;
  const int group = threadIdx.x / kPairs;
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
    const int64_t src = item * D;
    const int64_t base = (page * p.num_kv_heads + h) * static_cast<int64_t>(p.team_size) * D;
    const int64_t dst = base + static_cast<int64_t>(slot) * D;
    for (int e = threadIdx.x; e < D; e += kRepThreads) {
      if (p.is_bf16) {
        static_cast<uint16_t*>(p.k_pool)[dst + e] = static_cast<const uint16_t*>(p.k_new)[src + e];
        static_cast<uint16_t*>(p.v_pool)[dst + e] = static_cast<const uint16_t*>(p.v_new)[src + e];
      } else {
        static_cast<float*>(p.k_pool)[dst + e] = static_cast<const float*>(p.k_new)[src + e];
        static_cast<float*>(p.v_pool)[dst + e] = static_cast<const float*>(p.v_new)[src + e];
      }
    }
    // rows 0 .. slot-1 are not written by this launch (one writer per page and head)
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int t = group; t < slot; t += kGroups) {
      const float2 v = load_pair<D>(p.k_pool, p.is_bf16, base + static_cast<int64_t>(t) * D +
                                                              2 * pair);
      acc.x += v.x;
      acc.y += v.y;
    }
    if (slot % kGroups == group) {
      const float2 v = load_pair<D>(p.k_new, p.is_bf16, src + 2 * pair);
      acc.x += v.x;
      acc.y += v.y;
    }
    part[group][pair] = acc;
    __syncthreads();
    if (group == 0) {
      float2 s = part[0][pair];
#pragma unroll
      for (int g = 1; g < kGroups; ++g) {
        s.x += part[g][pair].x;
        s.y += part[g][pair].y;
      }
      const int fill = slot + 1;
      reinterpret_cast<float2*>(p.reps + (page * p.num_kv_heads + h) * D)[pair] =
          make_float2(s.x / fill, s.y / fill);
    }
    if (h == 0 && threadIdx.x == 0 && p.seq_lens_next) p.seq_lens_next[b] = L + 1;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.batch) * p.num_kv_heads;
  if (items == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(items < (1ll << 30) ? items : (1ll << 30));
  if (head_dim == 128)
    append_kernel<128><<<grid, kRepThreads, 0, stream>>>(p);
  else
    append_kernel<64><<<grid, kRepThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_reps(const RepsParams& p, int head_dim, cudaStream_t stream) {
  const int64_t items = static_cast<int64_t>(p.num_items) * p.num_kv_heads;
  if (items == 0) return cudaSuccess;
  const unsigned grid = static_cast<unsigned>(items < (1ll << 30) ? items : (1ll << 30));
  if (head_dim == 128)
    reps_kernel<128><<<grid, kRepThreads, 0, stream>>>(p);
  else
    reps_kernel<64><<<grid, kRepThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace santa
