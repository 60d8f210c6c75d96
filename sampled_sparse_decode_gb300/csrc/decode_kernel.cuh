// decode_kernel.cuh — one SANTA++ decode step per (sequence, KV head) unit in one kernel:
// representative scoring, GQA-mixed team softmax, Philox inverse-CDF sampling, the
// deduplicated sampled set with its weights, exact attention inside the sampled teams
// reweighted by 1/pi, and the Horvitz-Thompson combine.
//
// Method ("SANTA++: Sampling Attention through Representative Keys", abstract; explainer
// "SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%", section 三 steps 1-5, 3.1):
//   s_{g,i} = q_g . rep_i / sqrt(d);  p_{g,i} = softmax_i(s_{g,.});  p_i = (1/G) sum_g p_{g,i}
//   draw r: u = (word 0 of Philox4x32-10((r, h, b, 0), (lo32, hi32 of seed)) + 1/2) 2^-32,
//           team = smallest i with u*Z < C_i, decided exactly on the integer CDF of
//           round(p_i 2^62) (floor(u Z) from a 128-bit product)
//   S = distinct draws, pi_i = 1 - (1 - p_i)^M
//   out_g = sum_{i in S} (1/pi_i) sum_{j in i} e^{s_j} v_j / sum_{i in S} (1/pi_i) sum_{j in i} e^{s_j}
// (with the sampler variants of santa.h: systematic draws, Hansen-Hurwitz weights, and a
// defensive uniform mixture of p).
//
// GB300 mapping.  A unit is served by NC thread-block clusters of CL CTAs (NC = 1 unless a
// unit's work needs more CTAs than one cluster's tables hold).  Inside a cluster:
//   phase A  CTA r scores the representatives of its slice of teams (page ids read first,
//            rows staged with cp.async, 16 lanes per team), turns the slice into
//            e = exp(s - m_slice) and pushes e, the page ids and (m_slice, z_slice) into
//            every CTA of the cluster by distributed-shared-memory stores before one
//            cluster barrier.  Every CTA then holds the whole unit: per-head global
//            statistics (warp per head), p, the fixed-point CDF (one block scan), the M
//            draws and a ballot bit mask of the drawn teams (slot k = k-th set bit).  All
//            reductions run in a fixed order, so every CTA gets the same sampled set.
//            Units with more teams than one CTA holds use a distributed variant (slices'
//            totals and counts exchanged over three cluster barriers).
//   phase B  the unit's sampled teams form a list of 64-token chunks; CTA g of the unit owns
//            a contiguous range; each chunk's team, page and -log2 pi are resolved from the
//            mask in shared memory; rank 0 of the first cluster writes the outputs of S.
//   phase C  one thread streams each chunk's K and V into a ring of stages on mbarriers
//            (bf16: 2-D tensor copies with 128-byte swizzle; fp32: bulk copies).  bf16 is
//            consumed on tensor cores (mma.sync m16n8k16: scores S^T = K Q^T with the G
//            heads as N, base-2 online softmax with -log2 pi folded in, P transposed by
//            movmatrix and split bf16 hi + lo for O^T += V^T P^T); fp32 on CUDA cores.
//            W = false: two CTAs per SM, warps split token tiles and halves of d.
//            W = true (launches that fit one CTA per SM): six stages, two warp groups
//            consuming alternate chunks on their own stages.
//   phase D  the warps merge into a CTA partial; each CTA pushes the quads of the output
//            slice rank r owns, with its (m, l), into rank r's shared memory (st.async,
//            completing on rank r's mbarrier); each CTA merges its slice in rank order.
//            With NC > 1 the cluster partials go to global scratch and the last CTA of the
//            unit (an atomic ticket, no waiting) merges them in cluster order.
// Compact form (template flag FAST, bf16 steps with NC = 1).  FAST = 1 compiles a decode
// step with i.i.d. Horvitz-Thompson draws alone; FAST = 2 adds the sampler variants, the
// mixture and sampling-only steps.  Phases A and B are replaced by a shorter sequence: CTA r
// stages its slice's representative rows by one bulk copy each, scores them in base 2, and
// stores its [G + 1][slice] block (scores, page ids) into every CTA with st.async, completing
// on the receiver's mbarrier (no cluster barrier); each CTA then takes the per-head
// statistics (warp per head), p, pi and the CDF (one block scan), the draws (binary search,
// Philox words computed while the rows were in flight), and writes S with the chunk table in
// one pass, issuing the first copies at once.  In phase D each merging thread forms its
// head's weights itself.  Its code is kept short: it runs once per launch, and the SM waits
// on fetching cold instructions there.
// The kernel is launched with programmatic stream serialization and touches global memory
// only after griddepcontrol.wait.  No wait is unbounded: mbarrier waits give up after 2 s
// (status bit, clean exit through the remaining barriers); every CTA executes every cluster
// barrier on every path.
#pragma once

#include <cooperative_groups.h>

#include <cmath>

#include "kernels.h"

namespace santa {

namespace cgx = cooperative_groups;

// Chunk of the unit's work owned by this CTA: where it comes from and how it is weighted.
struct ChunkMeta {
  int page;   // physical page, -1 for a chunk that contributes nothing
  int valid;  // valid tokens in the chunk (0..64)
  float lw2;  // -log2(pi) of its team (0 in dense mode)
  int part;   // which 64-token part of the page
};

// A drawn team as published to the cluster.
struct ListEntry {
  int team;
  float lw2;
};

// Values a CTA publishes to its cluster peers.
struct Published {
  float m[kMaxGroup];   // per-head max score over the CTA's teams
  float z[kMaxGroup];   // per-head sum of exp(s - m) over them
  unsigned long long total;  // the CTA's CDF total (62-bit fixed point)
  int count;            // drawn teams in the CTA's slice
  int pad;
};

template <bool BF16, int D, int G, bool W = false>
struct DecodeTraits {
  static constexpr int kThreads = 256;
  static constexpr int kWarps = 8;
  static constexpr int kEsize = BF16 ? 2 : 4;
  static constexpr int kChunkBytes = kChunk * D * kEsize;
  static constexpr int kStageBytes = 2 * kChunkBytes;
  // W (wide): one CTA per SM, six stages, two warp groups consuming alternate chunks (each
  // group owns the even or the odd stages); otherwise up to two CTAs per SM
  static constexpr int kStages =
      W ? 6 : (kStageBytes >= 65536 ? 2 : (kStageBytes >= 32768 ? 3 : 4));
  static constexpr int kEplS = D / 16;
  static constexpr int kEplV = D / 32;
  static constexpr int kRing = kStages * kStageBytes;
  // phase A scratch inside the ring, for `cap` teams: cdf (uint64), es [8][cap], ps, flag,
  // page ids and room for the drawn-team bit mask (local path), then rows of
  // representatives (fp32 [rows][D]); rounded up to 128 bytes (the rows take 16-byte copies)
  static constexpr size_t sample_scratch(int cap) {
    return ((sizeof(unsigned long long) + sizeof(float) * kMaxGroup + sizeof(float) +
             2 * sizeof(int) + sizeof(ListEntry)) * static_cast<size_t>(cap) + 127) / 128 * 128;
  }
  static constexpr int rep_rows(int cap) {
    return static_cast<int>((static_cast<size_t>(kRing) - sample_scratch(cap)) / (D * 4));
  }
  static_assert(rep_rows(kMaxTeamsPerCta) >= 16, "representative buffer must hold 16 rows");
  static_assert(sizeof(ListEntry) * kMaxTeamsPerCta >= sizeof(float) * kPubScores,
                "the list region must hold the published scores");
  // phase D: warp merge buffer [8][G][D + 4] + m, l [8][8], then the CTA partial [G][D] + m, l.
  // The 4-float pad puts the rows of heads g and g + 2 four banks apart: a warp's store of its
  // mma accumulator fragment (8 rows of d x 4 heads per instruction) then hits 32 banks.
  static constexpr int kMrgStride = D + 4;
  static constexpr int kMergeFloats = kWarps * G * kMrgStride + 2 * kWarps * kMaxGroup;
  static constexpr int kPartialOff = kMergeFloats;                    // in floats
  static constexpr int kPartialFloats = G * D + 2 * kMaxGroup;
  static_assert((kMergeFloats + kPartialFloats) * 4 <= kRing, "merge buffers must fit");
  // combine buffers in the list region: [CL][ceil(G*D/4/CL)] float4 + [CL][G][2] floats
  static_assert((G * D / 4 + kMaxCluster) * 16 + kMaxCluster * kMaxGroup * 8 <=
                    sizeof(ListEntry) * kMaxTeamsPerCta,
                "combine buffers must fit the list region");
  // dynamic shared memory: ring | list | chunk table | p rows | alpha | bars
  static constexpr size_t kListOff = static_cast<size_t>(kRing);
  static constexpr size_t kTableOff = kListOff + sizeof(ListEntry) * kMaxTeamsPerCta;
  static constexpr size_t kPOff = kTableOff + sizeof(ChunkMeta) * kMaxChunksPerSplit;
  static constexpr size_t kAOff = kPOff + sizeof(float) * kWarps * 64;
  static constexpr size_t kBarOff = kAOff + sizeof(float) * kWarps * kMaxGroup;
  // mbarriers: one per stage, then three of the compact path (staged rows, score exchange,
  // the partials of the combine)
  static constexpr size_t kSmem = kBarOff + sizeof(uint64_t) * (kStages + 3);
  static constexpr int kMinBlocks = (!W && kSmem <= 112 * 1024) ? 2 : 1;
  static_assert(!W || (BF16 && kStages % 2 == 0), "wide: bf16 only, even stage count");

  // Compact path (a bf16 decode step with one cluster per unit).  CTA r scores the slice of `fast_per` teams starting at r * fast_per (a power
  // of two >= 4, so each slice is a whole number of 16-byte pieces and team j's rank and
  // place in it are shifts) and sends its block [G + 1][fast_per] (the G heads' scores, then
  // the page ids) from its list region to every CTA, into block r of the receive buffer
  // [cluster][G + 1][fast_per] at the end of the ring.  In front of it, from the first stage
  // the scratch needs: the CDF [cap] uint64, drawn flags and pi [cap] 4 B each.
  // The representative rows are staged from the start of the ring up to the receive buffer
  // (peers may send while this CTA still scores; everything else is written after).
  static constexpr int fast_per(int max_teams, int cluster) {
    int per = 4;
    while (per < (max_teams + cluster - 1) / cluster) per *= 2;
    return per;
  }
  static constexpr size_t fast_recv_bytes(int max_teams, int cluster) {
    return (G + 1) * static_cast<size_t>(cluster) * fast_per(max_teams, cluster) * 4;
  }
  static constexpr size_t fast_misc_bytes(int max_teams) {
    return (16 * static_cast<size_t>((max_teams + 3) / 4 * 4) + 127) / 128 * 128;
  }
  static constexpr int fast_scratch_stages(int max_teams, int cluster) {
    return static_cast<int>((fast_recv_bytes(max_teams, cluster) + fast_misc_bytes(max_teams) +
                             kStageBytes - 1) / kStageBytes);
  }
  // Whether a shape runs on the compact path: every team of the unit sampled in each CTA
  // (at most 1024), slices of at most 256 teams whose scores fit the list region and whose
  // representative rows fit in front of the receive buffer, at least one stage in front of
  // the scratch, and each CTA's chunks within its table.
  static constexpr bool fast_fits(int max_teams, int cluster, int team_size, int num_draws) {
    const int per = fast_per(max_teams, cluster);
    const int free_stages = kStages - fast_scratch_stages(max_teams, cluster);
    const int sel_max = num_draws < max_teams ? num_draws : max_teams;
    const int chunks = (sel_max * (team_size / kChunk) + cluster - 1) / cluster;
    return max_teams >= 1 && max_teams <= kMaxTeamsPerCta && per <= 256 && free_stages >= 1 &&
           static_cast<size_t>(G + 1) * per * 4 <= sizeof(ListEntry) * kMaxTeamsPerCta &&
           static_cast<size_t>(per) * D * 4 + fast_recv_bytes(max_teams, cluster) <=
               static_cast<size_t>(kRing) &&
           chunks <= kMaxChunksPerSplit;
  }
};

// ---------------------------------------------------------------- element loaders

template <bool BF16, int D>
__device__ __forceinline__ int score_elem(int lane16, int e) {
  if constexpr (BF16) {
    return lane16 * (D / 16) + e;
  } else {
    return (e >> 2) * 64 + lane16 * 4 + (e & 3);
  }
}

// Score-phase row slice of lane16: bf16 rows as one 8- or 16-byte vector per lane; fp32 rows
// with d = 128 as two 16-byte vectors 256 bytes apart (a quarter-warp always covers 128
// consecutive bytes, no bank conflicts).  Works on shared or global memory.
template <bool BF16, int D>
__device__ __forceinline__ void load_score_row(const unsigned char* row, int lane16,
                                               float (&x)[D / 16]) {
  if constexpr (BF16 && D == 128) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + lane16 * 16);
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  } else if constexpr (BF16 && D == 64) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + lane16 * 8);
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
  } else if constexpr (!BF16 && D == 128) {
    const float4 a = *reinterpret_cast<const float4*>(row + lane16 * 16);
    const float4 c = *reinterpret_cast<const float4*>(row + 256 + lane16 * 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = c.x; x[5] = c.y; x[6] = c.z; x[7] = c.w;
  } else {
    const float4 a = *reinterpret_cast<const float4*>(row + lane16 * 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  }
}

template <bool BF16, int D>
__device__ __forceinline__ void load_value_row(const unsigned char* row, int lane,
                                               float (&x)[D / 32]) {
  if constexpr (BF16 && D == 128) {
    const uint2 w = *reinterpret_cast<const uint2*>(row + lane * 8);
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
  } else if constexpr (BF16 && D == 64) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(row + lane * 4);
    x[0] = bf16_lo(w); x[1] = bf16_hi(w);
  } else if constexpr (!BF16 && D == 128) {
    const float4 a = *reinterpret_cast<const float4*>(row + lane * 16);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  } else {
    const float2 a = *reinterpret_cast<const float2*>(row + lane * 8);
    x[0] = a.x; x[1] = a.y;
  }
}

// Sum of v[0..7] over the 16 lanes of each half-warp, scattered: afterwards lane l holds
// the full sum of head (l >> 1) & 7 (lanes l and l^1 hold the same value).  8 shuffles.
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int lane) {
  const bool b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
  float w4[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float send = b3 ? v[k] : v[k + 4];
    const float keep = b3 ? v[k + 4] : v[k];
    w4[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  float w2[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float send = b2 ? w4[k] : w4[k + 2];
    const float keep = b2 ? w4[k + 2] : w4[k];
    w2[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  float w1 = (b1 ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? w2[0] : w2[1], 2);
  return w1 + __shfl_xor_sync(0xffffffffu, w1, 1);
}

// Inclusive scan of one value per thread over the 256-thread block, fixed order.
template <typename V>
__device__ __forceinline__ V block_inclusive_scan(V v, V* warp_tot, V& block_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    V w = lane < 8 ? warp_tot[lane] : V(0);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const V t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    if (lane < 8) warp_tot[lane] = w;
  }
  __syncthreads();
  const V pre = warp > 0 ? warp_tot[warp - 1] : V(0);
  block_total = warp_tot[7];
  const V res = pre + v;
  __syncthreads();
  return res;
}

// Exclusive scan of one value per thread over the 256-thread block with a single barrier:
// every warp sums the 8 warp totals itself (fixed order).  `total` receives the block sum.
// warp_tot must not be written again before another block-wide barrier.
template <typename V>
__device__ __forceinline__ V block_exclusive_scan(V v, V* warp_tot, V& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  V incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  V pre = V(0), tot = V(0);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const V t = warp_tot[w];
    if (w < warp) pre += t;
    tot += t;
  }
  total = tot;
  return pre + incl - v;
}

// Systematic draw point r: floor((r Z + t_u) / M), the fixed-point form of (r + u) Z / M
// (t_u = floor(u Z), Z < 2^63, M <= 4096).  The 128-bit numerator is divided by two 64-bit
// long-division steps; its high word is below M, so every partial numerator fits.
// Kept out of line: the default sampler never calls it, and its long divisions would
// otherwise lengthen the straight-line code every launch fetches.
static __device__ __noinline__ unsigned long long systematic_point(unsigned long long t_u, int r,
                                                                   int M, unsigned long long Z) {
  const unsigned long long ru = static_cast<unsigned long long>(r);
  const unsigned long long lo0 = ru * Z;
  const unsigned long long lo = lo0 + t_u;
  const unsigned long long hi = __umul64hi(ru, Z) + (lo < lo0 ? 1ull : 0ull);
  const unsigned long long m = static_cast<unsigned long long>(M);
  const unsigned long long x1 = (hi << 32) | (lo >> 32);
  const unsigned long long q1 = x1 / m;
  const unsigned long long x0 = ((x1 - q1 * m) << 32) | (lo & 0xffffffffull);
  return (q1 << 32) | (x0 / m);
}

// 1 / weight of a selected team under the sampler: Horvitz-Thompson 1 - (1 - q)^M,
// systematic min(1, M q), Hansen-Hurwitz M q / c (c draws of the team).
__device__ __forceinline__ float team_recip(int sampler, float Mf, float q, int c) {
  if (sampler == SANTA_SAMPLER_SYSTEMATIC) return fminf(1.f, Mf * q);
  if (sampler == SANTA_SAMPLER_IID_HH) return Mf * q / static_cast<float>(c);
  return -expm1f(Mf * log1pf(-q));
}

// Team of sampled slot k (0-based, k < the number of set bits): the k-th set bit of the
// team mask, whose 32-bit words are grouped in 8 runs of `wpw` words with set-bit counts
// gtot[0..7].  Slots follow ascending team order.
__device__ __forceinline__ int select_team(const uint32_t* mask, const int* gtot, int wpw, int k) {
  int g = 0;
  while (g < 7 && k >= gtot[g]) k -= gtot[g++];
  int w = g * wpw;
  for (;;) {
    const int c = __popc(mask[w]);
    if (k < c) break;
    k -= c;
    ++w;
  }
  uint32_t m = mask[w];
  int pos = 0;
#pragma unroll
  for (int half = 16; half; half >>= 1) {
    const uint32_t lo = m & ((1u << half) - 1u);
    const int c = __popc(lo);
    if (k >= c) {
      k -= c;
      m >>= half;
      pos += half;
    } else {
      m = lo;
    }
  }
  return 32 * w + pos;
}

// Scores s_{g,j} = q_g . rep_j / sqrt(d) of teams [t0, t0 + cnt) of unit (b, h), written
// to es[g * stride + j] (j relative to t0); pg[j] receives the team's page id, or -2 for a
// page id out of range (score -inf, status bit).  The page ids of a batch are read in one
// parallel pass first, so that the 16-byte asynchronous copies of the fp32 representative
// rows (issued by every thread, one round trip per batch of `rows_cap` rows) do not each
// wait on a dependent load; 16 lanes score one team (d/16 elements each, q in registers in
// the same layout) and an 8-shuffle reduce-scatter leaves lane l with head (l >> 1) & 7.
template <int D, int G>
__device__ __forceinline__ void score_teams(const DecodeParams& p, int b, int h, int t0, int cnt,
                                            const float (&qs)[G][D / 16], float* rows,
                                            int rows_cap, float* es, int stride, int* pg) {
  constexpr int kQuads = D / 4;                    // 16-byte pieces of a row
  constexpr float kNegInf = -INFINITY;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, lane16 = lane & 15;
  const int hh = (lane >> 1) & 7;
  for (int j0 = 0; j0 < cnt; j0 += rows_cap) {
    const int bc = min(rows_cap, cnt - j0);
    for (int j = tid; j < bc; j += 256) {
      const int page = p.page_table[static_cast<int64_t>(b) * p.max_teams + t0 + j0 + j];
      const bool ok = page >= 0 && page < p.num_pages;
      if (!ok) set_status(p.status, SANTA_DEV_BAD_PAGE);
      pg[j0 + j] = ok ? page : -2;
    }
    __syncthreads();
    for (int c = tid; c < bc * kQuads; c += 256) {
      const int j = c / kQuads, k = c - j * kQuads;
      const int64_t page = max(pg[j0 + j], 0);
      cp_async16(rows + static_cast<size_t>(j) * D + 4 * k,
                 p.reps + (page * p.num_kv_heads + h) * D + 4 * k);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int jj = 2 * warp; jj < bc; jj += 16) {
      const int j = jj + (lane >> 4);
      float x[D / 16];
      if (j < bc) {
        load_score_row<false, D>(reinterpret_cast<const unsigned char*>(rows + static_cast<size_t>(j) * D),
                                 lane16, x);
      } else {
#pragma unroll
        for (int e = 0; e < D / 16; ++e) x[e] = 0.f;
      }
      float part[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        part[g] = 0.f;
        if (g < G) {
#pragma unroll
          for (int e = 0; e < D / 16; ++e) part[g] = fmaf(qs[g][e], x[e], part[g]);
        }
      }
      const float sum = reduce_scatter8(part, lane);
      if (j < bc && !(lane & 1) && hh < G)
        es[hh * stride + j0 + j] = pg[j0 + j] >= 0 ? sum * p.scale : kNegInf;
    }
    __syncthreads();                               // rows may be refilled
  }
  fence_proxy_async_smem();    // the staging rows may next be overwritten by bulk copies
}

// ---------------------------------------------------------------- the kernel

template <bool BF16, int D, int G, bool W, int FAST = 0>
__global__ void __launch_bounds__(256, (DecodeTraits<BF16, D, G, W>::kMinBlocks))
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using Tr = DecodeTraits<BF16, D, G, W>;
  constexpr int S = Tr::kStages;
  constexpr float kNegInf = -INFINITY;
  cgx::cluster_group cluster = cgx::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int CL = static_cast<int>(cluster.num_blocks());
  const int NC = FAST ? 1 : p.clusters_per_unit;
  const int cidx = blockIdx.x / CL;
  const int h = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.num_kv_heads + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, lane16 = lane & 15;
  const int M = p.num_draws;
  const int mode = FAST == 1 ? kModeDecode : p.mode;   // FAST = 2: decode or sample only
  const bool sampling = mode == kModeDecode || mode == kModeSample;
  const bool attending = mode != kModeSample;
  const bool writer = cidx == 0;          // the cluster that writes the sampling outputs

  extern __shared__ __align__(1024) unsigned char smem[];  // 128-byte swizzle atoms: 1 KiB
  ListEntry* list = reinterpret_cast<ListEntry*>(smem + Tr::kListOff);
  ChunkMeta* table = reinterpret_cast<ChunkMeta*>(smem + Tr::kTableOff);
  float* prow = reinterpret_cast<float*>(smem + Tr::kPOff);
  float* arow = reinterpret_cast<float*>(smem + Tr::kAOff);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Tr::kBarOff);
  __shared__ Published pub;
  __shared__ float s_pm[16 * kMaxGroup], s_pz[16 * kMaxGroup];   // peers' (m, z)
  __shared__ float s_gm[kMaxGroup], s_gz[kMaxGroup];
  __shared__ unsigned long long s_wd[8];
  __shared__ int s_wi[8];
  __shared__ int s_base[17];
  __shared__ unsigned long long s_off, s_Z;
  __shared__ int s_abort, s_last;
  int L = 0;                  // the unit's sequence length
  int n_chunks = 0;           // 64-token chunks this CTA streams
  int early_n = 0;            // chunks already issued when the chunk table is complete
  // one chunk's K and V copies into its ring stage (or a bare arrival for an empty chunk)
  const unsigned char* kpool = static_cast<const unsigned char*>(p.k_pool);
  const unsigned char* vpool = static_cast<const unsigned char*>(p.v_pool);
  auto issue_meta = [&](int ci, const ChunkMeta& m) {
    const int stage = ci % S;
    if (m.page >= 0) {
      unsigned char* dst = smem + static_cast<size_t>(stage) * Tr::kStageBytes;
      mbar_arrive_expect_tx(&bar[stage], 2u * Tr::kChunkBytes);
      if constexpr (BF16) {
        // 64 rows x 64 elements (128 bytes, swizzled) per box; d = 128 takes two boxes
        const int row = (m.page * p.num_kv_heads + h) * p.team_size + m.part * kChunk;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx) {
          tma_load_2d(dst + bx * kChunk * 128, &p.tmap_k, bx * 64, row, &bar[stage]);
          tma_load_2d(dst + Tr::kChunkBytes + bx * kChunk * 128, &p.tmap_v, bx * 64, row,
                      &bar[stage]);
        }
      } else {
        const int64_t off = ((static_cast<int64_t>(m.page) * p.num_kv_heads + h) *
                                 static_cast<int64_t>(p.team_size) + m.part * kChunk) *
                            D * Tr::kEsize;
        bulk_g2s(dst, kpool + off, Tr::kChunkBytes, &bar[stage]);
        bulk_g2s(dst + Tr::kChunkBytes, vpool + off, Tr::kChunkBytes, &bar[stage]);
      }
    } else {
      mbar_arrive(&bar[stage]);
    }
  };
  if constexpr (FAST) {
    // ============================================================ compact path: phases A, B
    // A decode step with one cluster per unit, every team of the unit sampled in each CTA
    // (DecodeTraits::fast_fits).  FAST = 1: i.i.d. draws with Horvitz-Thompson weights and no
    // mixture; FAST = 2 also compiles the sampler variants and the mixture (separate
    // instantiations: the default sampler's prologue measured slower with their code in it).
    // This code runs once per launch, so it is kept short (rolled loops) and has few phases:
    // the SM waits on fetching straight-line instructions here more than on the arithmetic.
    const int n_max = p.max_teams;
    const int per = Tr::fast_per(n_max, CL);           // teams scored per CTA, power of 2
    const int lo = rank * per;
    const int nl = max(0, min(per, n_max - lo));
    const int cap = (n_max + 3) & ~3;
    early_n = S - Tr::fast_scratch_stages(n_max, CL);     // stages in front of the scratch
    const int RS = (G + 1) * per;                      // floats of one rank's block
    const int lp = __ffs(per) - 1;
    // team j's entry of row g (g = G: its page id) in the receive buffer: block j >> lp,
    // place j & (per - 1)
    auto at = [&](int j, int g) { return j + (((j >> lp) * G + g) << lp); };
    float* xs = reinterpret_cast<float*>(smem + Tr::kRing - Tr::fast_recv_bytes(n_max, CL));
    unsigned long long* cdf = reinterpret_cast<unsigned long long*>(
        smem + static_cast<size_t>(early_n) * Tr::kStageBytes);        // [cap]
    int* flg = reinterpret_cast<int*>(cdf + cap);                        // [cap] drawn
    float* ps = reinterpret_cast<float*>(flg + cap);                     // [cap] pi
    float* rows = reinterpret_cast<float*>(smem);      // [per][D] staged representatives
    float* mine = reinterpret_cast<float*>(list);      // [G + 1][per] this CTA's slice, sent
    uint64_t* rbar = &bar[S];                          // staged rows
    uint64_t* xbar = &bar[S + 1];                      // the received slices
    const bool bad_layout = BF16 && (smem_u32(smem) & 1023u) != 0;
    __shared__ uint32_t s_xw[Tr::kThreads];
    const uint2 key = make_uint2(static_cast<uint32_t>(p.seed),
                                 static_cast<uint32_t>(p.seed >> 32));
    if (!bad_layout) {
      // shared memory only: allowed before the previous kernel of the stream has finished
      if (tid == 0) {
        if (attending) {
          prefetch_tensormap(&p.tmap_k);
          prefetch_tensormap(&p.tmap_v);
        }
        for (int s2 = 0; s2 < S; ++s2) mbar_init(&bar[s2], 1);
        mbar_init(rbar, Tr::kThreads);
        mbar_init(xbar, 1);
        mbar_init(&bar[S + 2], 1);     // the combine's partials
        fence_mbar_init();
        s_abort = 0;
      }
      __syncthreads();                // the mbarriers are initialised
      if (tid == 0) mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(CL * RS * 4));
      cluster_arrive_relaxed();       // split barrier: this CTA runs, its mbarriers are set up
    }
    grid_dependency_wait();
    grid_launch_dependents();
    if (bad_layout) {                 // the same for every CTA: all leave together
      if (tid == 0 && rank == 0) set_status(p.status, SANTA_DEV_LAYOUT);
      return;
    }
    // ---- the loads that depend on nothing else: length, query, this thread's row of the
    // slice; the row's representative comes by one bulk copy on rbar
    L = p.seq_lens[b];
    const bool len_ok = L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(n_max) *
                                                                p.team_size;
    const int n = len_ok ? (L + p.team_size - 1) / p.team_size : 0;
    if (tid < nl) {
      const int page = p.page_table[static_cast<int64_t>(b) * n_max + lo + tid];
      const bool ok = page >= 0 && page < p.num_pages;
      mine[G * per + tid] = __int_as_float(ok ? page : -2);
      if (ok) {
        mbar_arrive_expect_tx(rbar, D * 4);
        bulk_g2s(rows + static_cast<size_t>(tid) * D,
                 p.reps + (static_cast<int64_t>(page) * p.num_kv_heads + h) * D, D * 4, rbar);
      } else {
        mbar_arrive(rbar);
        if (lo + tid < n) set_status(p.status, SANTA_DEV_BAD_PAGE);
      }
    } else {
      mbar_arrive(rbar);
    }
    if (!len_ok && rank == 0 && tid == 0) set_status(p.status, SANTA_DEV_BAD_SEQLEN);
    float qs[G][Tr::kEplS];           // the group's query in the fp32 score layout
    {
      const uint16_t* qh = static_cast<const uint16_t*>(p.q) +
                           (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e4 = 0; e4 < Tr::kEplS / 4; ++e4) {
          const uint2 w = *reinterpret_cast<const uint2*>(qh + g * D + e4 * 64 + lane16 * 4);
          qs[g][4 * e4] = bf16_lo(w.x);
          qs[g][4 * e4 + 1] = bf16_hi(w.x);
          qs[g][4 * e4 + 2] = bf16_lo(w.y);
          qs[g][4 * e4 + 3] = bf16_hi(w.y);
        }
    }
    // the Philox word of each draw r < 256 (it needs only the seed and the unit) while the
    // representative rows are in flight; draw r falls to thread (r mod 32) * 8 + r / 32, so
    // the first draws spread over all warps
    {
      const int r = (tid & 7) * 32 + (tid >> 3);
      if (r < M)
        s_xw[r] = philox4x32_10_compact(make_uint4(static_cast<uint32_t>(r),
                                                   static_cast<uint32_t>(h),
                                                   static_cast<uint32_t>(b), 0u), key).x;
    }
    if (!mbar_wait(rbar, 0)) set_status(p.status, SANTA_DEV_TIMEOUT);
    // ---- the slice's scores s_{g,j} = q_g . rep_j / sqrt(d), kept in base 2 (times log2 e,
    // so that exp(s - m) is one exp2): 16 lanes per team, lane l ends with head (l >> 1) & 7;
    // -inf past the sequence and for bad page ids
    {
      const int hh = (lane >> 1) & 7;
#pragma unroll 2
      for (int j0 = 0; j0 < nl; j0 += 16) {
        const int jl = j0 + 2 * warp + (lane >> 4);
        float x[Tr::kEplS];
        if (jl < nl) {
          load_score_row<false, D>(reinterpret_cast<const unsigned char*>(rows + static_cast<size_t>(jl) * D),
                                   lane16, x);
        } else {
#pragma unroll
          for (int e = 0; e < Tr::kEplS; ++e) x[e] = 0.f;
        }
        float part[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          part[g] = 0.f;
          if (g < G) {
#pragma unroll
            for (int e = 0; e < Tr::kEplS; ++e) part[g] = fmaf(qs[g][e], x[e], part[g]);
          }
        }
        const float sum = reduce_scatter8(part, lane);
        if (jl < nl && !(lane & 1) && hh < G) {
          const bool ok = __float_as_int(mine[G * per + jl]) >= 0 && lo + jl < n;
          mine[hh * per + jl] = ok ? sum * p.scale_log2 : kNegInf;   // base 2
        }
      }
    }
    // ---- send the slice to every CTA of the cluster (itself included), into block `rank`
    // of the receiver's buffer: 16-byte st.async stores from every thread, whose bytes
    // complete on the receiver's xbar (bulk copies took the issuing threads longer)
    fence_proxy_async_smem();         // staged rows read: the ring's start is refilled by copies later
    __syncthreads();
    cluster_wait();                   // every peer runs and has initialised its mbarriers
    {
      const int nq = RS / 4;                           // 16-byte quads of one block
      const float4* src = reinterpret_cast<const float4*>(mine);
#pragma unroll 1
      for (int i = tid; i < CL * nq; i += Tr::kThreads) {
        const int dst = i / nq, qd = i - dst * nq;
        st_async_v4(cluster_addr(smem_u32(xs + rank * RS + 4 * qd), dst), src[qd],
                    cluster_addr(smem_u32(xbar), dst));
      }
    }
    if (!mbar_wait(xbar, 0)) set_status(p.status, SANTA_DEV_TIMEOUT);
    // ---- per-head statistics over the unit, warp g on row g: m_g, e_gj = exp(s_gj - m_g)
    // (2^ of the base-2 scores) in place and 1 / (G z_g); four independent teams per lane at a
    // time, summed in a fixed order (the same in every CTA)
    const bool out_writer = rank == 0;
    const int tpt = (n_max + Tr::kThreads - 1) / Tr::kThreads;
    const int jt = tid * tpt;
    __shared__ float s_zinv[kMaxGroup];
    if (warp < G) {
      float m = kNegInf;
#pragma unroll 1
      for (int j0 = lane; j0 < n_max; j0 += 128) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = j0 + 32 * k < n_max ? xs[at(j0 + 32 * k, warp)] : kNegInf;
        m = fmaxf(m, fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3])));
      }
      m = warp_max(m);
      float z = 0.f;
#pragma unroll 1
      for (int j0 = lane; j0 < n_max; j0 += 128) {
        int a[4];
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {          // every load of the four before any store
          a[k] = at(j0 + 32 * k, warp);
          v[k] = j0 + 32 * k < n_max ? xs[a[k]] : kNegInf;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float ev = v[k] == kNegInf ? 0.f : ex2_approx(v[k] - m);
          if (j0 + 32 * k < n_max) xs[a[k]] = ev;
          z += ev;
        }
      }
      z = warp_sum(z);
      if (lane == 0) s_zinv[warp] = z > 0.f ? 1.f / (z * static_cast<float>(G)) : 0.f;
    }
    __syncthreads();
    float zg[G];
#pragma unroll
    for (int g = 0; g < G; ++g) zg[g] = s_zinv[g];
    // ---- p_j = sum_g e_gj / (G z_g), round(p_j 2^62) and the exact integer CDF (this
    // thread's inclusive sums, then one block-wide scan)
    unsigned long long run = 0ull;
    const float alpha = FAST == 2 ? p.mix_alpha : 0.f;  // defensive mixture: q = (1 - a) p + a / n
    const float alpha_n = n > 0 ? alpha / static_cast<float>(n) : 0.f;
#pragma unroll 1
    for (int u = 0; u < tpt; ++u) {
      const int j = jt + u;
      if (j < n_max) {
        float pj = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) pj = fmaf(xs[at(j, g)], zg[g], pj);
        if constexpr (FAST == 2)
          if (alpha != 0.f && j < n) pj = fmaf(1.f - alpha, pj, alpha_n);
        unsigned long long P = 0ull;
        if (pj > 0.f) {
          const float x = pj * 0x1p62f;                              // exact scaling
          const unsigned long long fl = __float2ull_rd(x);
          const float frac = x - __ull2float_rn(fl);                 // exact
          P = fl + (frac >= 0.5f ? 1ull : 0ull);
        }
        run += P;
        cdf[j] = run;                 // this thread's inclusive sum; its prefix is added below
        // 1 / weight and its -log2 (to the team's head-0 entry of the receive buffer, no
        // longer read), independent of the scan below: Horvitz-Thompson pi_j = 1 - (1 - q_j)^M,
        // systematic min(1, M q_j); Hansen-Hurwitz needs the draw counts, so q_j waits here
        const float Mf = static_cast<float>(M);
        float piv;
        if constexpr (FAST == 2)
          piv = p.sampler == SANTA_SAMPLER_SYSTEMATIC ? fminf(1.f, Mf * pj)
                : p.sampler == SANTA_SAMPLER_IID_HH   ? pj
                                                      : -expm1f(Mf * log1pf(-pj));
        else
          piv = -expm1f(Mf * log1pf(-pj));
        ps[j] = piv;
        xs[at(j, 0)] = -log2f(piv);
        flg[j] = 0;
        if (p.team_probs && out_writer)
          p.team_probs[static_cast<int64_t>(unit) * p.max_teams + j] = pj;
      }
    }
    unsigned long long Z;
    const unsigned long long before = block_exclusive_scan<unsigned long long>(run, s_wd, Z);
#pragma unroll 1
    for (int u = 0; u < tpt; ++u)
      if (jt + u < n_max) cdf[jt + u] += before;
    __syncthreads();
    // ---- M draws: the smallest j with floor(u Z) < C_j
    const bool valid = len_ok && Z > 0ull;
    if (valid) {
      // systematic: every point derives from the uniform of draw 0
      const bool systematic = FAST == 2 && p.sampler == SANTA_SAMPLER_SYSTEMATIC;
#pragma unroll 1
      for (int r = tid; r < M; r += Tr::kThreads) {
        uint32_t x;
        if constexpr (FAST == 2) {
          const int rw = systematic ? 0 : r;
          x = rw < Tr::kThreads
                  ? s_xw[rw]
                  : philox4x32_10_compact(make_uint4(static_cast<uint32_t>(rw),
                                                     static_cast<uint32_t>(h),
                                                     static_cast<uint32_t>(b), 0u), key).x;
        } else {
          x = r == tid ? s_xw[r]
                       : philox4x32_10_compact(make_uint4(static_cast<uint32_t>(r),
                                                          static_cast<uint32_t>(h),
                                                          static_cast<uint32_t>(b), 0u), key).x;
        }
        const unsigned long long a = 2ull * x + 1ull;                // u = a / 2^33
        unsigned long long t = (__umul64hi(a, Z) << 31) | ((a * Z) >> 33);
        if constexpr (FAST == 2)
          if (systematic) t = systematic_point(t, r, M, Z);
        int lo_i = 0, hi_i = n_max - 1;
#pragma unroll 1
        while (lo_i < hi_i) {
          const int mid = (lo_i + hi_i) >> 1;
          if (t < cdf[mid]) hi_i = mid; else lo_i = mid + 1;
        }
        if (out_writer) p.draw_ids[static_cast<int64_t>(unit) * M + r] = lo_i;
        if constexpr (FAST == 2) {
          if (p.sampler == SANTA_SAMPLER_IID_HH) atomicAdd(&flg[lo_i], 1);   // draws per team
          else flg[lo_i] = 1;
        } else {
          flg[lo_i] = 1;
        }
      }
    } else if (out_writer) {
#pragma unroll 1
      for (int r = tid; r < M; r += Tr::kThreads) p.draw_ids[static_cast<int64_t>(unit) * M + r] = -1;
    }
    __syncthreads();
    // ---- S in ascending team order (per-thread counts, a block scan: slot k of each drawn
    // team) and phase B at once: the thread holding a sampled team writes its outputs and the
    // table entries of its 64-token chunks that fall in this CTA's contiguous range, and
    // copies at once those that go to the stages in front of the scratch
    {
      int cnt = 0;
#pragma unroll 1
      for (int u = 0; u < tpt; ++u) cnt += (jt + u < n_max && flg[jt + u]) ? 1 : 0;
      int tot;
      int k = block_exclusive_scan<int>(cnt, s_wi, tot);
      const int cpt = p.team_size / kChunk;
      const int total_chunks = attending ? tot * cpt : 0;
      const int cps = (total_chunks + CL - 1) / CL;
      const int c_begin = min(rank * cps, total_chunks);
      n_chunks = min(total_chunks - c_begin, cps);
#pragma unroll 1
      for (int u = 0; u < tpt; ++u) {
        const int j = jt + u;
        if (j < n_max && flg[j]) {
          if constexpr (FAST == 2) {
            if (p.sampler == SANTA_SAMPLER_IID_HH) {   // 1 / weight = M q_j / c_j
              const float recip = static_cast<float>(M) * ps[j] / static_cast<float>(flg[j]);
              ps[j] = recip;
              xs[at(j, 0)] = -log2f(recip);
            }
          }
          if (out_writer) {
            p.sel_ids[static_cast<int64_t>(unit) * M + k] = j;
            p.pi[static_cast<int64_t>(unit) * M + k] = ps[j];
          }
          const int page = __float_as_int(xs[at(j, G)]);
          const bool pok = page >= 0 && page < p.num_pages;
#pragma unroll 1
          for (int part = 0; part < cpt; ++part) {
            const int ci = k * cpt + part - c_begin;
            if (ci >= 0 && ci < n_chunks) {
              const int vt = pok ? max(0, min(min(p.team_size, L - j * p.team_size) -
                                                  part * kChunk, kChunk))
                                 : 0;
              const ChunkMeta m{vt > 0 ? page : -1, vt, xs[at(j, 0)], part};
              table[ci] = m;
              if (ci < early_n) issue_meta(ci, m);
            }
          }
          ++k;
        }
      }
      if (out_writer) {
#pragma unroll 1
        for (int k2 = tot + tid; k2 < M; k2 += Tr::kThreads) {
          p.sel_ids[static_cast<int64_t>(unit) * M + k2] = -1;
          p.pi[static_cast<int64_t>(unit) * M + k2] = 0.f;
        }
        if (tid == 0) p.sel_count[unit] = tot;
      }
    }
  } else {
  // Launched with programmatic stream serialization: nothing of global memory is touched
  // before the previous kernel of the stream has completed, and the next one may be
  // scheduled (onto SMs this grid leaves free) from here on.
  if constexpr (BF16) {
    if (attending && tid == 0) {       // descriptors are launch constants: no wait needed
      prefetch_tensormap(&p.tmap_k);
      prefetch_tensormap(&p.tmap_v);
    }
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if constexpr (BF16) {
    // The 128-byte-swizzled tile copies and the fragment addressing below both assume
    // 1 KiB-aligned stages; the layout is the same for every CTA, so all leave together.
    if (attending && (smem_u32(smem) & 1023u) != 0) {
      if (tid == 0 && rank == 0 && cidx == 0) set_status(p.status, SANTA_DEV_LAYOUT);
      return;
    }
  }

  // ---- per-unit lengths
  L = p.seq_lens[b];
  const bool len_ok = L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_teams) *
                                                             p.team_size;
  const int n = len_ok ? (L + p.team_size - 1) / p.team_size : 0;
  const int cpt = p.team_size / kChunk;
  if (!len_ok && writer && rank == 0 && tid == 0) set_status(p.status, SANTA_DEV_BAD_SEQLEN);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    mbar_init(&bar[S + 2], 1);       // the combine's partials
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  // Decode steps sampled inside one CTA keep the phase-A scratch in the last stage(s) of the
  // ring, so that this CTA's first `early_n` chunks can be copied as soon as S is known,
  // while the chunk table is still being built from that scratch.

  // ================================================================ phase A: sampling
  int total_sel = 0;                      // |S| of the unit
  // Exchange path: each CTA scores its slice of the teams and publishes the raw scores in
  // its list region; after one cluster barrier every CTA reads all scores (one parallel
  // DSMEM read) and samples the whole unit locally, so all CTAs hold the same S without
  // further exchange.  Shapes whose slice scores do not fit the region use the
  // distributed path (softmax statistics, CDF totals and counts exchanged in three rounds).
  const int per = (n + CL - 1) / CL;
  const bool local = (G + 1) * per <= kPubScores && n <= kMaxTeamsPerCta;
  uint32_t* mask_area = nullptr;          // local sampling: room for the drawn-team mask
  const int* lpages = nullptr;            // local sampling: page id of every team of the unit
  const uint32_t* lmask = nullptr;        // local sampling: bit mask of the drawn teams
  const float* lps = nullptr;             // local sampling: team probabilities
  const int* lcnt = nullptr;              // local sampling: draws per team
  int lwpw = 1;                           // local sampling: mask words per warp
  if (sampling) {
    const int cap = local ? (max(n, 1) + 3) / 4 * 4 : p.teams_per_cta;   // rows 16-byte aligned
    const size_t scr = Tr::sample_scratch(cap);
    const int scr_stages = static_cast<int>((scr + Tr::kStageBytes - 1) / Tr::kStageBytes);
    if (local && mode == kModeDecode && scr_stages < S) early_n = S - scr_stages;
    unsigned char* scr_base = smem + static_cast<size_t>(early_n) * Tr::kStageBytes;
    unsigned long long* cdf = reinterpret_cast<unsigned long long*>(scr_base);   // [cap]
    float* es = reinterpret_cast<float*>(cdf + cap);                 // [8][cap] scores, exps
    float* ps = es + kMaxGroup * cap;                                // [cap] team probability
    int* flag = reinterpret_cast<int*>(ps + cap);                    // [cap] drawn / slot
    int* pages = flag + cap;                                         // [cap] page ids (local)
    mask_area = reinterpret_cast<uint32_t*>(pages + cap);            // [cap] (nw words used)
    if (local) lpages = pages;
    // staging rows for the representatives: the stages in front of the scratch, else the
    // rest of the ring behind it
    float* rows = reinterpret_cast<float*>(early_n > 0 ? smem : smem + scr);
    const int rows_cap = early_n > 0 ? early_n * Tr::kStageBytes / (D * 4) : Tr::rep_rows(cap);
    float* pub_scores = reinterpret_cast<float*>(list);              // [G][per], published
    int* pub_pages = reinterpret_cast<int*>(pub_scores + G * per);   // [per], published
    int lo = min(rank * per, n);
    int nl = min(lo + per, n) - lo;
    // q of the group in registers, in the fp32 score layout
    float qs[G][Tr::kEplS];
    {
      const int64_t qbase = (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < Tr::kEplS; ++e) {
          const int64_t idx = qbase + g * D + score_elem<false, D>(lane16, e);
          qs[g][e] = BF16 ? bf16_to_f32(static_cast<const uint16_t*>(p.q)[idx])
                          : static_cast<const float*>(p.q)[idx];
        }
    }
    if (local) {
      // Split cluster barrier, arrive: this CTA runs.  The wait below, before the first
      // remote store, guarantees that every peer runs too.
      cluster_arrive_relaxed();
      score_teams<D, G>(p, b, h, lo, nl, qs, rows, rows_cap, pub_scores, per, pub_pages);
      // the slice's per-head max m_r and sum of exp z_r; the staged scores become
      // e = exp(s - m_r), so that p needs no further exponentials once m and z are known
      if (warp < G) {
        float m = kNegInf;
        for (int j = lane; j < nl; j += 32) m = fmaxf(m, pub_scores[warp * per + j]);
        m = warp_max(m);
        float z = 0.f;
        for (int j = lane; j < nl; j += 32) {
          const float sc = pub_scores[warp * per + j];
          const float e = (m == kNegInf || sc == kNegInf) ? 0.f : expf(sc - m);
          pub_scores[warp * per + j] = e;
          z += e;
        }
        z = warp_sum(z);
        if (lane == 0) {
          pub.m[warp] = m;
          pub.z[warp] = z;
        }
      }
      __syncthreads();
      // push the slice (e rows [G][per], page ids [per]) and (m_r, z_r) into every CTA of the
      // cluster (this one included): remote stores, no round trip; barrier S1 publishes them
      cluster_wait();
      if ((per & 3) == 0) {
        const int q = per / 4;                                       // 16-byte words per row
        const int items = CL * (G + 1) * q;
        for (int i = tid; i < items; i += Tr::kThreads) {
          const int r = i / ((G + 1) * q), k = i - r * (G + 1) * q;
          const int g = k / q, jj = 4 * (k - g * q);
          if (jj >= nl) continue;
          const uint4 v = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(pub_scores) + g * per + jj);
          uint32_t* dst = g < G ? reinterpret_cast<uint32_t*>(es + g * cap) : reinterpret_cast<uint32_t*>(pages);
          *reinterpret_cast<uint4*>(cluster.map_shared_rank(dst, r) + lo + jj) = v;
        }
      } else {
        const int items = CL * (G + 1) * nl;
        for (int i = tid; i < items; i += Tr::kThreads) {
          const int r = i / ((G + 1) * nl), k = i - r * (G + 1) * nl;
          const int g = k / nl, jj = k - g * nl;
          const uint32_t v = reinterpret_cast<const uint32_t*>(pub_scores)[g * per + jj];
          uint32_t* dst = g < G ? reinterpret_cast<uint32_t*>(es + g * cap) : reinterpret_cast<uint32_t*>(pages);
          cluster.map_shared_rank(dst, r)[lo + jj] = v;
        }
      }
      if (tid < CL * G) {
        const int r = tid / G, g = tid - r * G;
        cluster.map_shared_rank(s_pm, r)[rank * G + g] = pub.m[g];
        cluster.map_shared_rank(s_pz, r)[rank * G + g] = pub.z[g];
      }
      cluster.sync();                                                // barrier S1
      // per-head max m and sum z over the CL slices (warp g, lane r), and the slice weights
      // w_rg = exp(m_rg - m_g) / (G z_g), so that p_j = sum_g e_gj w_(r(j))g
      if (warp < G) {
        const float mr = lane < CL ? s_pm[lane * G + warp] : kNegInf;
        const float m = warp_max(mr);
        const float er = (lane < CL && mr != kNegInf) ? expf(mr - m) : 0.f;
        const float z = warp_sum(lane < CL ? s_pz[lane * G + warp] * er : 0.f);
        if (lane < CL) s_pm[lane * G + warp] = z > 0.f ? er / (z * static_cast<float>(G)) : 0.f;
      }
      __syncthreads();
      // round(p_j 2^62) and the exact integer CDF: thread t takes teams [t*tpt, (t+1)*tpt),
      // a serial sum, then one block-wide scan
      constexpr int kTpt = kMaxTeamsPerCta / Tr::kThreads;
      const int tpt = (n + Tr::kThreads - 1) / Tr::kThreads;          // <= kTpt
      const int jt = tid * tpt;
      const bool out_writer = writer && rank == 0;
      unsigned long long run = 0ull, incl_t[kTpt];
      int rj = per > 0 ? jt / per : 0;                                // slice of team jt
      const float alpha = p.mix_alpha;                                // defensive mixture
      const float alpha_n = n > 0 ? alpha / static_cast<float>(n) : 0.f;
#pragma unroll
      for (int u = 0; u < kTpt; ++u) {
        const int j = jt + u;
        unsigned long long P = 0ull;
        if (u < tpt && j < n) {
          if (j >= (rj + 1) * per) ++rj;
          float pj = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) pj = fmaf(es[g * cap + j], s_pm[rj * G + g], pj);
          if (alpha != 0.f) pj = fmaf(1.f - alpha, pj, alpha_n);       // q_j
          ps[j] = pj;
          flag[j] = 0;
          if (p.team_probs && out_writer) p.team_probs[static_cast<int64_t>(unit) * p.max_teams + j] = pj;
          if (pj > 0.f) {
            const float x = pj * 0x1p62f;                            // exact scaling
            const unsigned long long fl = __float2ull_rd(x);
            const float frac = x - __ull2float_rn(fl);               // exact
            P = fl + (frac >= 0.5f ? 1ull : 0ull);
          }
        }
        run += P;
        incl_t[u] = run;
      }
      unsigned long long Z;
      const unsigned long long before = block_exclusive_scan<unsigned long long>(run, s_wd, Z);
#pragma unroll
      for (int u = 0; u < kTpt; ++u)
        if (u < tpt && jt + u < n) cdf[jt + u] = before + incl_t[u];
      if (p.team_probs && out_writer)
        for (int j = n + tid; j < p.max_teams; j += Tr::kThreads)
          p.team_probs[static_cast<int64_t>(unit) * p.max_teams + j] = 0.f;
      __syncthreads();
      // M draws: smallest j with floor(u Z) < C_j
      const bool valid = len_ok && Z > 0ull;
      if (valid) {
        const uint2 key = make_uint2(static_cast<uint32_t>(p.seed),
                                     static_cast<uint32_t>(p.seed >> 32));
        // systematic: every point derives from the uniform of draw 0
        const bool systematic = p.sampler == SANTA_SAMPLER_SYSTEMATIC;
        const bool count_draws = p.sampler == SANTA_SAMPLER_IID_HH;
        for (int r = tid; r < M; r += Tr::kThreads) {
          const uint4 w = philox4x32_10(make_uint4(systematic ? 0u : static_cast<uint32_t>(r),
                                                   static_cast<uint32_t>(h),
                                                   static_cast<uint32_t>(b), 0u),
                                        key);
          const unsigned long long a = 2ull * w.x + 1ull;            // u = a / 2^33
          unsigned long long t = (__umul64hi(a, Z) << 31) | ((a * Z) >> 33);
          if (systematic) t = systematic_point(t, r, M, Z);
          int lo_i = 0, hi_i = n - 1;
          while (lo_i < hi_i) {
            const int mid = (lo_i + hi_i) >> 1;
            if (t < cdf[mid]) hi_i = mid; else lo_i = mid + 1;
          }
          if (out_writer) p.draw_ids[static_cast<int64_t>(unit) * M + r] = lo_i;
          if (count_draws) atomicAdd(&flag[lo_i], 1);                 // draws per team
          else flag[lo_i] = 1;
        }
      } else if (out_writer) {
        for (int r = tid; r < M; r += Tr::kThreads) p.draw_ids[static_cast<int64_t>(unit) * M + r] = -1;
      }
      __syncthreads();
      // the distinct drawn teams as a bit mask over the teams (slot k = k-th set bit, so
      // slots follow ascending team order): warp w ballots its run of wpw words
      {
        const int nw = (n + 31) / 32, wpw = (nw + 7) / 8;
        uint32_t* mask = mask_area;                                  // [nw]
        int cnt = 0;
        for (int w = warp * wpw; w < min(nw, (warp + 1) * wpw); ++w) {
          const int j = 32 * w + lane;
          const uint32_t bits = __ballot_sync(0xffffffffu, valid && j < n && flag[j] > 0);
          if (lane == 0) mask[w] = bits;
          cnt += __popc(bits);
        }
        if (lane == 0) s_wi[warp] = cnt;
        lmask = mask;
        lps = ps;
        lcnt = flag;
        lwpw = wpw;
      }
      __syncthreads();
      int count = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) count += s_wi[w];
      total_sel = count;
      if (early_n > 0 && tid < early_n) {
        // this CTA's first chunks (the chunk range as phase B computes it), one per thread,
        // into the stages in front of the scratch; phase B fills the same table entries
        const int ctas = CL * NC, gidx = cidx * CL + rank;
        const int tot = count * cpt, per_cta = (tot + ctas - 1) / ctas;
        const int cb = min(gidx * per_cta, tot), nch = min(tot - cb, per_cta);
        const int ci = tid;
        if (ci < nch) {
          const int c = cb + ci, slot = c / cpt, part = c - slot * cpt;
          const int team = select_team(lmask, s_wi, lwpw, slot);
          const int page = pages[team];
          const bool pok = page >= 0 && page < p.num_pages;
          const int vt = pok ? max(0, min(min(p.team_size, L - team * p.team_size) - part * kChunk,
                                          kChunk))
                             : 0;
          issue_meta(ci, ChunkMeta{vt > 0 ? page : -1, vt, 0.f, part});
        }
      }
    } else {
      score_teams<D, G>(p, b, h, lo, nl, qs, rows, rows_cap, es, cap, flag);
      // per-head (max, sum of exp) over the scored teams
      if (warp < G) {
        float m = kNegInf;
        for (int j = lane; j < nl; j += 32) m = fmaxf(m, es[warp * cap + j]);
        m = warp_max(m);
        float z = 0.f;
        if (m != kNegInf)
          for (int j = lane; j < nl; j += 32) {
            const float sc = es[warp * cap + j];
            z += sc == kNegInf ? 0.f : expf(sc - m);
          }
        z = warp_sum(z);
        if (lane == 0) {
          pub.m[warp] = m;
          pub.z[warp] = z;
        }
      }
      {
        cluster.sync();                                                // barrier A1
        if (tid < CL * G) {
          const Published* peer = cluster.map_shared_rank(&pub, tid / G);
          s_pm[tid] = peer->m[tid % G];
          s_pz[tid] = peer->z[tid % G];
        }
        __syncthreads();
        if (tid < G) {
          float m = kNegInf;
          for (int r = 0; r < CL; ++r) m = fmaxf(m, s_pm[r * G + tid]);
          float z = 0.f;
          if (m != kNegInf)
            for (int r = 0; r < CL; ++r) {
              const float mr = s_pm[r * G + tid];
              z += mr == kNegInf ? 0.f : s_pz[r * G + tid] * expf(mr - m);
            }
          s_gm[tid] = m;
          s_gz[tid] = z;
        }
      }
      __syncthreads();
      // team probabilities p_j = (1/G) sum_g exp(s_gj - m_g) / z_g, and their 62-bit
      // fixed-point values round(p * 2^62) (ties away from zero); inclusive CDF
      const bool out_writer = writer;
      unsigned long long carry = 0;
      for (int base = 0; base < nl; base += Tr::kThreads) {
        const int j = base + tid;
        unsigned long long P = 0;
        if (j < nl) {
          float acc = 0.f;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float sc = es[g * cap + j];
            acc += (sc == kNegInf || !(s_gz[g] > 0.f)) ? 0.f : expf(sc - s_gm[g]) / s_gz[g];
          }
          const float pj = acc / static_cast<float>(G);
          ps[j] = pj;
          flag[j] = 0;                                                 // held page ids
          if (p.team_probs && out_writer)
            p.team_probs[static_cast<int64_t>(unit) * p.max_teams + lo + j] = pj;
          if (pj > 0.f) {
            const float x = pj * 0x1p62f;                              // exact scaling
            const unsigned long long fl = __float2ull_rd(x);
            const float frac = x - __ull2float_rn(fl);                 // exact
            P = fl + (frac >= 0.5f ? 1ull : 0ull);
          }
        }
        unsigned long long tot;
        const unsigned long long v = block_inclusive_scan<unsigned long long>(P, s_wd, tot);
        if (j < nl) cdf[j] = carry + v;
        carry += tot;
      }
      if (p.team_probs && writer && rank == 0)
        for (int j = n + tid; j < p.max_teams; j += Tr::kThreads)
          p.team_probs[static_cast<int64_t>(unit) * p.max_teams + j] = 0.f;
      {
        if (tid == 0) pub.total = nl > 0 ? cdf[nl - 1] : 0ull;
        cluster.sync();                                                // barrier A2
        if (warp == 0) {                                                // exclusive prefix over ranks
          const unsigned long long t = lane < CL ? cluster.map_shared_rank(&pub, lane)->total : 0ull;
          unsigned long long incl = t;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
          }
          if (lane == rank) s_off = incl - t;
          if (lane == 31) s_Z = incl;
        }
      }
      __syncthreads();
      // M draws; the CTA whose slice [off, off + total) holds floor(u Z) resolves the draw
      const unsigned long long off = s_off, Z = s_Z;
      const bool valid = len_ok && Z > 0ull;
      if (valid && nl > 0) {
        const unsigned long long tot = cdf[nl - 1];
        const uint2 key = make_uint2(static_cast<uint32_t>(p.seed),
                                     static_cast<uint32_t>(p.seed >> 32));
        for (int r = tid; r < M; r += Tr::kThreads) {
          const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(r), static_cast<uint32_t>(h),
                                                   static_cast<uint32_t>(b), 0u),
                                        key);
          const unsigned long long a = 2ull * w.x + 1ull;              // u = a / 2^33
          const unsigned long long t = (__umul64hi(a, Z) << 31) | ((a * Z) >> 33);
          if (t >= off && t - off < tot) {
            const unsigned long long tl = t - off;
            int lo_i = 0, hi_i = nl - 1;
            while (lo_i < hi_i) {
              const int mid = (lo_i + hi_i) >> 1;
              if (tl < cdf[mid]) hi_i = mid; else lo_i = mid + 1;
            }
            if (out_writer) p.draw_ids[static_cast<int64_t>(unit) * M + r] = lo + lo_i;
            flag[lo_i] = 1;
          }
        }
      }
      if (!valid && writer && rank == 0)
        for (int r = tid; r < M; r += Tr::kThreads) p.draw_ids[static_cast<int64_t>(unit) * M + r] = -1;
      __syncthreads();
      // number the drawn teams (ascending) and record them with -log2 pi
      ListEntry* mylist = list;
      int count = 0;
      const float Mf = static_cast<float>(M);
      for (int base = 0; base < nl; base += Tr::kThreads) {
        const int j = base + tid;
        const int f = j < nl ? (flag[j] == 1) : 0;
        int tot;
        const int incl = block_inclusive_scan<int>(f, s_wi, tot);
        if (f) {
          const int k = count + incl - 1;
          const float piv = -expm1f(Mf * log1pf(-ps[j]));
          mylist[k] = ListEntry{lo + j, -log2f(piv)};
          flag[j] = k;                       // keep the slot for the global outputs
          ps[j] = piv;
        } else if (j < nl) {
          flag[j] = -1;
        }
        count += tot;
      }
      if (!valid) count = 0;
      {
        if (tid == 0) pub.count = count;
        cluster.sync();                                                // barrier A3
        if (warp == 0) {
          const int c = lane < CL ? cluster.map_shared_rank(&pub, lane)->count : 0;
          int incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
          }
          if (lane < CL) s_base[lane] = incl - c;
          if (lane == 31) s_base[CL] = incl;
        }
      }
      __syncthreads();
      total_sel = s_base[CL];
      if (out_writer) {
        const int my_base = s_base[rank];
        if (valid)
          for (int j = tid; j < nl; j += Tr::kThreads) {
            if (flag[j] < 0) continue;
            const int64_t slot = static_cast<int64_t>(unit) * M + my_base + flag[j];
            p.sel_ids[slot] = lo + j;
            p.pi[slot] = ps[j];
          }
        if (rank == 0) {
          for (int s = total_sel + tid; s < M; s += Tr::kThreads) {
            p.sel_ids[static_cast<int64_t>(unit) * M + s] = -1;
            p.pi[static_cast<int64_t>(unit) * M + s] = 0.f;
          }
          if (tid == 0) p.sel_count[unit] = total_sel;
        }
      }
      __syncthreads();
    }
  } else if (mode == kModeAttend) {
    total_sel = p.sel_count[unit];
    if (total_sel < 0 || total_sel > min(M, n)) {
      if (writer && rank == 0 && tid == 0) set_status(p.status, SANTA_DEV_BAD_SEL);
      total_sel = 0;
    }
  } else {                                 // dense
    total_sel = n;
  }

  // ================================================================ phase B: chunk table
  const int ctas = CL * NC;
  const int gidx = cidx * CL + rank;
  const int total_chunks = attending ? total_sel * cpt : 0;
  const int cps = (total_chunks + ctas - 1) / ctas;
  const int c_begin = min(gidx * cps, total_chunks);
  n_chunks = min(total_chunks - c_begin, cps);
  const float Mf = static_cast<float>(M);
  if (lmask && writer && rank == 0) {
    // the sampling outputs of the unit: S in ascending order with pi, padded
    for (int k = tid; k < M; k += Tr::kThreads) {
      int team = -1;
      float piv = 0.f;
      if (k < total_sel) {
        team = select_team(lmask, s_wi, lwpw, k);
        piv = team_recip(p.sampler, Mf, lps[team], lcnt[team]);
      }
      p.sel_ids[static_cast<int64_t>(unit) * M + k] = team;
      p.pi[static_cast<int64_t>(unit) * M + k] = piv;
    }
    if (tid == 0) p.sel_count[unit] = total_sel;
  }
  for (int ci = tid; ci < n_chunks; ci += Tr::kThreads) {
    const int c = c_begin + ci;
    const int slot = c / cpt, part = c - slot * cpt;
    int team = slot;
    float lw2 = 0.f;
    bool ok = true;
    if (mode == kModeDecode) {
      ListEntry e;
      if (local) {
        e.team = select_team(lmask, s_wi, lwpw, slot);
        e.lw2 = -log2f(team_recip(p.sampler, Mf, lps[e.team], lcnt[e.team]));
      } else {
        int owner = 0;
        while (owner + 1 < CL && s_base[owner + 1] <= slot) ++owner;
        e = cluster.map_shared_rank(list, owner)[slot - s_base[owner]];
      }
      team = e.team;
      lw2 = e.lw2;
    } else if (mode == kModeAttend) {
      const int64_t sidx = static_cast<int64_t>(unit) * M + slot;
      team = p.sel_ids[sidx];
      const float piv = p.pi[sidx];
      ok = team >= 0 && team < n && piv > 0.f && isfinite(piv);   // pi = 1 / weight
      if (!ok) set_status(p.status, SANTA_DEV_BAD_SEL);
      lw2 = ok ? -log2f(piv) : 0.f;
    }
    int page = -1;
    if (ok) {
      page = lpages ? lpages[team] : p.page_table[static_cast<int64_t>(b) * p.max_teams + team];
      if (page < 0 || page >= p.num_pages) {
        set_status(p.status, SANTA_DEV_BAD_PAGE);
        ok = false;
      }
    }
    const int vt =
        ok ? max(0, min(min(p.team_size, L - team * p.team_size) - part * kChunk, kChunk)) : 0;
    table[ci] = ChunkMeta{vt > 0 ? page : -1, vt, lw2, part};
  }
  }
  fence_proxy_async_smem();      // the ring held phase-A scratch; the copies overwrite it
  __syncthreads();
  // Split cluster barrier: this CTA has finished every read of its peers' shared memory
  // (published scores, drawn-team lists).  The matching wait comes after the streaming loop,
  // before partials are pushed into the peers' list regions.
  cluster_arrive_relaxed();

  // ================================================================ phase C: stream + compute
  auto issue = [&](int ci) { issue_meta(ci, table[ci]); };
  if (tid >= early_n && tid < min(S, n_chunks)) issue(tid);   // chunks < early_n are out

  constexpr int kMS = Tr::kMrgStride;
  float* mrg_acc = reinterpret_cast<float*>(smem);                   // [8][G][kMS]
  float* mrg_m = mrg_acc + Tr::kWarps * G * kMS;                     // [8][8]
  float* mrg_l = mrg_m + Tr::kWarps * kMaxGroup;                     // [8][8]
  float* part = reinterpret_cast<float*>(smem) + Tr::kPartialOff;    // acc [G][D], m [8], l [8]
  float* part_m = part + G * D;
  float* part_l = part_m + kMaxGroup;
  if constexpr (BF16 && W) {
    // ---- bf16 K/V, wide variant: warp group grp = warp >> 2 consumes chunks ci = grp,
    // grp + 2, ... (the stage count is even, so each group owns its stages and refills them
    // itself); warp (grp, tile) computes the scores of its 16-token tile and P.V over all
    // of d.  Same fragments, swizzle and P hi/lo split as the two-CTA variant below.
    constexpr int kKS = D / 16;                  // k-steps of the scores
    constexpr int kDT = D / 16;                  // 16-row d-tiles (all of d)
    constexpr int kBox = kChunk * 128;           // bytes of one 64-row box
    const int grp = warp >> 2, tile = warp & 3, gtid = tid & 127;
    const int h0 = 2 * (lane & 3);               // this lane's heads h0, h0 + 1
    const int r0 = 16 * tile + (lane >> 2);      // this lane's tokens r0, r0 + 8
    uint32_t qfrag[kKS][2];
    {
      const int n = lane >> 2, kq = 2 * (lane & 3);
      const uint16_t* qh = static_cast<const uint16_t*>(p.q) +
                           (static_cast<int64_t>(b) * p.num_q_heads + h * G + (n < G ? n : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk) {
        qfrag[kk][0] = n < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + kq) : 0u;
        qfrag[kk][1] = n < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + kq) : 0u;
      }
    }
    float o[kDT][4];
#pragma unroll
    for (int t = 0; t < kDT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float mr0 = kNegInf, mr1 = kNegInf, lr0 = 0.f, lr1 = 0.f;   // lr: this lane's share
    const int mi = lane >> 3, lr = lane & 7;
    bool timed_out = false;
    int ci = grp;
    for (; ci < n_chunks; ci += 2) {
      const int stage = ci % S;
      if (!mbar_wait(&bar[stage], (ci / S) & 1)) {
        set_status(p.status, SANTA_DEV_TIMEOUT);
        timed_out = true;
      }
      const int vt = table[ci].valid;
      unsigned char* kst = smem + static_cast<size_t>(stage) * Tr::kStageBytes;
      if (vt < kChunk) {                         // rows past the valid tokens: zero V (P = 0)
        unsigned char* vst = kst + Tr::kChunkBytes;
        for (int i = gtid; i < (kChunk - vt) * 8 * (D / 64); i += 128) {
          const int bx = i / ((kChunk - vt) * 8), rem = i - bx * (kChunk - vt) * 8;
          const int row = vt + rem / 8, piece = rem & 7;
          *reinterpret_cast<uint4*>(vst + bx * kBox + row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();                // before a later copy into this stage
        bar_red_or(1 + grp, 128, false);
      }
      const float lw2 = table[ci].lw2;
      const uint32_t kb = smem_u32(kst), vb = kb + Tr::kChunkBytes;
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk) {
        const int bx = (16 * kk) / 64, c0 = ((16 * kk) & 63) / 8;
        const int r = 16 * tile + lr + ((mi & 1) << 3), pc = c0 + (mi >> 1);
        uint32_t a[4];
        ldmatrix_x4(a, kb + bx * kBox + r * 128 + ((pc ^ (r & 7)) << 4));
        mma_bf16_16816((kk & 1) ? c2 : c, a, qfrag[kk][0], qfrag[kk][1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] += c2[j];
      const bool t0ok = r0 < vt, t1ok = r0 + 8 < vt, g0ok = h0 < G, g1ok = h0 + 1 < G;
      const float s0 = (t0ok && g0ok) ? fmaf(c[0], p.scale_log2, lw2) : kNegInf;
      const float s1 = (t0ok && g1ok) ? fmaf(c[1], p.scale_log2, lw2) : kNegInf;
      const float s2 = (t1ok && g0ok) ? fmaf(c[2], p.scale_log2, lw2) : kNegInf;
      const float s3 = (t1ok && g1ok) ? fmaf(c[3], p.scale_log2, lw2) : kNegInf;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(mr0, mx0), mn1 = fmaxf(mr1, mx1);
      const float al0 = mn0 == kNegInf ? 1.f : ex2_approx(mr0 - mn0);
      const float al1 = mn1 == kNegInf ? 1.f : ex2_approx(mr1 - mn1);
      const float p0 = mn0 == kNegInf ? 0.f : ex2_approx(s0 - mn0);
      const float p1 = mn1 == kNegInf ? 0.f : ex2_approx(s1 - mn1);
      const float p2 = mn0 == kNegInf ? 0.f : ex2_approx(s2 - mn0);
      const float p3 = mn1 == kNegInf ? 0.f : ex2_approx(s3 - mn1);
      lr0 = fmaf(lr0, al0, p0 + p2);
      lr1 = fmaf(lr1, al1, p1 + p3);
      mr0 = mn0;
      mr1 = mn1;
#pragma unroll
      for (int t = 0; t < kDT; ++t) {
        o[t][0] *= al0;
        o[t][1] *= al1;
        o[t][2] *= al0;
        o[t][3] *= al1;
      }
      const uint32_t hi01 = pack_bf16(p0, p1), hi23 = pack_bf16(p2, p3);
      const uint32_t lo01 = pack_bf16(p0 - bf16_lo_f(hi01), p1 - bf16_hi_f(hi01));
      const uint32_t lo23 = pack_bf16(p2 - bf16_lo_f(hi23), p3 - bf16_hi_f(hi23));
      const uint32_t bh0 = movmatrix_trans(hi01), bh1 = movmatrix_trans(hi23);
      const uint32_t bl0 = movmatrix_trans(lo01), bl1 = movmatrix_trans(lo23);
#pragma unroll
      for (int t = 0; t < kDT; ++t) {
        const int d0 = 16 * t;
        const int bx = d0 / 64, cd = (d0 & 63) / 8;
        const int r = 16 * tile + lr + ((mi >> 1) << 3), pc = cd + (mi & 1);
        uint32_t a[4];
        ldmatrix_x4_trans(a, vb + bx * kBox + r * 128 + ((pc ^ (r & 7)) << 4));
        mma_bf16_16816(o[t], a, bh0, bh1);
        mma_bf16_16816(o[t], a, bl0, bl1);
      }
      // the group's barrier releases the stage (and reports a timed-out wait)
      if (bar_red_or(1 + grp, 128, timed_out)) break;
      if (gtid == 0 && ci + S < n_chunks) issue(ci + S);
    }
    if (ci < n_chunks) {
      // a wait of this group gave up at chunk ci: wait (bounded) for the group's copies that
      // may still be in flight (ci, ci + 2, .. below ci + S), and flag the CTA
      if (gtid == 0)
        for (int cj = ci; cj < min(ci + S, n_chunks); cj += 2)
          (void)mbar_wait(&bar[cj % S], (cj / S) & 1);
      s_abort = 1;
    }
    __syncthreads();                             // both groups done with the ring
    if (s_abort) {
      mr0 = mr1 = kNegInf;
      lr0 = lr1 = 0.f;
#pragma unroll
      for (int t = 0; t < kDT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lr0 += __shfl_xor_sync(0xffffffffu, lr0, off);
      lr1 += __shfl_xor_sync(0xffffffffu, lr1, off);
    }
    if (attending) {
      // warp partials over all of d; every warp has its own (m, l) per head
#pragma unroll
      for (int t = 0; t < kDT; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = 16 * t + (lane >> 2) + ((j >> 1) << 3);
          const int g = h0 + (j & 1);
          if (g < G) mrg_acc[(warp * G + g) * kMS + d] = o[t][j];
        }
      if (lane < 4) {
        mrg_m[warp * kMaxGroup + h0] = mr0;
        mrg_m[warp * kMaxGroup + h0 + 1] = mr1;
        mrg_l[warp * kMaxGroup + h0] = lr0;
        mrg_l[warp * kMaxGroup + h0 + 1] = lr1;
      }
      __syncthreads();      // the combine's push forms each partial quad from mrg_acc
    }
  } else if constexpr (BF16) {
    // ---- bf16 K/V: tensor-core scores and P.V (mma.sync m16n8k16, fp32 accumulate)
    // Warp w owns 16-token tile (w & 3) of every chunk for the scores S^T = K Q^T (the G <= 8
    // heads are the N = 8 dimension) and half (w >> 2) of d for O^T += V^T P^T.  The chunk's
    // K and V arrive as 64-row x 128-byte boxes with 128-byte swizzle: 16-byte piece c of row
    // r sits at piece c ^ (r & 7), so every ldmatrix is conflict-free.  P goes to the second
    // product as bf16 hi + lo (two MMAs), keeping ~16 bits of it.
    constexpr int kKS = D / 16;                  // k-steps of the scores
    constexpr int kDT = D / 32;                  // 16-row d-tiles per half of d
    constexpr int kBox = kChunk * 128;           // bytes of one 64-row box
    const int tile = warp & 3, dh = warp >> 2;
    const int h0 = 2 * (lane & 3);               // this lane's heads h0, h0 + 1
    const int r0 = 16 * tile + (lane >> 2);      // this lane's tokens r0, r0 + 8
    uint32_t qfrag[kKS][2];
    {
      const int n = lane >> 2, kq = 2 * (lane & 3);
      const uint16_t* qh = static_cast<const uint16_t*>(p.q) +
                           (static_cast<int64_t>(b) * p.num_q_heads + h * G + (n < G ? n : 0)) * D;
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk) {
        qfrag[kk][0] = n < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + kq) : 0u;
        qfrag[kk][1] = n < G ? *reinterpret_cast<const uint32_t*>(qh + 16 * kk + 8 + kq) : 0u;
      }
    }
    float o[kDT][4];
#pragma unroll
    for (int t = 0; t < kDT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    // lr0, lr1: this lane's share of the running denominators (its own tokens), summed over
    // the lanes of a head once after the loop
    float mr0 = kNegInf, mr1 = kNegInf, lr0 = 0.f, lr1 = 0.f;
    const int mi = lane >> 3, lr = lane & 7;
    // One CTA barrier per chunk: each thread waits on the chunk's mbarrier itself; the
    // barrier at the end of the chunk releases its stage and reports a timed-out wait, after
    // which every thread leaves the loop together (the chunk's results are discarded).
    bool timed_out = false;
    int ci = 0;
    for (; ci < n_chunks; ++ci) {
      const int stage = ci % S;
      if (!mbar_wait(&bar[stage], (ci / S) & 1)) {
        set_status(p.status, SANTA_DEV_TIMEOUT);
        timed_out = true;
      }
      const int vt = table[ci].valid;
      unsigned char* kst = smem + static_cast<size_t>(stage) * Tr::kStageBytes;
      if (vt < kChunk) {                         // rows past the valid tokens: zero V (P = 0)
        unsigned char* vst = kst + Tr::kChunkBytes;
        for (int i = tid; i < (kChunk - vt) * 8 * (D / 64); i += Tr::kThreads) {
          const int bx = i / ((kChunk - vt) * 8), rem = i - bx * (kChunk - vt) * 8;
          const int row = vt + rem / 8, piece = rem & 7;
          *reinterpret_cast<uint4*>(vst + bx * kBox + row * 128 + piece * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();  // before a later copy into this stage
        __syncthreads();
      }
      const float lw2 = table[ci].lw2;
      const uint32_t kb = smem_u32(kst), vb = kb + Tr::kChunkBytes;
      // scores of tokens r0, r0 + 8 for heads h0, h0 + 1 (even and odd k-steps in two
      // accumulators: two dependent MMA chains of half the length)
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < kKS; ++kk) {
        const int bx = (16 * kk) / 64, c0 = ((16 * kk) & 63) / 8;
        const int r = 16 * tile + lr + ((mi & 1) << 3), pc = c0 + (mi >> 1);
        uint32_t a[4];
        ldmatrix_x4(a, kb + bx * kBox + r * 128 + ((pc ^ (r & 7)) << 4));
        mma_bf16_16816((kk & 1) ? c2 : c, a, qfrag[kk][0], qfrag[kk][1]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) c[j] += c2[j];
      const bool t0ok = r0 < vt, t1ok = r0 + 8 < vt, g0ok = h0 < G, g1ok = h0 + 1 < G;
      const float s0 = (t0ok && g0ok) ? fmaf(c[0], p.scale_log2, lw2) : kNegInf;
      const float s1 = (t0ok && g1ok) ? fmaf(c[1], p.scale_log2, lw2) : kNegInf;
      const float s2 = (t1ok && g0ok) ? fmaf(c[2], p.scale_log2, lw2) : kNegInf;
      const float s3 = (t1ok && g1ok) ? fmaf(c[3], p.scale_log2, lw2) : kNegInf;
      // online softmax per head over the tile's 16 tokens (lanes sharing lane & 3)
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(mr0, mx0), mn1 = fmaxf(mr1, mx1);
      const float al0 = mn0 == kNegInf ? 1.f : ex2_approx(mr0 - mn0);
      const float al1 = mn1 == kNegInf ? 1.f : ex2_approx(mr1 - mn1);
      const float p0 = mn0 == kNegInf ? 0.f : ex2_approx(s0 - mn0);
      const float p1 = mn1 == kNegInf ? 0.f : ex2_approx(s1 - mn1);
      const float p2 = mn0 == kNegInf ? 0.f : ex2_approx(s2 - mn0);
      const float p3 = mn1 == kNegInf ? 0.f : ex2_approx(s3 - mn1);
      lr0 = fmaf(lr0, al0, p0 + p2);
      lr1 = fmaf(lr1, al1, p1 + p3);
      mr0 = mn0;
      mr1 = mn1;
#pragma unroll
      for (int t = 0; t < kDT; ++t) {
        o[t][0] *= al0;
        o[t][1] *= al1;
        o[t][2] *= al0;
        o[t][3] *= al1;
      }
      // P^T as B fragments: bf16 hi + lo, transposed 8x8 blocks
      const uint32_t hi01 = pack_bf16(p0, p1), hi23 = pack_bf16(p2, p3);
      const uint32_t lo01 = pack_bf16(p0 - bf16_lo_f(hi01), p1 - bf16_hi_f(hi01));
      const uint32_t lo23 = pack_bf16(p2 - bf16_lo_f(hi23), p3 - bf16_hi_f(hi23));
      const uint32_t bh0 = movmatrix_trans(hi01), bh1 = movmatrix_trans(hi23);
      const uint32_t bl0 = movmatrix_trans(lo01), bl1 = movmatrix_trans(lo23);
#pragma unroll
      for (int t = 0; t < kDT; ++t) {
        const int d0 = dh * (D / 2) + 16 * t;
        const int bx = d0 / 64, cd = (d0 & 63) / 8;
        const int r = 16 * tile + lr + ((mi >> 1) << 3), pc = cd + (mi & 1);
        uint32_t a[4];
        ldmatrix_x4_trans(a, vb + bx * kBox + r * 128 + ((pc ^ (r & 7)) << 4));
        mma_bf16_16816(o[t], a, bh0, bh1);
        mma_bf16_16816(o[t], a, bl0, bl1);
      }
      if (__syncthreads_or(timed_out)) break;
      if (tid == 0 && ci + S < n_chunks) issue(ci + S);
    }
    if (ci < n_chunks) {
      // a wait at chunk ci gave up: wait (bounded) for the copies that may still be in
      // flight (chunks ci .. ci + S - 1), and contribute nothing
      if (tid == 0)
        for (int cj = ci; cj < min(ci + S, n_chunks); ++cj)
          (void)mbar_wait(&bar[cj % S], (cj / S) & 1);
      mr0 = mr1 = kNegInf;
      lr0 = lr1 = 0.f;
#pragma unroll
      for (int t = 0; t < kDT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
      __syncthreads();
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lr0 += __shfl_xor_sync(0xffffffffu, lr0, off);
      lr1 += __shfl_xor_sync(0xffffffffu, lr1, off);
    }
    if (attending) {
      // warp partials: O^T elements (d = d0 + lane/4 (+8), head h0 / h0 + 1), (m, l) per head
#pragma unroll
      for (int t = 0; t < kDT; ++t)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int d = dh * (D / 2) + 16 * t + (lane >> 2) + ((j >> 1) << 3);
          const int g = h0 + (j & 1);
          if (g < G) mrg_acc[(warp * G + g) * kMS + d] = o[t][j];
        }
      if (lane < 4) {
        mrg_m[warp * kMaxGroup + h0] = mr0;
        mrg_m[warp * kMaxGroup + h0 + 1] = mr1;
        mrg_l[warp * kMaxGroup + h0] = lr0;
        mrg_l[warp * kMaxGroup + h0 + 1] = lr1;
      }
      __syncthreads();      // the combine's push forms each partial quad from mrg_acc
    }
  } else {
    // ---- fp32 K/V: CUDA-core scores and P.V
    // q of the group in registers, in the score layout
    float qr[G][Tr::kEplS];
    {
      const unsigned char* qbp = static_cast<const unsigned char*>(p.q) +
                                 (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D * Tr::kEsize;
#pragma unroll
      for (int g = 0; g < G; ++g) load_score_row<BF16, D>(qbp + g * D * Tr::kEsize, lane16, qr[g]);
    }
    const int hh = (lane >> 1) & 7;
    float m_run = kNegInf, l_run = 0.f;
    float acc[G][Tr::kEplV];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < Tr::kEplV; ++e) acc[g][e] = 0.f;
    float* pw = prow + warp * 64;
    float* aw = arow + warp * kMaxGroup;
    int consumed = 0;

    for (int ci = 0; ci < n_chunks; ++ci) {
      const int stage = ci % S;
      if (!mbar_wait(&bar[stage], (ci / S) & 1)) {
        set_status(p.status, SANTA_DEV_TIMEOUT);
        s_abort = 1;
      }
      __syncthreads();
      if (s_abort) break;
      consumed = ci + 1;
      const int vt = table[ci].valid;
      const float lw2 = table[ci].lw2;
      const unsigned char* ks = smem + static_cast<size_t>(stage) * Tr::kStageBytes;
      const unsigned char* vs = ks + Tr::kChunkBytes;

      float sc[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = warp * 8 + 2 * k + (lane >> 4);
        float x[Tr::kEplS];
        load_score_row<BF16, D>(ks + static_cast<size_t>(t) * D * Tr::kEsize, lane16, x);
        float part[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          part[g] = 0.f;
          if (g < G) {
#pragma unroll
            for (int e = 0; e < Tr::kEplS; ++e) part[g] = fmaf(qr[g][e], x[e], part[g]);
          }
        }
        const float sum = reduce_scatter8(part, lane);
        sc[k] = (t < vt && hh < G) ? fmaf(sum, p.scale_log2, lw2) : kNegInf;
      }
      float cm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
      const float m_new = fmaxf(m_run, cm);
      const float alpha = m_new == kNegInf ? 1.f : exp2f(m_run - m_new);
      float pv[4], psum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        pv[k] = m_new == kNegInf ? 0.f : exp2f(sc[k] - m_new);
        psum += pv[k];
      }
      psum += __shfl_xor_sync(0xffffffffu, psum, 16);
      l_run = fmaf(l_run, alpha, psum);
      m_run = m_new;
      if (!(lane & 1)) {
#pragma unroll
        for (int k = 0; k < 4; ++k) pw[(2 * k + (lane >> 4)) * 8 + hh] = pv[k];
      }
      if (!(lane & 0x11)) aw[hh] = alpha;
      __syncwarp();
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float a = aw[g];
#pragma unroll
        for (int e = 0; e < Tr::kEplV; ++e) acc[g][e] *= a;
      }
      const int nt = min(8, vt - warp * 8);
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        if (tt < nt) {
          float v[Tr::kEplV];
          load_value_row<BF16, D>(vs + static_cast<size_t>(warp * 8 + tt) * D * Tr::kEsize, lane,
                                  v);
          const float4 pa = *reinterpret_cast<const float4*>(pw + tt * 8);
          const float4 pb = *reinterpret_cast<const float4*>(pw + tt * 8 + 4);
          const float pg[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < Tr::kEplV; ++e) acc[g][e] = fmaf(pg[g], v[e], acc[g][e]);
        }
      }
      __syncthreads();
      if (tid == 0 && ci + S < n_chunks) issue(ci + S);
    }
    if (s_abort) {
      // wait (bounded) for the copies still in flight; contribute nothing
      if (tid == 0)
        for (int ci = consumed; ci < min(consumed + S, n_chunks); ++ci)
          (void)mbar_wait(&bar[ci % S], (ci / S) & 1);
      m_run = kNegInf;
      l_run = 0.f;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < Tr::kEplV; ++e) acc[g][e] = 0.f;
      __syncthreads();
    }

    if (attending) {
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < Tr::kEplV; ++e)
          mrg_acc[(warp * G + g) * kMS + lane * Tr::kEplV + e] = acc[g][e];
      if (!(lane & 0x11)) {
        mrg_m[warp * kMaxGroup + hh] = m_run;
        mrg_l[warp * kMaxGroup + hh] = l_run;
      }
      __syncthreads();
      if (tid < G) {
        float mx = kNegInf;
#pragma unroll
        for (int w = 0; w < Tr::kWarps; ++w) mx = fmaxf(mx, mrg_m[w * kMaxGroup + tid]);
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < Tr::kWarps; ++w) {
          const float mw = mrg_m[w * kMaxGroup + tid];
          l = fmaf(mw == kNegInf ? 0.f : exp2f(mw - mx), mrg_l[w * kMaxGroup + tid], l);
        }
        part_m[tid] = mx;
        part_l[tid] = l;
      }
      for (int i = tid; i < G * D; i += Tr::kThreads) {
        const int g = i / D, k = i - g * D;
        float mx = kNegInf;
#pragma unroll
        for (int w = 0; w < Tr::kWarps; ++w) mx = fmaxf(mx, mrg_m[w * kMaxGroup + g]);
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < Tr::kWarps; ++w) {
          const float mw = mrg_m[w * kMaxGroup + g];
          a = fmaf(mw == kNegInf ? 0.f : exp2f(mw - mx), mrg_acc[(w * G + g) * kMS + k], a);
        }
        part[i] = a;
      }
    }
  }
  // ---- combine: each CTA pushes the quads of its partial that rank r owns, with its (m, l),
  // into rank r's list region by st.async stores whose bytes complete on rank r's combine
  // mbarrier; each CTA waits for its own slice only (no cluster barrier), then merges its
  // slice of the G*D outputs from local shared memory, in rank order.
  constexpr int kQuads = G * D / 4;
  const int qper = (kQuads + CL - 1) / CL;
  float4* comb_q = reinterpret_cast<float4*>(list);                 // [CL][qper] partial quads
  float* comb_ml = reinterpret_cast<float*>(comb_q + CL * qper);    // [CL][G][2] (m, l)
  if constexpr (!BF16) __syncthreads();                             // part complete
  cluster_wait();                                                   // peers' reads are done
  if (attending) {
    for (int qi = tid; qi < kQuads; qi += Tr::kThreads) {
      const int r = qi / qper, k = qi - r * qper;
      float4 v;
      if constexpr (BF16) {
        // the CTA partial quad straight from the warp partials, weighted exp2(m_w - m) over
        // every warp (wide) or the four token tiles of this half of d (both halves share m
        // and l, kept by warps 0-3), each thread forming its head's weights itself
        const int g = (4 * qi) / D, k0 = 4 * qi - g * D;
        constexpr int kW = W ? Tr::kWarps : 4;
        const int w0 = W ? 0 : (k0 / (D / 2)) * 4;
        float mw[kW], mx = kNegInf;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
          mw[w] = mrg_m[w * kMaxGroup + g];
          mx = fmaxf(mx, mw[w]);
        }
        v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kW; ++w) {
          const float a = mw[w] == kNegInf ? 0.f : ex2_approx(mw[w] - mx);
          const float4 x = *reinterpret_cast<const float4*>(mrg_acc + ((w0 + w) * G + g) * kMS + k0);
          v.x = fmaf(a, x.x, v.x);
          v.y = fmaf(a, x.y, v.y);
          v.z = fmaf(a, x.z, v.z);
          v.w = fmaf(a, x.w, v.w);
        }
      } else {
        v = reinterpret_cast<const float4*>(part)[qi];
      }
      st_async_v4(cluster_addr(smem_u32(comb_q + rank * qper + k), r), v,
                  cluster_addr(smem_u32(&bar[S + 2]), r));
    }
    if (tid < CL * G) {
      const int r = tid / G, g = tid - r * G;
      float pm, pl;
      if constexpr (BF16) {
        // the CTA's (m, l) of head g from the warps' (the same weights as above)
        constexpr int kW = W ? Tr::kWarps : 4;
        pm = kNegInf;
        pl = 0.f;
#pragma unroll
        for (int w = 0; w < kW; ++w) pm = fmaxf(pm, mrg_m[w * kMaxGroup + g]);
#pragma unroll
        for (int w = 0; w < kW; ++w) {
          const float mw = mrg_m[w * kMaxGroup + g];
          pl = fmaf(mw == kNegInf ? 0.f : ex2_approx(mw - pm), mrg_l[w * kMaxGroup + g], pl);
        }
      } else {
        pm = part_m[g];
        pl = part_l[g];
      }
      st_async_v2(cluster_addr(smem_u32(comb_ml + (rank * G + g) * 2), r), pm, pl,
                  cluster_addr(smem_u32(&bar[S + 2]), r));
    }
    // this CTA's slice of every peer's partial (and their (m, l)) has arrived: the bytes
    // counted on its mbarrier, no cluster-wide barrier
    if (tid == 0) {
      const int nq_own = min(min(rank * qper, kQuads) + qper, kQuads) - min(rank * qper, kQuads);
      mbar_arrive_expect_tx(&bar[S + 2], static_cast<uint32_t>(CL * (nq_own * 16 + G * 8)));
    }
    if (!mbar_wait(&bar[S + 2], 0)) set_status(p.status, SANTA_DEV_TIMEOUT);
  }
  float* out_unit = p.out + (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D;
  if (attending && NC == 1) {
    // this CTA's slice of the output: each thread forms the CL ranks' weights of its quad's
    // head itself and merges in rank order (no barrier)
    const int q0 = min(rank * qper, kQuads);
    const int nq = min(q0 + qper, kQuads) - q0;
    for (int k = tid; k < nq; k += Tr::kThreads) {
      const int qi = q0 + k;
      const int g = (qi * 4) / D;
      float mx = kNegInf;
#pragma unroll 4
      for (int r = 0; r < CL; ++r) mx = fmaxf(mx, comb_ml[(r * G + g) * 2]);
      float l = 0.f;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int r = 0; r < CL; ++r) {
        const float mr = comb_ml[(r * G + g) * 2];
        const float w = mr == kNegInf ? 0.f : ex2_approx(mr - mx);
        l = fmaf(w, comb_ml[(r * G + g) * 2 + 1], l);
        const float4 v = comb_q[r * qper + k];
        a.x = fmaf(w, v.x, a.x);
        a.y = fmaf(w, v.y, a.y);
        a.z = fmaf(w, v.z, a.z);
        a.w = fmaf(w, v.w, a.w);
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      reinterpret_cast<float4*>(out_unit)[qi] =
          make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
    }
    return;
  }
  if (attending) {
    // weights of the CL partials per head: warp g, lane r
    if (warp < G) {
      const float mr = lane < CL ? comb_ml[(lane * G + warp) * 2] : kNegInf;
      const float mx = warp_max(mr);
      const float w = mr == kNegInf ? 0.f : exp2f(mr - mx);
      if (lane < CL) s_pm[lane * G + warp] = w;
      const float l = warp_sum(lane < CL ? w * comb_ml[(lane * G + warp) * 2 + 1] : 0.f);
      if (lane == 0) {
        s_gm[warp] = mx;
        s_gz[warp] = l;
      }
    }
    __syncthreads();
    const int q0 = min(rank * qper, kQuads);
    const int nq = min(q0 + qper, kQuads) - q0;
    for (int k = tid; k < nq; k += Tr::kThreads) {
      const int qi = q0 + k;
      const int g = (qi * 4) / D;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int r = 0; r < CL; ++r) {
        const float w = s_pm[r * G + g];
        const float4 v = comb_q[r * qper + k];
        a.x = fmaf(w, v.x, a.x);
        a.y = fmaf(w, v.y, a.y);
        a.z = fmaf(w, v.z, a.z);
        a.w = fmaf(w, v.w, a.w);
      }
      if (NC == 1) {
        const float l = s_gz[g];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        reinterpret_cast<float4*>(out_unit)[qi] =
            make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
      } else {
        reinterpret_cast<float4*>(p.part_acc +
                                  (static_cast<int64_t>(unit) * NC + cidx) * G * D)[qi] = a;
      }
    }
    if (NC > 1 && rank == 0 && tid < G) {
      p.part_ml[((static_cast<int64_t>(unit) * NC + cidx) * G + tid) * 2] = s_gm[tid];
      p.part_ml[((static_cast<int64_t>(unit) * NC + cidx) * G + tid) * 2 + 1] = s_gz[tid];
    }
  }
  if (!attending || NC == 1) return;

  // ---- several clusters per unit: the last CTA to arrive merges the cluster partials (its
  // arrival ticket releases this CTA's partial writes and acquires everyone's)
  __syncthreads();
  if (tid == 0)
    s_last = atomic_add_acq_rel_gpu(&p.counters[unit], 1u) == static_cast<unsigned>(CL * NC - 1);
  __syncthreads();
  if (!s_last) return;
  // every load of this CTA at once (one round trip): thread t's quad of every cluster partial
  // (G * d / 4 <= 256 quads) and the clusters' (m, l) of its head; each thread then forms
  // its head's weights itself and merges in cluster order (no barrier)
  static_assert(G * D / 4 <= 256, "one output quad per thread");
  const int qi = tid, gq = (qi * 4) / D;
  if (qi < kQuads) {
    float4 v[kMaxClustersPerUnit];
    float2 ml[kMaxClustersPerUnit];
    const float4* src =
        reinterpret_cast<const float4*>(p.part_acc + static_cast<int64_t>(unit) * NC * G * D) + qi;
    const float2* mls = reinterpret_cast<const float2*>(p.part_ml) +
                        static_cast<int64_t>(unit) * NC * G + gq;
#pragma unroll
    for (int c = 0; c < kMaxClustersPerUnit; ++c) {
      v[c] = c < NC ? __ldcg(src + c * (G * D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
      ml[c] = c < NC ? __ldcg(mls + c * G) : make_float2(kNegInf, 0.f);
    }
    float mx = kNegInf;
#pragma unroll
    for (int c = 0; c < kMaxClustersPerUnit; ++c) mx = fmaxf(mx, ml[c].x);
    float l = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < kMaxClustersPerUnit; ++c) {
      const float w = ml[c].x == kNegInf ? 0.f : ex2_approx(ml[c].x - mx);
      l = fmaf(w, ml[c].y, l);
      a.x = fmaf(w, v[c].x, a.x);
      a.y = fmaf(w, v[c].y, a.y);
      a.z = fmaf(w, v[c].z, a.z);
      a.w = fmaf(w, v[c].w, a.w);
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<float4*>(out_unit)[qi] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  }
  if (tid == 0) p.counters[unit] = 0u;
}

// ---------------------------------------------------------------- host-side launch helpers

template <bool BF16, int D, int G, bool W, int FAST = 0>
std::atomic<unsigned long long>& decode_smem_flag() {
  static std::atomic<unsigned long long> flag{0};
  return flag;
}

template <bool BF16, int D, int G, bool W, int FAST = 0>
cudaError_t decode_prepare_t() {
  using Tr = DecodeTraits<BF16, D, G, W>;
  auto* kern = decode_kernel<BF16, D, G, W, FAST>;
  static std::atomic<unsigned long long> cluster_flag{0};
  cudaError_t e = ensure_dynamic_smem(kern, Tr::kSmem, decode_smem_flag<BF16, D, G, W, FAST>());
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(cluster_flag.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cluster_flag.fetch_or(bit);
  }
  return cudaSuccess;
}

// How many clusters of `cluster` CTAs can be co-resident (0 if none / on error).
template <bool BF16, int D, int G, bool W, int FAST = 0>
int decode_max_clusters_t(int cluster) {
  using Tr = DecodeTraits<BF16, D, G, W>;
  if (decode_prepare_t<BF16, D, G, W, FAST>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(Tr::kThreads);
  cfg.dynamicSmemBytes = Tr::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<BF16, D, G, W, FAST>, &cfg) != cudaSuccess)
    return 0;
  return n;
}

template <bool BF16, int D, int G, bool W, int FAST = 0>
int decode_resident_t() {
  using Tr = DecodeTraits<BF16, D, G, W>;
  if (decode_prepare_t<BF16, D, G, W, FAST>() != cudaSuccess) return 0;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, decode_kernel<BF16, D, G, W, FAST>,
                                                    Tr::kThreads, Tr::kSmem) != cudaSuccess)
    return 0;
  return blocks;
}

template <bool BF16, int D, int G, bool W, int FAST = 0>
cudaError_t decode_launch_t(const DecodeParams& p, dim3 grid, int cluster, cudaStream_t stream) {
  using Tr = DecodeTraits<BF16, D, G, W>;
  cudaError_t e = decode_prepare_t<BF16, D, G, W, FAST>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Tr::kThreads);
  cfg.dynamicSmemBytes = Tr::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start while the previous kernel of the stream finishes (the kernel waits on it
  // before touching global memory)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, decode_kernel<BF16, D, G, W, FAST>, p);
}

// Dispatch on the group size (1..8) for one (dtype, head_dim).
#define SANTA_DISPATCH_G(G_VAR, CALL)        \
  switch (G_VAR) {                           \
    case 1: { constexpr int GG = 1; CALL; }  \
    case 2: { constexpr int GG = 2; CALL; }  \
    case 3: { constexpr int GG = 3; CALL; }  \
    case 4: { constexpr int GG = 4; CALL; }  \
    case 5: { constexpr int GG = 5; CALL; }  \
    case 6: { constexpr int GG = 6; CALL; }  \
    case 7: { constexpr int GG = 7; CALL; }  \
    default: { constexpr int GG = 8; CALL; } \
  }

}  // namespace santa
