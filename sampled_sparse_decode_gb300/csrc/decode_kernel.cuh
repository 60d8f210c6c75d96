// decode_kernel.cuh — one SANTA++ decode step per (sequence, KV head) unit in one kernel:
// representative scoring, GQA-mixed team softmax, Philox inverse-CDF sampling, the
// deduplicated sampled set with its inclusion probabilities, exact attention inside the
// sampled teams reweighted by 1/pi, and the Horvitz-Thompson combine.
//
// Method ("SANTA++: Sampling Attention through Representative Keys", abstract; explainer
// "SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%", section 三 steps 1-5, 3.1):
//   s_{g,i} = q_g . rep_i / sqrt(d);  p_{g,i} = softmax_i(s_{g,.});  p_i = (1/G) sum_g p_{g,i}
//   draw r: u = (word 0 of Philox4x32-10((r, h, b, 0), (lo32, hi32 of seed)) + 1/2) 2^-32,
//           team = smallest i with u*Z < C_i  (C the fp64 running sum of p, Z = C_{n-1})
//   S = distinct draws, pi_i = 1 - (1 - p_i)^M
//   out_g = sum_{i in S} (1/pi_i) sum_{j in i} e^{s_j} v_j / sum_{i in S} (1/pi_i) sum_{j in i} e^{s_j}
//
// GB300 mapping.  A unit is served by NC thread-block clusters of CL CTAs (NC = 1 unless a
// unit's work needs more CTAs than one cluster holds).  Inside a cluster:
//   phase A  CTA r scores the representatives of teams [r*per, (r+1)*per) (one warp per team,
//            coalesced 512-byte rows), publishes its per-head (max, sum) in shared memory;
//            after a cluster barrier every CTA reads all peers' values with one parallel
//            distributed-shared-memory (DSMEM) read and forms the same global softmax; the
//            fp64 CDF slices' totals are exchanged the same way; each CTA resolves the draws
//            whose u*Z falls in its slice by binary search, numbers its drawn teams and
//            publishes them (team, -log2 pi) as a list; a third barrier exchanges the counts.
//            Every reduction has a fixed order, so all CTAs (and all clusters of a unit)
//            compute bit-identical sampled sets.
//   phase B  the unit's sampled teams form a list of 64-token chunks; CTA g of the unit owns
//            chunks [g*cps, (g+1)*cps), cps = ceil(chunks / CTAs) — balanced for any S; each
//            chunk's team comes from its owner's list over DSMEM.
//   phase C  thread 0 streams each chunk's K and V rows (contiguous in the paged pool) into
//            a ring of shared-memory stages with two bulk copies (cp.async.bulk, the
//            non-tensor TMA form) on an mbarrier; warp w scores tokens 8w..8w+7 with q in
//            registers (16 lanes per token, 8-shuffle reduce-scatter to one head per lane),
//            keeps a base-2 online softmax with -log2 pi folded into the scores, and
//            accumulates P.V with lane l owning d/32 elements of every head.
//   phase D  the 8 warps merge in shared memory; after a cluster barrier each CTA combines
//            its slice of the outputs across the cluster's CTAs over DSMEM.  With NC > 1 the
//            cluster partials go to global scratch and the last CTA of the unit (an atomic
//            ticket, no waiting) merges them in cluster order.
// No wait is unbounded: mbarrier waits give up after 2 s (status bit, return through the
// remaining barriers); every CTA executes every cluster barrier on every path.
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

template <bool BF16, int D, int G>
struct DecodeTraits {
  static constexpr int kThreads = 256;
  static constexpr int kWarps = 8;
  static constexpr int kEsize = BF16 ? 2 : 4;
  static constexpr int kChunkBytes = kChunk * D * kEsize;
  static constexpr int kStageBytes = 2 * kChunkBytes;
  static constexpr int kStages = kStageBytes >= 65536 ? 2 : (kStageBytes >= 32768 ? 3 : 4);
  static constexpr int kEplS = D / 16;
  static constexpr int kEplV = D / 32;
  static constexpr int kRing = kStages * kStageBytes;
  // phase A scratch inside the ring: cdf (uint64) [tpc], es [8][tpc], ps [tpc], flag [tpc],
  // then a buffer of representative rows (fp32 [rows][D]) for as many rows as fit
  static constexpr size_t sample_scratch(int tpc) {
    return sizeof(unsigned long long) * tpc + sizeof(float) * kMaxGroup * tpc +
           sizeof(float) * tpc + sizeof(int) * tpc;
  }
  static constexpr int rep_rows(int tpc) {
    return static_cast<int>((static_cast<size_t>(kRing) - sample_scratch(tpc)) / (D * 4));
  }
  static_assert(rep_rows(kMaxTeamsPerCta) >= 32, "representative buffer must hold 32 rows");
  // phase D: warp merge buffer [8][G][D] + m, l [8][8], then the CTA partial [G][D] + m, l
  static constexpr int kMergeFloats = kWarps * G * D + 2 * kWarps * kMaxGroup;
  static constexpr int kPartialOff = kMergeFloats;                    // in floats
  static constexpr int kPartialFloats = G * D + 2 * kMaxGroup;
  static constexpr int kCombOff = kPartialOff + kPartialFloats;         // in floats, 16B aligned
  static constexpr int kCombFloats = 4 * kThreads;                      // [CL][qb] float4
  static_assert((kMergeFloats + kPartialFloats + kCombFloats) * 4 <= kRing,
                "merge buffers must fit");
  // dynamic shared memory: ring | list | chunk table | p rows | alpha | bars
  static constexpr size_t kListOff = static_cast<size_t>(kRing);
  static constexpr size_t kTableOff = kListOff + sizeof(ListEntry) * kMaxTeamsPerCta;
  static constexpr size_t kPOff = kTableOff + sizeof(ChunkMeta) * kMaxChunksPerSplit;
  static constexpr size_t kAOff = kPOff + sizeof(float) * kWarps * 64;
  static constexpr size_t kBarOff = kAOff + sizeof(float) * kWarps * kMaxGroup;
  static constexpr size_t kSmem = kBarOff + sizeof(uint64_t) * kStages;
  static constexpr int kMinBlocks = kSmem <= 112 * 1024 ? 2 : 1;
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

// ---------------------------------------------------------------- the kernel

template <bool BF16, int D, int G>
__global__ void __launch_bounds__(256, (DecodeTraits<BF16, D, G>::kMinBlocks))
    decode_kernel(const DecodeParams p) {
  using Tr = DecodeTraits<BF16, D, G>;
  constexpr int S = Tr::kStages;
  constexpr float kNegInf = -INFINITY;
  cgx::cluster_group cluster = cgx::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int CL = static_cast<int>(cluster.num_blocks());
  const int NC = p.clusters_per_unit;
  const int cidx = blockIdx.x / CL;
  const int h = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.num_kv_heads + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, lane16 = lane & 15;
  const int M = p.num_draws;
  const int mode = p.mode;
  const bool sampling = mode == kModeDecode || mode == kModeSample;
  const bool attending = mode != kModeSample;
  const bool writer = cidx == 0;          // the cluster that writes the sampling outputs

  extern __shared__ __align__(128) unsigned char smem[];
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
  __shared__ __align__(8) uint64_t s_rbar;

  // ---- per-unit lengths
  const int L = p.seq_lens[b];
  const bool len_ok = L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_teams) *
                                                             p.team_size;
  const int n = len_ok ? (L + p.team_size - 1) / p.team_size : 0;
  const int cpt = p.team_size / kChunk;
  if (!len_ok && writer && rank == 0 && tid == 0) set_status(p.status, SANTA_DEV_BAD_SEQLEN);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    mbar_init(&s_rbar, 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  // ================================================================ phase A: sampling
  int total_sel = 0;                      // |S| of the unit
  if (sampling) {
    const int tpc = p.teams_per_cta;
    unsigned long long* cdf = reinterpret_cast<unsigned long long*>(smem);   // [tpc]
    float* es = reinterpret_cast<float*>(cdf + tpc);                 // [8][tpc] scores, exps
    float* ps = es + kMaxGroup * tpc;                                // [tpc] team probability
    int* flag = reinterpret_cast<int*>(ps + tpc);                    // [tpc] drawn / slot
    float* rows = reinterpret_cast<float*>(smem + Tr::sample_scratch(tpc));  // rep rows
    const int max_rows = Tr::rep_rows(tpc);
    const int per = (n + CL - 1) / CL;
    const int lo = min(rank * per, n);
    const int nl = min(lo + per, n) - lo;
    constexpr int E = D / 32;

    // q of the group in registers, lane l holding d-elements [l*E, (l+1)*E)
    float qv[G][E];
    {
      const int64_t qbase = (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D + lane * E;
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < E; ++e)
          qv[g][e] = BF16 ? bf16_to_f32(static_cast<const uint16_t*>(p.q)[qbase + g * D + e])
                          : static_cast<const float*>(p.q)[qbase + g * D + e];
    }
    for (int j = tid; j < nl; j += Tr::kThreads) flag[j] = 0;

    // scores, in batches of representative rows staged by bulk copies (one round trip each)
    uint32_t rphase = 0;
    for (int j0 = 0; j0 < nl; j0 += max_rows) {
      const int cnt = min(max_rows, nl - j0);
      if (tid == 0) mbar_arrive_expect_tx(&s_rbar, static_cast<uint32_t>(cnt) * D * 4);
      __syncthreads();
      for (int j = tid; j < cnt; j += Tr::kThreads) {
        int64_t page = p.page_table[static_cast<int64_t>(b) * p.max_teams + lo + j0 + j];
        const bool ok = page >= 0 && page < p.num_pages;
        if (!ok) set_status(p.status, SANTA_DEV_BAD_PAGE);
        flag[j0 + j] = ok ? 0 : -2;                  // -2: unusable team
        bulk_g2s(rows + static_cast<size_t>(j) * D, p.reps + ((ok ? page : 0) * p.num_kv_heads + h) * D,
                 D * 4, &s_rbar);
      }
      if (!mbar_wait(&s_rbar, rphase)) set_status(p.status, SANTA_DEV_TIMEOUT);
      rphase ^= 1u;
      for (int j = warp; j < cnt; j += Tr::kWarps) {
        const float* rr = rows + static_cast<size_t>(j) * D + lane * E;
        float rv[E];
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4*>(rr);
          rv[0] = v.x; rv[1] = v.y; rv[2] = v.z; rv[3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(rr);
          rv[0] = v.x; rv[1] = v.y;
        }
        const bool ok = flag[j0 + j] == 0;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float part = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) part = fmaf(qv[g][e], rv[e], part);
          part = warp_sum(part);
          if (lane == 0) es[g * tpc + j0 + j] = ok ? part * p.scale : kNegInf;
        }
      }
      __syncthreads();                                  // rows reusable, scores visible
    }
    // local per-head (max, sum of exp) over this CTA's teams
    if (warp < G) {
      float m = kNegInf;
      for (int j = lane; j < nl; j += 32) m = fmaxf(m, es[warp * tpc + j]);
      m = warp_max(m);
      float z = 0.f;
      if (m != kNegInf)
        for (int j = lane; j < nl; j += 32) {
          const float sc = es[warp * tpc + j];
          z += sc == kNegInf ? 0.f : expf(sc - m);
        }
      z = warp_sum(z);
      if (lane == 0) {
        pub.m[warp] = m;
        pub.z[warp] = z;
      }
    }
    cluster.sync();                                                  // barrier A1
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
    __syncthreads();
    // team probabilities p_j = (1/G) sum_g exp(s_gj - m_g) / z_g, and their 62-bit
    // fixed-point values round(p * 2^62) (ties away from zero)
    unsigned long long carry = 0;
    for (int base = 0; base < nl; base += Tr::kThreads) {
      const int j = base + tid;
      unsigned long long P = 0;
      if (j < nl) {
        float acc = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float sc = es[g * tpc + j];
          acc += (sc == kNegInf || !(s_gz[g] > 0.f)) ? 0.f : expf(sc - s_gm[g]) / s_gz[g];
        }
        const float pj = acc / static_cast<float>(G);
        ps[j] = pj;
        if (p.team_probs && writer)
          p.team_probs[static_cast<int64_t>(unit) * p.max_teams + lo + j] = pj;
        if (pj > 0.f) {
          const float x = pj * 0x1p62f;                              // exact scaling
          const unsigned long long fl = __float2ull_rd(x);
          const float frac = x - __ull2float_rn(fl);                 // exact (x < 2^63)
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
    if (tid == 0) pub.total = nl > 0 ? cdf[nl - 1] : 0ull;
    cluster.sync();                                                  // barrier A2
    if (warp == 0) {                                                  // exclusive prefix over ranks
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
          if (writer) p.draw_ids[static_cast<int64_t>(unit) * M + r] = lo + lo_i;
          flag[lo_i] = 1;
        }
      }
    }
    if (!valid && writer && rank == 0)
      for (int r = tid; r < M; r += Tr::kThreads) p.draw_ids[static_cast<int64_t>(unit) * M + r] = -1;
    __syncthreads();
    // number this CTA's drawn teams and publish them (team, -log2 pi)
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
        list[k] = ListEntry{lo + j, -log2f(piv)};
        flag[j] = k;                       // keep the local slot for the global outputs
        ps[j] = piv;
      } else if (j < nl) {
        flag[j] = -1;
      }
      count += tot;
    }
    if (tid == 0) pub.count = valid ? count : 0;
    cluster.sync();                                                  // barrier A3
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
    __syncthreads();
    total_sel = s_base[CL];
    if (writer) {
      if (valid)
        for (int j = tid; j < nl; j += Tr::kThreads) {
          if (flag[j] < 0) continue;
          const int64_t slot = static_cast<int64_t>(unit) * M + s_base[rank] + flag[j];
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
    __syncthreads();                       // sampling scratch is dead from here on
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
  const int n_chunks = min(total_chunks - c_begin, cps);
  for (int ci = tid; ci < n_chunks; ci += Tr::kThreads) {
    const int c = c_begin + ci;
    const int slot = c / cpt, part = c - slot * cpt;
    int team = slot;
    float lw2 = 0.f;
    bool ok = true;
    if (mode == kModeDecode) {
      int owner = 0;
      while (owner + 1 < CL && s_base[owner + 1] <= slot) ++owner;
      const ListEntry e = cluster.map_shared_rank(list, owner)[slot - s_base[owner]];
      team = e.team;
      lw2 = e.lw2;
    } else if (mode == kModeAttend) {
      const int64_t sidx = static_cast<int64_t>(unit) * M + slot;
      team = p.sel_ids[sidx];
      const float piv = p.pi[sidx];
      ok = team >= 0 && team < n && piv > 0.f && piv <= 1.f;
      if (!ok) set_status(p.status, SANTA_DEV_BAD_SEL);
      lw2 = ok ? -log2f(piv) : 0.f;
    }
    int page = -1;
    if (ok) {
      page = p.page_table[static_cast<int64_t>(b) * p.max_teams + team];
      if (page < 0 || page >= p.num_pages) {
        set_status(p.status, SANTA_DEV_BAD_PAGE);
        ok = false;
      }
    }
    const int vt =
        ok ? max(0, min(min(p.team_size, L - team * p.team_size) - part * kChunk, kChunk)) : 0;
    table[ci] = ChunkMeta{vt > 0 ? page : -1, vt, lw2, part};
  }
  __syncthreads();

  // ================================================================ phase C: stream + compute
  // q of the group in registers, in the score layout
  float qr[G][Tr::kEplS];
  {
    const unsigned char* qb = static_cast<const unsigned char*>(p.q) +
                              (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D * Tr::kEsize;
#pragma unroll
    for (int g = 0; g < G; ++g) load_score_row<BF16, D>(qb + g * D * Tr::kEsize, lane16, qr[g]);
  }
  const unsigned char* kpool = static_cast<const unsigned char*>(p.k_pool);
  const unsigned char* vpool = static_cast<const unsigned char*>(p.v_pool);
  auto issue = [&](int ci) {
    const int stage = ci % S;
    const ChunkMeta m = table[ci];
    if (m.page >= 0) {
      const int64_t off = ((static_cast<int64_t>(m.page) * p.num_kv_heads + h) *
                               static_cast<int64_t>(p.team_size) + m.part * kChunk) *
                          D * Tr::kEsize;
      unsigned char* dst = smem + static_cast<size_t>(stage) * Tr::kStageBytes;
      mbar_arrive_expect_tx(&bar[stage], 2u * Tr::kChunkBytes);
      bulk_g2s(dst, kpool + off, Tr::kChunkBytes, &bar[stage]);
      bulk_g2s(dst + Tr::kChunkBytes, vpool + off, Tr::kChunkBytes, &bar[stage]);
    } else {
      mbar_arrive(&bar[stage]);
    }
  };
  if (tid < min(S, n_chunks)) issue(tid);

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

  // ================================================================ phase D: combine
  float* mrg_acc = reinterpret_cast<float*>(smem);                   // [8][G][D]
  float* mrg_m = mrg_acc + Tr::kWarps * G * D;                       // [8][8]
  float* mrg_l = mrg_m + Tr::kWarps * kMaxGroup;                     // [8][8]
  float* part = reinterpret_cast<float*>(smem) + Tr::kPartialOff;    // acc [G][D], m [8], l [8]
  float* part_m = part + G * D;
  float* part_l = part_m + kMaxGroup;
  if (attending) {
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < Tr::kEplV; ++e)
        mrg_acc[(warp * G + g) * D + lane * Tr::kEplV + e] = acc[g][e];
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
        a = fmaf(mw == kNegInf ? 0.f : exp2f(mw - mx), mrg_acc[(w * G + g) * D + k], a);
      }
      part[i] = a;
    }
  }
  cluster.sync();                                                    // barrier D1
  float* out_unit = p.out + (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D;
  if (attending) {
    // cluster-wide weights: peers' (m, l) per head
    if (tid < CL * G) {
      const float* peer = cluster.map_shared_rank(part, tid / G);
      s_pm[tid] = peer[G * D + tid % G];
      s_pz[tid] = peer[G * D + kMaxGroup + tid % G];
    }
    __syncthreads();
    if (tid < G) {
      float mx = kNegInf;
      for (int r = 0; r < CL; ++r) mx = fmaxf(mx, s_pm[r * G + tid]);
      float l = 0.f;
      for (int r = 0; r < CL; ++r) {
        const float mr = s_pm[r * G + tid];
        const float w = mr == kNegInf ? 0.f : exp2f(mr - mx);
        s_pm[r * G + tid] = w;                                       // becomes the weight
        l = fmaf(w, s_pz[r * G + tid], l);
      }
      s_gm[tid] = mx;
      s_gz[tid] = l;
    }
    __syncthreads();
    // this CTA's slice of the G*D/4 output quads: one thread per (peer, quad) fetches that
    // peer's weighted partial quad (all remote reads in flight at once), then per-quad sums
    // in rank order
    constexpr int kQuads = G * D / 4;
    const int qper = (kQuads + CL - 1) / CL;
    const int q0 = min(rank * qper, kQuads);
    const int nq = min(q0 + qper, kQuads) - q0;
    const int qb = Tr::kThreads / CL;                                // quads per block
    float4* comb = reinterpret_cast<float4*>(reinterpret_cast<float*>(smem) + Tr::kCombOff);
    for (int base = 0; base < nq; base += qb) {
      const int nb = min(qb, nq - base);
      {
        const int r = tid / qb, k = tid - r * qb;
        if (r < CL && k < nb) {
          const int qi = q0 + base + k;
          const float w = s_pm[r * G + (qi * 4) / D];
          const float4 v = reinterpret_cast<const float4*>(cluster.map_shared_rank(part, r))[qi];
          comb[r * qb + k] = make_float4(w * v.x, w * v.y, w * v.z, w * v.w);
        }
      }
      __syncthreads();
      if (tid < nb) {
        const int qi = q0 + base + tid;
        const int g = (qi * 4) / D;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < CL; ++r) {
          const float4 v = comb[r * qb + tid];
          a.x += v.x;
          a.y += v.y;
          a.z += v.z;
          a.w += v.w;
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
      __syncthreads();
    }
    if (NC > 1 && rank == 0 && tid < G) {
      p.part_ml[((static_cast<int64_t>(unit) * NC + cidx) * G + tid) * 2] = s_gm[tid];
      p.part_ml[((static_cast<int64_t>(unit) * NC + cidx) * G + tid) * 2 + 1] = s_gz[tid];
    }
  }
  cluster.sync();                                                    // barrier D2: peers done
  if (!attending || NC == 1) return;

  // ---- several clusters per unit: the last CTA to arrive merges the cluster partials
  __threadfence();
  __syncthreads();
  if (tid == 0)
    s_last = atomicAdd(&p.counters[unit], 1u) == static_cast<unsigned>(ctas - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < NC * G) {
    s_pm[tid] = __ldcg(&p.part_ml[(static_cast<int64_t>(unit) * NC * G + tid) * 2]);
    s_pz[tid] = __ldcg(&p.part_ml[(static_cast<int64_t>(unit) * NC * G + tid) * 2 + 1]);
  }
  __syncthreads();
  if (tid < G) {
    float mx = kNegInf;
    for (int c = 0; c < NC; ++c) mx = fmaxf(mx, s_pm[c * G + tid]);
    float l = 0.f;
    for (int c = 0; c < NC; ++c) {
      const float mc = s_pm[c * G + tid];
      const float w = mc == kNegInf ? 0.f : exp2f(mc - mx);
      s_pm[c * G + tid] = w;
      l = fmaf(w, s_pz[c * G + tid], l);
    }
    s_gz[tid] = l;
  }
  __syncthreads();
  constexpr int kQuads = G * D / 4;
  for (int qi = tid; qi < kQuads; qi += Tr::kThreads) {
    const int g = (qi * 4) / D;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < NC; ++c) {
      const float w = s_pm[c * G + g];
      const float4 v = __ldcg(
          reinterpret_cast<const float4*>(p.part_acc + (static_cast<int64_t>(unit) * NC + c) * G * D) + qi);
      a.x = fmaf(w, v.x, a.x);
      a.y = fmaf(w, v.y, a.y);
      a.z = fmaf(w, v.z, a.z);
      a.w = fmaf(w, v.w, a.w);
    }
    const float l = s_gz[g];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<float4*>(out_unit)[qi] = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  }
  if (tid == 0) p.counters[unit] = 0u;
}

// ---------------------------------------------------------------- host-side launch helpers

template <bool BF16, int D, int G>
std::atomic<unsigned long long>& decode_smem_flag() {
  static std::atomic<unsigned long long> flag{0};
  return flag;
}

template <bool BF16, int D, int G>
cudaError_t decode_prepare_t() {
  using Tr = DecodeTraits<BF16, D, G>;
  auto* kern = decode_kernel<BF16, D, G>;
  static std::atomic<unsigned long long> cluster_flag{0};
  cudaError_t e = ensure_dynamic_smem(kern, Tr::kSmem, decode_smem_flag<BF16, D, G>());
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
template <bool BF16, int D, int G>
int decode_max_clusters_t(int cluster) {
  using Tr = DecodeTraits<BF16, D, G>;
  if (decode_prepare_t<BF16, D, G>() != cudaSuccess) return 0;
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
  if (cudaOccupancyMaxActiveClusters(&n, decode_kernel<BF16, D, G>, &cfg) != cudaSuccess)
    return 0;
  return n;
}

template <bool BF16, int D, int G>
int decode_resident_t() {
  using Tr = DecodeTraits<BF16, D, G>;
  if (decode_prepare_t<BF16, D, G>() != cudaSuccess) return 0;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, decode_kernel<BF16, D, G>,
                                                    Tr::kThreads, Tr::kSmem) != cudaSuccess)
    return 0;
  return blocks;
}

template <bool BF16, int D, int G>
cudaError_t decode_launch_t(const DecodeParams& p, dim3 grid, int cluster, cudaStream_t stream) {
  using Tr = DecodeTraits<BF16, D, G>;
  cudaError_t e = decode_prepare_t<BF16, D, G>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Tr::kThreads);
  cfg.dynamicSmemBytes = Tr::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<BF16, D, G>, p);
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
