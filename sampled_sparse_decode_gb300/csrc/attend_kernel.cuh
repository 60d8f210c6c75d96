// attend_kernel.cuh — split-K exact attention inside the sampled teams, each team weighted
// by the inverse of its inclusion probability, combined as a Horvitz-Thompson ratio.
//
// Method ("SANTA++: Sampling Attention through Representative Keys", abstract: exact
// attention scores within the sampled teams, each team's contribution reweighted by the
// inverse of its inclusion probability; explainer section 三 steps 4-5): for every query
// head g of the group,
//   out_g = sum_{i in S} (1/pi_i) sum_{j in team i} e^{s_j} v_j
//         / sum_{i in S} (1/pi_i) sum_{j in team i} e^{s_j},   s_j = q_g . k_j / sqrt(d).
// The weight is folded into the exponent, e^{s_j}/pi_i = e^{s_j - ln pi_i}, so the running
// maximum of the online softmax sees the weighted scores and 1/pi never overflows.  Scores
// are kept in base 2 (s * log2 e) so every exponential is one exp2.  Dense mode (the speed
// reference) runs the same code over every team with weight 1.
//
// GB300 mapping (HBM-bound gather, no tensor cores in this version):
//  - the unit's sampled teams form a list of 64-token chunks; CTA `split` of a unit owns
//    chunks [split*CPS, (split+1)*CPS) of that list;
//  - thread 0 streams each chunk's K and V rows (64*d contiguous elements each, straight
//    from the paged pool) into a ring of shared-memory stages with two bulk copies
//    (cp.async.bulk, the non-tensor TMA form) completing on an mbarrier;
//  - warp w owns tokens 8w..8w+7 of every chunk: scores use 16 lanes per token (8 or 4
//    elements each, q held in registers) and a reduce-scatter across the 16 lanes that
//    leaves lane l with head (l>>1)&7; probabilities go through a per-warp scratch row to
//    the P.V phase, where lane l owns d-elements [l*d/32, (l+1)*d/32) of every head;
//  - each warp keeps its own running (max, sum, acc); at the end the 8 warps merge in shared
//    memory and the CTA writes one partial (m, l, acc[d]) per head, or the output directly
//    when the unit has a single split;
//  - the last CTA of a unit to finish (an atomic ticket, no waiting) merges the unit's
//    partials in split order — the result does not depend on which CTA is last — writes
//    out and resets the ticket counter.
#pragma once

#include <cmath>

#include "kernels.h"

namespace santa {

// Where a staged chunk comes from and how it is weighted.
struct ChunkMeta {
  int page;      // physical page, or -1 for a chunk that contributes nothing
  int valid;     // valid tokens in the chunk (0..64)
  float lw2;     // -log2(pi) of its team (0 in dense mode)
  int part;      // which 64-token half of the page
};

template <bool BF16, int D, int G>
struct AttendTraits {
  static constexpr int kThreads = 256;
  static constexpr int kWarps = 8;
  static constexpr int kEsize = BF16 ? 2 : 4;
  static constexpr int kChunkBytes = kChunk * D * kEsize;
  static constexpr int kStageBytes = 2 * kChunkBytes;                 // K chunk + V chunk
  static constexpr int kStages = kStageBytes >= 65536 ? 2 : (kStageBytes >= 32768 ? 3 : 4);
  static constexpr int kEplS = D / 16;                                // score-phase elements
  static constexpr int kEplV = D / 32;                                // P.V-phase elements
  static constexpr int kMergeFloats = kWarps * G * D + 2 * kWarps * kMaxGroup;
  static_assert(kMergeFloats * 4 <= kStages * kStageBytes, "merge buffer must fit the stages");
  // two CTAs per SM when their stages fit (bf16, and fp32 with d = 64)
  static constexpr int kMinBlocks = kStages * kStageBytes <= 100 * 1024 ? 2 : 1;
  static constexpr int kCombineFloats = 3 * kMaxSplits * G + 2 * kMaxGroup;
  static_assert(kCombineFloats * 4 <= kStages * kStageBytes, "combine scratch must fit");
  // dynamic shared memory: stages | p rows [8][64] | alpha [8][8] | chunk table | bars
  static constexpr size_t kPOff = static_cast<size_t>(kStages) * kStageBytes;
  static constexpr size_t kAOff = kPOff + sizeof(float) * kWarps * 64;
  static constexpr size_t kMetaOff = kAOff + sizeof(float) * kWarps * kMaxGroup;
  static constexpr size_t kBarOff = kMetaOff + sizeof(ChunkMeta) * kMaxChunksPerSplit;
  static constexpr size_t kSmem = kBarOff + sizeof(uint64_t) * kStages;
};

// Score-phase element e of lane16: bf16 rows are read as one contiguous 8- or 16-byte
// vector per lane; fp32 rows with d = 128 as two 16-byte vectors 256 bytes apart, so a
// quarter-warp always covers 128 consecutive bytes (no bank conflicts).
template <bool BF16, int D>
__device__ __forceinline__ int score_elem(int lane16, int e) {
  if constexpr (BF16) {
    return lane16 * (D / 16) + e;
  } else {
    return (e >> 2) * 64 + lane16 * 4 + (e & 3);
  }
}

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

__device__ __forceinline__ float load_q(const void* q, bool bf16, int64_t idx) {
  return bf16 ? bf16_to_f32(__ldg(static_cast<const uint16_t*>(q) + idx))
              : __ldg(static_cast<const float*>(q) + idx);
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

template <bool BF16, int D, int G>
__global__ void __launch_bounds__(256, (AttendTraits<BF16, D, G>::kMinBlocks))
    attend_kernel(const AttendParams p) {
  using Tr = AttendTraits<BF16, D, G>;
  constexpr int S = Tr::kStages;
  constexpr float kNegInf = -INFINITY;
  extern __shared__ __align__(128) unsigned char smem[];
  float* prow = reinterpret_cast<float*>(smem + Tr::kPOff);        // [warp][token 8][head 8]
  float* arow = reinterpret_cast<float*>(smem + Tr::kAOff);        // [warp][head 8]
  ChunkMeta* meta = reinterpret_cast<ChunkMeta*>(smem + Tr::kMetaOff);  // [chunks of split]
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + Tr::kBarOff);
  __shared__ int s_last;
  __shared__ int s_abort;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, lane16 = lane & 15;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.num_kv_heads + h;
  const int hh = (lane >> 1) & 7;                        // head this lane reduces to

  // ---- prologue independent of the sampling kernel: q in registers, barriers
  float qr[G][Tr::kEplS];
  {
    const int64_t qbase = (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < Tr::kEplS; ++e)
        qr[g][e] = load_q(p.q, BF16, qbase + g * D + score_elem<BF16, D>(lane16, e));
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  const int L = p.seq_lens[b];
  const bool len_ok = L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_teams) *
                                                             p.team_size;
  const int n = len_ok ? (L + p.team_size - 1) / p.team_size : 0;
  const int cpt = p.team_size / kChunk;                  // chunks per team

  pdl_wait();  // sel_ids / sel_count / pi / counters come from the sampling kernel

  int count = n;
  if (!p.dense) {
    count = p.sel_count[unit];
    const int cap = min(p.num_draws, n);
    if (count < 0 || count > cap) {
      if (tid == 0) set_status(p.status, SANTA_DEV_BAD_SEL);
      count = 0;
    }
  }
  if (!len_ok && split == 0 && tid == 0) set_status(p.status, SANTA_DEV_BAD_SEQLEN);
  const int total_chunks = count * cpt;
  const int active = (total_chunks + p.chunks_per_split - 1) / p.chunks_per_split;
  float* out_unit = p.out + (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D;
  if (active == 0) {                                      // nothing to attend: zeros
    if (split == 0)
      for (int i = tid; i < G * D; i += Tr::kThreads) out_unit[i] = 0.f;
    return;
  }
  if (split >= active) return;
  const int c_begin = split * p.chunks_per_split;
  const int n_chunks = min(c_begin + p.chunks_per_split, total_chunks) - c_begin;

  // ---- chunk table of this split, all chunks resolved in parallel
  for (int ci = tid; ci < n_chunks; ci += Tr::kThreads) {
    const int c = c_begin + ci;
    const int slot = c / cpt, part = c - slot * cpt;
    int team = slot;
    float lw2 = 0.f;
    bool ok = true;
    if (!p.dense) {
      const int64_t sidx = static_cast<int64_t>(unit) * p.num_draws + slot;
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
        page = -1;
      }
    }
    const int vt =
        ok ? max(0, min(min(p.team_size, L - team * p.team_size) - part * kChunk, kChunk)) : 0;
    meta[ci] = ChunkMeta{vt > 0 ? page : -1, vt, lw2, part};
  }
  __syncthreads();

  const unsigned char* kpool = static_cast<const unsigned char*>(p.k_pool);
  const unsigned char* vpool = static_cast<const unsigned char*>(p.v_pool);
  // Producer: stage chunk ci of this split (one thread per call).
  auto issue = [&](int ci) {
    const int stage = ci % S;
    const ChunkMeta m = meta[ci];
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
    const int vt = meta[ci].valid;
    const float lw2 = meta[ci].lw2;
    const unsigned char* ks = smem + static_cast<size_t>(stage) * Tr::kStageBytes;
    const unsigned char* vs = ks + Tr::kChunkBytes;

    // scores of tokens 8w + 2k + (lane >> 4), k = 0..3, for head hh
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
    // online softmax per head over this warp's tokens
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

    // P.V: lane owns d-elements [lane*kEplV, (lane+1)*kEplV) of every head
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
    __syncthreads();                                      // stage and p rows free again
    if (tid == 0 && ci + S < n_chunks) issue(ci + S);
  }

  if (s_abort) {
    // wait (bounded) for the copies this CTA still has in flight, then give up
    if (tid == 0)
      for (int ci = consumed; ci < min(consumed + S, n_chunks); ++ci)
        (void)mbar_wait(&bar[ci % S], (ci / S) & 1);
    __syncthreads();
    return;
  }

  // ---- merge the 8 warps of this CTA
  float* mrg_acc = reinterpret_cast<float*>(smem);                  // [8][G][D]
  float* mrg_m = mrg_acc + Tr::kWarps * G * D;                      // [8][8]
  float* mrg_l = mrg_m + Tr::kWarps * kMaxGroup;                    // [8][8]
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

  const int ms = p.max_splits;
  const int64_t part_base = static_cast<int64_t>(unit) * ms;
  for (int i = tid; i < G * D; i += Tr::kThreads) {
    const int g = i / D, k = i - g * D;
    float mx = kNegInf;
#pragma unroll
    for (int w = 0; w < Tr::kWarps; ++w) mx = fmaxf(mx, mrg_m[w * kMaxGroup + g]);
    float a = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < Tr::kWarps; ++w) {
      const float mw = mrg_m[w * kMaxGroup + g];
      const float f = mw == kNegInf ? 0.f : exp2f(mw - mx);
      a = fmaf(f, mrg_acc[(w * G + g) * D + k], a);
      l = fmaf(f, mrg_l[w * kMaxGroup + g], l);
    }
    if (active == 1) {
      out_unit[i] = l > 0.f ? a / l : 0.f;
    } else {
      p.part_acc[((part_base + split) * G + g) * D + k] = a;
      if (k == 0) {
        p.part_ml[((part_base + split) * G + g) * 2] = mx;
        p.part_ml[((part_base + split) * G + g) * 2 + 1] = l;
      }
    }
  }
  if (active == 1) return;

  // ---- last CTA of the unit combines all partials, in split order
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&p.counters[unit], 1u) == static_cast<unsigned>(active - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  float* cm_s = reinterpret_cast<float*>(smem);                     // [active][G] maxima
  float* cl_s = cm_s + kMaxSplits * G;                              // [active][G] sums
  float* cw_s = cl_s + kMaxSplits * G;                              // [active][G] weights
  float* gm_s = cw_s + kMaxSplits * G;                              // [G] overall maxima
  float* gl_s = gm_s + kMaxGroup;                                   // [G] overall sums
  for (int i = tid; i < active * G; i += Tr::kThreads) {
    cm_s[i] = __ldcg(&p.part_ml[(part_base * G + i) * 2]);
    cl_s[i] = __ldcg(&p.part_ml[(part_base * G + i) * 2 + 1]);
  }
  __syncthreads();
  if (warp < G) {
    float mx = kNegInf;
    for (int c = lane; c < active; c += 32) mx = fmaxf(mx, cm_s[c * G + warp]);
    mx = warp_max(mx);
    if (lane == 0) gm_s[warp] = mx;
  }
  __syncthreads();
  for (int i = tid; i < active * G; i += Tr::kThreads) {
    const float mc = cm_s[i];
    cw_s[i] = mc == kNegInf ? 0.f : exp2f(mc - gm_s[i % G]);
  }
  __syncthreads();
  if (warp < G) {
    float l = 0.f;
    for (int c = lane; c < active; c += 32) l = fmaf(cw_s[c * G + warp], cl_s[c * G + warp], l);
    l = warp_sum(l);
    if (lane == 0) gl_s[warp] = l;
  }
  __syncthreads();
  constexpr int kQuads = D / 4;
  for (int i = tid; i < G * kQuads; i += Tr::kThreads) {
    const int g = i / kQuads, k4 = i - g * kQuads;
    const float4* src =
        reinterpret_cast<const float4*>(p.part_acc + (part_base * G + g) * D) + k4;
    const int stride = G * kQuads;                                  // one split, in float4
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int c = 0; c < active; ++c) {
      const float w = cw_s[c * G + g];
      const float4 v = __ldcg(src + static_cast<int64_t>(c) * stride);
      a.x = fmaf(w, v.x, a.x);
      a.y = fmaf(w, v.y, a.y);
      a.z = fmaf(w, v.z, a.z);
      a.w = fmaf(w, v.w, a.w);
    }
    const float l = gl_s[g];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<float4*>(out_unit + g * D)[k4] =
        make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
  }
  if (tid == 0) p.counters[unit] = 0u;
}

template <bool BF16, int D, int G>
std::atomic<unsigned long long>& attend_smem_flag() {
  static std::atomic<unsigned long long> flag{0};
  return flag;
}

// CTAs of this instantiation that fit on one SM (0 on error).
template <bool BF16, int D, int G>
int attend_resident_t() {
  using Tr = AttendTraits<BF16, D, G>;
  auto* kern = attend_kernel<BF16, D, G>;
  if (ensure_dynamic_smem(kern, Tr::kSmem, attend_smem_flag<BF16, D, G>()) != cudaSuccess)
    return 0;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, Tr::kThreads, Tr::kSmem) !=
      cudaSuccess)
    return 0;
  return blocks;
}

template <bool BF16, int D, int G>
cudaError_t launch_attend_t(const AttendParams& p, dim3 grid, bool programmatic,
                            cudaStream_t stream) {
  using Tr = AttendTraits<BF16, D, G>;
  auto* kern = attend_kernel<BF16, D, G>;
  cudaError_t e = ensure_dynamic_smem(kern, Tr::kSmem, attend_smem_flag<BF16, D, G>());
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(Tr::kThreads);
  cfg.dynamicSmemBytes = Tr::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool BF16, int D>
cudaError_t launch_attend_g(const AttendParams& p, int group, dim3 grid, bool programmatic,
                            cudaStream_t stream) {
  switch (group) {
    case 1: return launch_attend_t<BF16, D, 1>(p, grid, programmatic, stream);
    case 2: return launch_attend_t<BF16, D, 2>(p, grid, programmatic, stream);
    case 3: return launch_attend_t<BF16, D, 3>(p, grid, programmatic, stream);
    case 4: return launch_attend_t<BF16, D, 4>(p, grid, programmatic, stream);
    case 5: return launch_attend_t<BF16, D, 5>(p, grid, programmatic, stream);
    case 6: return launch_attend_t<BF16, D, 6>(p, grid, programmatic, stream);
    case 7: return launch_attend_t<BF16, D, 7>(p, grid, programmatic, stream);
    case 8: return launch_attend_t<BF16, D, 8>(p, grid, programmatic, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <bool BF16, int D>
int attend_resident_g(int group) {
  switch (group) {
    case 1: return attend_resident_t<BF16, D, 1>();
    case 2: return attend_resident_t<BF16, D, 2>();
    case 3: return attend_resident_t<BF16, D, 3>();
    case 4: return attend_resident_t<BF16, D, 4>();
    case 5: return attend_resident_t<BF16, D, 5>();
    case 6: return attend_resident_t<BF16, D, 6>();
    case 7: return attend_resident_t<BF16, D, 7>();
    default: return attend_resident_t<BF16, D, 8>();
  }
}

template <bool BF16, int D>
size_t attend_smem_g(int group) {
  switch (group) {
    case 1: return AttendTraits<BF16, D, 1>::kSmem;
    case 2: return AttendTraits<BF16, D, 2>::kSmem;
    case 3: return AttendTraits<BF16, D, 3>::kSmem;
    case 4: return AttendTraits<BF16, D, 4>::kSmem;
    case 5: return AttendTraits<BF16, D, 5>::kSmem;
    case 6: return AttendTraits<BF16, D, 6>::kSmem;
    case 7: return AttendTraits<BF16, D, 7>::kSmem;
    default: return AttendTraits<BF16, D, 8>::kSmem;
  }
}

}  // namespace santa
