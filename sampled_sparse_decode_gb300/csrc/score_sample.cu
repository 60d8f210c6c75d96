// score_sample.cu — representative scoring, GQA-mixed team softmax, Philox inverse-CDF
// sampling, deduplication and inclusion probabilities for every (sequence, KV head) unit.
//
// Method ("SANTA++: Sampling Attention through Representative Keys", abstract; explainer
// "SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%", section 三 steps 2-3):
//   s_{g,i} = q_g . rep_i / sqrt(d)          for the G query heads g sharing KV head h
//   p_{g,i} = softmax_i(s_{g,.}),  p_i = (1/G) sum_g p_{g,i}
//   C_i = p_0 + ... + p_i (fp64), Z = C_{n-1}
//   draw r: x = word 0 of Philox4x32-10(counter (r, h, b, 0), key (lo32, hi32 of seed)),
//           u = (x + 1/2) 2^-32, team = smallest i with u*Z < C_i
//   S = distinct draws (ascending), pi_i = 1 - (1 - p_i)^M
//
// GB300 mapping: one thread-block cluster of CL CTAs per unit; CTA r of the cluster owns
// the contiguous team range [r*per, (r+1)*per).  Each warp scores its teams with one
// coalesced 512-byte read of the fp32 representative and warp-shuffle dot products; the
// per-head maxima, exponential sums, CDF totals and selected counts are exchanged between
// the CTAs through distributed shared memory at four cluster barriers.  Every reduction has
// a fixed order, so all CTAs agree bit for bit.  The CDF is a block scan in fp64; a draw
// is resolved by the one CTA whose [offset, offset + total) interval holds u*Z, by binary
// search over its own CDF slice.  The kernel lets the attention kernel launch early
// (programmatic dependent launch) so its prologue overlaps this kernel.
#include <cooperative_groups.h>

#include <cmath>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace santa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct Exchange {      // the values a CTA publishes to its cluster peers
  double total;        // its CDF total
  float m[kMaxGroup];  // per-head maximum score over its teams
  float z[kMaxGroup];  // per-head sum of exp(s - m)
  int count;           // its selected-team count
  int pad;
};

// Inclusive block scan of one value per thread over a 256-thread block (fixed order).
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
    V w = lane < kWarps ? warp_tot[lane] : V(0);
#pragma unroll
    for (int o = 1; o < kWarps; o <<= 1) {
      const V t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    if (lane < kWarps) warp_tot[lane] = w;
  }
  __syncthreads();
  const V pre = warp > 0 ? warp_tot[warp - 1] : V(0);
  block_total = warp_tot[kWarps - 1];
  const V res = pre + v;
  __syncthreads();
  return res;
}

template <int D>
__global__ void __launch_bounds__(kThreads) score_sample_kernel(const SampleParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int CL = static_cast<int>(cluster.num_blocks());
  const int h = blockIdx.y, b = blockIdx.z;
  const int unit = b * p.num_kv_heads + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.group, M = p.num_draws, tpc = p.teams_per_cta;
  constexpr float kNegInf = -INFINITY;

  extern __shared__ __align__(16) unsigned char smem[];
  double* cdf = reinterpret_cast<double*>(smem);                    // [tpc]
  Exchange* xs = reinterpret_cast<Exchange*>(cdf + tpc);             // published values
  float* qs = reinterpret_cast<float*>(xs + 1);                      // [G][D]
  float* es = qs + kMaxGroup * D;                                    // [G][tpc] scores, exps
  float* ps = es + kMaxGroup * tpc;                                  // [tpc] team probability
  int* flag = reinterpret_cast<int*>(ps + tpc);                      // [tpc] drawn / slot
  __shared__ double s_wd[kWarps];
  __shared__ int s_wi[kWarps];
  __shared__ float s_m[kMaxGroup], s_z[kMaxGroup];
  __shared__ double s_off, s_Z;
  __shared__ int s_base, s_total;

  pdl_trigger();

  const int L = p.seq_lens[b];
  const bool bad_len = L < 1 || static_cast<int64_t>(L) > static_cast<int64_t>(p.max_teams) *
                                                              p.team_size;
  const int n = bad_len ? 0 : (L + p.team_size - 1) / p.team_size;
  const int per = (n + CL - 1) / CL;
  const int lo = min(rank * per, n);
  const int nl = min(lo + per, n) - lo;   // teams owned by this CTA (<= tpc)

  // ---- query vectors of the group, fp32
  for (int i = tid; i < G * D; i += kThreads) {
    const int64_t idx = (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D + i;
    qs[i] = p.is_bf16 ? bf16_to_f32(static_cast<const uint16_t*>(p.q)[idx])
                      : static_cast<const float*>(p.q)[idx];
  }
  for (int j = tid; j < nl; j += kThreads) flag[j] = 0;
  __syncthreads();

  // ---- scores: one warp per team, lanes over d, four teams in flight per warp
  {
    constexpr int E = D / 32;
    float qr[kMaxGroup][E];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g)
#pragma unroll
      for (int e = 0; e < E; ++e) qr[g][e] = g < G ? qs[g * D + lane * E + e] : 0.f;
    constexpr int U = 4;
    for (int j0 = warp; j0 < nl; j0 += kWarps * U) {
      float rv[U][E];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * kWarps;
        ok[u] = false;
#pragma unroll
        for (int e = 0; e < E; ++e) rv[u][e] = 0.f;
        if (j < nl) {
          const int64_t page = p.page_table[static_cast<int64_t>(b) * p.max_teams + lo + j];
          ok[u] = page >= 0 && page < p.num_pages;
          if (ok[u]) {
            const float* rep = p.reps + (page * p.num_kv_heads + h) * D + lane * E;
            if constexpr (E == 4) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(rep));
              rv[u][0] = v.x; rv[u][1] = v.y; rv[u][2] = v.z; rv[u][3] = v.w;
            } else {
              const float2 v = __ldg(reinterpret_cast<const float2*>(rep));
              rv[u][0] = v.x; rv[u][1] = v.y;
            }
          } else if (lane == 0) {
            set_status(p.status, SANTA_DEV_BAD_PAGE);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * kWarps;
        if (j >= nl) continue;
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) {
          if (g >= G) break;
          float part = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) part = fmaf(qr[g][e], rv[u][e], part);
          part = warp_sum(part);
          if (lane == 0) es[g * tpc + j] = ok[u] ? part * p.scale : kNegInf;
        }
      }
    }
  }
  __syncthreads();

  // ---- per-head maximum over the cluster
  if (warp < G) {
    float m = kNegInf;
    for (int j = lane; j < nl; j += 32) m = fmaxf(m, es[warp * tpc + j]);
    m = warp_max(m);
    if (lane == 0) xs->m[warp] = m;
  }
  cluster.sync();
  if (tid < G) {
    float m = kNegInf;
    for (int r = 0; r < CL; ++r) m = fmaxf(m, cluster.map_shared_rank(xs, r)->m[tid]);
    s_m[tid] = m;
  }
  __syncthreads();

  // ---- exponentials and per-head sums over the cluster
  for (int i = tid; i < G * nl; i += kThreads) {
    const int g = i / nl, j = i - g * nl;
    const float s = es[g * tpc + j];
    es[g * tpc + j] = s == kNegInf ? 0.f : expf(s - s_m[g]);
  }
  __syncthreads();
  if (warp < G) {
    float z = 0.f;
    for (int j = lane; j < nl; j += 32) z += es[warp * tpc + j];
    z = warp_sum(z);
    if (lane == 0) xs->z[warp] = z;
  }
  cluster.sync();
  if (tid < G) {
    float z = 0.f;
    for (int r = 0; r < CL; ++r) z += cluster.map_shared_rank(xs, r)->z[tid];
    s_z[tid] = z;
  }
  __syncthreads();

  // ---- team probabilities p_i = (1/G) sum_g e_{g,i} / z_g
  for (int j = tid; j < nl; j += kThreads) {
    float acc = 0.f;
    for (int g = 0; g < G; ++g) acc += s_z[g] > 0.f ? es[g * tpc + j] / s_z[g] : 0.f;
    ps[j] = acc / static_cast<float>(G);
    if (p.team_probs) p.team_probs[static_cast<int64_t>(unit) * p.max_teams + lo + j] = ps[j];
  }
  if (p.team_probs && rank == 0)
    for (int j = n + tid; j < p.max_teams; j += kThreads)
      p.team_probs[static_cast<int64_t>(unit) * p.max_teams + j] = 0.f;
  __syncthreads();

  // ---- fp64 CDF of this CTA's slice
  {
    double carry = 0.0;
    for (int base = 0; base < nl; base += kThreads) {
      const int j = base + tid;
      double tot;
      const double v = block_inclusive_scan<double>(j < nl ? static_cast<double>(ps[j]) : 0.0,
                                                    s_wd, tot);
      if (j < nl) cdf[j] = carry + v;
      carry += tot;
    }
  }
  __syncthreads();
  if (tid == 0) xs->total = nl > 0 ? cdf[nl - 1] : 0.0;
  cluster.sync();
  if (tid == 0) {
    double acc = 0.0, off = 0.0;
    for (int r = 0; r < CL; ++r) {
      if (r == rank) off = acc;
      acc = acc + cluster.map_shared_rank(xs, r)->total;
    }
    s_off = off;
    s_Z = acc;
  }
  __syncthreads();

  // ---- M draws; the CTA whose interval holds u*Z resolves the draw
  const double off = s_off, Z = s_Z;
  const bool valid = !bad_len && Z > 0.0 && Z < INFINITY;
  if (valid && nl > 0) {
    const double hi_b = off + cdf[nl - 1];
    const uint2 key = make_uint2(static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32));
    for (int r = tid; r < M; r += kThreads) {
      const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(r), static_cast<uint32_t>(h),
                                               static_cast<uint32_t>(b), 0u),
                                    key);
      const double u = (static_cast<double>(w.x) + 0.5) * 0x1p-32;
      double t = u * Z;
      if (!(t < Z)) t = nextafter(Z, 0.0);
      if (off <= t && t < hi_b) {
        int a = 0, c = nl - 1;
        while (a < c) {
          const int mid = (a + c) >> 1;
          if (t < off + cdf[mid]) c = mid; else a = mid + 1;
        }
        p.draw_ids[static_cast<int64_t>(unit) * M + r] = lo + a;
        flag[a] = 1;
      }
    }
  }
  if (!valid && rank == 0) {
    for (int r = tid; r < M; r += kThreads) p.draw_ids[static_cast<int64_t>(unit) * M + r] = -1;
    if (tid == 0 && bad_len) set_status(p.status, SANTA_DEV_BAD_SEQLEN);
  }
  __syncthreads();

  // ---- deduplicate: ascending slots of the drawn teams across the cluster
  int count = 0;
  for (int base = 0; base < nl; base += kThreads) {
    const int j = base + tid;
    const int f = j < nl ? flag[j] : 0;
    int tot;
    const int incl = block_inclusive_scan<int>(f, s_wi, tot);
    if (j < nl) flag[j] = f ? count + incl - 1 : -1;
    count += tot;
  }
  if (tid == 0) xs->count = valid ? count : 0;
  cluster.sync();
  if (tid == 0) {
    int acc = 0, base = 0;
    for (int r = 0; r < CL; ++r) {
      if (r == rank) base = acc;
      acc += cluster.map_shared_rank(xs, r)->count;
    }
    s_base = base;
    s_total = acc;
  }
  __syncthreads();
  if (valid) {
    const float Mf = static_cast<float>(M);
    for (int j = tid; j < nl; j += kThreads) {
      if (flag[j] < 0) continue;
      const int64_t slot = static_cast<int64_t>(unit) * M + s_base + flag[j];
      p.sel_ids[slot] = lo + j;
      p.pi[slot] = -expm1f(Mf * log1pf(-ps[j]));
    }
  }
  if (rank == 0) {
    for (int s = s_total + tid; s < M; s += kThreads) {
      p.sel_ids[static_cast<int64_t>(unit) * M + s] = -1;
      p.pi[static_cast<int64_t>(unit) * M + s] = 0.f;
    }
    if (tid == 0) {
      p.sel_count[unit] = s_total;
      if (p.counters) p.counters[unit] = 0u;
    }
  }
  cluster.sync();  // peers may still be reading this CTA's published values
}

}  // namespace

size_t sample_smem_bytes(int head_dim, int teams_per_cta) {
  return sizeof(double) * teams_per_cta + sizeof(Exchange) + sizeof(float) * kMaxGroup * head_dim +
         sizeof(float) * kMaxGroup * teams_per_cta + sizeof(float) * teams_per_cta +
         sizeof(int) * teams_per_cta;
}

cudaError_t launch_sample(const SampleParams& p, int head_dim, int cluster, cudaStream_t stream) {
  const size_t smem = sample_smem_bytes(head_dim, p.teams_per_cta);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, p.num_kv_heads, p.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the limit is raised once to the largest size any supported shape needs: 16384 teams over
  // a cluster of 8 CTAs
  const size_t smem_max = sample_smem_bytes(head_dim, 2048);
  static std::atomic<unsigned long long> set128{0}, set64{0};
  cudaError_t e;
  if (head_dim == 128) {
    e = ensure_dynamic_smem(score_sample_kernel<128>, smem_max, set128);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, score_sample_kernel<128>, p);
  } else {
    e = ensure_dynamic_smem(score_sample_kernel<64>, smem_max, set64);
    if (e != cudaSuccess) return e;
    e = cudaLaunchKernelEx(&cfg, score_sample_kernel<64>, p);
  }
  return e;
}

}  // namespace santa
