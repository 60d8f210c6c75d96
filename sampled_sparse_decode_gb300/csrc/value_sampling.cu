// value_sampling.cu — attention over sampled teams with value-row sampling inside each team.
//
// "Stochastic Sparse Attention for Memory-Bound Inference", abstract: instead of the full
// P.V product, draw value rows from the post-softmax distribution and gather-add them.
// Here that replaces the P.V step inside every team the team sampler selected.  With
// grouped-query attention the G query heads share one set of rows per team: rows are drawn
// from the group-mean in-team distribution r_j = (1/G) sum_g exp(s_gj - m_g) / Z_g, and head
// g weighs a drawn row j by exp(s_gj - m_g) / r_j (an importance-sampling estimate of
// sum_j exp(s_gj - m_g) v_j that is unbiased given the team).  The denominators Z_g stay
// exact.  Row draw k of team i of unit (b, h) uses Philox4x32-10 word 0 of counter
// (k, h, b, 1 + i) and the exact fixed-point decision of the team draws.
//
// Two launches: vs_team_kernel, one CTA per (sampled slot, KV head, sequence), writes each
// team's (m_g, Z_g, acc_g) to the workspace; vs_combine_kernel merges the slots of a unit in
// slot order with the Horvitz-Thompson (or Hansen-Hurwitz) weight 1/pi of each team.
#include "decode_kernel.cuh"

namespace santa {

namespace {

constexpr int kVsThreads = 256;
constexpr int kMaxValueRows = 256;
constexpr int kMaxVsSlots = 1024;   // M for which value sampling is offered

struct VsParams {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* sel_ids;      // [units][M]
  const int32_t* sel_count;    // [units]
  const float* pi;             // [units][M], 1 / weight
  int num_q_heads;
  int num_kv_heads;
  int team_size;
  int max_teams;
  int num_draws;               // M, the slot dimension
  int value_rows;              // S
  int64_t num_pages;
  uint64_t seed;
  float scale;                 // 1 / sqrt(d)
  float* part_m;               // [units][M][G]
  float* part_z;               // [units][M][G]
  float* part_acc;             // [units][M][G][D]
  int32_t* value_ids;          // [units][M][S] or nullptr
  float* out;                  // [B][Hq][D]
  int32_t* status;
};

template <bool BF16, int D, int G>
struct VsLayout {
  static constexpr int kEsize = BF16 ? 2 : 4;
  static constexpr size_t kK = 0;                                            // K rows [T][D]
  static constexpr size_t kQ(int T) { return kK + static_cast<size_t>(T) * D * kEsize; }
  static constexpr size_t kS(int T) { return kQ(T) + sizeof(float) * G * D; }   // scores [G][T]
  static constexpr size_t kR(int T) { return kS(T) + sizeof(float) * G * T; }   // r [T]
  static constexpr size_t kC(int T) { return kR(T) + sizeof(float) * T; }       // CDF [T]
  static constexpr size_t kW(int T) { return kC(T) + sizeof(unsigned long long) * T; }
  static constexpr size_t kIdx(int T) { return kW(T) + sizeof(float) * G * kMaxValueRows; }
  static constexpr size_t kBytes(int T) { return kIdx(T) + sizeof(int) * kMaxValueRows; }
};

template <bool BF16, int D, int G>
__global__ void __launch_bounds__(kVsThreads) vs_team_kernel(const VsParams p) {
  using Ly = VsLayout<BF16, D, G>;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float s_m[kMaxGroup], s_z[kMaxGroup];
  __shared__ unsigned long long s_wd[8];
  const int slot = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int M = p.num_draws, S = p.value_rows, T = p.team_size;
  const int64_t unit = static_cast<int64_t>(b) * p.num_kv_heads + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, lane16 = lane & 15;
  // launched with programmatic serialisation: wait for the kernel that wrote the sampled set,
  // then let the combine kernel be scheduled (it waits for this grid to finish)
  grid_dependency_wait();
  grid_launch_dependents();
  const int count = p.sel_count[unit];
  if (slot >= count || slot >= M) return;
  float* pm = p.part_m + (unit * M + slot) * G;
  float* pz = p.part_z + (unit * M + slot) * G;
  // the team, validated as santa_attend validates it
  const int L = p.seq_lens[b];
  const int n = (L >= 1 && static_cast<int64_t>(L) <= static_cast<int64_t>(p.max_teams) * T)
                    ? (L + T - 1) / T : 0;
  const int team = p.sel_ids[unit * M + slot];
  const float recip = p.pi[unit * M + slot];
  const bool sel_ok = count <= min(M, n) && team >= 0 && team < n && recip > 0.f &&
                      isfinite(recip);
  const int page = sel_ok ? p.page_table[static_cast<int64_t>(b) * p.max_teams + team] : -1;
  const bool ok = sel_ok && page >= 0 && page < p.num_pages;
  if (!ok) {
    if (tid == 0) set_status(p.status, sel_ok ? SANTA_DEV_BAD_PAGE : SANTA_DEV_BAD_SEL);
    if (tid < G) {
      pm[tid] = -INFINITY;
      pz[tid] = 0.f;
    }
    return;
  }
  const int len = min(T, L - team * T);
  unsigned char* krows = smem + Ly::kK;
  float* qf = reinterpret_cast<float*>(smem + Ly::kQ(T));
  float* sc = reinterpret_cast<float*>(smem + Ly::kS(T));
  float* rr = reinterpret_cast<float*>(smem + Ly::kR(T));
  unsigned long long* cdf = reinterpret_cast<unsigned long long*>(smem + Ly::kC(T));
  float* wgt = reinterpret_cast<float*>(smem + Ly::kW(T));
  int* idx = reinterpret_cast<int*>(smem + Ly::kIdx(T));

  // K rows of the team (contiguous block of the (page, head)) into shared memory
  const int64_t base = (static_cast<int64_t>(page) * p.num_kv_heads + h) * T;
  const unsigned char* ksrc = static_cast<const unsigned char*>(p.k_pool) + base * D * Ly::kEsize;
  const int pieces = len * D * Ly::kEsize / 16;
  for (int i = tid; i < pieces; i += kVsThreads) cp_async16(krows + 16 * i, ksrc + 16 * i);
  // q of the group as fp32, in the score layout of load_score_row
  for (int i = tid; i < G * D; i += kVsThreads) {
    const int g = i / D, k = i - g * D;
    const int64_t qi = (static_cast<int64_t>(b) * p.num_q_heads + h * G + g) * D + k;
    qf[i] = BF16 ? bf16_to_f32(static_cast<const uint16_t*>(p.q)[qi])
                 : static_cast<const float*>(p.q)[qi];
  }
  cp_async_wait_all();
  __syncthreads();
  // scores s_gt = q_g . k_t / sqrt(d): 16 lanes per token, reduce-scatter over the heads
  {
    float qs[G][D / 16];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < D / 16; ++e) qs[g][e] = qf[g * D + score_elem<BF16, D>(lane16, e)];
    const int hh = (lane >> 1) & 7;
    for (int t0 = 2 * warp; t0 < T; t0 += 16) {
      const int t = t0 + (lane >> 4);
      float x[D / 16];
      if (t < len) {
        load_score_row<BF16, D>(krows + static_cast<size_t>(t) * D * Ly::kEsize, lane16, x);
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
      if (t < T && !(lane & 1) && hh < G) sc[hh * T + t] = t < len ? sum * p.scale : -INFINITY;
    }
  }
  __syncthreads();
  // per-head team max and sum of exp (warp per head)
  if (warp < G) {
    float m = -INFINITY;
    for (int t = lane; t < len; t += 32) m = fmaxf(m, sc[warp * T + t]);
    m = warp_max(m);
    float z = 0.f;
    for (int t = lane; t < len; t += 32) z += expf(sc[warp * T + t] - m);
    z = warp_sum(z);
    if (lane == 0) {
      s_m[warp] = m;
      s_z[warp] = z;
    }
  }
  __syncthreads();
  // r_t, its 62-bit fixed-point value and the exact integer CDF (one token per thread)
  unsigned long long P = 0ull;
  if (tid < len) {
    float r = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) r += expf(sc[g * T + tid] - s_m[g]) / s_z[g];
    r /= static_cast<float>(G);
    rr[tid] = r;
    if (r > 0.f) {
      const float x = r * 0x1p62f;
      const unsigned long long fl = __float2ull_rd(x);
      const float frac = x - __ull2float_rn(fl);
      P = fl + (frac >= 0.5f ? 1ull : 0ull);
    }
  }
  unsigned long long Z;
  const unsigned long long before = block_exclusive_scan<unsigned long long>(P, s_wd, Z);
  if (tid < len) cdf[tid] = before + P;
  __syncthreads();
  // S row draws, and each row's weight per head exp(s_gj - m_g) / r_j / S
  const uint2 key = make_uint2(static_cast<uint32_t>(p.seed), static_cast<uint32_t>(p.seed >> 32));
  for (int k = tid; k < S; k += kVsThreads) {
    const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(k), static_cast<uint32_t>(h),
                                             static_cast<uint32_t>(b), static_cast<uint32_t>(1 + team)),
                                  key);
    const unsigned long long a = 2ull * w.x + 1ull;
    const unsigned long long t = (__umul64hi(a, Z) << 31) | ((a * Z) >> 33);
    int lo = 0, hi = len - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (t < cdf[mid]) hi = mid; else lo = mid + 1;
    }
    idx[k] = lo;
    if (p.value_ids) p.value_ids[(unit * M + slot) * S + k] = lo;
    const float inv = 1.f / (rr[lo] * static_cast<float>(S));
#pragma unroll
    for (int g = 0; g < G; ++g) wgt[g * kMaxValueRows + k] = expf(sc[g * T + lo] - s_m[g]) * inv;
  }
  __syncthreads();
  // gather-add the drawn value rows: thread e of each half takes element e, the two halves
  // split the rows and are added in fixed order
  const int e = tid % D, half = tid / D;                       // D = 64: four quarters
  constexpr int kParts = kVsThreads / D;
  float acc[G];
#pragma unroll
  for (int g = 0; g < G; ++g) acc[g] = 0.f;
  const unsigned char* vsrc = static_cast<const unsigned char*>(p.v_pool) + base * D * Ly::kEsize;
  // rows in batches of 8: all loads of a batch are in flight before any is used
  for (int k0 = half; k0 < S; k0 += 8 * kParts) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u * kParts;
      v[u] = 0.f;
      if (k < S) {
        const int j = idx[k];
        v[u] = BF16 ? bf16_to_f32(reinterpret_cast<const uint16_t*>(vsrc)[j * D + e])
                    : reinterpret_cast<const float*>(vsrc)[j * D + e];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u * kParts;
      if (k < S) {
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = fmaf(wgt[g * kMaxValueRows + k], v[u], acc[g]);
      }
    }
  }
  float* red = reinterpret_cast<float*>(smem + Ly::kK);         // K rows are no longer needed
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) red[(half * G + g) * D + e] = acc[g];
  __syncthreads();
  float* pacc = p.part_acc + (unit * M + slot) * G * D;
  for (int i = tid; i < G * D; i += kVsThreads) {
    const int g = i / D, k = i - g * D;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < kParts; ++q) s += red[(q * G + g) * D + k];
    pacc[i] = s;
  }
  if (tid < G) {
    pm[tid] = s_m[tid];
    pz[tid] = s_z[tid];
  }
}

// out_g = sum_c (1/pi_c) e^(m_c - mx) acc_c / sum_c (1/pi_c) e^(m_c - mx) Z_c over the unit's
// slots c.  Warp g forms head g's slot weights (lanes over slots) into shared memory [G][M].
// Then four groups of threads each sum every fourth slot of every output quad, with the
// loads of 8 slots in flight at once, and the four group sums are added in fixed order.
constexpr int kCombThreads = 1024;
constexpr int kCombGroups = 4;

template <int D, int G>
__global__ void __launch_bounds__(kCombThreads) vs_combine_kernel(const VsParams p) {
  constexpr int kQuads = G * D / 4;
  extern __shared__ float s_w[];                       // [G][M]
  __shared__ float s_den[kMaxGroup];
  __shared__ float4 s_red[kCombGroups][kQuads];
  const int h = blockIdx.x, b = blockIdx.y;
  const int M = p.num_draws;
  const int64_t unit = static_cast<int64_t>(b) * p.num_kv_heads + h;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dependency_wait();                              // the team kernel's partials
  const int count = max(0, min(p.sel_count[unit], M));
  if (warp < G) {
    float mx = -INFINITY;
    for (int c = lane; c < count; c += 32) mx = fmaxf(mx, p.part_m[(unit * M + c) * G + warp]);
    mx = warp_max(mx);
    float den = 0.f;
    for (int c = lane; c < count; c += 32) {
      const float m = p.part_m[(unit * M + c) * G + warp];
      const float w = m == -INFINITY ? 0.f : expf(m - mx) / p.pi[unit * M + c];
      s_w[warp * M + c] = w;
      den = fmaf(w, p.part_z[(unit * M + c) * G + warp], den);
    }
    den = warp_sum(den);
    if (lane == 0) s_den[warp] = den;
  }
  __syncthreads();
  const float4* acc = reinterpret_cast<const float4*>(p.part_acc) + unit * M * kQuads;
  for (int item = tid; item < kCombGroups * kQuads; item += kCombThreads) {
    const int grp = item / kQuads, qi = item - grp * kQuads;
    const int g = (4 * qi) / D;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c0 = grp; c0 < count; c0 += 8 * kCombGroups) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * kCombGroups;
        v[u] = c < count ? acc[static_cast<int64_t>(c) * kQuads + qi] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * kCombGroups;
        const float w = c < count ? s_w[g * M + c] : 0.f;
        a.x = fmaf(w, v[u].x, a.x);
        a.y = fmaf(w, v[u].y, a.y);
        a.z = fmaf(w, v[u].z, a.z);
        a.w = fmaf(w, v[u].w, a.w);
      }
    }
    s_red[grp][qi] = a;
  }
  __syncthreads();
  float4* out = reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(b) * p.num_q_heads + h * G) * D);
  for (int qi = tid; qi < kQuads; qi += kCombThreads) {
    const int g = (4 * qi) / D;
    float4 sum = s_red[0][qi];
#pragma unroll
    for (int grp = 1; grp < kCombGroups; ++grp) {
      sum.x += s_red[grp][qi].x;
      sum.y += s_red[grp][qi].y;
      sum.z += s_red[grp][qi].z;
      sum.w += s_red[grp][qi].w;
    }
    const float den = s_den[g];
    const float inv = den > 0.f ? 1.f / den : 0.f;
    out[qi] = make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
  }
}

template <bool BF16, int D, int G>
cudaError_t vs_launch_t(const VsParams& p, int batch, cudaStream_t stream) {
  using Ly = VsLayout<BF16, D, G>;
  const size_t smem = Ly::kBytes(p.team_size);
  static std::atomic<unsigned long long> flag{0};
  // the attribute once per device, for the largest team size and slot count
  cudaError_t e = ensure_dynamic_smem(vs_team_kernel<BF16, D, G>, Ly::kBytes(128), flag);
  if (e != cudaSuccess) return e;
  // both kernels may be scheduled while the previous kernel of the stream finishes; each
  // waits on it before reading what it wrote
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_draws, p.num_kv_heads, batch);
  cfg.blockDim = dim3(kVsThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, vs_team_kernel<BF16, D, G>, p)) != cudaSuccess) return e;
  const size_t csmem = sizeof(float) * G * static_cast<size_t>(p.num_draws);
  static std::atomic<unsigned long long> cflag{0};
  if ((e = ensure_dynamic_smem(vs_combine_kernel<D, G>, sizeof(float) * G * kMaxVsSlots,
                               cflag)) != cudaSuccess)
    return e;
  cfg.gridDim = dim3(p.num_kv_heads, batch);
  cfg.blockDim = dim3(kCombThreads);
  cfg.dynamicSmemBytes = csmem;
  return cudaLaunchKernelEx(&cfg, vs_combine_kernel<D, G>, p);
}

}  // namespace

cudaError_t launch_value_sampled(const VsLaunch& l, cudaStream_t stream) {
  VsParams p;
  p.q = l.q;
  p.k_pool = l.k_pool;
  p.v_pool = l.v_pool;
  p.page_table = l.page_table;
  p.seq_lens = l.seq_lens;
  p.sel_ids = l.sel_ids;
  p.sel_count = l.sel_count;
  p.pi = l.pi;
  p.num_q_heads = l.num_q_heads;
  p.num_kv_heads = l.num_kv_heads;
  p.team_size = l.team_size;
  p.max_teams = l.max_teams;
  p.num_draws = l.num_draws;
  p.value_rows = l.value_rows;
  p.num_pages = l.num_pages;
  p.seed = l.seed;
  p.scale = l.scale;
  p.part_m = l.part_m;
  p.part_z = l.part_z;
  p.part_acc = l.part_acc;
  p.value_ids = l.value_ids;
  p.out = l.out;
  p.status = l.status;
  const int G = l.num_q_heads / l.num_kv_heads;
  if (l.bf16) {
    if (l.head_dim == 128) { SANTA_DISPATCH_G(G, return (vs_launch_t<true, 128, GG>(p, l.batch, stream))) }
    SANTA_DISPATCH_G(G, return (vs_launch_t<true, 64, GG>(p, l.batch, stream)))
  }
  if (l.head_dim == 128) { SANTA_DISPATCH_G(G, return (vs_launch_t<false, 128, GG>(p, l.batch, stream))) }
  SANTA_DISPATCH_G(G, return (vs_launch_t<false, 64, GG>(p, l.batch, stream)))
}

}  // namespace santa
