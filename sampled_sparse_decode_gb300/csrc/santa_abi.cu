// santa_abi.cu — the extern "C" entry points of libsanta.so (declared in include/santa.h):
// argument checks, the split plan and workspace layout, and the kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "kernels.h"

namespace {

// The driver's allocation id of a pointer into memory from a CUDA allocation API (0 if the
// driver does not know the pointer).
unsigned long long allocation_id(const void* ptr) {
  static std::once_flag once;
  static PFN_cuPointerGetAttribute_v4000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &f, 4000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(f);
  });
  unsigned long long id = 0;
  if (!fn || fn(&id, CU_POINTER_ATTRIBUTE_BUFFER_ID, reinterpret_cast<CUdeviceptr>(ptr)) !=
                 CUDA_SUCCESS)
    return 0;
  return id;
}

// `host` itself, if [host, host + bytes) lies in one page-locked allocation that the current
// device reaches at the same address (unified addressing) and the copy with `dev` can move
// 16-byte words (both pointers and the size multiples of 16); otherwise nullptr, and
// santa_decode_host uses the copy engine.  Pageable memory, memory pinned for another device,
// a range that leaves its allocation and unaligned copies all take the copy engine.
const void* mapped_host(const void* host, const void* dev, size_t bytes) {
  if (((reinterpret_cast<uintptr_t>(host) | reinterpret_cast<uintptr_t>(dev) | bytes) & 15) != 0)
    return nullptr;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  int cur = -1;
  if (at.type != cudaMemoryTypeHost || at.devicePointer != host ||
      cudaGetDevice(&cur) != cudaSuccess || at.device != cur)
    return nullptr;
  // the first and the last byte in the same allocation: the kernel stays inside it
  const unsigned long long id = allocation_id(host);
  if (id == 0 || allocation_id(static_cast<const unsigned char*>(host) + bytes - 1) != id)
    return nullptr;
  return host;  // unified addressing: the device reaches the memory at the host's address
}

using santa::DecodeParams;
using santa::RepsParams;

constexpr int kMaxTeams = 16384;
constexpr int kMaxDraws = 4096;
constexpr size_t kAlign = 256;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int map_cuda(cudaError_t e) { return e == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA; }

// Streaming multiprocessors of the current device (cached per device).
int current_sms() {
  static std::mutex mu;
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && cache[dev]) return cache[dev];
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = sms;
  return sms;
}

int check_shape(int dtype, int batch, int hq, int hkv, int d, int T, int max_teams) {
  if (dtype != SANTA_F32 && dtype != SANTA_BF16) return SANTA_ERR_UNSUPPORTED;
  if (batch < 1 || hq < 1 || hkv < 1 || max_teams < 1) return SANTA_ERR_INVALID_ARG;
  if (hq % hkv != 0) return SANTA_ERR_INVALID_ARG;
  if (hq / hkv > santa::kMaxGroup) return SANTA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return SANTA_ERR_UNSUPPORTED;
  if (T != 64 && T != 128) return SANTA_ERR_UNSUPPORTED;
  if (max_teams > kMaxTeams || batch > 65535 || hkv > 65535) return SANTA_ERR_UNSUPPORTED;
  return SANTA_OK;
}

int check_inputs(const santa_decode_args* a) {
  if (!a) return SANTA_ERR_INVALID_ARG;
  int rc = check_shape(a->dtype, a->batch, a->num_q_heads, a->num_kv_heads, a->head_dim,
                       a->team_size, a->max_teams);
  if (rc) return rc;
  if (a->num_pages < 1) return SANTA_ERR_INVALID_ARG;
  if (!a->q || !a->k_pool || !a->v_pool || !a->page_table || !a->seq_lens)
    return SANTA_ERR_INVALID_ARG;
  if (!aligned(a->q, 16) || !aligned(a->k_pool, 16) || !aligned(a->v_pool, 16) ||
      !aligned(a->page_table, 4) || !aligned(a->seq_lens, 4))
    return SANTA_ERR_INVALID_ARG;
  if (a->device_status && !aligned(a->device_status, 4)) return SANTA_ERR_INVALID_ARG;
  return SANTA_OK;
}

int check_draws(const santa_decode_args* a) {
  if (a->num_draws < 1 || a->num_draws > kMaxDraws) return SANTA_ERR_UNSUPPORTED;
  if (a->sampler < SANTA_SAMPLER_IID_HT || a->sampler > SANTA_SAMPLER_IID_HH)
    return SANTA_ERR_INVALID_ARG;
  if (!(a->mix_alpha >= 0.f && a->mix_alpha <= 1.f)) return SANTA_ERR_INVALID_ARG;
  if (!a->sel_ids || !a->sel_count || !a->pi) return SANTA_ERR_INVALID_ARG;
  if (!aligned(a->sel_ids, 4) || !aligned(a->sel_count, 4) || !aligned(a->pi, 4))
    return SANTA_ERR_INVALID_ARG;
  return SANTA_OK;
}

// ---------------------------------------------------------------- launch plan
//
// A unit (sequence, KV head) is served by NC clusters of CL CTAs.  CL is the largest power
// of two <= 16 that keeps the whole job within one wave of resident CTAs (and that the
// device can co-schedule); sampling needs CL >= max_teams / 1024.  NC > 1 only when one
// cluster would give each CTA more than 8 chunks and the wave has room, or when a CTA would
// own more than kMaxChunksPerSplit chunks.  Only NC > 1 uses the workspace:
//   counters  [B*Hkv] uint32                      (rounded up to 256 bytes)
//   part_ml   [B*Hkv][NC][G][2] fp32 (m, l)       (rounded up to 256 bytes)
//   part_acc  [B*Hkv][NC][G][d] fp32
// with the base rounded up to 256 bytes.

size_t counters_bytes(int64_t units) { return round_up(static_cast<size_t>(units) * 4, kAlign); }
size_t cluster_partial_bytes(int64_t units, int G, int d) {
  return static_cast<size_t>(units) * G * (d + 2) * sizeof(float);
}
size_t ws_bytes_for(int64_t units, int G, int d, int nc) {
  if (nc <= 1) return kAlign;
  return kAlign + counters_bytes(units) +
         round_up(static_cast<size_t>(units) * nc * G * 2 * sizeof(float), kAlign) +
         static_cast<size_t>(units) * nc * G * d * sizeof(float);
}

int64_t chunks_max_of(int T, int max_teams, int M, int mode) {
  if (mode == santa::kModeSample) return 0;
  const int64_t teams = mode == santa::kModeDense ? max_teams : std::min(M, max_teams);
  return teams * (T / santa::kChunk);
}

int pow2_at_least(int64_t x) {
  int c = 1;
  while (c < x) c <<= 1;
  return c;
}

// CTAs of the kernel one SM holds; `wide` selects the one-CTA-per-SM bf16 variant.
int resident_ctas(bool bf16, int d, int G, bool wide) {
  static std::mutex mu;
  static int cache[64][2][2][2][santa::kMaxGroup + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][bf16][wide][d == 128][G];
  if (!c)
    c = bf16 ? (wide ? santa::decode_resident_bf16_wide(d, G) : santa::decode_resident_bf16(d, G))
             : santa::decode_resident_f32(d, G);
  return c;
}

// CTAs of the compact form of the bf16 kernel one SM holds (cached per device and shape).
int compact_resident(int d, int G, bool wide, bool variants) {
  static std::mutex mu;
  static int cache[64][2][2][2][santa::kMaxGroup + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][variants][wide][d == 128][G];
  if (!c)
    c = variants ? (wide ? santa::decode_resident_bf16_wide_fast_var(d, G)
                         : santa::decode_resident_bf16_fast_var(d, G))
                 : (wide ? santa::decode_resident_bf16_wide_fast(d, G)
                         : santa::decode_resident_bf16_fast(d, G));
  return c;
}

// Clusters of `cl` CTAs the device can run at once (cached per device and shape).
int max_clusters(bool bf16, int d, int G, int cl, bool wide) {
  static std::mutex mu;
  static int cache[64][2][2][2][santa::kMaxGroup + 1][5] = {};  // 0 unknown, -1 none
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int li = 0;
  while ((1 << li) < cl) ++li;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][bf16][wide][d == 128][G][li];
  if (!c) {
    const int n = bf16 ? (wide ? santa::decode_max_clusters_bf16_wide(d, G, cl)
                               : santa::decode_max_clusters_bf16(d, G, cl))
                       : santa::decode_max_clusters_f32(d, G, cl);
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

struct Plan {
  int cluster = 1;       // CL
  int clusters = 1;      // NC
  int tpc = 1;           // teams per CTA in the sampling phase
  bool wide = false;     // bf16 one-CTA-per-SM variant
  uint32_t* counters = nullptr;
  float* part_ml = nullptr;
  float* part_acc = nullptr;
};

// Chooses CL and NC for a shape; nc_cap limits NC (the workspace's capacity).
int choose(int dtype, int64_t units, int G, int d, int T, int max_teams, int M, int mode,
           int64_t nc_cap, bool wide, Plan* pl) {
  const bool bf16 = dtype == SANTA_BF16;
  const int sms = current_sms();
  const int res = resident_ctas(bf16, d, G, wide);
  if (sms <= 0 || res <= 0) return SANTA_ERR_CUDA;
  const int64_t slots = static_cast<int64_t>(sms) * res;
  const int64_t spu = std::max<int64_t>(1, slots / units);
  const bool sampling = mode == santa::kModeDecode || mode == santa::kModeSample;
  const int64_t cmax = chunks_max_of(T, max_teams, M, mode);
  // smallest cluster that keeps per-CTA tables in bounds
  int64_t cl_min = 1;
  if (sampling) cl_min = std::max<int64_t>(cl_min, ceil_div(max_teams, santa::kMaxTeamsPerCta));
  const int64_t nc_limit = std::min<int64_t>(santa::kMaxClustersPerUnit, std::max<int64_t>(1, nc_cap));
  cl_min = std::max<int64_t>(cl_min, ceil_div(cmax, santa::kMaxChunksPerSplit * nc_limit));
  int cl_lo = pow2_at_least(cl_min);
  if (cl_lo > santa::kMaxCluster) return SANTA_ERR_UNSUPPORTED;
  int cl_start = 1;
  while (cl_start * 2 <= std::min<int64_t>(spu, santa::kMaxCluster)) cl_start *= 2;
  cl_start = std::max(cl_start, cl_lo);
  // Cluster size: the largest power of two (<= units' share of one wave, <= 16) whose
  // clusters can all be resident at once; failing that, the smallest allowed.  Clusters per
  // unit: as few as keep every CTA's chunk table in bounds.  A dense step (no sampling to
  // repeat per cluster) also takes more clusters when each CTA would otherwise stream more
  // than 8 chunks and the extra clusters still fit the wave.
  int cl = -1;
  int64_t nc = 1;
  for (int c = cl_start; c >= cl_lo; c >>= 1) {
    const int maxc = max_clusters(bf16, d, G, c, wide);
    if (maxc <= 0) continue;
    const int64_t nc_min = cmax > 0 ? ceil_div(cmax, static_cast<int64_t>(santa::kMaxChunksPerSplit) * c) : 1;
    if (nc_min > nc_limit) continue;
    int64_t n_c = nc_min;
    if (mode == santa::kModeDense) {
      const int64_t want = ceil_div(ceil_div(cmax, c), 8);
      const int64_t room = std::max<int64_t>(1, maxc / units);
      n_c = std::max(nc_min, std::min({want, room, nc_limit}));
    }
    cl = c;
    nc = n_c;
    if (units * n_c <= maxc) break;
  }
  if (cl < 0) return SANTA_ERR_UNSUPPORTED;
  pl->cluster = cl;
  pl->clusters = static_cast<int>(nc);
  pl->tpc = static_cast<int>(std::max<int64_t>(1, ceil_div(max_teams, cl)));
  pl->wide = wide;
  return SANTA_OK;
}

// A dense bf16 plan on the wide variant that fills the device: the largest units * CL * NC
// CTAs, at most one per SM, that the device can co-schedule (larger clusters on ties).
// Returns false if no such plan reaches three quarters of the SMs.
bool dense_fill_plan(int64_t units, int G, int d, int T, int max_teams, int64_t nc_cap,
                     Plan* pl) {
  const int64_t sms = current_sms();
  const int64_t cmax = chunks_max_of(T, max_teams, 1, santa::kModeDense);
  int64_t best = 0;
  for (int cl = santa::kMaxCluster; cl >= 1; cl >>= 1) {
    int64_t nc = std::min<int64_t>({santa::kMaxClustersPerUnit, std::max<int64_t>(1, nc_cap),
                                    sms / (units * cl)});
    const int maxc = max_clusters(true, d, G, cl, true);
    nc = std::min<int64_t>(nc, maxc / units);
    if (nc < 1 || ceil_div(cmax, cl * nc) > santa::kMaxChunksPerSplit) continue;
    if (units * cl * nc > best) {
      best = units * cl * nc;
      pl->cluster = cl;
      pl->clusters = static_cast<int>(nc);
      pl->tpc = static_cast<int>(std::max<int64_t>(1, ceil_div(max_teams, cl)));
      pl->wide = true;
    }
  }
  return best * 4 >= sms * 3;
}

// The two-CTA-per-SM plan, replaced by the wide variant's plan when the step is a bf16
// attending one and both plans need no more CTAs than the device has SMs (each CTA then has
// an SM to itself anyway, and the wide variant consumes two chunks at a time).  A dense step
// whose two-CTA-per-SM grid is under one and a half waves of SMs instead fills the device
// with the wide variant (dense_fill_plan): uneven pairs of CTAs per SM set its tail.
int choose_variant(int dtype, int64_t units, int G, int d, int T, int max_teams, int M,
                   int mode, int64_t nc_cap, Plan* pl) {
  int rc = choose(dtype, units, G, d, T, max_teams, M, mode, nc_cap, false, pl);
  if (rc || dtype != SANTA_BF16 || mode == santa::kModeSample) return rc;
  const int64_t sms = current_sms();
  if (mode == santa::kModeDense) {
    Plan w;
    if (2 * units * pl->cluster * pl->clusters < 3 * sms &&
        dense_fill_plan(units, G, d, T, max_teams, nc_cap, &w))
      *pl = w;
    return SANTA_OK;
  }
  if (units * pl->cluster * pl->clusters > sms) {
    // a decode step whose units still get clusters of at least 4 CTAs with one CTA per SM
    // takes the wide variant (more stages per SM; at Qwen B=8: 4 x 32 CTAs instead of 8 x 32
    // two per SM, 0.4 us faster); smaller clusters stay on the two-CTA-per-SM variant
    Plan w;
    if (mode == santa::kModeDecode &&
        choose(dtype, units, G, d, T, max_teams, M, mode, nc_cap, true, &w) == SANTA_OK &&
        w.cluster >= 4 && units * w.cluster * w.clusters <= sms)
      *pl = w;
    return SANTA_OK;
  }
  Plan w;
  if (choose(dtype, units, G, d, T, max_teams, M, mode, nc_cap, true, &w) == SANTA_OK &&
      units * w.cluster * w.clusters <= sms)
    *pl = w;
  return SANTA_OK;
}

int make_plan(const santa_decode_args* a, int mode, Plan* pl) {
  const int64_t units = static_cast<int64_t>(a->batch) * a->num_kv_heads;
  const int G = a->num_q_heads / a->num_kv_heads, d = a->head_dim;
  // clusters per unit the workspace can hold
  int64_t nc_cap = 1;
  uintptr_t base = 0;
  if (a->workspace && a->workspace_bytes > 0) {
    const uintptr_t raw = reinterpret_cast<uintptr_t>(a->workspace);
    base = round_up(raw, kAlign);
    const size_t fixed = (base - raw) + counters_bytes(units) + kAlign;
    if (a->workspace_bytes > fixed)
      nc_cap = std::max<int64_t>(1, static_cast<int64_t>((a->workspace_bytes - fixed) /
                                                         cluster_partial_bytes(units, G, d)));
  }
  int rc = choose_variant(a->dtype, units, G, d, a->team_size, a->max_teams, a->num_draws, mode,
                          nc_cap, pl);
  if (rc) return rc;
  if (pl->clusters > 1) {
    if (!base) return SANTA_ERR_INVALID_ARG;
    unsigned char* b = reinterpret_cast<unsigned char*>(base);
    pl->counters = reinterpret_cast<uint32_t*>(b);
    b += counters_bytes(units);
    pl->part_ml = reinterpret_cast<float*>(b);
    b += round_up(static_cast<size_t>(units) * pl->clusters * G * 2 * sizeof(float), kAlign);
    pl->part_acc = reinterpret_cast<float*>(b);
  }
  return SANTA_OK;
}

size_t default_ws_bytes(int dtype, int batch, int hq, int hkv, int d, int T, int max_teams,
                        int M, int mode) {
  if (check_shape(dtype, batch, hq, hkv, d, T, max_teams)) return 0;
  if (mode != santa::kModeDense && (M < 1 || M > kMaxDraws)) return 0;
  Plan pl;
  const int64_t units = static_cast<int64_t>(batch) * hkv;
  if (choose_variant(dtype, units, hq / hkv, d, T, max_teams, M, mode,
                     santa::kMaxClustersPerUnit, &pl))
    return 0;
  return ws_bytes_for(units, hq / hkv, d, pl.clusters);
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// A bf16 pool [P][Hkv][T][d] as a 2-D tensor [P*Hkv*T rows][d]: boxes of 64 rows x 64
// elements (128 bytes, the swizzle span) with 128-byte swizzle.
int encode_pool_map(CUtensorMap* map, const void* pool, int64_t rows, int d) {
  auto encode = tensor_map_encoder();
  if (!encode) return SANTA_ERR_CUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool),
                            dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SANTA_OK : SANTA_ERR_CUDA;
}

// Whether a compact-path call needs the instantiations with the sampler variants compiled in:
// a variant sampler, the mixture, or a sampling-only step.
bool compact_variants(const santa_decode_args* a, int mode) {
  return mode == santa::kModeSample || a->sampler != SANTA_SAMPLER_IID_HT || a->mix_alpha != 0.f;
}

// Whether a checked and planned call runs the compact path of the decode kernel: a bf16
// decode (or sampling-only) step with one cluster per unit whose shape the compact path's
// shared-memory layout holds.
bool uses_compact_path(const santa_decode_args* a, int mode, const Plan& pl) {
  if ((mode != santa::kModeDecode && mode != santa::kModeSample) || a->dtype != SANTA_BF16 ||
      pl.clusters != 1)
    return false;
  const bool variants = compact_variants(a, mode);
  const int G = a->num_q_heads / a->num_kv_heads;
  const bool fits =
      pl.wide ? santa::decode_fast_fits_bf16_wide(a->head_dim, G, a->max_teams, pl.cluster,
                                                  a->team_size, a->num_draws)
              : santa::decode_fast_fits_bf16(a->head_dim, G, a->max_teams, pl.cluster,
                                             a->team_size, a->num_draws);
  // the plan assumes the general kernel's resident CTAs per SM: the compact one must match
  return fits && compact_resident(a->head_dim, G, pl.wide, variants) >=
                     resident_ctas(true, a->head_dim, G, pl.wide);
}

// Every host-side check of a call in `mode`, then its plan; launches nothing.
int check_and_plan(const santa_decode_args* a, int mode, Plan* pl) {
  int rc = check_inputs(a);
  if (rc) return rc;
  const bool sampling = mode == santa::kModeDecode || mode == santa::kModeSample;
  if (mode != santa::kModeDense && (rc = check_draws(a))) return rc;
  if (sampling) {
    if (!a->reps || !aligned(a->reps, 16) || !a->draw_ids || !aligned(a->draw_ids, 4))
      return SANTA_ERR_INVALID_ARG;
    if (a->team_probs && !aligned(a->team_probs, 4)) return SANTA_ERR_INVALID_ARG;
  }
  if (mode != santa::kModeSample && (!a->out || !aligned(a->out, 16)))
    return SANTA_ERR_INVALID_ARG;
  if ((rc = make_plan(a, mode, pl))) return rc;
  const bool variant = a->sampler != SANTA_SAMPLER_IID_HT || a->mix_alpha != 0.f;
  if (sampling && variant) {
    // the variants are implemented where a CTA samples its whole unit in shared memory
    const int G = a->num_q_heads / a->num_kv_heads;
    const int64_t per = ceil_div(a->max_teams, pl->cluster);
    if (a->max_teams > santa::kMaxTeamsPerCta || (G + 1) * per > santa::kPubScores)
      return SANTA_ERR_UNSUPPORTED;
  }
  return SANTA_OK;
}

int launch(const santa_decode_args* a, int mode, cudaStream_t stream) {
  Plan pl;
  int rc = check_and_plan(a, mode, &pl);
  if (rc) return rc;
  const bool sampling = mode == santa::kModeDecode || mode == santa::kModeSample;
  DecodeParams p = {};
  p.q = a->q;
  p.k_pool = a->k_pool;
  p.v_pool = a->v_pool;
  p.reps = sampling ? a->reps : nullptr;
  p.page_table = a->page_table;
  p.seq_lens = a->seq_lens;
  p.batch = a->batch;
  p.num_q_heads = a->num_q_heads;
  p.num_kv_heads = a->num_kv_heads;
  p.team_size = a->team_size;
  p.max_teams = a->max_teams;
  p.num_draws = mode == santa::kModeDense ? 1 : a->num_draws;
  p.num_pages = a->num_pages;
  p.seed = a->seed;
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a->head_dim)));
  p.scale_log2 =
      static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a->head_dim)));
  p.mode = mode;
  p.teams_per_cta = pl.tpc;
  p.clusters_per_unit = pl.clusters;
  p.sampler = sampling ? a->sampler : SANTA_SAMPLER_IID_HT;
  p.mix_alpha = sampling ? a->mix_alpha : 0.f;
  p.out = a->out;
  p.draw_ids = a->draw_ids;
  p.sel_ids = a->sel_ids;
  p.sel_count = a->sel_count;
  p.pi = a->pi;
  p.team_probs = sampling ? a->team_probs : nullptr;
  p.part_ml = pl.part_ml;
  p.part_acc = pl.part_acc;
  p.counters = pl.counters;
  p.status = a->device_status;
  if (a->dtype == SANTA_BF16 && mode != santa::kModeSample) {
    const int64_t rows = a->num_pages * a->num_kv_heads * static_cast<int64_t>(a->team_size);
    if (rows > 0x7fffffffll) return SANTA_ERR_UNSUPPORTED;     // 32-bit row coordinates
    if ((rc = encode_pool_map(&p.tmap_k, a->k_pool, rows, a->head_dim))) return rc;
    if ((rc = encode_pool_map(&p.tmap_v, a->v_pool, rows, a->head_dim))) return rc;
  }
  const dim3 grid(pl.cluster * pl.clusters, a->num_kv_heads, a->batch);
  const int G = a->num_q_heads / a->num_kv_heads;
  if (uses_compact_path(a, mode, pl)) {
    if (compact_variants(a, mode))
      return map_cuda(pl.wide ? santa::decode_launch_bf16_wide_fast_var(p, a->head_dim, G, grid,
                                                                        pl.cluster, stream)
                              : santa::decode_launch_bf16_fast_var(p, a->head_dim, G, grid,
                                                                   pl.cluster, stream));
    return map_cuda(pl.wide ? santa::decode_launch_bf16_wide_fast(p, a->head_dim, G, grid,
                                                                  pl.cluster, stream)
                            : santa::decode_launch_bf16_fast(p, a->head_dim, G, grid,
                                                             pl.cluster, stream));
  }
  const cudaError_t e =
      a->dtype == SANTA_BF16
          ? (pl.wide ? santa::decode_launch_bf16_wide(p, a->head_dim, G, grid, pl.cluster, stream)
                     : santa::decode_launch_bf16(p, a->head_dim, G, grid, pl.cluster, stream))
          : santa::decode_launch_f32(p, a->head_dim, G, grid, pl.cluster, stream);
  return map_cuda(e);
}

int do_reps(const void* k_pool, int dtype, int64_t num_pages, int hkv, int T, int d,
            const int32_t* pages, int64_t num_listed, const int32_t* page_fill, float* reps,
            int32_t* status, cudaStream_t stream) {
  if (dtype != SANTA_F32 && dtype != SANTA_BF16) return SANTA_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return SANTA_ERR_UNSUPPORTED;
  if (T != 64 && T != 128) return SANTA_ERR_UNSUPPORTED;
  if (num_pages < 1 || hkv < 1 || num_listed < 0) return SANTA_ERR_INVALID_ARG;
  if (!k_pool || !reps || !aligned(k_pool, 16) || !aligned(reps, 16))
    return SANTA_ERR_INVALID_ARG;
  if ((page_fill && !aligned(page_fill, 4)) || (status && !aligned(status, 4)))
    return SANTA_ERR_INVALID_ARG;
  RepsParams p;
  p.k_pool = k_pool;
  p.is_bf16 = dtype == SANTA_BF16;
  p.num_pages = num_pages;
  p.num_kv_heads = hkv;
  p.team_size = T;
  p.pages = pages;
  p.num_items = num_listed;
  p.page_fill = page_fill;
  p.reps = reps;
  p.status = status;
  return map_cuda(santa::launch_reps(p, d, stream));
}

}  // namespace

namespace santa {
int check_and_plan_decode(const santa_decode_args* a, int* clusters_per_unit) {
  Plan pl;
  const int rc = check_and_plan(a, kModeDecode, &pl);
  if (rc == SANTA_OK && clusters_per_unit) *clusters_per_unit = pl.clusters;
  return rc;
}
}  // namespace santa

// Only the C ABI is exported (the library is built with -fvisibility=hidden).
#pragma GCC visibility push(default)
extern "C" {

int santa_abi_version(void) { return SANTA_ABI_VERSION; }

const char* santa_status_string(int status) {
  switch (status) {
    case SANTA_OK: return "ok";
    case SANTA_ERR_INVALID_ARG: return "invalid argument (null, misaligned, bad size or short workspace)";
    case SANTA_ERR_UNSUPPORTED: return "unsupported shape (dtype, head_dim, team_size, group, draws or teams), or a sampler variant for a shape sampled across CTAs";
    case SANTA_ERR_CUDA: return "CUDA runtime or launch error";
    case SANTA_ERR_DEVICE_STATUS: return "device status word reported an error";
    case SANTA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than santa_decode_noalloc's static buffer holds";
    default: return "unknown status";
  }
}

int santa_build_reps(const void* k_pool, int dtype, int64_t num_pages, int num_kv_heads,
                     int team_size, int head_dim, const int32_t* page_fill, float* reps,
                     int32_t* device_status, void* stream) {
  return do_reps(k_pool, dtype, num_pages, num_kv_heads, team_size, head_dim, nullptr,
                 num_pages, page_fill, reps, device_status, static_cast<cudaStream_t>(stream));
}

int santa_update_reps(const void* k_pool, int dtype, int64_t num_pages, int num_kv_heads,
                      int team_size, int head_dim, const int32_t* pages, int num_listed,
                      const int32_t* page_fill, float* reps, int32_t* device_status,
                      void* stream) {
  if (!pages || !aligned(pages, 4)) return SANTA_ERR_INVALID_ARG;
  return do_reps(k_pool, dtype, num_pages, num_kv_heads, team_size, head_dim, pages, num_listed,
                 page_fill, reps, device_status, static_cast<cudaStream_t>(stream));
}

size_t santa_attend_vs_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                       int head_dim, int num_draws) {
  if (check_shape(SANTA_F32, batch, num_q_heads, num_kv_heads, head_dim, 64, 1)) return 0;
  if (num_draws < 1 || num_draws > 1024) return 0;
  const size_t units = static_cast<size_t>(batch) * num_kv_heads;
  const size_t G = static_cast<size_t>(num_q_heads / num_kv_heads);
  const size_t ml = round_up(units * num_draws * G * sizeof(float), kAlign);
  return kAlign + 2 * ml + units * num_draws * G * head_dim * sizeof(float);
}

int santa_attend_vs(const santa_decode_args* a, int value_rows, int32_t* value_ids,
                    void* stream) {
  int rc = check_inputs(a);
  if (rc) return rc;
  if (a->num_draws < 1 || a->num_draws > 1024 || value_rows < 1 || value_rows > 256)
    return SANTA_ERR_UNSUPPORTED;
  if (!a->sel_ids || !a->sel_count || !a->pi || !aligned(a->sel_ids, 4) ||
      !aligned(a->sel_count, 4) || !aligned(a->pi, 4))
    return SANTA_ERR_INVALID_ARG;
  if (!a->out || !aligned(a->out, 16) || (value_ids && !aligned(value_ids, 4)))
    return SANTA_ERR_INVALID_ARG;
  const size_t need = santa_attend_vs_workspace_bytes(a->batch, a->num_q_heads, a->num_kv_heads,
                                                      a->head_dim, a->num_draws);
  if (!a->workspace || a->workspace_bytes < need) return SANTA_ERR_INVALID_ARG;
  const size_t units = static_cast<size_t>(a->batch) * a->num_kv_heads;
  const size_t G = static_cast<size_t>(a->num_q_heads / a->num_kv_heads);
  const uintptr_t raw = reinterpret_cast<uintptr_t>(a->workspace);
  unsigned char* base = reinterpret_cast<unsigned char*>(round_up(raw, kAlign));
  const size_t ml = round_up(units * a->num_draws * G * sizeof(float), kAlign);
  santa::VsLaunch l;
  l.q = a->q;
  l.k_pool = a->k_pool;
  l.v_pool = a->v_pool;
  l.page_table = a->page_table;
  l.seq_lens = a->seq_lens;
  l.sel_ids = a->sel_ids;
  l.sel_count = a->sel_count;
  l.pi = a->pi;
  l.bf16 = a->dtype == SANTA_BF16;
  l.batch = a->batch;
  l.num_q_heads = a->num_q_heads;
  l.num_kv_heads = a->num_kv_heads;
  l.head_dim = a->head_dim;
  l.team_size = a->team_size;
  l.max_teams = a->max_teams;
  l.num_draws = a->num_draws;
  l.value_rows = value_rows;
  l.num_pages = a->num_pages;
  l.seed = a->seed;
  l.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a->head_dim)));
  l.part_m = reinterpret_cast<float*>(base);
  l.part_z = reinterpret_cast<float*>(base + ml);
  l.part_acc = reinterpret_cast<float*>(base + 2 * ml);
  l.value_ids = value_ids;
  l.out = a->out;
  l.status = a->device_status;
  return map_cuda(santa::launch_value_sampled(l, static_cast<cudaStream_t>(stream)));
}

int santa_append_kv(const void* k_new, const void* v_new, int dtype, int batch,
                    int num_kv_heads, int team_size, int head_dim, int max_teams,
                    int64_t num_pages, const int32_t* page_table, const int32_t* seq_lens,
                    void* k_pool, void* v_pool, float* reps, int32_t* seq_lens_next,
                    int32_t* device_status, void* stream) {
  if (dtype != SANTA_F32 && dtype != SANTA_BF16) return SANTA_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return SANTA_ERR_UNSUPPORTED;
  if (team_size != 64 && team_size != 128) return SANTA_ERR_UNSUPPORTED;
  if (batch < 1 || num_kv_heads < 1 || max_teams < 1 || num_pages < 1)
    return SANTA_ERR_INVALID_ARG;
  if (max_teams > kMaxTeams) return SANTA_ERR_UNSUPPORTED;
  if (!k_new || !v_new || !page_table || !seq_lens || !k_pool || !v_pool || !reps)
    return SANTA_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pool, 16) ||
      !aligned(v_pool, 16) || !aligned(reps, 16) || !aligned(page_table, 4) ||
      !aligned(seq_lens, 4))
    return SANTA_ERR_INVALID_ARG;
  if ((seq_lens_next && !aligned(seq_lens_next, 4)) ||
      (device_status && !aligned(device_status, 4)))
    return SANTA_ERR_INVALID_ARG;
  if (seq_lens_next == seq_lens) return SANTA_ERR_INVALID_ARG;   // read while written
  santa::AppendParams p;
  p.k_new = k_new;
  p.v_new = v_new;
  p.is_bf16 = dtype == SANTA_BF16;
  p.batch = batch;
  p.num_kv_heads = num_kv_heads;
  p.team_size = team_size;
  p.max_teams = max_teams;
  p.num_pages = num_pages;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.reps = reps;
  p.seq_lens_next = seq_lens_next;
  p.status = device_status;
  return map_cuda(santa::launch_append(p, head_dim, static_cast<cudaStream_t>(stream)));
}

size_t santa_decode_workspace_bytes(int dtype, int batch, int num_q_heads, int num_kv_heads,
                                    int head_dim, int team_size, int max_teams, int num_draws) {
  return default_ws_bytes(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size,
                          max_teams, num_draws, santa::kModeDecode);
}

size_t santa_decode_workspace_min_bytes(int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int team_size, int max_teams,
                                        int num_draws) {
  if (check_shape(SANTA_F32, batch, num_q_heads, num_kv_heads, head_dim, team_size, max_teams))
    return 0;
  if (num_draws < 1 || num_draws > kMaxDraws) return 0;
  // with the largest cluster, a unit needs ceil(chunks / (16 * kMaxChunksPerSplit)) clusters
  const int64_t units = static_cast<int64_t>(batch) * num_kv_heads;
  const int64_t cmax = chunks_max_of(team_size, max_teams, num_draws, santa::kModeDecode);
  const int64_t nc = ceil_div(cmax, static_cast<int64_t>(santa::kMaxCluster) *
                                        santa::kMaxChunksPerSplit);
  return ws_bytes_for(units, num_q_heads / num_kv_heads, head_dim, static_cast<int>(nc));
}

size_t santa_dense_workspace_bytes(int dtype, int batch, int num_q_heads, int num_kv_heads,
                                   int head_dim, int team_size, int max_teams) {
  return default_ws_bytes(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size,
                          max_teams, 1, santa::kModeDense);
}

int santa_decode_plan(const santa_decode_args* a, int which, int32_t* out) {
  if (!a || !out || which < santa::kModeDecode || which > santa::kModeDense)
    return SANTA_ERR_INVALID_ARG;
  int rc = check_shape(a->dtype, a->batch, a->num_q_heads, a->num_kv_heads, a->head_dim,
                       a->team_size, a->max_teams);
  if (rc) return rc;
  if (which != santa::kModeDense && (a->num_draws < 1 || a->num_draws > kMaxDraws))
    return SANTA_ERR_UNSUPPORTED;
  Plan pl;
  if ((rc = make_plan(a, which, &pl))) return rc;
  out[0] = pl.cluster;
  out[1] = pl.clusters;
  out[2] = pl.tpc;
  out[3] = max_clusters(a->dtype == SANTA_BF16, a->head_dim, a->num_q_heads / a->num_kv_heads,
                        pl.cluster, pl.wide);
  out[4] = pl.wide ? 1 : 0;
  return SANTA_OK;
}

int santa_decode_path(const santa_decode_args* a) {
  if (!a) return -SANTA_ERR_INVALID_ARG;
  int rc = check_shape(a->dtype, a->batch, a->num_q_heads, a->num_kv_heads, a->head_dim,
                       a->team_size, a->max_teams);
  if (rc) return -rc;
  if (a->num_draws < 1 || a->num_draws > kMaxDraws) return -SANTA_ERR_UNSUPPORTED;
  Plan pl;
  if ((rc = make_plan(a, santa::kModeDecode, &pl))) return -rc;
  return uses_compact_path(a, santa::kModeDecode, pl) ? 1 : 0;
}

int santa_sample(const santa_decode_args* a, void* stream) {
  return launch(a, santa::kModeSample, static_cast<cudaStream_t>(stream));
}

int santa_attend(const santa_decode_args* a, void* stream) {
  return launch(a, santa::kModeAttend, static_cast<cudaStream_t>(stream));
}

int santa_decode(const santa_decode_args* a, void* stream) {
  return launch(a, santa::kModeDecode, static_cast<cudaStream_t>(stream));
}

int santa_dense_decode(const santa_decode_args* a, void* stream) {
  return launch(a, santa::kModeDense, static_cast<cudaStream_t>(stream));
}

int santa_host_copy_route(const void* host, const void* dev, size_t bytes) {
  return bytes && host && dev && mapped_host(host, dev, bytes) ? 1 : 0;
}

int santa_decode_host(const santa_decode_args* a, const void* host_in, void* dev_in,
                      size_t in_bytes, void* host_out, const void* dev_out, size_t out_bytes,
                      void* stream) {
  if (!a || (in_bytes && (!host_in || !dev_in)) || (out_bytes && (!host_out || !dev_out)))
    return SANTA_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (in_bytes) {
    const void* src = mapped_host(host_in, dev_in, in_bytes);
    const cudaError_t e =
        src ? santa::launch_stage_in(src, dev_in, in_bytes, s)
            : cudaMemcpyAsync(dev_in, host_in, in_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return SANTA_ERR_CUDA;
  }
  const int rc = launch(a, santa::kModeDecode, s);
  if (rc != SANTA_OK) return rc;
  if (out_bytes) {
    void* dst = const_cast<void*>(mapped_host(host_out, dev_out, out_bytes));
    const cudaError_t e =
        dst ? santa::launch_stage_out(dev_out, dst, out_bytes, s)
            : cudaMemcpyAsync(host_out, dev_out, out_bytes, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return SANTA_ERR_CUDA;
  }
  return cudaStreamSynchronize(s) == cudaSuccess ? SANTA_OK : SANTA_ERR_CUDA;
}

}  // extern "C"
#pragma GCC visibility pop
