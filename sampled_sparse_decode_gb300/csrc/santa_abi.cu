// santa_abi.cu — the extern "C" entry points of libsanta.so (declared in include/santa.h):
// argument checks, the split plan and workspace layout, and the kernel launches.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.h"

namespace {

using santa::AttendParams;
using santa::AttendShape;
using santa::RepsParams;
using santa::SampleParams;

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
  if (!a->sel_ids || !a->sel_count || !a->pi) return SANTA_ERR_INVALID_ARG;
  if (!aligned(a->sel_ids, 4) || !aligned(a->sel_count, 4) || !aligned(a->pi, 4))
    return SANTA_ERR_INVALID_ARG;
  return SANTA_OK;
}

// ---------------------------------------------------------------- workspace and split plan
//
// Workspace layout (base rounded up to 256 bytes):
//   counters  [B*Hkv] uint32                      (rounded up to 256 bytes)
//   part_ml   [B*Hkv][cap][G][2] fp32 (m, l)       (rounded up to 256 bytes)
//   part_acc  [B*Hkv][cap][G][d] fp32
// where cap, the splits a unit may use, is whatever the given size holds.

size_t counters_bytes(int64_t units) { return round_up(static_cast<size_t>(units) * 4, kAlign); }
size_t split_bytes(int64_t units, int G, int d) {
  return static_cast<size_t>(units) * G * (d + 2) * sizeof(float) + kAlign;
}
size_t ws_bytes_for(int64_t units, int G, int d, int splits) {
  return kAlign + counters_bytes(units) +
         round_up(static_cast<size_t>(units) * splits * G * 2 * sizeof(float), kAlign) +
         static_cast<size_t>(units) * splits * G * d * sizeof(float);
}

int64_t chunks_max_of(int T, int max_teams, int M, bool dense) {
  const int64_t teams = dense ? max_teams : std::min(M, max_teams);
  return teams * (T / santa::kChunk);
}

// Splits needed so that no CTA owns more than kMaxChunksPerSplit chunks.
int64_t min_splits_of(int64_t chunks_max) {
  return ceil_div(chunks_max, santa::kMaxChunksPerSplit);
}

// Resident attention CTAs per SM for a shape (cached per device and shape).
int resident_ctas(bool bf16, int d, int G) {
  static std::mutex mu;
  static int cache[64][2][2][santa::kMaxGroup + 1] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  int& c = cache[dev][bf16 ? 1 : 0][d == 128 ? 1 : 0][G];
  if (!c) c = std::max(1, santa::attend_resident_ctas(santa::AttendShape{bf16, d, G}));
  return c;
}

// Default split: one wave of resident CTAs over the whole job, i.e. each unit gets
// floor(SMs * resident / units) splits (at least one, at most kMaxSplits).
void default_split(int64_t units, int64_t chunks_max, int sms, int resident, int64_t* cps,
                   int64_t* splits) {
  const int64_t slots = std::max<int64_t>(1, static_cast<int64_t>(sms) * resident);
  const int64_t per_unit = std::min<int64_t>(santa::kMaxSplits, std::max<int64_t>(1, slots / units));
  *cps = std::max<int64_t>(ceil_div(chunks_max, per_unit), 1);
  *cps = std::min<int64_t>(*cps, santa::kMaxChunksPerSplit);
  *splits = ceil_div(chunks_max, *cps);
}

struct Plan {
  int chunks_per_split = 1;
  int splits = 1;
  int cap = 0;
  uint32_t* counters = nullptr;
  float* part_ml = nullptr;
  float* part_acc = nullptr;
};

int make_plan(const santa_decode_args* a, bool dense, Plan* pl) {
  const int64_t units = static_cast<int64_t>(a->batch) * a->num_kv_heads;
  const int G = a->num_q_heads / a->num_kv_heads, d = a->head_dim;
  if (!a->workspace) return SANTA_ERR_INVALID_ARG;
  const uintptr_t raw = reinterpret_cast<uintptr_t>(a->workspace);
  const uintptr_t base = round_up(raw, kAlign);
  const size_t lead = base - raw;
  const size_t fixed = lead + counters_bytes(units);
  if (a->workspace_bytes < fixed + split_bytes(units, G, d)) return SANTA_ERR_INVALID_ARG;
  int64_t cap = static_cast<int64_t>((a->workspace_bytes - fixed - kAlign) /
                                     (static_cast<size_t>(units) * G * (d + 2) * sizeof(float)));
  const int64_t cmax = chunks_max_of(a->team_size, a->max_teams, a->num_draws, dense);
  cap = std::min<int64_t>({cap, cmax, static_cast<int64_t>(santa::kMaxSplits)});
  if (cap < min_splits_of(cmax)) return SANTA_ERR_INVALID_ARG;
  const int sms = current_sms();
  if (sms <= 0) return SANTA_ERR_CUDA;
  int64_t cps, splits;
  default_split(units, cmax, sms, resident_ctas(a->dtype == SANTA_BF16, d, G), &cps, &splits);
  if (splits > cap) {
    cps = ceil_div(cmax, cap);
    splits = ceil_div(cmax, cps);
  }
  pl->chunks_per_split = static_cast<int>(cps);
  pl->splits = static_cast<int>(splits);
  pl->cap = static_cast<int>(cap);
  unsigned char* b = reinterpret_cast<unsigned char*>(base);
  pl->counters = reinterpret_cast<uint32_t*>(b);
  b += counters_bytes(units);
  pl->part_ml = reinterpret_cast<float*>(b);
  b += round_up(static_cast<size_t>(units) * cap * G * 2 * sizeof(float), kAlign);
  pl->part_acc = reinterpret_cast<float*>(b);
  return SANTA_OK;
}

size_t default_ws_bytes(int dtype, int batch, int hq, int hkv, int d, int T, int max_teams,
                        int M, bool dense) {
  if (check_shape(dtype, batch, hq, hkv, d, T, max_teams)) return 0;
  if (!dense && (M < 1 || M > kMaxDraws)) return 0;
  const int64_t units = static_cast<int64_t>(batch) * hkv;
  const int G = hq / hkv;
  const int sms = current_sms();
  if (sms <= 0) return 0;
  const int64_t cmax = chunks_max_of(T, max_teams, M, dense);
  int64_t cps, splits;
  default_split(units, cmax, sms, resident_ctas(dtype == SANTA_BF16, d, G), &cps, &splits);
  return ws_bytes_for(units, G, d, static_cast<int>(splits));
}

// Cluster size of the sampling kernel: enough CTAs that each scores about 32 teams, at most
// 8 (so at most 2048 teams per CTA for the longest supported sequence).
int sample_cluster(int max_teams) {
  int cl = 1;
  while (cl < 8 && cl * 32 < max_teams) cl <<= 1;
  return cl;
}

int do_sample(const santa_decode_args* a, cudaStream_t stream) {
  int rc = check_inputs(a);
  if (rc) return rc;
  if ((rc = check_draws(a))) return rc;
  if (!a->reps || !aligned(a->reps, 16) || !a->draw_ids || !aligned(a->draw_ids, 4))
    return SANTA_ERR_INVALID_ARG;
  if (a->team_probs && !aligned(a->team_probs, 4)) return SANTA_ERR_INVALID_ARG;
  uint32_t* counters = nullptr;
  if (a->workspace) {
    Plan pl;
    if ((rc = make_plan(a, false, &pl))) return rc;
    counters = pl.counters;
  }
  const int cl = sample_cluster(a->max_teams);
  SampleParams p;
  p.q = a->q;
  p.reps = a->reps;
  p.page_table = a->page_table;
  p.seq_lens = a->seq_lens;
  p.is_bf16 = a->dtype == SANTA_BF16;
  p.batch = a->batch;
  p.num_q_heads = a->num_q_heads;
  p.num_kv_heads = a->num_kv_heads;
  p.group = a->num_q_heads / a->num_kv_heads;
  p.team_size = a->team_size;
  p.max_teams = a->max_teams;
  p.num_draws = a->num_draws;
  p.num_pages = a->num_pages;
  p.seed = a->seed;
  p.scale = static_cast<float>(1.0 / std::sqrt(static_cast<double>(a->head_dim)));
  p.teams_per_cta = static_cast<int>(ceil_div(a->max_teams, cl));
  p.draw_ids = a->draw_ids;
  p.sel_ids = a->sel_ids;
  p.sel_count = a->sel_count;
  p.pi = a->pi;
  p.team_probs = a->team_probs;
  p.counters = counters;
  p.status = a->device_status;
  return map_cuda(santa::launch_sample(p, a->head_dim, cl, stream));
}

int do_attend(const santa_decode_args* a, bool dense, bool programmatic, cudaStream_t stream) {
  int rc = check_inputs(a);
  if (rc) return rc;
  if (!dense && (rc = check_draws(a))) return rc;
  if (!a->out || !aligned(a->out, 16)) return SANTA_ERR_INVALID_ARG;
  Plan pl;
  if ((rc = make_plan(a, dense, &pl))) return rc;
  AttendParams p;
  p.q = a->q;
  p.k_pool = a->k_pool;
  p.v_pool = a->v_pool;
  p.page_table = a->page_table;
  p.seq_lens = a->seq_lens;
  p.sel_ids = dense ? nullptr : a->sel_ids;
  p.sel_count = dense ? nullptr : a->sel_count;
  p.pi = dense ? nullptr : a->pi;
  p.batch = a->batch;
  p.num_q_heads = a->num_q_heads;
  p.num_kv_heads = a->num_kv_heads;
  p.team_size = a->team_size;
  p.max_teams = a->max_teams;
  p.num_draws = dense ? 0 : a->num_draws;
  p.num_pages = a->num_pages;
  p.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(a->head_dim)));
  p.dense = dense ? 1 : 0;
  p.chunks_per_split = pl.chunks_per_split;
  p.max_splits = pl.cap;
  p.part_ml = pl.part_ml;
  p.part_acc = pl.part_acc;
  p.counters = pl.counters;
  p.out = a->out;
  p.status = a->device_status;
  AttendShape s{a->dtype == SANTA_BF16, a->head_dim, a->num_q_heads / a->num_kv_heads};
  const dim3 grid(pl.splits, a->num_kv_heads, a->batch);
  return map_cuda(santa::launch_attend(p, s, grid, programmatic, stream));
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

cudaError_t launch_attend(const AttendParams& p, const AttendShape& s, dim3 grid,
                          bool programmatic, cudaStream_t stream) {
  return s.is_bf16 ? launch_attend_bf16(p, s.head_dim, s.group, grid, programmatic, stream)
                   : launch_attend_f32(p, s.head_dim, s.group, grid, programmatic, stream);
}

int attend_resident_ctas(const AttendShape& s) {
  return s.is_bf16 ? attend_resident_ctas_bf16(s.head_dim, s.group)
                   : attend_resident_ctas_f32(s.head_dim, s.group);
}

size_t attend_smem_bytes(const AttendShape& s) {
  return s.is_bf16 ? attend_smem_bytes_bf16(s.head_dim, s.group)
                   : attend_smem_bytes_f32(s.head_dim, s.group);
}

}  // namespace santa

extern "C" {

int santa_abi_version(void) { return SANTA_ABI_VERSION; }

const char* santa_status_string(int status) {
  switch (status) {
    case SANTA_OK: return "ok";
    case SANTA_ERR_INVALID_ARG: return "invalid argument (null, misaligned, bad size or short workspace)";
    case SANTA_ERR_UNSUPPORTED: return "unsupported shape (dtype, head_dim, team_size, group, draws or teams)";
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

size_t santa_decode_workspace_bytes(int dtype, int batch, int num_q_heads, int num_kv_heads,
                                    int head_dim, int team_size, int max_teams, int num_draws) {
  return default_ws_bytes(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size,
                          max_teams, num_draws, false);
}

size_t santa_decode_workspace_min_bytes(int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int team_size, int max_teams,
                                        int num_draws) {
  if (check_shape(SANTA_F32, batch, num_q_heads, num_kv_heads, head_dim, team_size, max_teams))
    return 0;
  if (num_draws < 1 || num_draws > kMaxDraws) return 0;
  const int64_t units = static_cast<int64_t>(batch) * num_kv_heads;
  const int64_t splits = min_splits_of(chunks_max_of(team_size, max_teams, num_draws, false));
  return kAlign + counters_bytes(units) +
         static_cast<size_t>(splits) * (split_bytes(units, num_q_heads / num_kv_heads, head_dim) -
                                        kAlign) + kAlign;
}

size_t santa_dense_workspace_bytes(int dtype, int batch, int num_q_heads, int num_kv_heads,
                                   int head_dim, int team_size, int max_teams) {
  return default_ws_bytes(dtype, batch, num_q_heads, num_kv_heads, head_dim, team_size,
                          max_teams, 1, true);
}

int santa_sample(const santa_decode_args* a, void* stream) {
  return do_sample(a, static_cast<cudaStream_t>(stream));
}

int santa_attend(const santa_decode_args* a, void* stream) {
  return do_attend(a, false, false, static_cast<cudaStream_t>(stream));
}

int santa_decode(const santa_decode_args* a, void* stream) {
  if (!a || !a->workspace) return SANTA_ERR_INVALID_ARG;
  int rc = do_sample(a, static_cast<cudaStream_t>(stream));
  if (rc) return rc;
  return do_attend(a, false, true, static_cast<cudaStream_t>(stream));
}

int santa_dense_decode(const santa_decode_args* a, void* stream) {
  return do_attend(a, true, false, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
