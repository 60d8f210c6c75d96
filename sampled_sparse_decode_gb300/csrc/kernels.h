// kernels.h — parameter blocks and launchers of the SANTA++ kernels (internal to libsanta).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace santa {

// ---------------------------------------------------------------- representatives
struct RepsParams {
  const void* k_pool;       // [P][Hkv][T][d]
  bool is_bf16;
  int64_t num_pages;
  int num_kv_heads;
  int team_size;
  const int32_t* pages;     // listed page ids, or nullptr for pages 0..num_items-1
  int64_t num_items;        // listed pages (or num_pages)
  const int32_t* page_fill; // [P] or nullptr
  float* reps;              // [P][Hkv][d]
  int32_t* status;
};
cudaError_t launch_reps(const RepsParams& p, int head_dim, cudaStream_t stream);

// ---------------------------------------------------------------- value-row sampling
struct VsLaunch {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* sel_ids;
  const int32_t* sel_count;
  const float* pi;
  bool bf16;
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int team_size;
  int max_teams;
  int num_draws;
  int value_rows;
  int64_t num_pages;
  uint64_t seed;
  float scale;
  float* part_m;
  float* part_z;
  float* part_acc;
  int32_t* value_ids;
  float* out;
  int32_t* status;
};
cudaError_t launch_value_sampled(const VsLaunch& l, cudaStream_t stream);

// ---------------------------------------------------------------- token append
struct AppendParams {
  const void* k_new;        // [B][Hkv][d]
  const void* v_new;        // [B][Hkv][d]
  bool is_bf16;
  int batch;
  int num_kv_heads;
  int team_size;
  int max_teams;
  int64_t num_pages;
  const int32_t* page_table;  // [B][max_teams]
  const int32_t* seq_lens;    // [B] current lengths: the new token goes to position L
  void* k_pool;
  void* v_pool;
  float* reps;                // [P][Hkv][d]
  int32_t* seq_lens_next;     // [B] L + 1, or nullptr
  int32_t* status;
};
cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream);

// ---------------------------------------------------------------- host slabs of santa_decode_host
// bytes / 16 words from src to dst (both 16-byte aligned; one of them host memory mapped into
// the device's address space).  stage-in lets the next launch be scheduled early; stage-out
// is a programmatic dependent of the previous launch and reads nothing before it completed.
cudaError_t launch_stage_in(const void* src, void* dst, size_t bytes, cudaStream_t stream);
cudaError_t launch_stage_out(const void* src, void* dst, size_t bytes, cudaStream_t stream);

// ---------------------------------------------------------------- fused decode step
constexpr int kModeDecode = 0;   // sample, then attend over the sampled teams
constexpr int kModeSample = 1;   // sample only
constexpr int kModeAttend = 2;   // attend over the caller's sel_ids / sel_count / pi
constexpr int kModeDense = 3;    // attend over every team with weight 1

struct DecodeParams {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const float* reps;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int batch, num_q_heads, num_kv_heads, team_size, max_teams, num_draws;
  int64_t num_pages;
  uint64_t seed;
  float scale;              // 1/sqrt(d): representative scores (natural base)
  float scale_log2;         // log2(e)/sqrt(d): in-team scores (base 2)
  int mode;                 // kMode*
  int teams_per_cta;        // sampling: ceil(max_teams / cluster size) <= kMaxTeamsPerCta
  int clusters_per_unit;    // NC
  int sampler;              // SANTA_SAMPLER_*
  float mix_alpha;          // q = (1 - alpha) p + alpha / n
  float* out;               // [B][Hq][d]
  int32_t* draw_ids;        // [B*Hkv][M]
  int32_t* sel_ids;         // [B*Hkv][M]  (read in attend mode)
  int32_t* sel_count;       // [B*Hkv]     (read in attend mode)
  float* pi;                // [B*Hkv][M]  (read in attend mode)
  float* team_probs;        // [B*Hkv][max_teams] or nullptr
  float* part_ml;           // NC > 1: [B*Hkv][NC][G][2]
  float* part_acc;          // NC > 1: [B*Hkv][NC][G][d]
  uint32_t* counters;       // NC > 1: [B*Hkv], zero between calls
  int32_t* status;
  // bf16 attending modes: 2-D tensor maps of the K and V pools viewed as
  // [P*Hkv*T rows][d] with 64-row x 64-element boxes and 128-byte swizzle
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
};

cudaError_t decode_launch_bf16(const DecodeParams& p, int head_dim, int group, dim3 grid,
                               int cluster, cudaStream_t stream);
cudaError_t decode_launch_f32(const DecodeParams& p, int head_dim, int group, dim3 grid,
                              int cluster, cudaStream_t stream);
int decode_resident_bf16(int head_dim, int group);
int decode_resident_f32(int head_dim, int group);
int decode_max_clusters_bf16(int head_dim, int group, int cluster);
int decode_max_clusters_f32(int head_dim, int group, int cluster);
// wide variant (bf16 only): one CTA per SM, six stages, two warp groups
cudaError_t decode_launch_bf16_wide(const DecodeParams& p, int head_dim, int group, dim3 grid,
                                    int cluster, cudaStream_t stream);
int decode_resident_bf16_wide(int head_dim, int group);
int decode_max_clusters_bf16_wide(int head_dim, int group, int cluster);
// compact path (bf16 decode steps with one cluster per unit, every team sampled in each CTA;
// these instantiations: i.i.d. Horvitz-Thompson draws, no mixture): launchers of both
// variants, the shape test and the resident CTAs per SM (the plan is made for the general
// kernel's)
cudaError_t decode_launch_bf16_fast(const DecodeParams& p, int head_dim, int group, dim3 grid,
                                    int cluster, cudaStream_t stream);
cudaError_t decode_launch_bf16_wide_fast(const DecodeParams& p, int head_dim, int group,
                                         dim3 grid, int cluster, cudaStream_t stream);
bool decode_fast_fits_bf16(int head_dim, int group, int max_teams, int cluster, int team_size,
                           int num_draws);
bool decode_fast_fits_bf16_wide(int head_dim, int group, int max_teams, int cluster,
                                int team_size, int num_draws);
int decode_resident_bf16_fast(int head_dim, int group);
int decode_resident_bf16_wide_fast(int head_dim, int group);
// the compact path with the sampler variants compiled in (systematic, Hansen-Hurwitz, the
// defensive mixture): separate instantiations, so the default sampler's prologue stays short
cudaError_t decode_launch_bf16_fast_var(const DecodeParams& p, int head_dim, int group,
                                        dim3 grid, int cluster, cudaStream_t stream);
cudaError_t decode_launch_bf16_wide_fast_var(const DecodeParams& p, int head_dim, int group,
                                             dim3 grid, int cluster, cudaStream_t stream);
int decode_resident_bf16_fast_var(int head_dim, int group);
int decode_resident_bf16_wide_fast_var(int head_dim, int group);

// Every host-side check santa_decode makes on `a`, then its launch plan; launches nothing
// and touches no device memory.  On SANTA_OK *clusters_per_unit receives the plan's NC (> 1:
// the partials and arrival counters go through a->workspace).
int check_and_plan_decode(const santa_decode_args* a, int* clusters_per_unit);

}  // namespace santa
