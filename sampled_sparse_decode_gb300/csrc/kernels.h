// kernels.h — parameter blocks and launchers of the SANTA++ kernels (internal to libsanta).
#pragma once

#include <cstdint>
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

// ---------------------------------------------------------------- score + sample
struct SampleParams {
  const void* q;
  const float* reps;
  const int32_t* page_table;
  const int32_t* seq_lens;
  bool is_bf16;
  int batch, num_q_heads, num_kv_heads, group, team_size, max_teams, num_draws;
  int64_t num_pages;
  uint64_t seed;
  float scale;              // 1/sqrt(d)
  int teams_per_cta;        // shared-memory capacity: ceil(max_teams / cluster size)
  int32_t* draw_ids;
  int32_t* sel_ids;
  int32_t* sel_count;
  float* pi;
  float* team_probs;        // may be nullptr
  uint32_t* counters;       // [B*Hkv] split-arrival counters to reset (may be nullptr)
  int32_t* status;
};
size_t sample_smem_bytes(int head_dim, int teams_per_cta);
cudaError_t launch_sample(const SampleParams& p, int head_dim, int cluster, cudaStream_t stream);

// ---------------------------------------------------------------- split-K attention
struct AttendParams {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* sel_ids;   // sampled mode: [B*Hkv][M]
  const int32_t* sel_count; // sampled mode: [B*Hkv]
  const float* pi;          // sampled mode: [B*Hkv][M]
  int batch, num_q_heads, num_kv_heads, team_size, max_teams, num_draws;
  int64_t num_pages;
  float scale_log2;         // log2(e) / sqrt(d): scores live in the base-2 domain
  int dense;                // 1: every token of every team, weight 1
  int chunks_per_split;     // 64-token chunks handled by one CTA
  int max_splits;           // splits held per unit by the workspace
  float* part_ml;           // [B*Hkv][max_splits][G][2]  (running max, running sum)
  float* part_acc;          // [B*Hkv][max_splits][G][d]
  uint32_t* counters;       // [B*Hkv] arrival counters, zero between calls
  float* out;               // [B][Hq][d]
  int32_t* status;
};
struct AttendShape {
  bool is_bf16;
  int head_dim;
  int group;
};
size_t attend_smem_bytes(const AttendShape& s);
cudaError_t launch_attend(const AttendParams& p, const AttendShape& s, dim3 grid,
                          bool programmatic, cudaStream_t stream);
// per-dtype launchers (one translation unit each)
cudaError_t launch_attend_bf16(const AttendParams& p, int head_dim, int group, dim3 grid,
                               bool programmatic, cudaStream_t stream);
cudaError_t launch_attend_f32(const AttendParams& p, int head_dim, int group, dim3 grid,
                              bool programmatic, cudaStream_t stream);
size_t attend_smem_bytes_bf16(int head_dim, int group);
size_t attend_smem_bytes_f32(int head_dim, int group);
int attend_resident_ctas(const AttendShape& s);
int attend_resident_ctas_bf16(int head_dim, int group);
int attend_resident_ctas_f32(int head_dim, int group);

}  // namespace santa
