// santa_noalloc.cu — santa_decode for callers that cannot allocate device memory.
//
// santa_decode needs a caller-provided workspace for its split-K partials and arrival
// counters.  Some callers cannot obtain one: code that runs where cudaMalloc is forbidden
// or unavailable (a plug-in inside an inference engine that owns all device memory and
// hands out none after start-up, a real-time loop that must not allocate once running,
// or a runtime whose allocator is not reachable from C).  santa_decode_noalloc serves them
// with a scratch buffer that lives in this library's own device image: a file-scope
// __device__ array, created when the library's module is loaded on a device and held until
// the process exits.  The call itself allocates nothing.
#include <mutex>

#include "kernels.h"

// Upper bound of the scratch this entry point can use.  4 MiB holds the default split plan
// of every workload in this repository (about 1 MiB each); larger problems run with fewer,
// longer splits, and problems whose minimum need exceeds it are rejected.
static constexpr size_t kStaticScratchBytes = size_t(4) << 20;

// The scratch itself: zero-initialised when the module loads on a device.  In host code
// this name is only a stand-in; kernels get the address from scratch_address().
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

// Device address of g_static_scratch on each device, looked up once per device (the host
// symbol itself is only a stand-in and must never be handed to a kernel).
void* scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

// Only the C ABI is exported (the library is built with -fvisibility=hidden).
#pragma GCC visibility push(default)
extern "C" int santa_decode_noalloc(const santa_decode_args* a, void* stream) {
  if (!a) return SANTA_ERR_INVALID_ARG;
  // 1. Size checks, before any CUDA call: the shape's minimum split scratch, and the arrival
  //    counters (one 32-bit word per unit, padded to 256 bytes), must both fit the array.
  const size_t need = santa_decode_workspace_min_bytes(a->batch, a->num_q_heads,
                                                       a->num_kv_heads, a->head_dim,
                                                       a->team_size, a->max_teams,
                                                       a->num_draws);
  if (need == 0) return SANTA_ERR_UNSUPPORTED;
  const size_t units = static_cast<size_t>(a->batch) * static_cast<size_t>(a->num_kv_heads);
  const size_t counters = (units * sizeof(uint32_t) + 255) / 256 * 256;
  if (need > kStaticScratchBytes || counters + 256 > kStaticScratchBytes)
    return SANTA_ERR_SCRATCH_LIMIT;
  void* scratch = scratch_address();
  if (!scratch) return SANTA_ERR_CUDA;
  santa_decode_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = kStaticScratchBytes;
  // 2. Every argument check and the launch plan, still without touching the array.
  int clusters = 1;
  const int rc = santa::check_and_plan_decode(&b, &clusters);
  if (rc != SANTA_OK) return rc;
  // 3. The array keeps the previous call's contents.  Partials are always written before
  //    they are read; the arrival counters (at the array's start: it is 256-byte aligned,
  //    so the plan puts them at offset 0) are used only when several clusters share a unit,
  //    and must then start at zero.  Clear them on the call's stream.
  if (clusters > 1 &&
      cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SANTA_ERR_CUDA;
  return santa_decode(&b, stream);
}

extern "C" size_t santa_noalloc_scratch_bytes(void) { return kStaticScratchBytes; }
#pragma GCC visibility pop
