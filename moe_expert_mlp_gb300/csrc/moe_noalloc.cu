// Routing + permutation for callers that cannot allocate device memory.
//
// moe_route_permute needs a small scratch buffer (the per-chunk expert
// histogram) that the caller normally allocates.  Some callers have no way
// to do that: a host program that hands all device memory to its own fixed
// pool, or a runtime that forbids allocation once it is set up.  For them
// moe_route_permute_noalloc uses a scratch array that lives in this library's
// own device memory (a file-scope __device__ array, reserved on every GPU
// that loads the library for as long as the process runs) and otherwise does
// exactly what moe_route_permute does.
//
// Limits and caveats:
//   * the histogram must fit: ceil(T/256) * E * 4 bytes <= kStaticScratchBytes
//     (256 KiB, e.g. T = 65536 tokens with E = 256, or T = 262144 with E = 64);
//     larger problems are rejected with MOE_ERR_WORKSPACE before any work;
//   * every call on a device shares the one array, so two calls whose work
//     overlaps on the GPU (different streams, no ordering) race on it; calls
//     ordered on one stream are fine (the histogram is zeroed at the start of
//     every call, so nothing left by the previous call is read);
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current; make that first call
//     before any stream capture.  The address is kept for the life of the
//     process, so resetting the device (cudaDeviceReset) after the first
//     call is not supported.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kStaticScratchBytes = 256 * 1024;

// Device-side scratch.  In host code this name is only a handle for the
// runtime; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_route_scratch[kStaticScratchBytes / sizeof(int32_t)];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {};
std::mutex g_scratch_mu;

// Device address of g_route_scratch on the current device (looked up once).
moe_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_permute_noalloc(
    const moe_mlp_desc_t* desc, const float* logits, const float* bias, const void* x,
    int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
    int32_t* padded_offsets, int32_t* tile_prefix, int32_t* row_src, int32_t* row_of,
    void* x_perm, cudaStream_t stream) {
  // the rest of the descriptor is checked by moe_route_permute below
  if (!desc) return MOE_ERR_NULL;
  if (desc->T < 0 || desc->E < 1) return MOE_ERR_SHAPE;
  moe_status_t st;
  const size_t chunks =
      (static_cast<size_t>(desc->T) + moe::kTokensPerChunk - 1) / moe::kTokensPerChunk;
  if (chunks * static_cast<size_t>(desc->E) * sizeof(int32_t) > moe::kStaticScratchBytes)
    return MOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = moe::scratch_for_current_device(&scratch)) != MOE_OK) return st;
  return moe_route_permute(desc, logits, bias, x, topk_idx, topk_w, counts, offsets,
                           padded_offsets, tile_prefix, row_src, row_of, x_perm, scratch,
                           moe::kStaticScratchBytes, stream);
}
