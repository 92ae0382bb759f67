// C-ABI entry points of libmoe: argument checks, TMA tensor-map encoding
// and kernel launches.  See include/moe.h for the contract of each call.
//
// Nothing here allocates device memory, synchronises, or reads device data
// on the host (except moe_read_device_status, which exists to do exactly
// that outside any graph), so every call can be captured in a CUDA graph
// ("Improving MoE training throughput with advanced fused kernels",
// "Eliminating host-device synchronisation and CPU launch overhead").
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <mutex>

#include "moe_internal.h"
#include "moe_mx.cuh"
#include "moe_ptx.cuh"

namespace moe {

// Sticky device status word (one per device that loaded the library).
__device__ int g_status_word;

namespace {

// One CTA waits, with the pipelines' bounded wait, on an mbarrier phase that
// nothing completes; the wait gives up after limit_ns and records a timeout.
__global__ void k_wait_selftest(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, &abort_flag, limit_ns);
}

// One CTA arrives at a grid barrier that expects a second arrival nobody
// makes (the fused router's barrier); the wait gives up after limit_ns and
// records a timeout.
__device__ unsigned int g_selftest_grid_ctr;

__global__ void k_grid_wait_selftest(int* status, unsigned long long limit_ns) {
  __shared__ int fail;
  if (threadIdx.x == 0) {
    fail = 0;
    g_selftest_grid_ctr = 0;
  }
  grid_sync(&g_selftest_grid_ctr, 2u, status, &fail, limit_ns);
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int major = 0, minor = 0;
  int* status = nullptr;
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

moe_status_t device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    if (cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MOE_ERR_CUDA;
    di.status = static_cast<int*>(p);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return MOE_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    di.ready = true;
  }
  if (di.major != 10 || di.minor != 3) return MOE_ERR_ARCH;
  *out = &di;
  return MOE_OK;
}

// 3-D bf16 tensor map with 128-byte swizzle.  dims innermost first; the
// innermost dimension is contiguous; row_bytes / plane_bytes are the strides
// of dims 1 and 2.  Out-of-range box elements read as zero.
bool encode_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                uint64_t row_bytes, uint64_t plane_bytes, uint32_t box0, uint32_t box1,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B,
                CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (row_bytes & 15) || (plane_bytes & 15))
    return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {row_bytes, plane_bytes};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estride[3] = {1, 1, 1};
  CUresult r = g_encode(map, dtype, 3, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

moe_status_t check_desc(const moe_mlp_desc_t* d, bool need_tokens) {
  if (!d) return MOE_ERR_NULL;
  if (d->E < 1 || d->E > kMaxExperts) return MOE_ERR_SHAPE;
  if (d->d < 64 || d->d % 64 != 0) return MOE_ERR_SHAPE;
  if (d->F < 32 || d->F % 32 != 0) return MOE_ERR_SHAPE;
  if (d->align != kAlign) return MOE_ERR_UNSUPPORTED;
  if (d->dtype != MOE_DTYPE_BF16 && d->dtype != MOE_DTYPE_MXFP8 && d->dtype != MOE_DTYPE_NVFP4 &&
      d->dtype != MOE_DTYPE_FP32)
    return MOE_ERR_UNSUPPORTED;
  if (d->act != MOE_ACT_SWIGLU && d->act != MOE_ACT_GEGLU && d->act != MOE_ACT_SREGLU &&
      d->act != MOE_ACT_SRELU)
    return MOE_ERR_UNSUPPORTED;
  if (d->capacity < kAlign || d->capacity % kAlign != 0) return MOE_ERR_SHAPE;
  if (d->sm_margin < 0) return MOE_ERR_SHAPE;
  if (need_tokens) {
    if (d->T < 0 || d->k < 1 || d->k > kMaxTopK || d->k > d->E) return MOE_ERR_SHAPE;
    const long long need = static_cast<long long>(d->T) * d->k +
                           static_cast<long long>(d->E) * (kAlign - 1);
    if (d->capacity < need) return MOE_ERR_SHAPE;
  }
  return MOE_OK;
}

// Calls whose tensors are bf16 (every GEMM call without a type suffix, and
// the quantizers of bf16 tensors): not for a descriptor of fp32 tensors.
moe_status_t check_bf16_desc(const moe_mlp_desc_t* d, bool need_tokens = false) {
  moe_status_t st = check_desc(d, need_tokens);
  if (st != MOE_OK) return st;
  return d->dtype == MOE_DTYPE_FP32 ? MOE_ERR_UNSUPPORTED : MOE_OK;
}

// Bytes per element of the activation, weight and gradient tensors.
size_t act_bytes(const moe_mlp_desc_t* d) { return d->dtype == MOE_DTYPE_FP32 ? 4 : 2; }

// Workspace of the fp32 backward (moe_mlp_bwd with MOE_DTYPE_FP32): the
// transposed weights W1p^T [E][d][W1] and W2^T [E][F][d], and the transposed
// activations x_perm^T, dY^T [d][cap], A^T [F][cap], dH^T [W1][cap], each
// rounded up to 256 bytes.
size_t tf32_bwd_ws_bytes(const moe_mlp_desc_t* d) {
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t E = d->E, dm = d->d, F = d->F, W1 = fc1_width(d->act, d->F), cap = d->capacity;
  return r(E * dm * W1 * 4) + r(E * F * dm * 4) + 2 * r(dm * cap * 4) + r(F * cap * 4) +
         r(W1 * cap * 4);
}

moe_status_t mlp_fwd_tf32(const moe_mlp_desc_t* desc, const void* x_perm, const int32_t* counts,
                          const int32_t* padded_offsets, const void* w1p, const void* b1p,
                          const void* w2, const void* b2, void* h, void* a, void* y,
                          const moe_mx_out_t* a_mx, const moe_mx_out_t* y_mx,
                          cudaStream_t stream);
moe_status_t mlp_bwd_tf32(const moe_mlp_desc_t* desc, const void* dy, const void* x_perm,
                          const void* h, const void* a, const int32_t* counts,
                          const int32_t* padded_offsets, const void* w1p, const void* b1p,
                          const void* w2, void* dh, void* dx_perm, void* dw1p, void* db1p,
                          void* dw2, void* db2, const moe_mx_out_t* dh_mx, void* ws,
                          size_t ws_bytes, cudaStream_t stream);

int grid_for(const DeviceInfo* di, const moe_mlp_desc_t* d) {
  int g = di->sms - d->sm_margin;
  return g < 1 ? 1 : g;
}

size_t route_ws_bytes(const moe_mlp_desc_t* d) {
  const size_t nchunks = (static_cast<size_t>(d->T) + kTokensPerChunk - 1) / kTokensPerChunk;
  return (nchunks * d->E * sizeof(int32_t) + 255) / 256 * 256;
}

// MN-major operand [E][K rows][W] (W contiguous, W % 64 == 0) viewed as
// [E][W/64 atoms][K][64] so that one box {64, 64 rows, atoms, 1} fetches
// several 64-column atoms; the atom stride (128 B) is smaller than the row
// stride.  Returns false if the driver does not accept the view.
bool encode_mn_atoms(CUtensorMap* map, const void* base, uint64_t W, uint64_t K, uint64_t E,
                     uint64_t row_bytes, uint64_t plane_bytes, uint32_t atoms) {
  if (W % 64 != 0 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[4] = {64, K, W / 64, E};
  cuuint64_t strides[3] = {row_bytes, 128, plane_bytes};
  cuuint32_t box[4] = {64, 64, atoms, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims,
                        strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Output [E][rows][W] viewed as [E][W/32][rows][32]: box {32, 128, 2, 1}
// stores two adjacent 32-column chunks staged back to back.
bool encode_out2(CUtensorMap* map, const void* base, uint64_t W, uint64_t rows, uint64_t E) {
  if (W % 32 != 0 || (reinterpret_cast<uintptr_t>(base) & 15)) return false;
  cuuint64_t dims[4] = {32, rows, W / 32, E};
  cuuint64_t strides[3] = {W * 2, 64, rows * W * 2};
  cuuint32_t box[4] = {32, 128, 2, 1};
  cuuint32_t estride[4] = {1, 1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map: 32-column x 128-row boxes with 64-byte swizzle (the epilogue
// staging layout).
bool encode_out(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2) {
  return encode_map(map, base, d0, d1, d2, d0 * 2, d1 * d0 * 2, 32, 128,
                    CU_TENSOR_MAP_SWIZZLE_64B);
}

// Copy the optional MX outputs into the kernel arguments; zero the amax.
moe_status_t set_mx(GemmArgs& g, const moe_mx_out_t* mx, long long width, cudaStream_t stream) {
  if (!mx) return MOE_OK;
  if ((mx->q && !mx->scale) || (mx->qt && !mx->scale_t)) return MOE_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(mx->q) & 15) || width % 32 != 0) return MOE_ERR_SHAPE;
  if (mx->layout != MOE_MX_SCALES_ROWMAJOR && mx->layout != MOE_MX_SCALES_MMA)
    return MOE_ERR_UNSUPPORTED;
  g.mx_mma_layout = mx->layout == MOE_MX_SCALES_MMA;
  g.mx_q = mx->q;
  g.mx_s = mx->scale;
  g.mx_qt = mx->qt;
  g.mx_st = mx->scale_t;
  g.mx_amax = mx->amax;
  g.mx_width = width;
  if (mx->amax && cudaMemsetAsync(mx->amax, 0, 2 * sizeof(float), stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

void fill_common(GemmArgs& a, const moe_mlp_desc_t* d, const DeviceInfo* di,
                 const int32_t* counts, const int32_t* padded_offsets) {
  memset(&a, 0, sizeof(a));
  a.padded_offsets = padded_offsets;
  a.counts = counts;
  a.status = di->status;
  a.E = d->E;
  a.f_real = d->F;
  a.f_pad = fc1_pad(d->F);
  a.capacity = d->capacity;
  a.act = d->act;
  a.alpha = d->alpha;
  a.limit = d->limit;
  a.lin_off = d->linear_offset;
  a.out_scale = d->out_scale;
}

}  // namespace
}  // namespace moe

namespace moe {
bool encode_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t row_bytes, uint64_t plane_bytes, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle swizzle, CUtensorMapDataType dtype) {
  return g_encode != nullptr &&
         encode_map(map, base, d0, d1, d2, row_bytes, plane_bytes, box0, box1, swizzle, dtype);
}
}  // namespace moe

using namespace moe;

extern "C" {

int32_t moe_fc1_padded_width(int32_t F) { return fc1_pad(F); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_NULL: return "required pointer is NULL";
    case MOE_ERR_SHAPE: return "sizes out of the supported range";
    case MOE_ERR_UNSUPPORTED: return "option not supported";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_ARCH: return "current device is not sm_103";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE: return "device status word is set";
  }
  return "unknown status";
}

moe_status_t moe_workspace_size(const moe_mlp_desc_t* desc, size_t* bytes) {
  if (!desc || !bytes) return MOE_ERR_NULL;
  moe_status_t st = check_desc(desc, false);
  if (st != MOE_OK) return st;
  *bytes = route_ws_bytes(desc) + 256;
  if (desc->recompute_h && desc->act == MOE_ACT_SRELU)   // H regenerated into the workspace
    *bytes += static_cast<size_t>(desc->capacity) * fc1_width(desc->act, desc->F) * 2 + 256;
  if (desc->dtype == MOE_DTYPE_FP32)   // transposed operands of the fp32 backward
    *bytes = (*bytes + 255) / 256 * 256 + tf32_bwd_ws_bytes(desc);
  return MOE_OK;
}

moe_status_t moe_repack_fc1(const moe_mlp_desc_t* desc, const void* w1, const void* b1,
                            void* w1p, void* b1p, cudaStream_t stream) {
  moe_status_t st = check_desc(desc, false);
  if (st != MOE_OK) return st;
  if (!w1 || !w1p) return MOE_ERR_NULL;
  if ((b1 == nullptr) != (b1p == nullptr)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  cudaError_t e;
  const size_t eb = act_bytes(desc);   // rows move as 2-byte units
  if (desc->act == MOE_ACT_SRELU) {   // no halves to interleave: a plain copy
    const size_t n = static_cast<size_t>(desc->E) * desc->F;
    e = cudaMemcpyAsync(w1p, w1, n * desc->d * eb, cudaMemcpyDeviceToDevice, stream);
    if (e == cudaSuccess && b1) e = cudaMemcpyAsync(b1p, b1, n * eb, cudaMemcpyDeviceToDevice, stream);
    return cuda_status(e);
  }
  const int units = static_cast<int>(eb / 2);
  e = launch_repack_fc1(w1, w1p, desc->E, desc->F, desc->d * units, stream);
  if (e == cudaSuccess && b1) e = launch_repack_fc1(b1, b1p, desc->E, desc->F, units, stream);
  return cuda_status(e);
}

moe_status_t moe_unpack_fc1(const moe_mlp_desc_t* desc, const void* w1p, void* w1,
                            int32_t rows_width, cudaStream_t stream) {
  moe_status_t st = check_desc(desc, false);
  if (st != MOE_OK) return st;
  if (!w1p || !w1) return MOE_ERR_NULL;
  if (rows_width < 1) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const size_t eb = act_bytes(desc);
  if (desc->act == MOE_ACT_SRELU)
    return cuda_status(cudaMemcpyAsync(w1, w1p,
                                       static_cast<size_t>(desc->E) * desc->F * rows_width * eb,
                                       cudaMemcpyDeviceToDevice, stream));
  return cuda_status(launch_unpack_fc1(w1p, w1, desc->E, desc->F,
                                       rows_width * static_cast<int>(eb / 2), stream));
}

static moe_status_t route_permute_impl(const moe_mlp_desc_t* desc, const float* logits,
                               const float* bias, const void* x, int32_t* topk_idx,
                               float* topk_w, int32_t* counts, int32_t* offsets,
                               int32_t* padded_offsets, int32_t* tile_prefix,
                               int32_t* row_src, int32_t* row_of, void* x_perm, void* ws,
                               size_t ws_bytes, cudaStream_t stream, uint8_t* xq,
                               uint8_t* xs) {
  moe_status_t st = check_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!logits || !x || !topk_idx || !topk_w || !counts || !offsets || !padded_offsets ||
      !tile_prefix || !row_src || !row_of || !x_perm)
    return MOE_ERR_NULL;
  if (desc->T > 0 && !ws) return MOE_ERR_NULL;
  if (ws_bytes < route_ws_bytes(desc)) return MOE_ERR_WORKSPACE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const int T = desc->T, E = desc->E, k = desc->k;
  int32_t* chunk = static_cast<int32_t*>(ws);
  cudaError_t e = cudaMemsetAsync(row_src, 0xFF, sizeof(int32_t) * desc->capacity, stream);
  if (e == cudaSuccess && T > 0)
    e = launch_topk(logits, bias, T, E, k, topk_idx, topk_w, chunk, di->status, stream);
  if (e == cudaSuccess) {
    if (T > 0) {
      e = launch_scan_assign(topk_idx, T, E, k, chunk, desc->capacity, counts, offsets,
                             padded_offsets, tile_prefix, row_src, row_of, di->status, stream);
    } else {
      e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream);
      if (e == cudaSuccess)
        e = launch_offsets_from_counts(counts, E, desc->capacity, offsets, padded_offsets,
                                       tile_prefix, di->status, stream);
    }
  }
  if (e == cudaSuccess)
    e = xq ? launch_gather_rows_mx(x, row_src, padded_offsets, E, desc->d, T, desc->capacity,
                                   x_perm, xq, xs, di->sms, stream)
           : launch_gather_rows(x, row_src, padded_offsets, E,
                                desc->d * static_cast<int>(act_bytes(desc) / 2), T,
                                desc->capacity, x_perm, di->sms, stream);
  return cuda_status(e);
}

moe_status_t moe_route_permute(const moe_mlp_desc_t* desc, const float* logits,
                               const float* bias, const void* x, int32_t* topk_idx,
                               float* topk_w, int32_t* counts, int32_t* offsets,
                               int32_t* padded_offsets, int32_t* tile_prefix,
                               int32_t* row_src, int32_t* row_of, void* x_perm, void* ws,
                               size_t ws_bytes, cudaStream_t stream) {
  return route_permute_impl(desc, logits, bias, x, topk_idx, topk_w, counts, offsets,
                            padded_offsets, tile_prefix, row_src, row_of, x_perm, ws, ws_bytes,
                            stream, nullptr, nullptr);
}

moe_status_t moe_route_permute_mx(const moe_mlp_desc_t* desc, const float* logits,
                                  const float* bias, const void* x, int32_t* topk_idx,
                                  float* topk_w, int32_t* counts, int32_t* offsets,
                                  int32_t* padded_offsets, int32_t* tile_prefix,
                                  int32_t* row_src, int32_t* row_of, void* x_perm,
                                  const moe_mx_out_t* x_mx, void* ws, size_t ws_bytes,
                                  cudaStream_t stream) {
  if (!x_mx || !x_mx->q || !x_mx->scale) return MOE_ERR_NULL;
  if (x_mx->layout != MOE_MX_SCALES_MMA || x_mx->qt || x_mx->amax) return MOE_ERR_UNSUPPORTED;
  if (desc && desc->dtype == MOE_DTYPE_FP32) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x_mx->q) & 15) return MOE_ERR_SHAPE;
  return route_permute_impl(desc, logits, bias, x, topk_idx, topk_w, counts, offsets,
                            padded_offsets, tile_prefix, row_src, row_of, x_perm, ws, ws_bytes,
                            stream, x_mx->q, x_mx->scale);
}

moe_status_t moe_route_permute_fused(const moe_mlp_desc_t* desc, const void* x,
                                     const void* w_router, const float* bias, float* logits,
                                     int32_t* topk_idx, float* topk_w, int32_t* counts,
                                     int32_t* offsets, int32_t* padded_offsets,
                                     int32_t* tile_prefix, int32_t* row_src, int32_t* row_of,
                                     void* x_perm, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!x || !w_router || !topk_idx || !topk_w || !counts || !offsets || !padded_offsets ||
      !tile_prefix || !row_src || !row_of || !x_perm)
    return MOE_ERR_NULL;
  if (desc->T > 0 && !ws) return MOE_ERR_NULL;
  // the chunk histogram, then the grid-barrier counter of the routing tail
  const size_t ctr_off = route_ws_bytes(desc);
  if (ws_bytes < ctr_off + 256) return MOE_ERR_WORKSPACE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const int T = desc->T, E = desc->E, k = desc->k;
  const uint64_t d = desc->d;
  const int nchunks = (T + kTokensPerChunk - 1) / kTokensPerChunk;
  int32_t* chunk = static_cast<int32_t*>(ws);
  cudaError_t e = cudaMemsetAsync(row_src, 0xFF, sizeof(int32_t) * desc->capacity, stream);
  if (e == cudaSuccess && T > 0) {
    unsigned int* grid_ctr = reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + ctr_off);
    e = cudaMemsetAsync(chunk, 0, sizeof(int32_t) * nchunks * E, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(grid_ctr, 0, sizeof(unsigned int), stream);
    // one cooperative launch: logits = x W_r^T on the tensor cores, top-k +
    // softmax + histogram in the epilogue, then (after grid-wide barriers)
    // the group tables, the row assignment and the gather of x_perm
    GemmArgs g;
    memset(&g, 0, sizeof(g));
    g.status = di->status;
    g.E = 1;
    g.capacity = (T + kAlign - 1) / kAlign * kAlign;
    g.dense_rows = T;
    if (!encode_map(&g.tma_a, x, d, T, 1, d * 2, static_cast<uint64_t>(T) * d * 2, 64, 128) ||
        !encode_map(&g.tma_b, w_router, d, E, 1, d * 2, static_cast<uint64_t>(E) * d * 2, 64,
                    static_cast<uint32_t>((E + 15) / 16 * 16)))
      return MOE_ERR_SHAPE;
    g.K = desc->d;
    g.n_ext = E;
    g.b_ext = E;
    g.topk = k;
    g.r_bias = bias;
    g.r_idx = topk_idx;
    g.r_w = topk_w;
    g.r_hist = chunk;
    g.r_logits = logits;
    g.r_grid = grid_ctr;
    g.r_counts = counts;
    g.r_offsets = offsets;
    g.r_padded = padded_offsets;
    g.r_tiles = tile_prefix;
    g.r_row_src = row_src;
    g.r_row_of = row_of;
    g.r_x = x;
    g.r_x_perm = x_perm;
    g.r_tokens = T;
    g.r_vec_per_row = desc->d / 8;
    g.r_capacity = desc->capacity;
    g.r_nchunks = nchunks;
    if (e == cudaSuccess) e = launch_grouped_gemm(kRouter, g, grid_for(di, desc), stream);
    return cuda_status(e);
  }
  // no tokens: every group is empty
  if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * E, stream);
  if (e == cudaSuccess)
    e = launch_offsets_from_counts(counts, E, desc->capacity, offsets, padded_offsets,
                                   tile_prefix, di->status, stream);
  if (e == cudaSuccess)
    e = launch_gather_rows(x, row_src, padded_offsets, E, desc->d, T, desc->capacity, x_perm,
                           di->sms, stream);
  return cuda_status(e);
}

moe_status_t moe_group_offsets(const moe_mlp_desc_t* desc, const int32_t* counts,
                               int32_t* offsets, int32_t* padded_offsets,
                               int32_t* tile_prefix, cudaStream_t stream) {
  moe_status_t st = check_desc(desc, false);
  if (st != MOE_OK) return st;
  if (!counts || !offsets || !padded_offsets || !tile_prefix) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return cuda_status(launch_offsets_from_counts(counts, desc->E, desc->capacity, offsets,
                                                padded_offsets, tile_prefix, di->status, stream));
}

moe_status_t moe_fc1_glu_fwd(const moe_mlp_desc_t* desc, const void* x_perm,
                             const int32_t* counts, const int32_t* padded_offsets,
                             const void* w1p, const void* b1p, void* h, void* a,
                             const moe_mx_out_t* a_mx, cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!x_perm || !counts || !padded_offsets || !w1p || !a) return MOE_ERR_NULL;
  if (!h && !desc->recompute_h) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, x_perm, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_map(&g.tma_b, w1p, d, W1, E, d * 2, W1 * d * 2, 64, 256) ||
      (h && !encode_out(&g.tma_out0, h, W1, cap, 1)) ||
      !encode_out(&g.tma_out1, a, F, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.out1 = a;
  g.ld1 = F;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  if ((st = set_mx(g, a_mx, desc->F, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm(desc->act == MOE_ACT_SRELU ? kFc1Act : kFc1Glu, g,
                                         grid_for(di, desc), stream));
}

moe_status_t moe_fc2_fwd(const moe_mlp_desc_t* desc, const void* a, const int32_t* counts,
                         const int32_t* padded_offsets, const void* w2, const void* b2, void* y,
                         const moe_mx_out_t* y_mx, cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!a || !counts || !padded_offsets || !w2 || !y) return MOE_ERR_NULL;
  if (desc->has_b2 && !b2) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F;
  const uint64_t cap = desc->capacity;
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, a, F, cap, 1, F * 2, cap * F * 2, 64, 128) ||
      !encode_map(&g.tma_b, w2, F, d, E, F * 2, d * F * 2, 64, 256) ||
      !encode_out(&g.tma_out0, y, d, cap, 1) || !encode_out2(&g.tma_out2, y, d, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->F;
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = y;
  g.ld0 = d;
  g.bias = desc->has_b2 ? b2 : nullptr;
  g.bias_ld = d;
  if ((st = set_mx(g, y_mx, desc->d, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_mlp_fwd(const moe_mlp_desc_t* desc, const void* x_perm,
                         const int32_t* counts, const int32_t* padded_offsets,
                         const void* w1p, const void* b1p, const void* w2, const void* b2,
                         void* h, void* a, void* y, const moe_mx_out_t* a_mx,
                         const moe_mx_out_t* y_mx, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  if (desc && desc->dtype == MOE_DTYPE_FP32)
    return mlp_fwd_tf32(desc, x_perm, counts, padded_offsets, w1p, b1p, w2, b2, h, a, y, a_mx,
                        y_mx, stream);
  if (!w2 || !y || (desc && desc->has_b2 && !b2)) return MOE_ERR_NULL;
  moe_status_t st =
      moe_fc1_glu_fwd(desc, x_perm, counts, padded_offsets, w1p, b1p, h, a, a_mx, stream);
  if (st != MOE_OK) return st;
  return moe_fc2_fwd(desc, a, counts, padded_offsets, w2, b2, y, y_mx, stream);
}

moe_status_t moe_unpermute_combine(const moe_mlp_desc_t* desc, const void* y,
                                   const int32_t* row_of, const float* topk_w, void* out,
                                   cudaStream_t stream) {
  moe_status_t st = check_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!y || !row_of || !topk_w || !out) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  if (desc->dtype == MOE_DTYPE_FP32)
    return cuda_status(
        launch_combine_f32(y, row_of, topk_w, desc->T, desc->k, desc->d, out, stream));
  return cuda_status(launch_combine(y, row_of, topk_w, desc->T, desc->k, desc->d, out, stream));
}

moe_status_t moe_unpermute_combine_bwd(const moe_mlp_desc_t* desc, const void* dout,
                                       const void* y, const int32_t* row_of,
                                       const float* topk_w, const int32_t* row_src,
                                       const int32_t* padded_offsets, void* dy, float* dw,
                                       cudaStream_t stream) {
  moe_status_t st = check_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!dout || !y || !row_of || !topk_w || !row_src || !padded_offsets || !dy || !dw)
    return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const bool f32 = desc->dtype == MOE_DTYPE_FP32;
  cudaError_t e = launch_zero_pad_rows(row_src, padded_offsets, desc->E,
                                       f32 ? 2 * desc->d : desc->d, desc->capacity, dy, di->sms,
                                       stream);
  if (e == cudaSuccess)
    e = f32 ? launch_combine_bwd_f32(dout, y, row_of, topk_w, desc->T, desc->k, desc->d, dy, dw,
                                     stream)
            : launch_combine_bwd(dout, y, row_of, topk_w, desc->T, desc->k, desc->d, dy, dw,
                                 stream);
  return cuda_status(e);
}

moe_status_t moe_unpermute_combine_bwd_mx(const moe_mlp_desc_t* desc, const void* dout,
                                          const void* y, const int32_t* row_of,
                                          const float* topk_w, const int32_t* row_src,
                                          const int32_t* padded_offsets, void* dy,
                                          const moe_mx_out_t* dy_mx, float* dw,
                                          cudaStream_t stream) {
  moe_status_t st = check_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!dout || !y || !row_of || !topk_w || !row_src || !padded_offsets || !dy || !dw)
    return MOE_ERR_NULL;
  if (!dy_mx || !dy_mx->q || !dy_mx->scale) return MOE_ERR_NULL;
  if (dy_mx->layout != MOE_MX_SCALES_MMA || dy_mx->qt || dy_mx->amax) return MOE_ERR_UNSUPPORTED;
  if (desc->dtype == MOE_DTYPE_FP32) return MOE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(dy_mx->q) & 15) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  cudaError_t e = launch_zero_pad_rows(row_src, padded_offsets, desc->E, desc->d,
                                       desc->capacity, dy, di->sms, stream, dy_mx->q,
                                       dy_mx->scale);
  if (e == cudaSuccess)
    e = launch_combine_bwd_mx(dout, y, row_of, topk_w, desc->T, desc->k, desc->d,
                              desc->capacity, dy, dw, dy_mx->q, dy_mx->scale, stream);
  return cuda_status(e);
}

moe_status_t moe_fc2_dgrad_dglu(const moe_mlp_desc_t* desc, const void* dy, const void* h,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const void* w2, void* dh, const moe_mx_out_t* dh_mx,
                                cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!dy || !h || !counts || !padded_offsets || !w2 || !dh) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dA = dY W2 with W2 [d,F] read MN-major (F contiguous); dH from H
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, dy, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_out(&g.tma_out0, dh, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.b_atoms4d = encode_mn_atoms(&g.tma_b, w2, F, d, E, F * 2, d * F * 2, 4);
  if (!g.b_atoms4d && !encode_map(&g.tma_b, w2, F, d, E, F * 2, d * F * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = desc->act == MOE_ACT_SRELU ? desc->F : static_cast<int>(Fp);
  g.b_ext = desc->F;
  g.out0 = dh;
  g.ld0 = W1;
  g.aux = h;
  g.ld_aux = W1;
  if ((st = set_mx(g, dh_mx, W1, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm(desc->act == MOE_ACT_SRELU ? kDgradAct : kDgradDglu, g,
                                         grid_for(di, desc), stream));
}

moe_status_t moe_fc2_dgrad_dglu_recompute(const moe_mlp_desc_t* desc, const void* x_perm,
                                          const void* dy, const int32_t* counts,
                                          const int32_t* padded_offsets, const void* w1p,
                                          const void* b1p, const void* w2, void* dh,
                                          const moe_mx_out_t* dh_mx, cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;   // GLU activations
  if (!x_perm || !dy || !counts || !padded_offsets || !w1p || !w2 || !dh) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // H = X W1p^T (+b1) for the tile's packed block and dA = dY W2 (W2 read
  // MN-major, two 64-feature atoms per stage), both K = d; dH from them
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, x_perm, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_map(&g.tma_b, w1p, d, W1, E, d * 2, W1 * d * 2, 64, 256) ||
      !encode_map(&g.tma_a2, dy, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_out(&g.tma_out0, dh, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.b2_atoms4d = encode_mn_atoms(&g.tma_b2, w2, F, d, E, F * 2, d * F * 2, 2);
  if (!g.b2_atoms4d && !encode_map(&g.tma_b2, w2, F, d, E, F * 2, d * F * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = fc1_pad(desc->F);
  g.b_ext = desc->F;
  g.out0 = dh;
  g.ld0 = W1;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  if ((st = set_mx(g, dh_mx, W1, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm(kDgradDgluRc, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_wgrad(const moe_mlp_desc_t* desc, const void* dy, const void* a,
                           const int32_t* counts, const int32_t* padded_offsets, void* dw2,
                           cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!dy || !a || !counts || !padded_offsets || !dw2) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F;
  const uint64_t cap = desc->capacity;
  // dW2[e] (d x F) = sum over the group's rows of dY^T A (both read MN-major)
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_out(&g.tma_out0, dw2, F, d, E) || !encode_out2(&g.tma_out2, dw2, F, d, E))
    return MOE_ERR_SHAPE;
  g.a_atoms4d = encode_mn_atoms(&g.tma_a, dy, d, cap, 1, d * 2, cap * d * 2, 2);
  if (!g.a_atoms4d && !encode_map(&g.tma_a, dy, d, cap, 1, d * 2, cap * d * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.b_atoms4d = encode_mn_atoms(&g.tma_b, a, F, cap, 1, F * 2, cap * F * 2, 2);
  if (!g.b_atoms4d && !encode_map(&g.tma_b, a, F, cap, 1, F * 2, cap * F * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.m_ext = desc->d;
  g.n_ext = desc->F;
  g.b_ext = desc->F;
  g.out0 = dw2;
  g.ld0 = F;
  return cuda_status(launch_grouped_gemm(kWgradPair, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_dgrad(const moe_mlp_desc_t* desc, const void* dh, const int32_t* counts,
                           const int32_t* padded_offsets, const void* w1p, void* dx_perm,
                           cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!dh || !counts || !padded_offsets || !w1p || !dx_perm) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dX = dH W1p with W1p [2F_pad,d] read MN-major (d contiguous)
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, dh, W1, cap, 1, W1 * 2, cap * W1 * 2, 64, 128) ||
      !encode_out(&g.tma_out0, dx_perm, d, cap, 1) ||
      !encode_out2(&g.tma_out2, dx_perm, d, cap, 1))
    return MOE_ERR_SHAPE;
  g.b_atoms4d = encode_mn_atoms(&g.tma_b, w1p, d, W1, E, d * 2, W1 * d * 2, 4);
  if (!g.b_atoms4d && !encode_map(&g.tma_b, w1p, d, W1, E, d * 2, W1 * d * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.K = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dx_perm;
  g.ld0 = d;
  return cuda_status(launch_grouped_gemm(kDgradFc1, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_wgrad(const moe_mlp_desc_t* desc, const void* dh, const void* x_perm,
                           const int32_t* counts, const int32_t* padded_offsets, void* dw1p,
                           cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!dh || !x_perm || !counts || !padded_offsets || !dw1p) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dW1p[e] (2F_pad x d) = sum over the group's rows of dH^T X
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_out(&g.tma_out0, dw1p, d, W1, E) ||
      !encode_out2(&g.tma_out2, dw1p, d, W1, E))
    return MOE_ERR_SHAPE;
  g.a_atoms4d = encode_mn_atoms(&g.tma_a, dh, W1, cap, 1, W1 * 2, cap * W1 * 2, 2);
  if (!g.a_atoms4d &&
      !encode_map(&g.tma_a, dh, W1, cap, 1, W1 * 2, cap * W1 * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.b_atoms4d = encode_mn_atoms(&g.tma_b, x_perm, d, cap, 1, d * 2, cap * d * 2, 2);
  if (!g.b_atoms4d && !encode_map(&g.tma_b, x_perm, d, cap, 1, d * 2, cap * d * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.m_ext = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dw1p;
  g.ld0 = d;
  return cuda_status(launch_grouped_gemm(kWgradPair, g, grid_for(di, desc), stream));
}

moe_status_t moe_bias_grads(const moe_mlp_desc_t* desc, const void* dy, const void* dh,
                            const int32_t* counts, const int32_t* padded_offsets, void* db1p,
                            void* db2, cudaStream_t stream) {
  moe_status_t st = check_desc(desc, false);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || (db2 && !dy) || (db1p && !dh)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  cudaError_t e = cudaSuccess;
  const auto colsum = desc->dtype == MOE_DTYPE_FP32 ? launch_group_colsum_f32 : launch_group_colsum;
  if (db2) e = colsum(dy, counts, padded_offsets, desc->E, desc->d, db2, stream);
  if (e == cudaSuccess && db1p)
    e = colsum(dh, counts, padded_offsets, desc->E, fc1_width(desc->act, desc->F), db1p, stream);
  return cuda_status(e);
}

moe_status_t moe_mlp_bwd(const moe_mlp_desc_t* desc, const void* dy, const void* x_perm,
                         const void* h, const void* a, const int32_t* counts,
                         const int32_t* padded_offsets, const void* w1p, const void* b1p,
                         const void* w2, void* dh, void* dx_perm, void* dw1p, void* db1p,
                         void* dw2, void* db2, const moe_mx_out_t* dh_mx, void* ws,
                         size_t ws_bytes, cudaStream_t stream) {
  if (desc && desc->dtype == MOE_DTYPE_FP32)
    return mlp_bwd_tf32(desc, dy, x_perm, h, a, counts, padded_offsets, w1p, b1p, w2, dh,
                        dx_perm, dw1p, db1p, dw2, db2, dh_mx, ws, ws_bytes, stream);
  moe_status_t st = check_desc(desc, false);
  if (st != MOE_OK) return st;
  if (!dy || !x_perm || !a || !counts || !padded_offsets || !w1p || !w2 || !dh ||
      !dx_perm || !dw1p || !dw2)
    return MOE_ERR_NULL;
  if ((desc->has_b1 && !db1p) || (desc->has_b2 && !db2)) return MOE_ERR_NULL;
  if (!h && !desc->recompute_h) return MOE_ERR_NULL;
  if (!h && desc->act != MOE_ACT_SRELU) {
    // activation recompute inside the dGLU kernel: H never reaches HBM
    if ((st = moe_fc2_dgrad_dglu_recompute(desc, x_perm, dy, counts, padded_offsets, w1p, b1p,
                                           w2, dh, dh_mx, stream)) != MOE_OK)
      return st;
  } else {
    if (!h) {
      // non-gated activation: regenerate H in the workspace first
      size_t need = 0;
      if ((st = moe_workspace_size(desc, &need)) != MOE_OK) return st;
      if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
      const size_t off = (route_ws_bytes(desc) + 256 + 255) / 256 * 256;
      void* h_ws = static_cast<uint8_t*>(ws) + off;
      if ((st = moe_fc1_recompute_h(desc, x_perm, counts, padded_offsets, w1p, b1p, h_ws,
                                    stream)) != MOE_OK)
        return st;
      h = h_ws;
    }
    if ((st = moe_fc2_dgrad_dglu(desc, dy, h, counts, padded_offsets, w2, dh, dh_mx, stream)) !=
        MOE_OK)
      return st;
  }
  if ((st = moe_fc2_wgrad(desc, dy, a, counts, padded_offsets, dw2, stream)) != MOE_OK) return st;
  if ((st = moe_fc1_dgrad(desc, dh, counts, padded_offsets, w1p, dx_perm, stream)) != MOE_OK)
    return st;
  if ((st = moe_fc1_wgrad(desc, dh, x_perm, counts, padded_offsets, dw1p, stream)) != MOE_OK)
    return st;
  if (desc->has_b1 || desc->has_b2)
    st = moe_bias_grads(desc, dy, dh, counts, padded_offsets, desc->has_b1 ? db1p : nullptr,
                        desc->has_b2 ? db2 : nullptr, stream);
  return st;
}

moe_status_t moe_fc1_glu_fwd_unfused(const moe_mlp_desc_t* desc, const void* x_perm,
                                     const int32_t* counts, const int32_t* padded_offsets,
                                     const void* w1p, const void* b1p, void* h, void* a,
                                     cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;   // GLU passes only
  if (!x_perm || !counts || !padded_offsets || !w1p || !h || !a) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // plain grouped GEMM H = X W1p^T (+b1): the FC2-shaped kernel with W1p as B
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, x_perm, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_map(&g.tma_b, w1p, d, W1, E, d * 2, W1 * d * 2, 64, 256) ||
      !encode_out(&g.tma_out0, h, W1, cap, 1) || !encode_out2(&g.tma_out2, h, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  cudaError_t e = launch_grouped_gemm(kFc2, g, grid_for(di, desc), stream);
  if (e == cudaSuccess)
    e = launch_glu_rows(h, counts, padded_offsets, desc->E, desc->F, static_cast<int>(Fp), a,
                        desc->act, desc->alpha, desc->limit, desc->linear_offset,
                        desc->out_scale, di->sms, stream);
  return cuda_status(e);
}

moe_status_t moe_fc1_recompute_h(const moe_mlp_desc_t* desc, const void* x_perm,
                                 const int32_t* counts, const int32_t* padded_offsets,
                                 const void* w1p, const void* b1p, void* h, cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!x_perm || !counts || !padded_offsets || !w1p || !h) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  GemmArgs g;   // the FC2-shaped plain kernel with W1p as B
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, x_perm, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_map(&g.tma_b, w1p, d, W1, E, d * 2, W1 * d * 2, 64, 256) ||
      !encode_out(&g.tma_out0, h, W1, cap, 1) || !encode_out2(&g.tma_out2, h, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  return cuda_status(launch_grouped_gemm(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_dgrad_dglu_unfused(const moe_mlp_desc_t* desc, const void* dy,
                                        const void* h, const int32_t* counts,
                                        const int32_t* padded_offsets, const void* w2, void* da,
                                        void* dh, cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;   // GLU passes only
  if (!dy || !h || !counts || !padded_offsets || !w2 || !da || !dh) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // plain grouped GEMM dA = dY W2: the FC1-dgrad-shaped kernel with W2 as B
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_map(&g.tma_a, dy, d, cap, 1, d * 2, cap * d * 2, 64, 128) ||
      !encode_out(&g.tma_out0, da, F, cap, 1) || !encode_out2(&g.tma_out2, da, F, cap, 1))
    return MOE_ERR_SHAPE;
  g.b_atoms4d = encode_mn_atoms(&g.tma_b, w2, F, d, E, F * 2, d * F * 2, 4);
  if (!g.b_atoms4d && !encode_map(&g.tma_b, w2, F, d, E, F * 2, d * F * 2, 64, 64))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = desc->F;
  g.b_ext = desc->F;
  g.out0 = da;
  g.ld0 = F;
  cudaError_t e = launch_grouped_gemm(kDgradFc1, g, grid_for(di, desc), stream);
  if (e == cudaSuccess)
    e = launch_dglu_rows(da, h, counts, padded_offsets, desc->E, desc->F, static_cast<int>(Fp),
                         dh, desc->act, desc->alpha, desc->limit, desc->linear_offset,
                         desc->out_scale, di->sms, stream);
  return cuda_status(e);
}

moe_status_t moe_permute_bwd(const moe_mlp_desc_t* desc, const void* dx_perm,
                             const int32_t* row_of, void* dx, cudaStream_t stream) {
  moe_status_t st = check_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!dx_perm || !row_of || !dx) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  if (desc->dtype == MOE_DTYPE_FP32)
    return cuda_status(
        launch_combine_f32(dx_perm, row_of, nullptr, desc->T, desc->k, desc->d, dx, stream));
  return cuda_status(launch_permute_bwd(dx_perm, row_of, desc->T, desc->k, desc->d, dx, stream));
}

moe_status_t moe_route_bwd(const moe_mlp_desc_t* desc, const float* dw, const float* topk_w,
                           const int32_t* topk_idx, float* dlogits, cudaStream_t stream) {
  moe_status_t st = check_desc(desc, true);
  if (st != MOE_OK) return st;
  if (!dw || !topk_w || !topk_idx || !dlogits) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return cuda_status(
      launch_route_bwd(dw, topk_w, topk_idx, desc->T, desc->E, desc->k, dlogits, stream));
}

moe_status_t moe_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 5000000) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  k_wait_selftest<<<1, 32, 0, stream>>>(di->status, 1000ull * limit_us);
  return cuda_status(cudaGetLastError());
}

moe_status_t moe_selftest_grid_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
  if (limit_us == 0 || limit_us > 5000000) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  k_grid_wait_selftest<<<1, 64, 0, stream>>>(di->status, 1000ull * limit_us);
  return cuda_status(cudaGetLastError());
}

moe_status_t moe_read_device_status(int32_t* host_status, int32_t clear) {
  if (!host_status) return MOE_ERR_NULL;
  DeviceInfo* di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, di->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (clear && cudaMemset(di->status, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  *host_status = v;
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// MXFP8 path: the same grouped-GEMM modes with E4M3 operands (K-major, the
// transposed operands of the backward come from transposed MXFP8 copies) and
// E8M0 scales in the MMA layout.
namespace moe {
namespace {

long long sf_bytes(long long rows, long long cols) {
  return (cols + 127) / 128 * sf_row_atoms(rows) * 512;
}

// MXFP8 tensor described by `m`: the rowwise and/or transposed parts the
// caller needs, in the MMA layout, codes 16-byte aligned.
bool mx_ok(const moe_mx_out_t* m, bool row, bool col) {
  if (!m || m->layout != MOE_MX_SCALES_MMA) return false;
  if (row && (!m->q || !m->scale || (reinterpret_cast<uintptr_t>(m->q) & 15))) return false;
  if (col && (!m->qt || !m->scale_t || (reinterpret_cast<uintptr_t>(m->qt) & 15))) return false;
  return true;
}

bool mx_weights_ok(const moe_mx_weights_t* w) {
  return w && w->w1 && w->w1_s && w->w1t && w->w1t_s && w->w2 && w->w2_s && w->w2t && w->w2t_s;
}

// E4M3 operand [E][rows][K] (K contiguous), boxes of 128 K x box_rows rows.
bool encode_u8(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint64_t E,
               uint32_t box_rows) {
  return encode_map(map, base, K, rows, E, K, rows * K, 128, box_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8);
}

void set_scales(GemmArgs& g, const uint8_t* sfa, long long a_rows, const uint8_t* sfb,
                long long b_rows, long long b_expert_bytes) {
  g.sfa = sfa;
  g.sfa_atoms = sf_row_atoms(a_rows);
  g.sfb = sfb;
  g.sfb_atoms = sf_row_atoms(b_rows);
  g.sfb_expert_bytes = b_expert_bytes;
}

moe_status_t check_mx_desc(const moe_mlp_desc_t* d) {
  moe_status_t st = check_desc(d, false);
  if (st != MOE_OK) return st;
  if (d->dtype != MOE_DTYPE_MXFP8) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_mx_scale_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return static_cast<size_t>(sf_bytes(rows, cols));
}

moe_status_t moe_quantize_mx_bf16(const void* in, int64_t batch, int64_t rows, int64_t cols,
                                  const moe_mx_out_t* out, cudaStream_t stream) {
  if (!in || !out) return MOE_ERR_NULL;
  if ((out->q && !out->scale) || (out->qt && !out->scale_t) || (!out->q && !out->qt))
    return MOE_ERR_NULL;
  if (out->amax) return MOE_ERR_UNSUPPORTED;
  if (out->layout != MOE_MX_SCALES_ROWMAJOR && out->layout != MOE_MX_SCALES_MMA)
    return MOE_ERR_UNSUPPORTED;
  if (batch < 0 || rows < 0 || cols < 0 || rows % 32 != 0 || cols % 32 != 0)
    return MOE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out->q) & 15) ||
      (reinterpret_cast<uintptr_t>(out->qt) & 15))
    return MOE_ERR_SHAPE;
  DeviceInfo* di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_quant_bf16_mx(in, batch, rows, cols, out->q, out->scale, out->qt,
                                          out->scale_t, out->layout == MOE_MX_SCALES_MMA,
                                          nullptr, di->sms, di->status, stream));
}

moe_status_t moe_quantize_act_mx(const moe_mlp_desc_t* desc, const void* in, int32_t width,
                                 const int32_t* padded_offsets, const moe_mx_out_t* out,
                                 cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!in || !padded_offsets || !out) return MOE_ERR_NULL;
  if ((out->q && !out->scale) || (out->qt && !out->scale_t) || (!out->q && !out->qt))
    return MOE_ERR_NULL;
  if (out->amax) return MOE_ERR_UNSUPPORTED;
  if (out->layout != MOE_MX_SCALES_MMA) return MOE_ERR_UNSUPPORTED;
  if (width < 32 || width % 32 != 0) return MOE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(out->q) & 15) ||
      (reinterpret_cast<uintptr_t>(out->qt) & 15))
    return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return cuda_status(launch_quant_bf16_mx(in, 1, desc->capacity, width, out->q, out->scale,
                                          out->qt, out->scale_t, 1, padded_offsets + desc->E,
                                          di->sms, di->status, stream));
}

moe_status_t moe_quantize_weights_mx(const moe_mlp_desc_t* desc, const void* w1p,
                                     const void* w2, const moe_mx_weights_t* out,
                                     cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!w1p || !w2 || !mx_weights_ok(out)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const long long E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  cudaError_t e = launch_quant_bf16_mx(w1p, E, W1, d, out->w1, out->w1_s, out->w1t,
                                       out->w1t_s, 1, nullptr, di->sms, di->status, stream);
  if (e == cudaSuccess)
    e = launch_quant_bf16_mx(w2, E, d, F, out->w2, out->w2_s, out->w2t, out->w2t_s, 1, nullptr,
                             di->sms, di->status, stream);
  return cuda_status(e);
}

moe_status_t moe_fc1_glu_fwd_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const moe_mx_weights_t* w, const void* b1p, void* h, void* a,
                                const moe_mx_out_t* a_mx, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !mx_weights_ok(w)) return MOE_ERR_NULL;
  if (!h && !desc->recompute_h) return MOE_ERR_NULL;   // H kept unless recomputed
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!mx_ok(x_mx, true, false) || !mx_ok(a_mx, true, a_mx && a_mx->qt)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // x_perm (codes [cap, d]) x W1p (codes [E, 2F_pad, d]); GLU epilogue
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, x_mx->q, d, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w1, d, W1, E, 256) ||
      (h && !encode_out(&g.tma_out0, h, W1, cap, 1)) ||
      (a && !encode_out(&g.tma_out1, a, F, cap, 1)))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.out1 = a;
  g.ld1 = F;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  set_scales(g, x_mx->scale, cap, w->w1_s, W1, sf_bytes(W1, d));
  if ((st = set_mx(g, a_mx, desc->F, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm_mx(desc->act == MOE_ACT_SRELU ? kFc1Act : kFc1Glu, g,
                                            grid_for(di, desc), stream));
}

moe_status_t moe_fc2_fwd_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* a_mx,
                            const int32_t* counts, const int32_t* padded_offsets,
                            const moe_mx_weights_t* w, const void* b2, void* y,
                            cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !mx_weights_ok(w) || !y) return MOE_ERR_NULL;
  if (desc->has_b2 && !b2) return MOE_ERR_NULL;
  if (!mx_ok(a_mx, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F;
  const uint64_t cap = desc->capacity;
  // A (codes [cap, F]) x W2 (codes [E, d, F])
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, a_mx->q, F, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w2, F, d, E, 256) || !encode_out(&g.tma_out0, y, d, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->F;
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = y;
  g.ld0 = d;
  g.bias = desc->has_b2 ? b2 : nullptr;
  g.bias_ld = d;
  set_scales(g, a_mx->scale, cap, w->w2_s, d, sf_bytes(d, F));
  return cuda_status(launch_grouped_gemm_mx(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_dgrad_dglu_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_mx,
                                   const void* h, const int32_t* counts,
                                   const int32_t* padded_offsets, const moe_mx_weights_t* w,
                                   void* dh, const moe_mx_out_t* dh_mx, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!h || !counts || !padded_offsets || !mx_weights_ok(w)) return MOE_ERR_NULL;
  if (!mx_ok(dy_mx, true, false) || !mx_ok(dh_mx, true, true)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dY (codes [cap, d]) x W2^T (codes [E, F, d]); dGLU epilogue reads H;
  // the bf16 dH is stored only when dh is given
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dy_mx->q, d, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w2t, d, F, E, 256) ||
      (dh && !encode_out(&g.tma_out0, dh, W1, cap, 1)))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = desc->act == MOE_ACT_SRELU ? desc->F : static_cast<int>(Fp);
  g.b_ext = desc->F;
  g.out0 = dh;
  g.ld0 = W1;
  g.aux = h;
  g.ld_aux = W1;
  set_scales(g, dy_mx->scale, cap, w->w2t_s, F, sf_bytes(F, d));
  if ((st = set_mx(g, dh_mx, W1, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm_mx(desc->act == MOE_ACT_SRELU ? kDgradAct : kDgradDglu,
                                            g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_wgrad_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_mx,
                              const moe_mx_out_t* a_mx, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw2, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !dw2) return MOE_ERR_NULL;
  if (!mx_ok(dy_mx, false, true) || !mx_ok(a_mx, false, true)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F;
  const uint64_t cap = desc->capacity;
  // dW2[e] = dY^T A over the group's rows: codes [d, cap] and [F, cap]
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dy_mx->qt, cap, d, 1, 128) ||
      !encode_u8(&g.tma_b, a_mx->qt, cap, F, 1, 256) || !encode_out(&g.tma_out0, dw2, F, d, E))
    return MOE_ERR_SHAPE;
  g.m_ext = desc->d;
  g.n_ext = desc->F;
  g.b_ext = desc->F;
  g.out0 = dw2;
  g.ld0 = F;
  set_scales(g, dy_mx->scale_t, d, a_mx->scale_t, F, 0);
  return cuda_status(launch_grouped_gemm_mx(kWgrad, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_dgrad_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_mx,
                              const int32_t* counts, const int32_t* padded_offsets,
                              const moe_mx_weights_t* w, void* dx_perm, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !mx_weights_ok(w) || !dx_perm) return MOE_ERR_NULL;
  if (!mx_ok(dh_mx, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dH (codes [cap, 2F_pad]) x W1p^T (codes [E, d, 2F_pad])
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dh_mx->q, W1, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w1t, W1, d, E, 256) ||
      !encode_out(&g.tma_out0, dx_perm, d, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dx_perm;
  g.ld0 = d;
  set_scales(g, dh_mx->scale, cap, w->w1t_s, d, sf_bytes(d, W1));
  return cuda_status(launch_grouped_gemm_mx(kDgradFc1, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_wgrad_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_mx,
                              const moe_mx_out_t* x_mx, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw1p, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !dw1p) return MOE_ERR_NULL;
  if (!mx_ok(dh_mx, false, true) || !mx_ok(x_mx, false, true)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dW1p[e] = dH^T X over the group's rows: codes [2F_pad, cap] and [d, cap]
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dh_mx->qt, cap, W1, 1, 128) ||
      !encode_u8(&g.tma_b, x_mx->qt, cap, d, 1, 256) ||
      !encode_out(&g.tma_out0, dw1p, d, W1, E))
    return MOE_ERR_SHAPE;
  g.m_ext = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dw1p;
  g.ld0 = d;
  set_scales(g, dh_mx->scale_t, W1, x_mx->scale_t, d, 0);
  return cuda_status(launch_grouped_gemm_mx(kWgrad, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_recompute_h_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                                    const int32_t* counts, const int32_t* padded_offsets,
                                    const moe_mx_weights_t* w, const void* b1p, void* h,
                                    cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !mx_weights_ok(w) || !h) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!mx_ok(x_mx, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // the FC2-shaped plain kernel with W1p as B, on the forward's operands:
  // the same MMAs in the same order as FC1, so H comes out bitwise the same
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, x_mx->q, d, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w1, d, W1, E, 256) || !encode_out(&g.tma_out0, h, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  set_scales(g, x_mx->scale, cap, w->w1_s, W1, sf_bytes(W1, d));
  return cuda_status(launch_grouped_gemm_mx(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_dgrad_dglu_recompute_mx(const moe_mlp_desc_t* desc,
                                             const moe_mx_out_t* x_mx,
                                             const moe_mx_out_t* dy_mx, const int32_t* counts,
                                             const int32_t* padded_offsets,
                                             const moe_mx_weights_t* w, const void* b1p,
                                             void* dh, const moe_mx_out_t* dh_mx,
                                             cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;   // GLU activations
  if (!counts || !padded_offsets || !mx_weights_ok(w)) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!mx_ok(x_mx, true, false) || !mx_ok(dy_mx, true, false) || !mx_ok(dh_mx, true, true))
    return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // H = X W1p^T (+b1) on the forward's MXFP8 operands (the same MMAs as the
  // forward), dA = dY W2 on dY's codes and W2's transposed copy [E, F, d]
  // (128-row boxes: the tile's 128 features); dH and its MXFP8 copies
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, x_mx->q, d, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w1, d, W1, E, 256) ||
      !encode_u8(&g.tma_a2, dy_mx->q, d, cap, 1, 128) ||
      !encode_u8(&g.tma_b2, w->w2t, d, F, E, 128) ||
      (dh && !encode_out(&g.tma_out0, dh, W1, cap, 1)))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = fc1_pad(desc->F);
  g.b_ext = desc->F;
  g.out0 = dh;
  g.ld0 = W1;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  set_scales(g, x_mx->scale, cap, w->w1_s, W1, sf_bytes(W1, d));
  g.sfa2 = dy_mx->scale;
  g.sfa2_atoms = sf_row_atoms(cap);
  g.sfb2 = w->w2t_s;
  g.sfb2_atoms = sf_row_atoms(F);
  g.sfb2_expert_bytes = sf_bytes(F, d);
  if ((st = set_mx(g, dh_mx, W1, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm_mx(kDgradDgluRc, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_glu_fwd_mx_unfused(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                                        const int32_t* counts, const int32_t* padded_offsets,
                                        const moe_mx_weights_t* w, const void* b1p, void* h,
                                        void* a, const moe_mx_out_t* a_mx, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;   // GLU passes only
  if (!counts || !padded_offsets || !mx_weights_ok(w) || !h || !a) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!mx_ok(x_mx, true, false) || !mx_ok(a_mx, true, true)) return MOE_ERR_NULL;
  // 1. plain grouped GEMM H = X W1p^T (+b1) on the MXFP8 operands
  if ((st = moe_fc1_recompute_h_mx(desc, x_mx, counts, padded_offsets, w, b1p, h, stream)) !=
      MOE_OK)
    return st;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  // 2. the GLU as its own pass over the stored bf16 H
  cudaError_t e = launch_glu_rows(h, counts, padded_offsets, desc->E, desc->F,
                                  fc1_pad(desc->F), a, desc->act, desc->alpha, desc->limit,
                                  desc->linear_offset, desc->out_scale, di->sms, stream);
  // 3. MXFP8 quantization of A, rowwise and transposed, as its own pass
  if (e == cudaSuccess)
    e = launch_quant_bf16_mx(a, 1, desc->capacity, desc->F, a_mx->q, a_mx->scale, a_mx->qt,
                             a_mx->scale_t, 1, padded_offsets + desc->E, di->sms, di->status,
                             stream);
  return cuda_status(e);
}

moe_status_t moe_fc2_dgrad_dglu_mx_unfused(const moe_mlp_desc_t* desc,
                                           const moe_mx_out_t* dy_mx, const void* h,
                                           const int32_t* counts, const int32_t* padded_offsets,
                                           const moe_mx_weights_t* w, void* da, void* dh,
                                           const moe_mx_out_t* dh_mx, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (desc->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;   // GLU passes only
  if (!h || !counts || !padded_offsets || !mx_weights_ok(w) || !da || !dh) return MOE_ERR_NULL;
  if (!mx_ok(dy_mx, true, false) || !mx_ok(dh_mx, true, true)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // 1. plain grouped GEMM dA = dY W2 on the MXFP8 operands (dY codes [cap, d]
  //    x W2^T codes [E, F, d]): the plain-output kernel, dA [cap, F] bf16
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dy_mx->q, d, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->w2t, d, F, E, 256) || !encode_out(&g.tma_out0, da, F, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = desc->F;
  g.b_ext = desc->F;
  g.out0 = da;
  g.ld0 = F;
  set_scales(g, dy_mx->scale, cap, w->w2t_s, F, sf_bytes(F, d));
  cudaError_t e = launch_grouped_gemm_mx(kFc2, g, grid_for(di, desc), stream);
  // 2. the dGLU as its own pass over dA and the stored bf16 H
  if (e == cudaSuccess)
    e = launch_dglu_rows(da, h, counts, padded_offsets, desc->E, desc->F, fc1_pad(desc->F), dh,
                         desc->act, desc->alpha, desc->limit, desc->linear_offset,
                         desc->out_scale, di->sms, stream);
  // 3. MXFP8 quantization of dH, rowwise and transposed, as its own pass
  if (e == cudaSuccess)
    e = launch_quant_bf16_mx(dh, 1, desc->capacity, static_cast<long long>(W1), dh_mx->q,
                             dh_mx->scale, dh_mx->qt, dh_mx->scale_t, 1,
                             padded_offsets + desc->E, di->sms, di->status, stream);
  return cuda_status(e);
}

moe_status_t moe_mlp_fwd_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                            const int32_t* counts, const int32_t* padded_offsets,
                            const moe_mx_weights_t* w, const void* b1p, const void* b2, void* h,
                            void* a, const moe_mx_out_t* a_mx, void* y, cudaStream_t stream) {
  if (!y) return MOE_ERR_NULL;
  moe_status_t st =
      moe_fc1_glu_fwd_mx(desc, x_mx, counts, padded_offsets, w, b1p, h, a, a_mx, stream);
  if (st != MOE_OK) return st;
  return moe_fc2_fwd_mx(desc, a_mx, counts, padded_offsets, w, b2, y, stream);
}

moe_status_t moe_mlp_bwd_mx(const moe_mlp_desc_t* desc, const void* dy,
                            const moe_mx_out_t* dy_mx, const moe_mx_out_t* x_mx, const void* h,
                            const moe_mx_out_t* a_mx, const int32_t* counts,
                            const int32_t* padded_offsets, const moe_mx_weights_t* w, void* dh,
                            const moe_mx_out_t* dh_mx, void* dx_perm, void* dw1p, void* db1p,
                            void* dw2, void* db2, cudaStream_t stream) {
  moe_status_t st = check_mx_desc(desc);
  if (st != MOE_OK) return st;
  if (!dy || !dx_perm || !dw1p || !dw2) return MOE_ERR_NULL;
  if (db1p && !dh) return MOE_ERR_NULL;            // the FC1 bias gradient sums dH
  if (!mx_ok(dy_mx, true, true) || !mx_ok(x_mx, false, true) || !mx_ok(a_mx, false, true) ||
      !mx_ok(dh_mx, true, true))
    return MOE_ERR_NULL;
  if ((st = moe_fc2_dgrad_dglu_mx(desc, dy_mx, h, counts, padded_offsets, w, dh, dh_mx,
                                  stream)) != MOE_OK ||
      (st = moe_fc2_wgrad_mx(desc, dy_mx, a_mx, counts, padded_offsets, dw2, stream)) != MOE_OK ||
      (st = moe_fc1_dgrad_mx(desc, dh_mx, counts, padded_offsets, w, dx_perm, stream)) !=
          MOE_OK ||
      (st = moe_fc1_wgrad_mx(desc, dh_mx, x_mx, counts, padded_offsets, dw1p, stream)) != MOE_OK)
    return st;
  if (db1p || db2) return moe_bias_grads(desc, dy, dh, counts, padded_offsets, db1p, db2, stream);
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// NVFP4 path: the same grouped-GEMM modes with packed E2M1 operands (K-major;
// 128-byte boxes hold 256 values), UE4M3 scales per 16 values in the MMA
// layout, and the operands' encode amax values for the epilogue's 1/(g_a g_b).
namespace moe {
namespace {

moe_status_t check_nv_desc(const moe_mlp_desc_t* d) {
  moe_status_t st = check_desc(d, false);
  if (st != MOE_OK) return st;
  if (d->dtype != MOE_DTYPE_NVFP4) return MOE_ERR_UNSUPPORTED;
  if (d->F % 64 != 0) return MOE_ERR_SHAPE;
  return MOE_OK;
}

// NVFP4 tensor: the needed parts, the MMA layout, 16-byte aligned codes and
// the encode amax pair.
bool nv_ok(const moe_mx_out_t* m, bool row, bool col) {
  return mx_ok(m, row, col) && m->amax != nullptr;
}

bool nv_weights_ok(const moe_nv_weights_t* w) { return w && mx_weights_ok(&w->q) && w->amax; }

void set_nv_scales(GemmArgs& g, const uint8_t* sfa, long long a_rows, const uint8_t* sfb,
                   long long b_rows, long long b_expert_bytes, const float* amax_a,
                   const float* amax_b) {
  set_scales(g, sfa, a_rows, sfb, b_rows, b_expert_bytes);
  g.nv_amax_a = amax_a;
  g.nv_amax_b = amax_b;
}

// epilogue amax outputs only (plain and rotated amax of the bf16 result)
moe_status_t set_amax_out(GemmArgs& g, float* amax, long long width, cudaStream_t stream) {
  moe_mx_out_t m;
  memset(&m, 0, sizeof(m));
  m.amax = amax;
  m.layout = MOE_MX_SCALES_MMA;
  return set_mx(g, &m, width, stream);
}

}  // namespace
}  // namespace moe

extern "C" {

size_t moe_nvfp4_scale_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return static_cast<size_t>(nv_sf_bytes(rows, cols));
}

moe_status_t moe_amax_nvfp4(const void* in, int64_t batch, int64_t rows, int64_t cols,
                            const int32_t* row_limit, float* amax, cudaStream_t stream) {
  if (!in || !amax) return MOE_ERR_NULL;
  if (batch < 0 || rows < 0 || cols < 0 || rows % 16 != 0 || cols % 8 != 0) return MOE_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(in) & 15) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_amax_nv(in, batch, rows, cols, row_limit, amax, di->sms, stream));
}

moe_status_t moe_quantize_nvfp4_bf16(const void* in, int64_t batch, int64_t rows, int64_t cols,
                                     const moe_mx_out_t* out, int32_t rotate_t,
                                     cudaStream_t stream) {
  if (!in || !out) return MOE_ERR_NULL;
  if (!nv_ok(out, out->q != nullptr, out->qt != nullptr) || (!out->q && !out->qt))
    return MOE_ERR_NULL;
  if (batch < 0 || rows < 0 || cols < 0 || rows % 32 != 0 || cols % 32 != 0)
    return MOE_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(in) & 15) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  moe_status_t st = device_info(&di);
  if (st != MOE_OK) return st;
  return cuda_status(launch_quant_nv(in, batch, rows, cols, static_cast<uint8_t*>(out->q),
                                     static_cast<uint8_t*>(out->scale),
                                     static_cast<uint8_t*>(out->qt),
                                     static_cast<uint8_t*>(out->scale_t), out->amax,
                                     out->amax + 1, rotate_t != 0, nullptr, di->sms, stream));
}

moe_status_t moe_quantize_act_nvfp4(const moe_mlp_desc_t* desc, const void* in, int32_t width,
                                    const int32_t* padded_offsets, const moe_mx_out_t* out,
                                    int32_t compute_amax, cudaStream_t stream) {
  moe_status_t st = check_bf16_desc(desc);
  if (st != MOE_OK) return st;
  if (!in || !padded_offsets || !out) return MOE_ERR_NULL;
  if (!nv_ok(out, out->q != nullptr, out->qt != nullptr) || (!out->q && !out->qt))
    return MOE_ERR_NULL;
  if (width < 64 || width % 64 != 0) return MOE_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(in) & 15) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const int32_t* lim = padded_offsets + desc->E;
  cudaError_t e = cudaSuccess;
  if (compute_amax) e = launch_amax_nv(in, 1, desc->capacity, width, lim, out->amax, di->sms, stream);
  if (e == cudaSuccess)
    e = launch_quant_nv(in, 1, desc->capacity, width, static_cast<uint8_t*>(out->q),
                        static_cast<uint8_t*>(out->scale), static_cast<uint8_t*>(out->qt),
                        static_cast<uint8_t*>(out->scale_t), out->amax, out->amax + 1, 1, lim,
                        di->sms, stream);
  return cuda_status(e);
}

moe_status_t moe_quantize_weights_nvfp4(const moe_mlp_desc_t* desc, const void* w1p,
                                        const void* w2, const moe_nv_weights_t* out,
                                        cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!w1p || !w2 || !nv_weights_ok(out)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const long long E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  const moe_mx_weights_t& q = out->q;
  cudaError_t e = launch_amax_nv(w1p, 1, E * W1, d, nullptr, out->amax, di->sms, stream);
  if (e == cudaSuccess)
    e = launch_amax_nv(w2, 1, E * d, F, nullptr, out->amax + 2, di->sms, stream);
  if (e == cudaSuccess)
    e = launch_quant_nv(w1p, E, W1, d, static_cast<uint8_t*>(q.w1), static_cast<uint8_t*>(q.w1_s),
                        static_cast<uint8_t*>(q.w1t), static_cast<uint8_t*>(q.w1t_s), out->amax,
                        out->amax, 0, nullptr, di->sms, stream);
  if (e == cudaSuccess)
    e = launch_quant_nv(w2, E, d, F, static_cast<uint8_t*>(q.w2), static_cast<uint8_t*>(q.w2_s),
                        static_cast<uint8_t*>(q.w2t), static_cast<uint8_t*>(q.w2t_s),
                        out->amax + 2, out->amax + 2, 0, nullptr, di->sms, stream);
  return cuda_status(e);
}

moe_status_t moe_fc1_glu_fwd_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_nv,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const moe_nv_weights_t* w, const void* b1p, void* h, void* a,
                                float* a_amax, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !nv_weights_ok(w) || !a || !a_amax) return MOE_ERR_NULL;
  if (!h && !desc->recompute_h) return MOE_ERR_NULL;   // H kept unless recomputed
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!nv_ok(x_nv, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // x_perm (codes [cap, d/2]) x W1p (codes [E, W1, d/2]); GLU epilogue
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, x_nv->q, d / 2, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->q.w1, d / 2, W1, E, 256) ||
      (h && !encode_out(&g.tma_out0, h, W1, cap, 1)) || !encode_out(&g.tma_out1, a, F, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.out1 = a;
  g.ld1 = F;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  set_nv_scales(g, x_nv->scale, cap, w->q.w1_s, W1, nv_sf_bytes(W1, d), x_nv->amax, w->amax);
  if ((st = set_amax_out(g, a_amax, desc->F, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm_nv(desc->act == MOE_ACT_SRELU ? kFc1Act : kFc1Glu, g,
                                            grid_for(di, desc), stream));
}

moe_status_t moe_fc1_recompute_h_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_nv,
                                    const int32_t* counts, const int32_t* padded_offsets,
                                    const moe_nv_weights_t* w, const void* b1p, void* h,
                                    cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !nv_weights_ok(w) || !h) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!nv_ok(x_nv, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // the FC2-shaped plain kernel with W1p as B on the forward's NVFP4 operands
  // (same MMAs, same 1/(g_a g_b) and bias): bitwise the H FC1 would store
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, x_nv->q, d / 2, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->q.w1, d / 2, W1, E, 256) || !encode_out(&g.tma_out0, h, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  set_nv_scales(g, x_nv->scale, cap, w->q.w1_s, W1, nv_sf_bytes(W1, d), x_nv->amax, w->amax);
  return cuda_status(launch_grouped_gemm_nv(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_fwd_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* a_nv,
                            const int32_t* counts, const int32_t* padded_offsets,
                            const moe_nv_weights_t* w, const void* b2, void* y,
                            cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !nv_weights_ok(w) || !y) return MOE_ERR_NULL;
  if (desc->has_b2 && !b2) return MOE_ERR_NULL;
  if (!nv_ok(a_nv, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F;
  const uint64_t cap = desc->capacity;
  // A (codes [cap, F/2]) x W2 (codes [E, d, F/2])
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, a_nv->q, F / 2, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->q.w2, F / 2, d, E, 256) || !encode_out(&g.tma_out0, y, d, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->F;
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = y;
  g.ld0 = d;
  g.bias = desc->has_b2 ? b2 : nullptr;
  g.bias_ld = d;
  set_nv_scales(g, a_nv->scale, cap, w->q.w2_s, d, nv_sf_bytes(d, F), a_nv->amax, w->amax + 2);
  return cuda_status(launch_grouped_gemm_nv(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_dgrad_dglu_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_nv,
                                   const void* h, const int32_t* counts,
                                   const int32_t* padded_offsets, const moe_nv_weights_t* w,
                                   void* dh, float* dh_amax, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!h || !counts || !padded_offsets || !nv_weights_ok(w) || !dh || !dh_amax)
    return MOE_ERR_NULL;
  if (!nv_ok(dy_nv, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, Fp = fc1_pad(desc->F),
                 W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dY (codes [cap, d/2]) x W2^T (codes [E, F, d/2]); dGLU epilogue reads H
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dy_nv->q, d / 2, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->q.w2t, d / 2, F, E, 256) ||
      !encode_out(&g.tma_out0, dh, W1, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = desc->act == MOE_ACT_SRELU ? desc->F : static_cast<int>(Fp);
  g.b_ext = desc->F;
  g.out0 = dh;
  g.ld0 = W1;
  g.aux = h;
  g.ld_aux = W1;
  set_nv_scales(g, dy_nv->scale, cap, w->q.w2t_s, F, nv_sf_bytes(F, d), dy_nv->amax,
                w->amax + 2);
  if ((st = set_amax_out(g, dh_amax, W1, stream)) != MOE_OK) return st;
  return cuda_status(launch_grouped_gemm_nv(desc->act == MOE_ACT_SRELU ? kDgradAct : kDgradDglu,
                                            g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_wgrad_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_nv,
                              const moe_mx_out_t* a_nv, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw2, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !dw2) return MOE_ERR_NULL;
  if (!nv_ok(dy_nv, false, true) || !nv_ok(a_nv, false, true)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F;
  const uint64_t cap = desc->capacity;
  // dW2[e] = (H dY)^T (H A) over the group's rows: codes [d, cap/2], [F, cap/2]
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dy_nv->qt, cap / 2, d, 1, 128) ||
      !encode_u8(&g.tma_b, a_nv->qt, cap / 2, F, 1, 256) || !encode_out(&g.tma_out0, dw2, F, d, E))
    return MOE_ERR_SHAPE;
  g.m_ext = desc->d;
  g.n_ext = desc->F;
  g.b_ext = desc->F;
  g.out0 = dw2;
  g.ld0 = F;
  set_nv_scales(g, dy_nv->scale_t, d, a_nv->scale_t, F, 0, dy_nv->amax + 1, a_nv->amax + 1);
  return cuda_status(launch_grouped_gemm_nv(kWgrad, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_dgrad_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_nv,
                              const int32_t* counts, const int32_t* padded_offsets,
                              const moe_nv_weights_t* w, void* dx_perm, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !nv_weights_ok(w) || !dx_perm) return MOE_ERR_NULL;
  if (!nv_ok(dh_nv, true, false)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dH (codes [cap, W1/2]) x W1p^T (codes [E, d, W1/2])
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dh_nv->q, W1 / 2, cap, 1, 128) ||
      !encode_u8(&g.tma_b, w->q.w1t, W1 / 2, d, E, 256) ||
      !encode_out(&g.tma_out0, dx_perm, d, cap, 1))
    return MOE_ERR_SHAPE;
  g.K = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dx_perm;
  g.ld0 = d;
  set_nv_scales(g, dh_nv->scale, cap, w->q.w1t_s, d, nv_sf_bytes(d, W1), dh_nv->amax, w->amax);
  return cuda_status(launch_grouped_gemm_nv(kDgradFc1, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_wgrad_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_nv,
                              const moe_mx_out_t* x_nv, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw1p, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!counts || !padded_offsets || !dw1p) return MOE_ERR_NULL;
  if (!nv_ok(dh_nv, false, true) || !nv_ok(x_nv, false, true)) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dW1p[e] = (H dH)^T (H X) over the group's rows: codes [W1, cap/2], [d, cap/2]
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_u8(&g.tma_a, dh_nv->qt, cap / 2, W1, 1, 128) ||
      !encode_u8(&g.tma_b, x_nv->qt, cap / 2, d, 1, 256) ||
      !encode_out(&g.tma_out0, dw1p, d, W1, E))
    return MOE_ERR_SHAPE;
  g.m_ext = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dw1p;
  g.ld0 = d;
  set_nv_scales(g, dh_nv->scale_t, W1, x_nv->scale_t, d, 0, dh_nv->amax + 1, x_nv->amax + 1);
  return cuda_status(launch_grouped_gemm_nv(kWgrad, g, grid_for(di, desc), stream));
}

moe_status_t moe_mlp_fwd_nv(const moe_mlp_desc_t* desc, const void* x_perm,
                            const moe_mx_out_t* x_nv, const int32_t* counts,
                            const int32_t* padded_offsets, const moe_nv_weights_t* w,
                            const void* b1p, const void* b2, void* h, void* a,
                            const moe_mx_out_t* a_nv, void* y, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!x_perm || !a || !y || !a_nv) return MOE_ERR_NULL;   // h may be NULL with recompute_h
  if ((st = moe_quantize_act_nvfp4(desc, x_perm, desc->d, padded_offsets, x_nv, 1, stream)) !=
          MOE_OK ||
      (st = moe_fc1_glu_fwd_nv(desc, x_nv, counts, padded_offsets, w, b1p, h, a, a_nv->amax,
                               stream)) != MOE_OK ||
      (st = moe_quantize_act_nvfp4(desc, a, desc->F, padded_offsets, a_nv, 0, stream)) != MOE_OK)
    return st;
  return moe_fc2_fwd_nv(desc, a_nv, counts, padded_offsets, w, b2, y, stream);
}

moe_status_t moe_mlp_bwd_nv(const moe_mlp_desc_t* desc, const void* dy,
                            const moe_mx_out_t* dy_nv, const moe_mx_out_t* x_nv, const void* h,
                            const moe_mx_out_t* a_nv, const int32_t* counts,
                            const int32_t* padded_offsets, const moe_nv_weights_t* w, void* dh,
                            const moe_mx_out_t* dh_nv, void* dx_perm, void* dw1p, void* db1p,
                            void* dw2, void* db2, cudaStream_t stream) {
  moe_status_t st = check_nv_desc(desc);
  if (st != MOE_OK) return st;
  if (!dy || !dh || !dh_nv || !dx_perm || !dw1p || !dw2) return MOE_ERR_NULL;
  const int32_t W1 = fc1_width(desc->act, desc->F);
  if ((st = moe_quantize_act_nvfp4(desc, dy, desc->d, padded_offsets, dy_nv, 1, stream)) !=
          MOE_OK ||
      (st = moe_fc2_dgrad_dglu_nv(desc, dy_nv, h, counts, padded_offsets, w, dh, dh_nv->amax,
                                  stream)) != MOE_OK ||
      (st = moe_quantize_act_nvfp4(desc, dh, W1, padded_offsets, dh_nv, 0, stream)) != MOE_OK ||
      (st = moe_fc2_wgrad_nv(desc, dy_nv, a_nv, counts, padded_offsets, dw2, stream)) != MOE_OK ||
      (st = moe_fc1_dgrad_nv(desc, dh_nv, counts, padded_offsets, w, dx_perm, stream)) !=
          MOE_OK ||
      (st = moe_fc1_wgrad_nv(desc, dh_nv, x_nv, counts, padded_offsets, dw1p, stream)) != MOE_OK)
    return st;
  if (db1p || db2) return moe_bias_grads(desc, dy, dh, counts, padded_offsets, db1p, db2, stream);
  return MOE_OK;
}

}  // extern "C"

// ===========================================================================
// fp32 tensors (MOE_DTYPE_FP32): the grouped GEMMs on TF32 tensor cores
// (tcgen05 kind::tf32) with the same fused epilogues; every operand K-major,
// the backward's transposed operands from transposed copies.
namespace moe {
namespace {

// fp32 operand [E][rows][K] (K contiguous), boxes of 32 K x box_rows rows.
bool encode_f32(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint64_t E,
                uint32_t box_rows) {
  return encode_map(map, base, K, rows, E, K * 4, rows * K * 4, 32, box_rows,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

moe_status_t check_f32_desc(const moe_mlp_desc_t* d) {
  moe_status_t st = check_desc(d, false);
  if (st != MOE_OK) return st;
  if (d->dtype != MOE_DTYPE_FP32 || d->recompute_h) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status_t moe_transpose_weights_tf32(const moe_mlp_desc_t* desc, const void* w1p,
                                        const void* w2, void* w1t, void* w2t,
                                        cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!w1p || !w2 || !w1t || !w2t) return MOE_ERR_NULL;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const long long E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  cudaError_t e = launch_transpose_f32(w1p, E, W1, d, w1t, nullptr, stream);
  if (e == cudaSuccess) e = launch_transpose_f32(w2, E, d, F, w2t, nullptr, stream);
  return cuda_status(e);
}

moe_status_t moe_transpose_rows_f32(const moe_mlp_desc_t* desc, const void* in, int32_t width,
                                    const int32_t* padded_offsets, void* out,
                                    cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!in || !padded_offsets || !out) return MOE_ERR_NULL;
  if (width < 1) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  return cuda_status(launch_transpose_f32(in, 1, desc->capacity, width, out,
                                          padded_offsets + desc->E, stream));
}

moe_status_t moe_fc1_glu_fwd_tf32(const moe_mlp_desc_t* desc, const void* x_perm,
                                  const int32_t* counts, const int32_t* padded_offsets,
                                  const void* w1p, const void* b1p, void* h, void* a, void* a_t,
                                  cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!x_perm || !counts || !padded_offsets || !w1p || !h || !a) return MOE_ERR_NULL;
  if (desc->has_b1 && !b1p) return MOE_ERR_NULL;
  if (!al16(h) || !al16(a) || !al16(a_t)) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // x_perm [cap, d] x W1p [E, W1, d]^T; GLU epilogue (A^T optional)
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_f32(&g.tma_a, x_perm, d, cap, 1, 128) || !encode_f32(&g.tma_b, w1p, d, W1, E, 256))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = static_cast<int>(W1);
  g.b_ext = g.n_ext;
  g.out0 = h;
  g.ld0 = W1;
  g.out1 = a;
  g.ld1 = desc->F;
  g.out1_t = static_cast<float*>(a_t);
  g.bias = desc->has_b1 ? b1p : nullptr;
  g.bias_ld = W1;
  return cuda_status(launch_grouped_gemm_tf32(desc->act == MOE_ACT_SRELU ? kFc1Act : kFc1Glu, g,
                                              grid_for(di, desc), stream));
}

moe_status_t moe_fc2_fwd_tf32(const moe_mlp_desc_t* desc, const void* a, const int32_t* counts,
                              const int32_t* padded_offsets, const void* w2, const void* b2,
                              void* y, cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!a || !counts || !padded_offsets || !w2 || !y) return MOE_ERR_NULL;
  if (desc->has_b2 && !b2) return MOE_ERR_NULL;
  if (!al16(y)) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, cap = desc->capacity;
  // A [cap, F] x W2 [E, d, F]^T
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_f32(&g.tma_a, a, F, cap, 1, 128) || !encode_f32(&g.tma_b, w2, F, d, E, 256))
    return MOE_ERR_SHAPE;
  g.K = desc->F;
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = y;
  g.ld0 = d;
  g.bias = desc->has_b2 ? b2 : nullptr;
  g.bias_ld = d;
  return cuda_status(launch_grouped_gemm_tf32(kFc2, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_dgrad_dglu_tf32(const moe_mlp_desc_t* desc, const void* dy, const void* h,
                                     const int32_t* counts, const int32_t* padded_offsets,
                                     const void* w2t, void* dh, void* dh_t, cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!dy || !h || !counts || !padded_offsets || !w2t || (!dh && !dh_t)) return MOE_ERR_NULL;
  if (!al16(h) || !al16(dh) || !al16(dh_t)) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dY [cap, d] x W2^T [E, F, d]^T; the dGLU epilogue reads H
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_f32(&g.tma_a, dy, d, cap, 1, 128) || !encode_f32(&g.tma_b, w2t, d, F, E, 256))
    return MOE_ERR_SHAPE;
  g.K = desc->d;
  g.n_ext = desc->act == MOE_ACT_SRELU ? desc->F : fc1_pad(desc->F);
  g.b_ext = desc->F;
  g.out0 = dh;
  g.ld0 = W1;
  g.out0_t = static_cast<float*>(dh_t);
  g.aux = h;
  g.ld_aux = W1;
  return cuda_status(launch_grouped_gemm_tf32(desc->act == MOE_ACT_SRELU ? kDgradAct : kDgradDglu,
                                              g, grid_for(di, desc), stream));
}

moe_status_t moe_fc2_wgrad_tf32(const moe_mlp_desc_t* desc, const void* dy_t, const void* a_t,
                                const int32_t* counts, const int32_t* padded_offsets, void* dw2,
                                cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!dy_t || !a_t || !counts || !padded_offsets || !dw2) return MOE_ERR_NULL;
  if (!al16(dw2)) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t d = desc->d, F = desc->F, cap = desc->capacity;
  // dW2[e] = dY^T A over the group's rows: [d, cap] and [F, cap]
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_f32(&g.tma_a, dy_t, cap, d, 1, 128) || !encode_f32(&g.tma_b, a_t, cap, F, 1, 256))
    return MOE_ERR_SHAPE;
  g.m_ext = desc->d;
  g.n_ext = desc->F;
  g.b_ext = desc->F;
  g.out0 = dw2;
  g.ld0 = F;
  return cuda_status(launch_grouped_gemm_tf32(kWgrad, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_dgrad_tf32(const moe_mlp_desc_t* desc, const void* dh,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const void* w1t, void* dx_perm, cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!dh || !counts || !padded_offsets || !w1t || !dx_perm) return MOE_ERR_NULL;
  if (!al16(dx_perm)) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t E = desc->E, d = desc->d, W1 = fc1_width(desc->act, desc->F);
  const uint64_t cap = desc->capacity;
  // dH [cap, W1] x W1p^T [E, d, W1]^T
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_f32(&g.tma_a, dh, W1, cap, 1, 128) || !encode_f32(&g.tma_b, w1t, W1, d, E, 256))
    return MOE_ERR_SHAPE;
  g.K = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dx_perm;
  g.ld0 = d;
  return cuda_status(launch_grouped_gemm_tf32(kDgradFc1, g, grid_for(di, desc), stream));
}

moe_status_t moe_fc1_wgrad_tf32(const moe_mlp_desc_t* desc, const void* dh_t, const void* x_t,
                                const int32_t* counts, const int32_t* padded_offsets,
                                void* dw1p, cudaStream_t stream) {
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (!dh_t || !x_t || !counts || !padded_offsets || !dw1p) return MOE_ERR_NULL;
  if (!al16(dw1p)) return MOE_ERR_SHAPE;
  DeviceInfo* di;
  if ((st = device_info(&di)) != MOE_OK) return st;
  const uint64_t d = desc->d, W1 = fc1_width(desc->act, desc->F), cap = desc->capacity;
  // dW1p[e] = dH^T X over the group's rows: [W1, cap] and [d, cap]
  GemmArgs g;
  fill_common(g, desc, di, counts, padded_offsets);
  if (!encode_f32(&g.tma_a, dh_t, cap, W1, 1, 128) || !encode_f32(&g.tma_b, x_t, cap, d, 1, 256))
    return MOE_ERR_SHAPE;
  g.m_ext = static_cast<int>(W1);
  g.n_ext = desc->d;
  g.b_ext = desc->d;
  g.out0 = dw1p;
  g.ld0 = d;
  return cuda_status(launch_grouped_gemm_tf32(kWgrad, g, grid_for(di, desc), stream));
}

}  // extern "C"

namespace moe {
namespace {

moe_status_t mlp_fwd_tf32(const moe_mlp_desc_t* desc, const void* x_perm, const int32_t* counts,
                          const int32_t* padded_offsets, const void* w1p, const void* b1p,
                          const void* w2, const void* b2, void* h, void* a, void* y,
                          const moe_mx_out_t* a_mx, const moe_mx_out_t* y_mx,
                          cudaStream_t stream) {
  if (a_mx || y_mx) return MOE_ERR_UNSUPPORTED;
  moe_status_t st = moe_fc1_glu_fwd_tf32(desc, x_perm, counts, padded_offsets, w1p, b1p, h, a,
                                         nullptr, stream);
  if (st != MOE_OK) return st;
  return moe_fc2_fwd_tf32(desc, a, counts, padded_offsets, w2, b2, y, stream);
}

moe_status_t mlp_bwd_tf32(const moe_mlp_desc_t* desc, const void* dy, const void* x_perm,
                          const void* h, const void* a, const int32_t* counts,
                          const int32_t* padded_offsets, const void* w1p, const void* b1p,
                          const void* w2, void* dh, void* dx_perm, void* dw1p, void* db1p,
                          void* dw2, void* db2, const moe_mx_out_t* dh_mx, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  (void)b1p;
  moe_status_t st = check_f32_desc(desc);
  if (st != MOE_OK) return st;
  if (dh_mx) return MOE_ERR_UNSUPPORTED;
  if (!dy || !x_perm || !h || !a || !counts || !padded_offsets || !w1p || !w2 || !dh ||
      !dx_perm || !dw1p || !dw2)
    return MOE_ERR_NULL;
  if ((desc->has_b1 && !db1p) || (desc->has_b2 && !db2)) return MOE_ERR_NULL;
  size_t need = 0;
  if ((st = moe_workspace_size(desc, &need)) != MOE_OK) return st;
  if (!ws || ws_bytes < need || !al16(ws)) return MOE_ERR_WORKSPACE;
  auto r = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t E = desc->E, d = desc->d, F = desc->F, W1 = fc1_width(desc->act, desc->F),
               cap = desc->capacity;
  uint8_t* p = static_cast<uint8_t*>(ws) + r(route_ws_bytes(desc) + 256);
  void* w1t = p;  p += r(E * d * W1 * 4);
  void* w2t = p;  p += r(E * F * d * 4);
  void* x_t = p;  p += r(d * cap * 4);
  void* dy_t = p; p += r(d * cap * 4);
  void* a_t = p;  p += r(F * cap * 4);
  void* dh_t = p;
  const int32_t dd = desc->d, ff = desc->F;
  if ((st = moe_transpose_weights_tf32(desc, w1p, w2, w1t, w2t, stream)) != MOE_OK ||
      (st = moe_transpose_rows_f32(desc, x_perm, dd, padded_offsets, x_t, stream)) != MOE_OK ||
      (st = moe_transpose_rows_f32(desc, dy, dd, padded_offsets, dy_t, stream)) != MOE_OK ||
      (st = moe_transpose_rows_f32(desc, a, ff, padded_offsets, a_t, stream)) != MOE_OK ||
      (st = moe_fc2_dgrad_dglu_tf32(desc, dy, h, counts, padded_offsets, w2t, dh, dh_t,
                                    stream)) != MOE_OK ||
      (st = moe_fc2_wgrad_tf32(desc, dy_t, a_t, counts, padded_offsets, dw2, stream)) != MOE_OK ||
      (st = moe_fc1_dgrad_tf32(desc, dh, counts, padded_offsets, w1t, dx_perm, stream)) !=
          MOE_OK ||
      (st = moe_fc1_wgrad_tf32(desc, dh_t, x_t, counts, padded_offsets, dw1p, stream)) != MOE_OK)
    return st;
  if (desc->has_b1 || desc->has_b2)
    st = moe_bias_grads(desc, dy, dh, counts, padded_offsets, desc->has_b1 ? db1p : nullptr,
                        desc->has_b2 ? db2 : nullptr, stream);
  return st;
}

}  // namespace
}  // namespace moe
