// Standalone MXFP8 quantization (rowwise, or columnwise written transposed),
// using the same device quantizer as the fused GEMM epilogues.  It exists so
// that codes and scales can be checked bit for bit against the oracle on
// identical fp32 inputs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "moe_mx.cuh"
#include "moe_ptx.cuh"

namespace moe {
namespace {

// Rowwise: one thread per 32-element block of a row.
__global__ void __launch_bounds__(256) k_quant_rows(const float* __restrict__ in, int rows,
                                                    int cols, uint8_t* __restrict__ q,
                                                    uint8_t* __restrict__ scales) {
  const int bpr = cols / 32;
  const long long nblk = static_cast<long long>(rows) * bpr;
  for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nblk;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = b / bpr, c = (b - r * bpr) * 32;
    const float4* src = reinterpret_cast<const float4*>(in + r * cols + c);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = __ldg(src + i);
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    scales[b] = mx_quant32(v, q + r * cols + c);
  }
}

// Columnwise: one thread per (column, 32-row block); codes go to the
// transposed tensor qT [cols, rows], scales to [cols, rows/32].
__global__ void __launch_bounds__(256) k_quant_cols(const float* __restrict__ in, int rows,
                                                    int cols, uint8_t* __restrict__ qt,
                                                    uint8_t* __restrict__ scales) {
  const int rb_n = rows / 32;
  const long long nblk = static_cast<long long>(cols) * rb_n;
  for (long long b = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; b < nblk;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long rb = b / cols, c = b - rb * cols;     // adjacent threads: adjacent columns
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __ldg(in + (rb * 32 + i) * cols + c);
    scales[c * rb_n + rb] = mx_quant32(v, qt + c * rows + rb * 32);
  }
}

// bf16 [batch][rows][cols] -> MXFP8, one warp per 32 x 32 block,
// consecutive warps on consecutive column blocks of the same rows.  The
// block is read coalesced (lane l: 16-byte chunk l % 4 of rows l / 4 + 8k)
// into the warp's shared box (64-byte rows, 64-byte swizzle), from which
// lane l quantizes row l and column l.  Rowwise codes [batch][rows][cols];
// columnwise codes written transposed [batch][cols][rows]; scales row-major
// or in the MMA layout.
__global__ void __launch_bounds__(256) k_quant_bf16(const __nv_bfloat16* __restrict__ in,
                                                    long long batch, long long rows,
                                                    long long cols, uint8_t* q, uint8_t* s,
                                                    uint8_t* qt, uint8_t* st, int mma_layout,
                                                    const int32_t* row_limit) {
  __shared__ __align__(128) uint8_t boxes[8][32 * 64];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint8_t* const box = boxes[wid];
  const long long rbn = rows / 32, cbn = cols / 32;
  const long long per_batch = rbn * cbn;
  const long long nblk = batch * per_batch;
  const long long s_bytes = mma_layout ? (cols + 127) / 128 * sf_row_atoms(rows) * 512
                                       : rows * cols / 32;
  const long long st_bytes = mma_layout ? (rows + 127) / 128 * sf_row_atoms(cols) * 512
                                        : rows * cols / 32;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const long long rlim = row_limit ? __ldg(row_limit) : rows;   // rows past it are skipped
  for (long long w = blockIdx.x * static_cast<long long>(blockDim.x / 32) + wid; w < nblk;
       w += warps) {
    const long long b = w / per_batch;
    const long long rem = w - b * per_batch;
    const long long rb = rem / cbn, cb = rem - rb * cbn;
    if (rb * 32 >= rlim) continue;
    const __nv_bfloat16* src = in + (b * rows + rb * 32) * cols + cb * 32;
    __syncwarp();                       // the previous block's reads are done
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = (lane >> 2) + 8 * k, ch = lane & 3;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + r * cols) + ch);
      *reinterpret_cast<uint4*>(box + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4)) = v;
    }
    __syncwarp();
    const MxOut mx{q ? q + b * rows * cols : nullptr, s ? s + b * s_bytes : nullptr,
                   qt ? qt + b * rows * cols : nullptr, st ? st + b * st_bytes : nullptr,
                   nullptr, cols, rows, mma_layout};
    mx_block_from_box(mx, box, 0, rb * 32, static_cast<int>(cb * 32), lane);
  }
}

}  // namespace

cudaError_t launch_quant_bf16_mx(const void* in, long long batch, long long rows, long long cols,
                                 uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                                 int mma_layout, const int32_t* row_limit, int num_sms,
                                 cudaStream_t stream) {
  const long long nblk = batch * (rows / 32) * (cols / 32);
  if (nblk == 0) return cudaSuccess;
  long long grid = (nblk + 7) / 8;
  if (grid > static_cast<long long>(num_sms) * 16) grid = static_cast<long long>(num_sms) * 16;
  k_quant_bf16<<<static_cast<int>(grid), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(in), batch, rows, cols, q, s, qt, st, mma_layout,
      row_limit);
  return cudaGetLastError();
}

}  // namespace moe

extern "C" moe_status_t moe_quantize_mx(const float* in, int32_t rows, int32_t cols,
                                        int32_t colwise, uint8_t* q, uint8_t* scales,
                                        cudaStream_t stream) {
  if (!in || !q || !scales) return MOE_ERR_NULL;
  if (rows < 0 || cols < 0) return MOE_ERR_SHAPE;
  if (colwise ? (rows % 32 != 0) : (cols % 32 != 0)) return MOE_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(in) & 15) || (reinterpret_cast<uintptr_t>(q) & 15))
    return MOE_ERR_SHAPE;
  if (rows == 0 || cols == 0) return MOE_OK;
  const long long nblk = static_cast<long long>(rows) * cols / 32;
  const int grid = static_cast<int>((nblk + 255) / 256 < 65535 ? (nblk + 255) / 256 : 65535);
  if (colwise)
    moe::k_quant_cols<<<grid, 256, 0, stream>>>(in, rows, cols, q, scales);
  else
    moe::k_quant_rows<<<grid, 256, 0, stream>>>(in, rows, cols, q, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
