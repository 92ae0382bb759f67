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

// bf16 [batch][rows][cols] -> MXFP8 (rows, cols multiples of 32).  A CTA
// (8 warps) walks 128 x 128 tiles; each tile is loaded coalesced into four
// shared boxes of 128 rows x 32 columns (64-byte rows, 64-byte swizzle) with
// cp.async, double-buffered so that the next tile streams in while the
// current one is quantized and stored; each warp quantizes 32 x 32 blocks
// rowwise (lane = row) or columnwise (lane = column) into shared code
// tiles; the codes then leave as whole 128-byte lines and, in the MMA scale
// layout, each tile's scales as one 512-byte atom per direction.  Rowwise
// codes [batch][rows][cols]; columnwise codes transposed [batch][cols][rows].
// Rows at or past *row_limit (when given; in every batch entry) are not
// visited.
constexpr int kQT = 128;                       // tile edge
constexpr int kQThreads = 256;                 // 8 warps, two CTAs per SM
constexpr int kQIn = 4 * 8192;                 // one bf16 input tile (four boxes)
constexpr int kQuantSmem = 2 * kQIn + 2 * kQT * kQT + 2 * 512;

__device__ __forceinline__ void quant_block_to_smem(const float (&v)[32], uint8_t* code_row,
                                                    int line, int c32, uint8_t& scale) {
  // codes of one block row (32 bytes) into line `line` of a 128 x 128 code
  // tile at column c32*32; 16-byte chunks swizzled by (line & 7)
  uint32_t w[8];
  scale = mx_quant32_words(v, w);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int ch = (c32 * 2 + h) ^ (line & 7);
    *reinterpret_cast<uint4*>(code_row + line * kQT + ch * 16) =
        make_uint4(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
  }
}

struct QuantTile {
  long long b, r0, c0;
  int nr, nc;
};

__device__ __forceinline__ QuantTile quant_tile(long long t, long long rtn, long long ctn,
                                                long long rows, long long cols) {
  QuantTile q;
  q.b = t / (rtn * ctn);
  const long long rem = t - q.b * rtn * ctn;
  q.r0 = (rem / ctn) * kQT;
  q.c0 = (rem % ctn) * kQT;
  q.nr = static_cast<int>(min(static_cast<long long>(kQT), rows - q.r0));   // multiples of 32
  q.nc = static_cast<int>(min(static_cast<long long>(kQT), cols - q.c0));
  return q;
}

// Asynchronous load of one tile into `boxes` (thread -> 16-byte chunks; the
// chunks outside the tensor are zero-filled).
__device__ __forceinline__ void quant_load_async(const __nv_bfloat16* __restrict__ in,
                                                 const QuantTile& q, long long rows,
                                                 long long cols, uint8_t* boxes, int tid) {
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(boxes));
  for (int i = tid; i < kQT * 16; i += kQThreads) {
    const int r = i >> 4, ch = i & 15;
    const bool ok = r < q.nr && ch * 8 < q.nc;
    const __nv_bfloat16* src = ok ? in + (q.b * rows + q.r0 + r) * cols + q.c0 + ch * 8 : in;
    cp_async16_zfill(base + (ch >> 2) * 8192 + r * 64 + (((ch & 3) ^ ((r >> 1) & 3)) << 4),
                     src, ok);
  }
}

__global__ void __launch_bounds__(kQThreads, 2) k_quant_bf16(const __nv_bfloat16* __restrict__ in,
                                                    long long batch, long long rows,
                                                    long long cols, uint8_t* q, uint8_t* s,
                                                    uint8_t* qt, uint8_t* st, int mma_layout,
                                                    const int32_t* row_limit) {
  extern __shared__ __align__(1024) uint8_t qsm[];
  uint8_t* in_buf = qsm;                             // 2 x (4 x [128][64 B])
  uint8_t* code_r = qsm + 2 * kQIn;                  // [128 rows][128 B]
  uint8_t* code_c = code_r + kQT * kQT;              // [128 cols][128 B]
  uint8_t* atom_r = code_c + kQT * kQT;              // scale atoms (MMA layout)
  uint8_t* atom_c = atom_r + 512;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const long long rlim = row_limit ? min(rows, static_cast<long long>(__ldg(row_limit))) : rows;
  const long long rtn = (rlim + kQT - 1) / kQT, ctn = (cols + kQT - 1) / kQT;
  const long long ntiles = batch * rtn * ctn;
  const long long s_bytes = mma_layout ? (cols + 127) / 128 * sf_row_atoms(rows) * 512
                                       : rows * cols / 32;
  const long long st_bytes = mma_layout ? (rows + 127) / 128 * sf_row_atoms(cols) * 512
                                        : rows * cols / 32;
  for (int i = tid; i < 1024; i += kQThreads) atom_r[i] = 0;     // both atoms
  long long t = blockIdx.x;
  if (t < ntiles) quant_load_async(in, quant_tile(t, rtn, ctn, rows, cols), rows, cols, in_buf, tid);
  cp_async_commit();
  for (int it = 0; t < ntiles; t += gridDim.x, ++it) {
    const QuantTile qt_ = quant_tile(t, rtn, ctn, rows, cols);
    const long long b = qt_.b, r0 = qt_.r0, c0 = qt_.c0;
    const int nr = qt_.nr, nc = qt_.nc;
    // the next tile streams into the other buffer (its last reader, the
    // previous iteration's quantization, finished before that iteration's
    // second barrier)
    const long long tn = t + gridDim.x;
    if (tn < ntiles)
      quant_load_async(in, quant_tile(tn, rtn, ctn, rows, cols), rows, cols,
                       in_buf + ((it + 1) & 1) * kQIn, tid);
    cp_async_commit();
    cp_async_wait<1>();                              // this thread's chunks of tile t landed
    __syncthreads();                                 // all of tile t; previous tile stored
    const uint8_t* boxes = in_buf + (it & 1) * kQIn;
    // quantize: 16 blocks x {rowwise, columnwise}; warp w takes items w + 8k
    for (int item = wid; item < 32; item += kQThreads / 32) {
      const int colwise = item >> 4, blk = item & 15;
      const int bi = blk >> 2, bj = blk & 3;         // block row / column in the tile
      if (bi * 32 >= nr || bj * 32 >= nc) continue;  // warp-uniform
      if ((colwise ? qt : q) == nullptr) continue;
      const uint8_t* box = boxes + bj * 8192;
      float v[32];
      if (!colwise) {
        const int r = bi * 32 + lane;
        const uint4* rowp = reinterpret_cast<const uint4*>(box + r * 64);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const uint4 w4 = rowp[c4 ^ ((r >> 1) & 3)];
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * c4 + 2 * k] = __uint_as_float(w[k] << 16);
            v[8 * c4 + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
          }
        }
        uint8_t sc;
        quant_block_to_smem(v, code_r, r, bj, sc);
        if (mma_layout)
          atom_r[(r & 31) * 16 + (r >> 5) * 4 + bj] = sc;
        else
          s[b * s_bytes + (r0 + r) * (cols / 32) + c0 / 32 + bj] = sc;
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int r = bi * 32 + i;
          const uint16_t h = *reinterpret_cast<const uint16_t*>(
              box + r * 64 + ((((lane >> 3) ^ ((r >> 1) & 3))) << 4) + (lane & 7) * 2);
          v[i] = __uint_as_float(static_cast<uint32_t>(h) << 16);
        }
        const int c = bj * 32 + lane;                // column inside the tile
        uint8_t sc;
        quant_block_to_smem(v, code_c, c, bi, sc);
        if (mma_layout)
          atom_c[(c & 31) * 16 + (c >> 5) * 4 + bi] = sc;
        else
          st[b * st_bytes + (c0 + c) * (rows / 32) + r0 / 32 + bi] = sc;
      }
    }
    __syncthreads();
    // store codes as whole lines: thread -> 16-byte chunk (line i / 8)
    for (int i = tid; i < kQT * 8; i += kQThreads) {
      const int line = i >> 3, ch = i & 7;
      const int sch = ch ^ (line & 7);
      if (q && line < nr && ch * 16 < nc)
        *reinterpret_cast<uint4*>(q + (b * rows + r0 + line) * cols + c0 + ch * 16) =
            *reinterpret_cast<const uint4*>(code_r + line * kQT + sch * 16);
      if (qt && line < nc && ch * 16 < nr)
        *reinterpret_cast<uint4*>(qt + (b * cols + c0 + line) * rows + r0 + ch * 16) =
            *reinterpret_cast<const uint4*>(code_c + line * kQT + sch * 16);
    }
    if (mma_layout && tid < 64) {                    // one 512-byte atom per direction
      const int h = tid >> 5, k = tid & 31;
      if (h == 0 && q)
        reinterpret_cast<uint4*>(s + b * s_bytes + sf_mma_offset(r0, c0 / 32, sf_row_atoms(rows)))[k] =
            reinterpret_cast<const uint4*>(atom_r)[k];
      if (h == 1 && qt)
        reinterpret_cast<uint4*>(st + b * st_bytes + sf_mma_offset(c0, r0 / 32, sf_row_atoms(cols)))[k] =
            reinterpret_cast<const uint4*>(atom_c)[k];
    }
    __syncthreads();                                 // code tiles and atoms free again
    for (int i = tid; i < 1024; i += kQThreads) atom_r[i] = 0;   // both atoms, for the next tile
  }
  cp_async_wait<0>();
}

}  // namespace

cudaError_t launch_quant_bf16_mx(const void* in, long long batch, long long rows, long long cols,
                                 uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                                 int mma_layout, const int32_t* row_limit, int num_sms,
                                 cudaStream_t stream) {
  const long long ntiles = batch * ((rows + kQT - 1) / kQT) * ((cols + kQT - 1) / kQT);
  if (ntiles == 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(k_quant_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kQuantSmem);
  if (err != cudaSuccess) return err;
  long long grid = ntiles;
  if (grid > static_cast<long long>(num_sms) * 2) grid = static_cast<long long>(num_sms) * 2;
  k_quant_bf16<<<static_cast<int>(grid), kQThreads, kQuantSmem, stream>>>(
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
