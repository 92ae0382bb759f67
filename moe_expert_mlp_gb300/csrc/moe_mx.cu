// Standalone MXFP8 quantization (rowwise, or columnwise written transposed),
// using the same device quantizer as the fused GEMM epilogues.  It exists so
// that codes and scales can be checked bit for bit against the oracle on
// identical fp32 inputs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <string.h>

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
// (8 warps, two CTAs per SM) walks 128 x 128 tiles.  One thread moves the
// data with TMA: a tile arrives as four boxes of 128 rows x 32 columns
// (64-byte rows, 64-byte swizzle), two tiles in flight per CTA, and its
// codes leave as one 128 x 128-byte box per direction (128-byte swizzle),
// clipped at the tensor's edges.  Each warp quantizes two 32 x 32 blocks
// rowwise (lane = row) and two columnwise (lane = column) from shared
// memory into the code boxes; with the scales in the MMA layout each tile's
// scales leave as one 512-byte atom per direction.  Rowwise codes
// [batch][rows][cols]; columnwise codes transposed [batch][cols][rows].
// Tiles that start at or past *row_limit (when given; in every batch entry)
// are not visited.
constexpr int kQT = 128;                       // tile edge
constexpr int kQThreads = 256;                 // 8 warps, two CTAs per SM
constexpr int kQIn = 4 * 8192;                 // one bf16 input tile (four boxes)
constexpr int kQuantSmem = 1024 + 2 * kQIn + 2 * kQT * kQT + 2 * 512;

struct QuantMaps {
  CUtensorMap in;    // bf16 (cols, rows, batch), box 32 x 128, 64-byte swizzle
  CUtensorMap q;     // u8 (cols, rows, batch), box 128 x 128, 128-byte swizzle
  CUtensorMap qt;    // u8 (rows, cols, batch), box 128 x 128, 128-byte swizzle
};

// 32 codes into line `line` of a 128 x 128-byte code box at byte column
// 32 * blk (16-byte chunks swizzled by line & 7, the 128-byte TMA swizzle)
__device__ __forceinline__ void put_codes(uint8_t* box, int line, int blk, const uint32_t (&c)[8]) {
  uint8_t* row = box + line * kQT;
  const int sw = line & 7;
  *reinterpret_cast<uint4*>(row + (((2 * blk) ^ sw) << 4)) = make_uint4(c[0], c[1], c[2], c[3]);
  *reinterpret_cast<uint4*>(row + (((2 * blk + 1) ^ sw) << 4)) = make_uint4(c[4], c[5], c[6], c[7]);
}

__device__ __forceinline__ void quant_tile_coords(long long t, long long rtn, long long ctn,
                                                  long long& b, int& r0, int& c0) {
  b = t / (rtn * ctn);
  const long long rem = t - b * rtn * ctn;
  r0 = static_cast<int>(rem / ctn) * kQT;
  c0 = static_cast<int>(rem % ctn) * kQT;
}

__device__ __forceinline__ void quant_issue_load(const QuantMaps& maps, uint8_t* dst, uint64_t* bar,
                                                 long long b, int r0, int c0) {
  mbar_arrive_expect_tx(bar, kQIn);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    tma_load_3d(dst + j * 8192, &maps.in, bar, c0 + 32 * j, r0, static_cast<int>(b));
}

__global__ void __launch_bounds__(kQThreads, 2)
    k_quant_bf16(const __grid_constant__ QuantMaps maps, long long batch, long long rows,
                 long long cols, int has_q, int has_qt, uint8_t* s, uint8_t* st, int mma_layout,
                 const int32_t* row_limit, int* status) {
  extern __shared__ uint8_t qsm_raw[];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int abort_flag;
  // 1024-byte aligned: the swizzle patterns repeat every 512 / 1024 bytes
  uint8_t* qsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(qsm_raw) + 1023) &
                                            ~static_cast<uintptr_t>(1023));
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
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
    tma_prefetch_desc(&maps.in);
    for (int k = 0; k < 2; ++k) {
      const long long t = blockIdx.x + static_cast<long long>(k) * gridDim.x;
      if (t < ntiles) {
        long long b;
        int r0, c0;
        quant_tile_coords(t, rtn, ctn, b, r0, c0);
        quant_issue_load(maps, in_buf + k * kQIn, &full[k], b, r0, c0);
      }
    }
  }
  __syncthreads();
  // per-lane offsets of the two block kinds inside a 64-byte-swizzled box:
  // rowwise, the lane's row chunks sit at q ^ ((lane >> 1) & 3); columnwise,
  // row i's chunk holding column `lane` is (lane >> 3) ^ ((i >> 1) & 3)
  const int rsw = (lane >> 1) & 3;
  const int csub = (lane & 7) * 2;
  int it = 0;
  for (long long t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
    const int buf = it & 1;
    long long b;
    int r0, c0;
    quant_tile_coords(t, rtn, ctn, b, r0, c0);
    const int nr = static_cast<int>(min(static_cast<long long>(kQT), rows - r0));
    const int nc = static_cast<int>(min(static_cast<long long>(kQT), cols - c0));
    const bool ok = mbar_wait(&full[buf], (it >> 1) & 1, status, &abort_flag);
    if (tid == 0) bulk_wait_read<0>();               // the previous tile's code boxes were read
    if (!__syncthreads_and(ok)) break;
    const uint8_t* boxes = in_buf + buf * kQIn;
    if (has_q) {
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        const int blk = wid + 8 * k, bi = blk >> 2, bj = blk & 3;
        const int r = bi * 32 + lane;                // row inside the tile
        uint8_t sc = 0;
        if (bi * 32 < nr && bj * 32 < nc) {          // warp-uniform
          const uint4* rowp = reinterpret_cast<const uint4*>(boxes + bj * 8192 + r * 64);
          uint32_t w[16], c[8];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 v = rowp[q4 ^ rsw];
            w[4 * q4] = v.x;
            w[4 * q4 + 1] = v.y;
            w[4 * q4 + 2] = v.z;
            w[4 * q4 + 3] = v.w;
          }
          sc = mx_quant32_packed(w, c);
          put_codes(code_r, r, bj, c);
          if (!mma_layout) s[b * s_bytes + (r0 + r) * (cols / 32) + c0 / 32 + bj] = sc;
        }
        if (mma_layout) atom_r[lane * 16 + bi * 4 + bj] = sc;
      }
    }
    if (has_qt) {
#pragma unroll 1
      for (int k = 0; k < 2; ++k) {
        const int blk = wid + 8 * k, bi = blk >> 2, bj = blk & 3;
        const int c = bj * 32 + lane;                // column inside the tile
        uint8_t sc = 0;
        if (bi * 32 < nr && bj * 32 < nc) {          // warp-uniform
          const uint8_t* base = boxes + bj * 8192 + bi * 2048 + csub;
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint16_t h = *reinterpret_cast<const uint16_t*>(
                base + i * 64 + ((((lane >> 3) ^ ((i >> 1) & 3))) << 4));
            v[i] = __uint_as_float(static_cast<uint32_t>(h) << 16);
          }
          uint32_t cw[8];
          sc = mx_quant32_words(v, cw);
          put_codes(code_c, c, bi, cw);
          if (!mma_layout) st[b * st_bytes + (c0 + c) * (rows / 32) + r0 / 32 + bi] = sc;
        }
        if (mma_layout) atom_c[lane * 16 + bj * 4 + bi] = sc;
      }
    }
    fence_proxy_async_smem();                        // code boxes -> the TMA stores
    __syncthreads();
    if (tid == 0) {
      if (has_q) tma_store_3d(&maps.q, smem_u32(code_r), c0, r0, static_cast<int>(b));
      if (has_qt) tma_store_3d(&maps.qt, smem_u32(code_c), r0, c0, static_cast<int>(b));
      bulk_commit();
      // the tile after next into the buffer just read
      const long long tn = t + 2ll * gridDim.x;
      if (tn < ntiles) {
        long long bn;
        int rn, cn;
        quant_tile_coords(tn, rtn, ctn, bn, rn, cn);
        quant_issue_load(maps, in_buf + buf * kQIn, &full[buf], bn, rn, cn);
      }
    }
    if (mma_layout && tid < 64) {                    // one 512-byte atom per direction
      const int h = tid >> 5, k = tid & 31;
      if (h == 0 && has_q)
        reinterpret_cast<uint4*>(s + b * s_bytes + sf_mma_offset(r0, c0 / 32, sf_row_atoms(rows)))[k] =
            reinterpret_cast<const uint4*>(atom_r)[k];
      if (h == 1 && has_qt)
        reinterpret_cast<uint4*>(st + b * st_bytes + sf_mma_offset(c0, r0 / 32, sf_row_atoms(cols)))[k] =
            reinterpret_cast<const uint4*>(atom_c)[k];
    }
  }
  if (tid == 0) {
    bulk_wait_all();                                 // code stores done before the CTA exits
    // after an abort, loads still in flight land before the CTA leaves
    // (bounded: a load that never completes is given up on)
    if (abort_flag) {
      int dummy = 0;
      for (int k = 0; k < 2; ++k) mbar_wait(&full[k], (it >> 1) & 1, &dummy, &dummy, 50000000ull);
    }
  }
}

}  // namespace

cudaError_t launch_quant_bf16_mx(const void* in, long long batch, long long rows, long long cols,
                                 uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                                 int mma_layout, const int32_t* row_limit, int num_sms,
                                 int* status, cudaStream_t stream) {
  const long long ntiles = batch * ((rows + kQT - 1) / kQT) * ((cols + kQT - 1) / kQT);
  if (ntiles == 0) return cudaSuccess;
  QuantMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (!encode_map_3d(&maps.in, in, cols, rows, batch, cols * 2, rows * cols * 2, 32, 128,
                     CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) ||
      (q && !encode_map_3d(&maps.q, q, cols, rows, batch, cols, rows * cols, 128, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8)) ||
      (qt && !encode_map_3d(&maps.qt, qt, rows, cols, batch, rows, rows * cols, 128, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_DATA_TYPE_UINT8)))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(k_quant_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kQuantSmem);
  if (err != cudaSuccess) return err;
  long long grid = ntiles;
  if (grid > static_cast<long long>(num_sms) * 2) grid = static_cast<long long>(num_sms) * 2;
  k_quant_bf16<<<static_cast<int>(grid), kQThreads, kQuantSmem, stream>>>(
      maps, batch, rows, cols, q != nullptr, qt != nullptr, s, st, mma_layout, row_limit, status);
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
