// NVFP4 quantization of bf16 tensors for the block-scaled FP4 GEMMs.
//
// "Improving MoE training throughput with advanced fused kernels", "Reducing
// exposed memory overhead by fusing MXFP8 and NVFP4 quantization": for NVFP4
// the GEMM epilogues emit the BF16 output with its per-tensor amax and, in
// the backward, the amax of the output's transposed Hadamard rotation; the
// tensor is then quantized with the per-tensor scale those amax values give.
//
// Format (readings, the pages name NVFP4 only): E2M1 values in blocks of 16
// along the contraction axis, one UE4M3 scale per block, one fp32 encode
// scale per tensor g = 2688 / amax (448 * 6; 1 for amax 0).  In fp32:
//   block scale code = E4M3(RNE, saturating)((amax_block / 6) * g), s = its
//   value; codes = E2M1(RNE, saturating)(x * (g / s)), all zero for s = 0.
// A product of two such operands carries g_a g_b, which the GEMM epilogue
// divides out.  Transposed copies for the weight gradients (contraction over
// tokens) are rotated first by H16 / 4 along the tokens in 16-row segments --
// the same segments as the quantization blocks -- with g from the rotated
// tensor's amax.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "moe_internal.h"
#include "moe_mx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float nv_encode_scale_q(const float* amax) {
  const float a = __ldg(amax);
  return a > 0.0f ? __fdiv_rn(2688.0f, a) : 1.0f;
}

// In-place Walsh-Hadamard transform of 16 values (Sylvester order: output i
// is sum_j (-1)^popcount(i & j) v_j).
__device__ __forceinline__ void fwht16(float (&v)[16]) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
}

// g / s for every non-negative UE4M3 scale code (s = the code's value; 0 for
// s = 0), correctly rounded as the per-block division would be: the block
// quantizer looks the factor up instead of dividing.  128 threads fill it.
__device__ __forceinline__ void nv_inv_table(float* table, float g, int tid) {
  if (tid < 128) {
    const float s = __half2float(
        __half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(tid), __NV_E4M3)));
    table[tid] = s > 0.0f ? __fdiv_rn(g, s) : 0.0f;
  }
}

// One block of 16 values with encode scale g (inv_of = its nv_inv_table):
// returns the UE4M3 scale code and the 16 E2M1 codes packed two per byte
// (element 2i in the low nibble).
__device__ __forceinline__ uint8_t nv_quant16(const float (&v)[16], float g, const float* inv_of,
                                              uint2& codes) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
  const float target = __fmul_rn(__fdiv_rn(m, 6.0f), g);
  const __nv_fp8_storage_t sc = __nv_cvt_float_to_fp8(target, __NV_SATFINITE, __NV_E4M3);
  const float inv = inv_of[sc & 0x7F];      // target >= 0: a non-negative, finite code
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t b = __nv_cvt_float2_to_fp4x2(
        make_float2(__fmul_rn(v[2 * i], inv), __fmul_rn(v[2 * i + 1], inv)), __NV_E2M1,
        cudaRoundNearest);
    w[i >> 2] |= (b & 0xFFu) << (8 * (i & 3));
  }
  codes = make_uint2(w[0], w[1]);
  return static_cast<uint8_t>(sc);
}

// Per-tensor amax of bf16 [batch, rows, cols] (rows % 16 == 0, cols % 8 ==
// 0) over rows below *row_limit: amax[0] = max |x|, amax[1] = max |H16 x / 4|
// over 16-row segments (each column rotated along the rows).  One thread
// per (segment, 8 columns): sixteen 16-byte row loads; both outputs must be
// zero on entry.
__global__ void __launch_bounds__(256) k_amax_nv(const __nv_bfloat16* __restrict__ in,
                                                 long long batch, long long rows, long long cols,
                                                 const int32_t* row_limit, float* amax) {
  const long long rlim = row_limit ? __ldg(row_limit) : rows;
  const long long segs = (rlim < rows ? rlim : rows) / 16;
  const long long c8_n = cols / 8;
  const long long n = batch * segs * c8_n;
  float m0 = 0.0f, m1 = 0.0f;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long c8 = i % c8_n, rest = i / c8_n;
    const long long sg = rest % segs, b = rest / segs;
    const uint4* p = reinterpret_cast<const uint4*>(in + (b * rows + sg * 16) * cols) + c8;
    uint4 w[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) w[r] = __ldg(p + r * c8_n);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      float v[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        const uint32_t word = (c < 2) ? w[r].x : (c < 4) ? w[r].y : (c < 6) ? w[r].z : w[r].w;
        v[r] = __uint_as_float((c & 1) ? (word & 0xFFFF0000u) : (word << 16));
        m0 = fmaxf(m0, fabsf(v[r]));
      }
      fwht16(v);
#pragma unroll
      for (int r = 0; r < 16; ++r) m1 = fmaxf(m1, fabsf(v[r]));
    }
  }
  m1 *= 0.25f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xFFFFFFFFu, m0, o));
    m1 = fmaxf(m1, __shfl_xor_sync(0xFFFFFFFFu, m1, o));
  }
  if ((threadIdx.x & 31) == 0) {
    atomic_max_nonneg(amax, m0);
    atomic_max_nonneg(amax + 1, m1);
  }
}

// bf16 [batch][rows][cols] -> NVFP4, one CTA (8 warps) per 128 x 128 tile.
// Rowwise (q != null): blocks of 16 along each row, codes [batch][rows]
// [cols/2], scales in the MMA layout of a [rows, cols] operand.  Columnwise
// (qt != null): blocks of 16 down each column -- rotated by H16/4 first when
// `rotate` -- codes written transposed [batch][cols][rows/2], scales in the
// MMA layout of a [cols, rows] operand.  rows, cols multiples of 32; tiles at
// or past *row_limit are skipped.
constexpr int kNT = 128;                       // tile edge
constexpr int kTilePitch = 272;                // bytes per staged row (256 + 16 pad)
constexpr int kNvQuantSmem = kNT * kTilePitch + 2 * kNT * 64 + 4 * 512;

__global__ void __launch_bounds__(256, 3) k_quant_nv(const __nv_bfloat16* __restrict__ in,
                                                  long long batch, long long rows, long long cols,
                                                  uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                                                  const float* amax_row, const float* amax_col,
                                                  int rotate, const int32_t* row_limit) {
  extern __shared__ __align__(16) uint8_t nsm[];
  uint8_t* tile = nsm;                               // [128][272 B]
  uint8_t* code_r = tile + kNT * kTilePitch;         // [128 rows][64 B]
  uint8_t* code_c = code_r + kNT * 64;               // [128 cols][64 B], 8-byte pieces swizzled
  uint8_t* atom_r = code_c + kNT * 64;               // 2 atoms (K groups) x 512 B
  uint8_t* atom_c = atom_r + 1024;
  const int tid = threadIdx.x;
  const long long rtn = (rows + kNT - 1) / kNT, ctn = (cols + kNT - 1) / kNT;
  const long long ntiles = batch * rtn * ctn;
  const long long ra_r = sf_row_atoms(rows), ra_c = sf_row_atoms(cols);
  const long long s_bytes = (cols + 63) / 64 * ra_r * 512;
  const long long st_bytes = (rows + 63) / 64 * ra_c * 512;
  const long long rlim = row_limit ? __ldg(row_limit) : rows;
  const float g_row = q ? nv_encode_scale_q(amax_row) : 1.0f;
  const float g_col = qt ? nv_encode_scale_q(amax_col) : 1.0f;
  __shared__ float inv_row[128], inv_col[128];
  nv_inv_table(inv_row, g_row, tid);
  nv_inv_table(inv_col, g_col, tid);           // visible after the tile loop's first barrier
  // the tile's 2048 16-byte chunks, eight per thread, are loaded one tile
  // ahead into registers so that the loads overlap the previous tile's work
  auto load_tile = [&](long long t, uint4 (&v)[8]) {
    const long long b = t / (rtn * ctn);
    const long long rem = t - b * rtn * ctn;
    const long long r0 = (rem / ctn) * kNT, c0 = (rem % ctn) * kNT;
    const int nr = static_cast<int>(min(static_cast<long long>(kNT), rows - r0));
    const int nc = static_cast<int>(min(static_cast<long long>(kNT), cols - c0));
    const bool live = t < ntiles && r0 < rlim;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = tid + 256 * k;
      const int r = i >> 4, ch = i & 15;
      v[k] = make_uint4(0, 0, 0, 0);
      if (live && r < nr && ch * 8 < nc)
        v[k] = __ldg(reinterpret_cast<const uint4*>(in + (b * rows + r0 + r) * cols + c0) + ch);
    }
  };
  uint4 pre[8];
  load_tile(blockIdx.x, pre);
  for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const long long b = t / (rtn * ctn);
    const long long rem = t - b * rtn * ctn;
    const long long r0 = (rem / ctn) * kNT, c0 = (rem % ctn) * kNT;
    if (r0 >= rlim) {                                // uniform across the CTA
      load_tile(t + gridDim.x, pre);
      continue;
    }
    const int nr = static_cast<int>(min(static_cast<long long>(kNT), rows - r0));
    const int nc = static_cast<int>(min(static_cast<long long>(kNT), cols - c0));
    __syncthreads();                                 // previous tile fully stored
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = tid + 256 * k;
      *reinterpret_cast<uint4*>(tile + (i >> 4) * kTilePitch + (i & 15) * 16) = pre[k];
    }
    load_tile(t + gridDim.x, pre);
    if (tid < 128) reinterpret_cast<uint4*>(atom_r)[tid] = make_uint4(0, 0, 0, 0);   // both
    __syncthreads();
    if (q) {
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int item = tid + 256 * k;
        const int r = item >> 3, blk = item & 7;
        if (r >= nr || blk * 16 >= nc) continue;
        const uint4* src = reinterpret_cast<const uint4*>(tile + r * kTilePitch + blk * 32);
        float v[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 w4 = src[h];
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[8 * h + 2 * e] = __uint_as_float(w[e] << 16);
            v[8 * h + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
          }
        }
        uint2 c;
        const uint8_t sc = nv_quant16(v, g_row, inv_row, c);
        *reinterpret_cast<uint2*>(code_r + r * 64 + blk * 8) = c;
        atom_r[(blk >> 2) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (blk & 3)] = sc;
      }
    }
    if (qt) {
#pragma unroll 1
      for (int k = 0; k < 4; ++k) {
        const int item = tid + 256 * k;
        const int c = item & 127, rb = item >> 7;    // a warp: 32 adjacent columns
        if (c >= nc || rb * 16 >= nr) continue;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint16_t h =
              *reinterpret_cast<const uint16_t*>(tile + (rb * 16 + i) * kTilePitch + c * 2);
          v[i] = __uint_as_float(static_cast<uint32_t>(h) << 16);
        }
        if (rotate) {
          fwht16(v);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] *= 0.25f;
        }
        uint2 cw;
        const uint8_t sc = nv_quant16(v, g_col, inv_col, cw);
        *reinterpret_cast<uint2*>(code_c + c * 64 + ((rb ^ (c & 7)) * 8)) = cw;
        atom_c[(rb >> 2) * 512 + (c & 31) * 16 + ((c >> 5) & 3) * 4 + (rb & 3)] = sc;
      }
    }
    __syncthreads();
    // codes out as 16-byte pieces of whole lines (each piece = 32 values)
    for (int i = tid; i < kNT * 4; i += 256) {
      const int line = i >> 2, ch = i & 3;
      if (q && line < nr && ch * 32 < nc)
        *reinterpret_cast<uint4*>(q + (b * rows + r0 + line) * (cols / 2) + c0 / 2 + ch * 16) =
            *reinterpret_cast<const uint4*>(code_r + line * 64 + ch * 16);
      if (qt && line < nc && ch * 32 < nr) {
        const uint2 lo = *reinterpret_cast<const uint2*>(code_c + line * 64 +
                                                         (((2 * ch) ^ (line & 7)) * 8));
        const uint2 hi = *reinterpret_cast<const uint2*>(code_c + line * 64 +
                                                         (((2 * ch + 1) ^ (line & 7)) * 8));
        *reinterpret_cast<uint4*>(qt + (b * cols + c0 + line) * (rows / 2) + r0 / 2 + ch * 16) =
            make_uint4(lo.x, lo.y, hi.x, hi.y);
      }
    }
    // scale atoms: K groups of 64 values that start inside the tensor
    if (tid < 128) {
      const int dir = tid >> 6, a = (tid >> 5) & 1, k = tid & 31;
      if (dir == 0 && q && c0 + 64 * a < cols)
        reinterpret_cast<uint4*>(s + b * s_bytes + ((c0 / 64 + a) * ra_r + r0 / 128) * 512)[k] =
            reinterpret_cast<const uint4*>(atom_r + a * 512)[k];
      if (dir == 1 && qt && r0 + 64 * a < rows)
        reinterpret_cast<uint4*>(st + b * st_bytes + ((r0 / 64 + a) * ra_c + c0 / 128) * 512)[k] =
            reinterpret_cast<const uint4*>(atom_c + a * 512)[k];
    }
  }
}

}  // namespace

long long nv_sf_bytes(long long rows, long long cols) {
  return (cols + 63) / 64 * sf_row_atoms(rows) * 512;
}

cudaError_t launch_amax_nv(const void* in, long long batch, long long rows, long long cols,
                           const int32_t* row_limit, float* amax, int num_sms,
                           cudaStream_t stream) {
  cudaError_t err = cudaMemsetAsync(amax, 0, 2 * sizeof(float), stream);
  if (err != cudaSuccess) return err;
  const long long n = batch * (rows / 16) * (cols / 8);
  if (n == 0) return cudaSuccess;
  long long grid = (n + 255) / 256;
  if (grid > static_cast<long long>(num_sms) * 8) grid = static_cast<long long>(num_sms) * 8;
  k_amax_nv<<<static_cast<int>(grid), 256, 0, stream>>>(static_cast<const __nv_bfloat16*>(in),
                                                         batch, rows, cols, row_limit, amax);
  return cudaGetLastError();
}

cudaError_t launch_quant_nv(const void* in, long long batch, long long rows, long long cols,
                            uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                            const float* amax_row, const float* amax_col, int rotate,
                            const int32_t* row_limit, int num_sms, cudaStream_t stream) {
  const long long ntiles = batch * ((rows + kNT - 1) / kNT) * ((cols + kNT - 1) / kNT);
  if (ntiles == 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(k_quant_nv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kNvQuantSmem);
  if (err != cudaSuccess) return err;
  long long grid = ntiles;
  if (grid > static_cast<long long>(num_sms) * 3) grid = static_cast<long long>(num_sms) * 3;
  k_quant_nv<<<static_cast<int>(grid), 256, kNvQuantSmem, stream>>>(
      static_cast<const __nv_bfloat16*>(in), batch, rows, cols, q, s, qt, st, amax_row, amax_col,
      rotate, row_limit);
  return cudaGetLastError();
}

}  // namespace moe
