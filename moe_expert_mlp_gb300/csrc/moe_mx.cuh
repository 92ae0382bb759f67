// MXFP8 (OCP Microscaling: E4M3 payload, one E8M0 scale per 32 elements)
// and NVFP4-preparation amax helpers shared by the quantize kernel and the
// GEMM epilogues.
//
// "Improving MoE training throughput with advanced fused kernels", "Reducing
// exposed memory overhead by fusing MXFP8 and NVFP4 quantization": the
// activation output (BF16) is written in MXFP8 together with a transposed
// MXFP8 copy for the backward; for NVFP4 a per-tensor amax of the output and
// of its transposed Hadamard-rotated form is produced in the same pass.
//
// Scale rule: X = 2^(floor(log2 amax) - 8), exponent clamped to [-127, 127],
// E8M0 code = exponent + 127 (code 0 for an all-zero block).  Payload: v / X
// rounded to nearest-even E4M3 with saturation to +-448 (the hardware
// cvt.rn.satfinite conversion); dividing by X is an exact power-of-two scale.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// floor(log2(a)) of a finite a > 0, exact (handles fp32 subnormals).
__device__ __forceinline__ int floor_log2_f32(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = static_cast<int>((b >> 23) & 0xFFu);
  if (e != 0) return e - 127;
  return (31 - __clz(static_cast<int>(b & 0x7FFFFFu))) - 149;
}

// Unbiased E8M0 exponent of the block scale for block abs-max `amax`.
__device__ __forceinline__ int mx_scale_exponent(float amax) {
  if (!(amax > 0.0f)) return -127;
  const int s = floor_log2_f32(amax) - 8;
  return s < -127 ? -127 : (s > 127 ? 127 : s);
}

// 2^-s as fp32 (s in [-127, 119] for finite fp32 amax, so 2^-s is normal).
__device__ __forceinline__ float mx_inv_scale(int s) {
  return __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
}

// Two fp32 values -> two E4M3 codes (a in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  const __nv_fp8x2_storage_t r =
      __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  return static_cast<uint32_t>(r);
}

// Quantize one block of 32 values into eight 32-bit words of codes (code i
// in byte i % 4 of word i / 4); returns the E8M0 scale code.
__device__ __forceinline__ uint8_t mx_quant32_words(const float (&v)[32], uint32_t (&w)[8]) {
  float m[16];                                   // block max as a tree (depth 5)
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
#pragma unroll
  for (int k = 8; k >= 1; k >>= 1)
#pragma unroll
    for (int i = 0; i < k; ++i) m[i] = fmaxf(m[i], m[i + k]);
  const int s = mx_scale_exponent(m[0]);
  const float inv = mx_inv_scale(s);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t lo = e4m3x2(v[4 * j] * inv, v[4 * j + 1] * inv);
    const uint32_t hi = e4m3x2(v[4 * j + 2] * inv, v[4 * j + 3] * inv);
    w[j] = lo | (hi << 16);
  }
  return static_cast<uint8_t>(s + 127);
}

// max(|a|, |b|) per bf16 half (the sign bit of the result is not used)
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Block of 32 bf16 (value 2i in the low half of word i, 2i+1 in the high
// half) -> eight words of E4M3 codes; returns the E8M0 scale code.  The
// scale and the codes follow mx_quant32_words exactly: the block maximum is
// taken on the bf16 magnitudes, which order like the values.
__device__ __forceinline__ uint8_t mx_quant32_packed(const uint32_t (&w)[16], uint32_t (&c)[8]) {
  uint32_t m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = bf16x2_absmax(w[2 * i], w[2 * i + 1]);
#pragma unroll
  for (int k = 4; k >= 1; k >>= 1)
#pragma unroll
    for (int i = 0; i < k; ++i) m[i] = bf16x2_absmax(m[i], m[i + k]);
  const uint32_t lo = m[0] & 0x7FFFu, hi = (m[0] >> 16) & 0x7FFFu;
  const float amax = __uint_as_float((lo > hi ? lo : hi) << 16);
  const int s = mx_scale_exponent(amax);
  const float inv = mx_inv_scale(s);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t a = w[2 * j], b = w[2 * j + 1];
    const uint32_t c0 = e4m3x2(__uint_as_float(a << 16) * inv, __uint_as_float(a & 0xFFFF0000u) * inv);
    const uint32_t c1 = e4m3x2(__uint_as_float(b << 16) * inv, __uint_as_float(b & 0xFFFF0000u) * inv);
    c[j] = c0 | (c1 << 16);
  }
  return static_cast<uint8_t>(s + 127);
}

// Quantize one block of 32 values: writes 32 codes (16-byte aligned
// destination) and returns the E8M0 scale code.
__device__ __forceinline__ uint8_t mx_quant32(const float (&v)[32], uint8_t* q) {
  uint32_t w[8];
  const uint8_t sc = mx_quant32_words(v, w);
  uint4* d = reinterpret_cast<uint4*>(q);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return sc;
}

// Non-negative float max into a global word (bit patterns of non-negative
// floats order like the floats, so an integer max is exact and order-free).
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
}

// Byte offset of the scale of row r, K block j (32 elements) in the layout
// the block-scaled MMA consumes: atoms of 128 rows x 4 K blocks (512 bytes,
// row r at (r % 32) * 16 + ((r / 32) % 4) * 4 + j % 4), atoms ordered by K
// group (j / 4) and then by row group (r / 128); `row_atoms` is the number
// of row groups, rounded up to even so that a 256-row operand tile reads
// two adjacent atoms.
__host__ __device__ __forceinline__ long long sf_mma_offset(long long r, long long j,
                                                            long long row_atoms) {
  return ((j >> 2) * row_atoms + (r >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

__host__ __device__ __forceinline__ long long sf_row_atoms(long long rows) {
  return 2 * ((rows + 255) / 256);
}

// Optional MXFP8 / amax outputs of a GEMM epilogue (all-null = none).
struct MxOut {
  uint8_t* q;        // rowwise codes [cap, width]
  uint8_t* s;        // rowwise scales [cap, width/32] or MMA layout
  uint8_t* qt;       // columnwise codes, transposed [width, cap]
  uint8_t* st;       // columnwise scales [width, cap/32] or MMA layout
  float* amax;       // [2]: max |x|, max |H16 x^T / 4|
  long long width;
  long long cap;
  int mma_layout;    // scales in the block-scaled MMA layout (sf_mma_offset)
};

// MXFP8 of one staged 32 x 32 bf16 block.  The block sits in a
// shared-memory box of 64-byte rows with the 64-byte swizzle (16-byte chunk
// q of row r at chunk q ^ ((r >> 1) & 3)) -- the GEMM epilogue's output
// staging layout -- as the box's rows row0 .. row0+31; they are the
// tensor's rows r0 .. r0+31, columns col0 .. col0+31.  Lane l quantizes row
// r0+l (rowwise) and column col0+l (columnwise, written to the transposed
// tensor), reading shared memory only: no cross-lane shuffles.  Whole warp
// calls; the box must be visible to the warp.
__device__ __forceinline__ void mx_block_from_box(const MxOut& mx, const uint8_t* box, int row0,
                                                  long long r0, int col0, int lane) {
  if (mx.q) {
    // the lane's own row: four 16-byte chunks (the swizzle spreads the 8
    // rows of a quarter warp over distinct banks)
    uint32_t w[16], c[8];
    const int r = row0 + lane;
    const uint4* rowp = reinterpret_cast<const uint4*>(box + r * 64);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 c4 = rowp[q ^ ((r >> 1) & 3)];
      w[4 * q] = c4.x;
      w[4 * q + 1] = c4.y;
      w[4 * q + 2] = c4.z;
      w[4 * q + 3] = c4.w;
    }
    const long long row = r0 + lane;
    const uint8_t sc = mx_quant32_packed(w, c);
    uint4* dq = reinterpret_cast<uint4*>(mx.q + row * mx.width + col0);
    dq[0] = make_uint4(c[0], c[1], c[2], c[3]);
    dq[1] = make_uint4(c[4], c[5], c[6], c[7]);
    mx.s[mx.mma_layout ? sf_mma_offset(row, col0 / 32, sf_row_atoms(mx.cap))
                       : row * (mx.width / 32) + col0 / 32] = sc;
  }
  if (mx.qt) {
    // column `lane` down the 32 rows (consecutive lanes read consecutive
    // bf16 of one 64-byte row: no bank conflicts)
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = row0 + i;
      const uint16_t b = *reinterpret_cast<const uint16_t*>(
          box + r * 64 + ((((lane >> 3) ^ ((r >> 1) & 3))) << 4) + (lane & 7) * 2);
      v[i] = __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    const long long c = col0 + lane;
    const uint8_t sc = mx_quant32(v, mx.qt + c * mx.cap + r0);
    mx.st[mx.mma_layout ? sf_mma_offset(c, r0 / 32, sf_row_atoms(mx.width))
                        : c * (mx.cap / 32) + r0 / 32] = sc;
  }
}

__device__ __forceinline__ float bf16_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

}  // namespace moe
