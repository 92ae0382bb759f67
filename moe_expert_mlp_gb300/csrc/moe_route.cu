// Memory-bound steps of the routed-expert MLP: top-k routing, group offsets,
// the stable permutation into expert-contiguous ragged groups, the weighted
// combine, their backward passes, the FC1 weight repack and the per-group
// bias-gradient column sums.
//
// Sources: "Improving MoE training throughput with advanced fused kernels",
// "Overcoming training bottlenecks in the MoE block" (tokens per expert are
// computed at run time) and "Eliminating host-device synchronisation and CPU
// launch overhead" (group sizes are kept in GPU memory so nothing here reads
// device data on the host); "Accelerating dropless MoE training with JAX and
// NVIDIA Transformer Engine", "Claims and evidence" (ragged tensors; the
// combine step).
//
// All kernels are deterministic: no floating-point atomics, fixed reduction
// trees, and the permutation is a stable counting sort.
#include <cuda_bf16.h>
#include <float.h>
#include <math.h>

#include "moe_internal.h"
#include "moe_mx.cuh"
#include "moe_ptx.cuh"
#include "moe_route.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// ------------------------------------------------------------ top-k
// One warp per token, 8 tokens per block.  Lane l holds the scores of
// experts l, l+32, ...; k rounds of a warp arg-max (larger score wins, equal
// scores go to the lower expert index) give the slots in descending score.
// The weights are the softmax of the selected raw logits.  The per-expert
// histogram of each chunk of kTokensPerChunk tokens is accumulated with
// integer atomics into chunk_counts (zeroed beforehand); integer sums do
// not depend on the order, so the counts are exact and reproducible.
__global__ void __launch_bounds__(256) k_topk(
    const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    int32_t* __restrict__ chunk_counts, int* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float* lrow = logits + static_cast<size_t>(t) * E;
  float sc[kMaxExperts / 32];
#pragma unroll
  for (int q = 0; q < kMaxExperts / 32; ++q) {
    const int e = lane + 32 * q;
    sc[q] = -INFINITY;
    if (e < E) sc[q] = lrow[e] + (bias ? bias[e] : 0.0f);
  }
  uint32_t taken = 0;
  int my_idx = 0;
  for (int s = 0; s < k; ++s) {
    float best = -INFINITY;
    int bi = E;                           // sentinel: nothing selectable
#pragma unroll
    for (int q = 0; q < kMaxExperts / 32; ++q) {
      const int e = lane + 32 * q;
      if (e < E && !((taken >> q) & 1u)) {
        if (sc[q] > best || (sc[q] == best && e < bi)) {
          best = sc[q];
          bi = e;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xFFFFFFFFu, best, o);
      const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    if (bi >= E) {                        // non-finite scores left nothing to pick
      if (lane == 0) set_status(status, MOE_DEV_BAD_EXPERT);
      bi = s;
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == s) my_idx = bi;
  }
  const float z = (lane < k) ? lrow[my_idx] : -INFINITY;
  const float m = warp_max(z);
  const float ex = (lane < k) ? expf(z - m) : 0.0f;
  const float sum = warp_sum(ex);
  if (lane < k) {
    topk_idx[static_cast<size_t>(t) * k + lane] = my_idx;
    topk_w[static_cast<size_t>(t) * k + lane] = ex / sum;
    atomicAdd(&chunk_counts[static_cast<size_t>(t / kTokensPerChunk) * E + my_idx], 1);
  }
}

// ------------------------------------------------------------- scans
__global__ void k_offsets_from_counts(const int32_t* __restrict__ counts, int E, int capacity,
                                      int32_t* offsets, int32_t* padded_offsets,
                                      int32_t* tile_prefix, int* status) {
  __shared__ int32_t s_c[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_c[e] = counts[e];
  __syncthreads();
  if (threadIdx.x == 0) scan_experts(s_c, E, capacity, offsets, padded_offsets, tile_prefix, status);
}

// ------------------------------------------- group offsets + stable assignment
// One thread per token, one block per chunk (scan_assign_chunk).
__global__ void __launch_bounds__(kTokensPerChunk) k_scan_assign(
    const int32_t* __restrict__ topk_idx, int T, int E, int k,
    const int32_t* __restrict__ chunk_counts, int nchunks, int capacity,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ padded_offsets, int32_t* __restrict__ tile_prefix,
    int32_t* __restrict__ row_src, int32_t* __restrict__ row_of, int* status) {
  __shared__ AssignSmem sm;
  scan_assign_chunk(static_cast<int>(blockIdx.x), static_cast<int>(threadIdx.x), topk_idx, T, E,
                    k, chunk_counts, nchunks, capacity, counts, offsets, padded_offsets,
                    tile_prefix, row_src, row_of, status, sm, [] { __syncthreads(); });
}

// ---------------------------------------------------------- row gather
// x_perm[j] = x[row_src[j]] (zero on padding), one warp per row, 16-byte
// vectors.  The grid strides over the rows up to padded_offsets[E], which is
// read on the device.
__global__ void __launch_bounds__(256) k_gather_rows(
    const uint4* __restrict__ x, const int32_t* __restrict__ row_src,
    const int32_t* __restrict__ padded_offsets, int E, int vec_per_row, int T, int capacity,
    uint4* __restrict__ x_perm) {
  const int rows = min(padded_offsets[E], capacity);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = blockIdx.x * 8 + warp; j < rows; j += gridDim.x * 8)
    gather_row_warp(x, row_src, j, vec_per_row, T, x_perm, lane);
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&v)[8]) {
  v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
  v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
  v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  uint4 w;
  w.x = pack_bf16x2(v[0], v[1]);
  w.y = pack_bf16x2(v[2], v[3]);
  w.z = pack_bf16x2(v[4], v[5]);
  w.w = pack_bf16x2(v[6], v[7]);
  return w;
}

// MXFP8 (rowwise) of the eight bf16 values a lane holds: groups of four
// lanes hold one 32-element block (16-byte chunks 4b .. 4b+3 of a row), whose
// abs-max the group shares with two shuffles; the codes and the scale are
// those of the standalone quantizer (same scale rule, same conversions).
// The whole warp calls (inactive lanes pass zeros and store nothing).
__device__ __forceinline__ void mx_row_chunk(const float (&v)[8], bool active, int lane,
                                             uint8_t* q_row, uint8_t* sf, long long row,
                                             int chunk, long long row_atoms) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  if (!active) return;
  const int s = mx_scale_exponent(m);
  const float inv = mx_inv_scale(s);
  const uint32_t w0 = e4m3x2(v[0] * inv, v[1] * inv) | (e4m3x2(v[2] * inv, v[3] * inv) << 16);
  const uint32_t w1 = e4m3x2(v[4] * inv, v[5] * inv) | (e4m3x2(v[6] * inv, v[7] * inv) << 16);
  *reinterpret_cast<uint2*>(q_row + chunk * 8) = make_uint2(w0, w1);
  if ((lane & 3) == 0) sf[sf_mma_offset(row, chunk >> 2, row_atoms)] = static_cast<uint8_t>(s + 127);
}

// The gather with the rowwise MXFP8 copy of every row it writes (codes
// [capacity, d], scales in the MMA layout); padding rows get zero codes and
// scales.
__global__ void __launch_bounds__(256) k_gather_rows_mx(
    const uint4* __restrict__ x, const int32_t* __restrict__ row_src,
    const int32_t* __restrict__ padded_offsets, int E, int vec_per_row, int T, int capacity,
    uint4* __restrict__ x_perm, uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
    long long row_atoms) {
  const int rows = min(padded_offsets[E], capacity);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = blockIdx.x * 8 + warp; j < rows; j += gridDim.x * 8) {
    const int t = row_src[j];
    const bool real = t >= 0 && t < T;
    uint4* dst = x_perm + static_cast<size_t>(j) * vec_per_row;
    const uint4* src = x + static_cast<size_t>(real ? t : 0) * vec_per_row;
    uint8_t* q_row = q + static_cast<size_t>(j) * vec_per_row * 8;
    // four 16-byte loads per lane in flight before the first is used
    for (int c0 = 0; c0 < vec_per_row; c0 += 128) {
      uint4 w[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u + lane;
        w[u] = c < vec_per_row && real ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (c0 + 32 * u >= vec_per_row) break;     // warp-uniform
        const int c = c0 + 32 * u + lane;
        const bool active = c < vec_per_row;
        if (active) dst[c] = w[u];
        float v[8];
        unpack8(w[u], v);
        mx_row_chunk(v, active, lane, q_row, sf, j, c, row_atoms);
      }
    }
  }
}

__global__ void __launch_bounds__(256) k_zero_pad_rows(
    const int32_t* __restrict__ row_src, const int32_t* __restrict__ padded_offsets, int E,
    int vec_per_row, int capacity, uint4* __restrict__ rows_out, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sf, long long row_atoms) {
  const int rows = min(padded_offsets[E], capacity);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int j = blockIdx.x * 8 + warp; j < rows; j += gridDim.x * 8) {
    if (row_src[j] >= 0) continue;
    uint4* dst = rows_out + static_cast<size_t>(j) * vec_per_row;
    for (int c = lane; c < vec_per_row; c += 32) dst[c] = make_uint4(0, 0, 0, 0);
    if (q) {                      // the row's MXFP8 codes (8 per chunk) and scales
      uint2* qr = reinterpret_cast<uint2*>(q + static_cast<size_t>(j) * vec_per_row * 8);
      for (int c = lane; c < vec_per_row; c += 32) qr[c] = make_uint2(0, 0);
      for (int b = lane; b < vec_per_row / 4; b += 32) sf[sf_mma_offset(j, b, row_atoms)] = 0;
    }
  }
}

// ------------------------------------------------------------- combine
// out[t] = sum_s w[t,s] * y[row_of[t,s]]: one block per token, fp32 sums in
// slot order.  With w == nullptr the weights are 1 (permute backward).
__global__ void __launch_bounds__(128) k_combine(
    const uint4* __restrict__ y, const int32_t* __restrict__ row_of,
    const float* __restrict__ w, int k, int vec_per_row, uint4* __restrict__ out) {
  __shared__ int s_r[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    s_r[threadIdx.x] = row_of[static_cast<size_t>(t) * k + threadIdx.x];
    s_w[threadIdx.x] = w ? w[static_cast<size_t>(t) * k + threadIdx.x] : 1.0f;
  }
  __syncthreads();
  for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    // four slots' rows in flight at a time; accumulated in slot order
    int s = 0;
    for (; s + 4 <= k; s += 4) {
      uint4 v4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v4[u] = __ldg(y + static_cast<size_t>(s_r[s + u]) * vec_per_row + c);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float v[8];
        unpack8(v4[u], v);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(s_w[s + u], v[i], acc[i]);
      }
    }
    for (; s < k; ++s) {
      float v[8];
      unpack8(__ldg(y + static_cast<size_t>(s_r[s]) * vec_per_row + c), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(s_w[s], v[i], acc[i]);
    }
    out[static_cast<size_t>(t) * vec_per_row + c] = pack8(acc);
  }
}

// dy[row_of[t,s]] = bf16(w[t,s] * dout[t]); dw[t,s] = <dout[t], y[row_of[t,s]]>
// with a fixed-shape block reduction (deterministic).
__global__ void __launch_bounds__(128) k_combine_bwd(
    const uint4* __restrict__ dout, const uint4* __restrict__ y,
    const int32_t* __restrict__ row_of, const float* __restrict__ w, int k, int vec_per_row,
    uint4* __restrict__ dy, float* __restrict__ dw) {
  __shared__ float s_part[4][kMaxTopK];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int s = 0; s < k; ++s) {
    const int r = row_of[static_cast<size_t>(t) * k + s];
    const float ws = w[static_cast<size_t>(t) * k + s];
    float dot = 0.0f;
    for (int c = threadIdx.x; c < vec_per_row; c += blockDim.x) {
      float g[8], v[8], o[8];
      unpack8(__ldg(dout + static_cast<size_t>(t) * vec_per_row + c), g);
      unpack8(__ldg(y + static_cast<size_t>(r) * vec_per_row + c), v);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dot = fmaf(g[i], v[i], dot);
        o[i] = ws * g[i];
      }
      dy[static_cast<size_t>(r) * vec_per_row + c] = pack8(o);
    }
    dot = warp_sum(dot);
    if (lane == 0) s_part[warp][s] = dot;            // each warp its own entries
  }
  __syncthreads();                                  // one barrier per token
  if (threadIdx.x < k)
    dw[static_cast<size_t>(t) * k + threadIdx.x] =
        (s_part[0][threadIdx.x] + s_part[1][threadIdx.x]) +
        (s_part[2][threadIdx.x] + s_part[3][threadIdx.x]);
}

// The combine backward with the rowwise MXFP8 copy of each dY row it writes,
// quantized from the stored (bf16-rounded) values.
__global__ void __launch_bounds__(128) k_combine_bwd_mx(
    const uint4* __restrict__ dout, const uint4* __restrict__ y,
    const int32_t* __restrict__ row_of, const float* __restrict__ w, int k, int vec_per_row,
    uint4* __restrict__ dy, float* __restrict__ dw, uint8_t* __restrict__ q,
    uint8_t* __restrict__ sf, long long row_atoms) {
  __shared__ float s_part[4][kMaxTopK];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int s = 0; s < k; ++s) {
    const int r = row_of[static_cast<size_t>(t) * k + s];
    const float ws = w[static_cast<size_t>(t) * k + s];
    uint8_t* q_row = q + static_cast<size_t>(r) * vec_per_row * 8;
    float dot = 0.0f;
    for (int c0 = 0; c0 < vec_per_row; c0 += blockDim.x) {
      const int c = c0 + threadIdx.x;
      const bool active = c < vec_per_row;
      float g[8], v[8], o[8];
      if (active) {
        unpack8(__ldg(dout + static_cast<size_t>(t) * vec_per_row + c), g);
        unpack8(__ldg(y + static_cast<size_t>(r) * vec_per_row + c), v);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = v[i] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dot = fmaf(g[i], v[i], dot);
        o[i] = ws * g[i];
      }
      const uint4 packed = pack8(o);
      if (active) dy[static_cast<size_t>(r) * vec_per_row + c] = packed;
      float ob[8];
      unpack8(packed, ob);                       // the stored bf16 values
      mx_row_chunk(ob, active, lane, q_row, sf, r, c, row_atoms);
    }
    dot = warp_sum(dot);
    if (lane == 0) s_part[warp][s] = dot;            // each warp its own entries
  }
  __syncthreads();                                  // one barrier per token
  if (threadIdx.x < k)
    dw[static_cast<size_t>(t) * k + threadIdx.x] =
        (s_part[0][threadIdx.x] + s_part[1][threadIdx.x]) +
        (s_part[2][threadIdx.x] + s_part[3][threadIdx.x]);
}

// dlogits[t, idx[t,s]] = w_s * (dw_s - sum_s' w_s' dw_s'), zero elsewhere.
__global__ void __launch_bounds__(256) k_route_bwd(
    const float* __restrict__ dw, const float* __restrict__ w, const int32_t* __restrict__ idx,
    int T, int E, int k, float* __restrict__ dlogits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float ws = 0.0f, dws = 0.0f;
  int e = -1;
  if (lane < k) {
    ws = w[static_cast<size_t>(t) * k + lane];
    dws = dw[static_cast<size_t>(t) * k + lane];
    e = idx[static_cast<size_t>(t) * k + lane];
  }
  const float inner = warp_sum(ws * dws);
  float* row = dlogits + static_cast<size_t>(t) * E;
  for (int c = lane; c < E; c += 32) row[c] = 0.0f;
  __syncwarp();
  if (lane < k && e >= 0 && e < E) row[e] = ws * (dws - inner);
}

// --------------------------------------------------------- FC1 repack
// Packed row p of an expert: block b = p / 256, j = p % 256; j < 128 is gate
// feature 128b+j (logical row f), else linear feature 128b+j-128 (logical
// row F+f); features >= F are zero rows.
__device__ __forceinline__ int packed_to_logical(int p, int F) {
  const int b = p / (2 * kGluHalf), j = p % (2 * kGluHalf);
  const int f = b * kGluHalf + (j % kGluHalf);
  if (f >= F) return -1;
  return j < kGluHalf ? f : F + f;
}

// Copy with 2-byte elements; `width` elements per row (d for weights, 1 for
// biases).  One block per packed row.
__global__ void k_repack_fc1(const uint16_t* __restrict__ w1, uint16_t* __restrict__ w1p, int F,
                             int F_pad, int width) {
  const int e = blockIdx.y;
  const int p = blockIdx.x;
  const int src = packed_to_logical(p, F);
  uint16_t* dst = w1p + (static_cast<size_t>(e) * 2 * F_pad + p) * width;
  const uint16_t* s = w1 + (static_cast<size_t>(e) * 2 * F + (src < 0 ? 0 : src)) * width;
  for (int c = threadIdx.x; c < width; c += blockDim.x) dst[c] = src < 0 ? 0 : s[c];
}

__global__ void k_unpack_fc1(const uint16_t* __restrict__ w1p, uint16_t* __restrict__ w1, int F,
                             int F_pad, int width) {
  const int e = blockIdx.y;
  const int r = blockIdx.x;                    // logical row in [0, 2F)
  const int f = r < F ? r : r - F;
  const int p = (f / kGluHalf) * 2 * kGluHalf + (r < F ? 0 : kGluHalf) + f % kGluHalf;
  const uint16_t* s = w1p + (static_cast<size_t>(e) * 2 * F_pad + p) * width;
  uint16_t* dst = w1 + (static_cast<size_t>(e) * 2 * F + r) * width;
  for (int c = threadIdx.x; c < width; c += blockDim.x) dst[c] = s[c];
}

// db[e, c] = sum over the group's rows of g[r, c], in fp32 with a fixed
// order: a block owns 32 column pairs of one expert; warp w sums rows
// w, w+8, w+16, ... in order (a warp reads 128 contiguous bytes per row),
// then the eight partial sums are added in warp order.
__global__ void __launch_bounds__(256) k_group_colsum(
    const uint32_t* __restrict__ g, const int32_t* __restrict__ counts,
    const int32_t* __restrict__ padded_offsets, int pairs_per_row, uint32_t* __restrict__ out) {
  __shared__ float s_part[8][32][2];
  const int e = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  const int r0 = padded_offsets[e], m = counts[e];
  float a0 = 0.0f, a1 = 0.0f;
  if (c < pairs_per_row) {
    for (int r = warp; r < m; r += 8) {
      const uint32_t v = __ldg(g + static_cast<size_t>(r0 + r) * pairs_per_row + c);
      a0 += bf16_lo(v);
      a1 += bf16_hi(v);
    }
  }
  s_part[warp][lane][0] = a0;
  s_part[warp][lane][1] = a1;
  __syncthreads();
  if (warp == 0 && c < pairs_per_row) {
    float b0 = 0.0f, b1 = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      b0 += s_part[w][lane][0];
      b1 += s_part[w][lane][1];
    }
    out[static_cast<size_t>(e) * pairs_per_row + c] = pack_bf16x2(b0, b1);
  }
}

}  // namespace

// ---------------------------------------------------------------- launchers
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k,
                        int32_t* topk_idx, float* topk_w, int32_t* chunk_counts, int* status,
                        cudaStream_t s) {
  const int nchunks = (T + kTokensPerChunk - 1) / kTokensPerChunk;
  if (nchunks == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(chunk_counts, 0, sizeof(int32_t) * nchunks * E, s);
  if (e != cudaSuccess) return e;
  k_topk<<<(T + 7) / 8, 256, 0, s>>>(logits, bias, T, E, k, topk_idx, topk_w, chunk_counts,
                                     status);
  return cudaGetLastError();
}

cudaError_t launch_offsets_from_counts(const int32_t* counts, int E, int capacity,
                                       int32_t* offsets, int32_t* padded_offsets,
                                       int32_t* tile_prefix, int* status, cudaStream_t s) {
  k_offsets_from_counts<<<1, 256, 0, s>>>(counts, E, capacity, offsets, padded_offsets,
                                          tile_prefix, status);
  return cudaGetLastError();
}

cudaError_t launch_scan_assign(const int32_t* topk_idx, int T, int E, int k,
                               const int32_t* chunk_counts, int capacity, int32_t* counts,
                               int32_t* offsets, int32_t* padded_offsets, int32_t* tile_prefix,
                               int32_t* row_src, int32_t* row_of, int* status, cudaStream_t s) {
  const int nchunks = (T + kTokensPerChunk - 1) / kTokensPerChunk;
  if (nchunks == 0) return cudaSuccess;
  k_scan_assign<<<nchunks, kTokensPerChunk, 0, s>>>(topk_idx, T, E, k, chunk_counts, nchunks,
                                                    capacity, counts, offsets, padded_offsets,
                                                    tile_prefix, row_src, row_of, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* x, const int32_t* row_src,
                               const int32_t* padded_offsets, int E, int d, int T, int capacity,
                               void* x_perm, int num_sms, cudaStream_t s) {
  k_gather_rows<<<num_sms * 8, 256, 0, s>>>(static_cast<const uint4*>(x), row_src, padded_offsets,
                                            E, d / 8, T, capacity, static_cast<uint4*>(x_perm));
  return cudaGetLastError();
}

cudaError_t launch_zero_pad_rows(const int32_t* row_src, const int32_t* padded_offsets, int E,
                                 int width, int capacity, void* rows, int num_sms,
                                 cudaStream_t s, uint8_t* q, uint8_t* sf) {
  k_zero_pad_rows<<<num_sms * 4, 256, 0, s>>>(row_src, padded_offsets, E, width / 8, capacity,
                                              static_cast<uint4*>(rows), q, sf,
                                              sf_row_atoms(capacity));
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_mx(const void* x, const int32_t* row_src,
                                  const int32_t* padded_offsets, int E, int d, int T,
                                  int capacity, void* x_perm, uint8_t* q, uint8_t* sf,
                                  int num_sms, cudaStream_t s) {
  k_gather_rows_mx<<<num_sms * 8, 256, 0, s>>>(static_cast<const uint4*>(x), row_src,
                                               padded_offsets, E, d / 8, T, capacity,
                                               static_cast<uint4*>(x_perm), q, sf,
                                               sf_row_atoms(capacity));
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd_mx(const void* dout, const void* y, const int32_t* row_of,
                                  const float* w, int T, int k, int d, int capacity, void* dy,
                                  float* dw, uint8_t* q, uint8_t* sf, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_combine_bwd_mx<<<T, 128, 0, s>>>(static_cast<const uint4*>(dout),
                                     static_cast<const uint4*>(y), row_of, w, k, d / 8,
                                     static_cast<uint4*>(dy), dw, q, sf, sf_row_atoms(capacity));
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* y, const int32_t* row_of, const float* w, int T, int k,
                           int d, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_combine<<<T, 128, 0, s>>>(static_cast<const uint4*>(y), row_of, w, k, d / 8,
                              static_cast<uint4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd(const void* dout, const void* y, const int32_t* row_of,
                               const float* w, int T, int k, int d, void* dy, float* dw,
                               cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_combine_bwd<<<T, 128, 0, s>>>(static_cast<const uint4*>(dout), static_cast<const uint4*>(y),
                                  row_of, w, k, d / 8, static_cast<uint4*>(dy), dw);
  return cudaGetLastError();
}

cudaError_t launch_permute_bwd(const void* dx_perm, const int32_t* row_of, int T, int k, int d,
                               void* dx, cudaStream_t s) {
  return launch_combine(dx_perm, row_of, nullptr, T, k, d, dx, s);
}

cudaError_t launch_route_bwd(const float* dw, const float* w, const int32_t* idx, int T, int E,
                             int k, float* dlogits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_route_bwd<<<(T + 7) / 8, 256, 0, s>>>(dw, w, idx, T, E, k, dlogits);
  return cudaGetLastError();
}

cudaError_t launch_repack_fc1(const void* w1, void* w1p, int E, int F, int width,
                              cudaStream_t s) {
  const int F_pad = fc1_pad(F);
  dim3 grid(2 * F_pad, E);
  k_repack_fc1<<<grid, width >= 256 ? 256 : 32, 0, s>>>(static_cast<const uint16_t*>(w1),
                                                       static_cast<uint16_t*>(w1p), F, F_pad,
                                                       width);
  return cudaGetLastError();
}

cudaError_t launch_unpack_fc1(const void* w1p, void* w1, int E, int F, int width,
                              cudaStream_t s) {
  const int F_pad = fc1_pad(F);
  dim3 grid(2 * F, E);
  k_unpack_fc1<<<grid, width >= 256 ? 256 : 32, 0, s>>>(static_cast<const uint16_t*>(w1p),
                                                       static_cast<uint16_t*>(w1), F, F_pad,
                                                       width);
  return cudaGetLastError();
}

cudaError_t launch_group_colsum(const void* g, const int32_t* counts,
                                const int32_t* padded_offsets, int E, int width, void* out,
                                cudaStream_t s) {
  const int pairs = width / 2;
  dim3 grid((pairs + 31) / 32, E);
  k_group_colsum<<<grid, 256, 0, s>>>(static_cast<const uint32_t*>(g), counts, padded_offsets,
                                      pairs, static_cast<uint32_t*>(out));
  return cudaGetLastError();
}

}  // namespace moe
