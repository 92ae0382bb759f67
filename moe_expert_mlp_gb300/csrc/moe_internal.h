// Internal interface between the C-ABI entry points and the kernel
// translation units.  Not installed; not part of the public boundary.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kTokensPerChunk = 256;   // routing: tokens per histogram chunk
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 32;
constexpr int kAlign = 128;            // group alignment = GEMM tile rows
constexpr int kGluHalf = 128;          // packed FC1 block: 128 gate + 128 linear rows

inline int fc1_pad(int F) { return (F + kGluHalf - 1) / kGluHalf * kGluHalf; }

// ------------------------------------------------ memory-bound kernels
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k,
                        int32_t* topk_idx, float* topk_w, int32_t* chunk_counts, int* status,
                        cudaStream_t s);
cudaError_t launch_offsets_from_counts(const int32_t* counts, int E, int capacity,
                                       int32_t* offsets, int32_t* padded_offsets,
                                       int32_t* tile_prefix, int* status, cudaStream_t s);
// Group offsets from the per-chunk histogram and the stable assignment of
// (token, slot) pairs to rows, in one launch (one block per chunk).
cudaError_t launch_scan_assign(const int32_t* topk_idx, int T, int E, int k,
                               const int32_t* chunk_counts, int capacity, int32_t* counts,
                               int32_t* offsets, int32_t* padded_offsets, int32_t* tile_prefix,
                               int32_t* row_src, int32_t* row_of, int* status, cudaStream_t s);
cudaError_t launch_gather_rows(const void* x, const int32_t* row_src,
                               const int32_t* padded_offsets, int E, int d, int T, int capacity,
                               void* x_perm, int num_sms, cudaStream_t s);
cudaError_t launch_combine(const void* y, const int32_t* row_of, const float* w, int T, int k,
                           int d, void* out, cudaStream_t s);
cudaError_t launch_combine_bwd(const void* dout, const void* y, const int32_t* row_of,
                               const float* w, int T, int k, int d, void* dy, float* dw,
                               cudaStream_t s);
// Zero the padding rows (row_src < 0) of a per-row tensor, and when q / sf
// are given the rows' MXFP8 rowwise codes and scales (MMA layout).
cudaError_t launch_zero_pad_rows(const int32_t* row_src, const int32_t* padded_offsets, int E,
                                 int width, int capacity, void* rows, int num_sms,
                                 cudaStream_t s, uint8_t* q = nullptr, uint8_t* sf = nullptr);
// The gather / combine backward that also write the rowwise MXFP8 copy of
// the rows they write (codes [capacity, d], scales in the MMA layout).
cudaError_t launch_gather_rows_mx(const void* x, const int32_t* row_src,
                                  const int32_t* padded_offsets, int E, int d, int T,
                                  int capacity, void* x_perm, uint8_t* q, uint8_t* sf,
                                  int num_sms, cudaStream_t s);
cudaError_t launch_combine_bwd_mx(const void* dout, const void* y, const int32_t* row_of,
                                  const float* w, int T, int k, int d, int capacity, void* dy,
                                  float* dw, uint8_t* q, uint8_t* sf, cudaStream_t s);
cudaError_t launch_permute_bwd(const void* dx_perm, const int32_t* row_of, int T, int k, int d,
                               void* dx, cudaStream_t s);
cudaError_t launch_route_bwd(const float* dw, const float* w, const int32_t* idx, int T, int E,
                             int k, float* dlogits, cudaStream_t s);
cudaError_t launch_repack_fc1(const void* w1, void* w1p, int E, int F, int width,
                              cudaStream_t s);
cudaError_t launch_unpack_fc1(const void* w1p, void* w1, int E, int F, int width,
                              cudaStream_t s);
cudaError_t launch_group_colsum(const void* g, const int32_t* counts,
                                const int32_t* padded_offsets, int E, int width, void* out,
                                cudaStream_t s);

cudaError_t launch_glu_rows(const void* h, const int32_t* counts, const int32_t* padded_offsets,
                            int E, int F, int F_pad, void* a, int act, float alpha, float limit,
                            float lin_off, float out_scale, int num_sms, cudaStream_t s);
cudaError_t launch_dglu_rows(const void* da, const void* h, const int32_t* counts,
                             const int32_t* padded_offsets, int E, int F, int F_pad, void* dh,
                             int act, float alpha, float limit, float lin_off, float out_scale,
                             int num_sms, cudaStream_t s);

// ------------------------------------------------ grouped GEMM (tcgen05)
enum GemmMode : int {
  kFc1Glu = 0,     // H = X W1p^T (+b1), A = GLU(H)             ragged M
  kFc2 = 1,        // Y = A W2^T (+b2)                          ragged M
  kDgradDglu = 2,  // dA = dY W2, dH = dGLU(dA, H)              ragged M
  kDgradFc1 = 3,   // dX = dH W1p                               ragged M
  kWgrad = 4,      // dW[e] = sum over group rows of P^T Q      ragged K
  kWgradPair = 5,  // same on CTA pairs (2-SM MMA, 256x256 tiles)
  kFc1Act = 6,     // non-gated: H = X W1^T (+b1), A = act(H)   ragged M
  kDgradAct = 7,   // non-gated: dA = dY W2, dH = act'(H) dA     ragged M
  kRouter = 8,     // logits = x W_r^T, top-k in the epilogue    one dense group
  kDgradDgluRc = 9 // dA = dY W2 and H = X W1p^T (+b1) recomputed ragged M
                   // for the same tile, dH = dGLU(dA, H): H never in HBM
};

// FC1 output width: 2*F_pad (gate and linear halves, packed) for the GLU
// activations, F for the non-gated squared ReLU.
inline int fc1_width(int act, int F) { return act == MOE_ACT_SRELU ? F : 2 * fc1_pad(F); }

struct GemmArgs {
  CUtensorMap tma_a;
  CUtensorMap tma_b;
  CUtensorMap tma_out0;   // primary output, 32x32 boxes, 64-byte swizzle
  CUtensorMap tma_out1;   // GLU output A (FC1 mode only)
  CUtensorMap tma_out2;   // primary output as [E][W/32][rows][32]: two-chunk boxes
  const int32_t* padded_offsets;
  const int32_t* counts;
  int* status;
  int E;
  int K;            // contraction length (ragged-M modes)
  int n_ext;        // output columns covered by tiles
  int b_ext;        // real extent of B's N dimension (MN-major box count)
  int m_ext;        // ragged-K mode: output rows
  int f_real;       // F
  int f_pad;        // F_pad
  int capacity;
  int act;
  float alpha, limit, lin_off, out_scale;
  void* out0;
  long long ld0;
  void* out1;
  long long ld1;
  const void* aux;
  long long ld_aux;
  const void* bias;
  long long bias_ld;
  // optional MXFP8 / amax outputs of the epilogue's bf16 result
  uint8_t* mx_q;
  uint8_t* mx_s;
  uint8_t* mx_qt;
  uint8_t* mx_st;
  float* mx_amax;
  long long mx_width;
  // MN-major operands given as [E][atom][K][64] views (one TMA per stage
  // fetches all atoms) instead of one 64x64 box per atom: 1 = yes.
  int a_atoms4d;
  int b_atoms4d;
  int mx_mma_layout;      // epilogue MX scales in the MMA layout
  // MXFP8 operands (launch_grouped_gemm_mx): E4M3 codes through tma_a /
  // tma_b (K-major, 128-element boxes), scales in the MMA layout.  A's scale
  // tensor has sfa_atoms row groups; B's has sfb_atoms, and sfb_expert_bytes
  // between experts (ragged-M modes; 0 for weight gradients).
  const uint8_t* sfa;
  const uint8_t* sfb;
  long long sfa_atoms;
  long long sfb_atoms;
  long long sfb_expert_bytes;
  // one dense group of `dense_rows` rows instead of device offsets (router)
  int dense_rows;
  // kRouter outputs: per token the top-`topk` experts by logit + bias
  // (fp32), their softmax weights over the raw logits, the per-chunk expert
  // histogram, and optionally the logits themselves
  int topk;
  const float* r_bias;
  int32_t* r_idx;
  float* r_w;
  int32_t* r_hist;
  float* r_logits;
  // kRouter with the permutation in the same launch (a cooperative launch:
  // after the logits GEMM every CTA meets at grid-wide barriers on r_grid, a
  // counter zeroed before the launch; nullptr: top-k only): the group
  // tables, the row maps and the gathered rows x_perm of the r_tokens bf16
  // token rows r_x (r_vec_per_row 16-byte vectors each)
  unsigned int* r_grid;
  int32_t* r_counts;
  int32_t* r_offsets;
  int32_t* r_padded;
  int32_t* r_tiles;
  int32_t* r_row_src;
  int32_t* r_row_of;
  const void* r_x;
  void* r_x_perm;
  int r_tokens;
  int r_vec_per_row;
  int r_capacity;
  int r_nchunks;
  // NVFP4 operands (launch_grouped_gemm_nv): per-tensor amax of the
  // quantized A and B operands; the epilogue scales the accumulator by
  // 1 / (g_a g_b), g = 2688 / amax (1 for amax 0)
  const float* nv_amax_a;
  const float* nv_amax_b;
  // kDgradDgluRc: the second GEMM's operands (tma_a / tma_b and sfa / sfb
  // hold the H GEMM's X and W1p): dY (K-major) and W2 (bf16: MN-major
  // [E][d][F], as 2-atom 4-D boxes when b2_atoms4d, else 64 x 64 boxes;
  // MXFP8: the transposed copy [E][F][d], 128-row boxes), with their scales
  CUtensorMap tma_a2;
  CUtensorMap tma_b2;
  const uint8_t* sfa2;
  const uint8_t* sfb2;
  long long sfa2_atoms;
  long long sfb2_atoms;
  long long sfb2_expert_bytes;
  int b2_atoms4d;
  // TF32 path (launch_grouped_gemm_tf32): optional transposed fp32 copies
  // [width][capacity] of out0 / out1, written by the epilogue
  float* out0_t;
  float* out1_t;
};

cudaError_t launch_grouped_gemm(int mode, const GemmArgs& args, int grid, cudaStream_t s);
// The same modes with block-scaled MXFP8 operands (kWgrad: 1-CTA tiles).
cudaError_t launch_grouped_gemm_mx(int mode, const GemmArgs& args, int grid, cudaStream_t s);
// The ragged-M modes and kWgrad with NVFP4 operands: packed E2M1 codes
// (K-major, 128-byte boxes = 256 values) and UE4M3 scales per 16 values in
// the MMA layout (sf_mma_offset with 16-element blocks).
cudaError_t launch_grouped_gemm_nv(int mode, const GemmArgs& args, int grid, cudaStream_t s);
cudaError_t launch_quant_bf16_mx(const void* in, long long batch, long long rows, long long cols,
                                 uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                                 int mma_layout, const int32_t* row_limit, int num_sms,
                                 int* status, cudaStream_t stream);
// 3-D tensor map (moe_api.cu): dims innermost first, the innermost
// contiguous, row_bytes / plane_bytes the strides of dims 1 and 2; false when
// the driver rejects it (alignment, extents) or the encoder is not loaded yet.
bool encode_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t row_bytes, uint64_t plane_bytes, uint32_t box0, uint32_t box1,
                   CUtensorMapSwizzle swizzle, CUtensorMapDataType dtype);
// NVFP4 quantization (moe_nvfp4.cu): scale-buffer bytes of a [rows, cols]
// operand; per-tensor plain and 16-row-Hadamard amax (zeroed first); the
// rowwise / (rotated) transposed quantizer with encode amax pointers.
long long nv_sf_bytes(long long rows, long long cols);
cudaError_t launch_amax_nv(const void* in, long long batch, long long rows, long long cols,
                           const int32_t* row_limit, float* amax, int num_sms,
                           cudaStream_t stream);
cudaError_t launch_quant_nv(const void* in, long long batch, long long rows, long long cols,
                            uint8_t* q, uint8_t* s, uint8_t* qt, uint8_t* st,
                            const float* amax_row, const float* amax_col, int rotate,
                            const int32_t* row_limit, int num_sms, cudaStream_t stream);
size_t grouped_gemm_smem_bytes();

// ------------------------------------------------ fp32 tensors (moe_tf32.cu)
// The ragged-M modes (kFc1Glu, kFc1Act, kFc2, kDgradDglu, kDgradAct,
// kDgradFc1) and kWgrad on TF32 tensor cores: fp32 operands, all K-major
// (tma_a / tma_b: 32-value boxes, 128-byte swizzle), fp32 outputs.
cudaError_t launch_grouped_gemm_tf32(int mode, const GemmArgs& args, int grid, cudaStream_t s);
cudaError_t launch_combine_f32(const void* y, const int32_t* row_of, const float* w, int T, int k,
                               int d, void* out, cudaStream_t s);
cudaError_t launch_combine_bwd_f32(const void* dout, const void* y, const int32_t* row_of,
                                   const float* w, int T, int k, int d, void* dy, float* dw,
                                   cudaStream_t s);
cudaError_t launch_group_colsum_f32(const void* g, const int32_t* counts,
                                    const int32_t* padded_offsets, int E, int width, void* out,
                                    cudaStream_t s);
// out[b][c][r] = in[b][r][c] for r < rows (and r < *row_limit when given).
cudaError_t launch_transpose_f32(const void* in, long long batch, long long rows, long long cols,
                                 void* out, const int32_t* row_limit, cudaStream_t s);

}  // namespace moe
