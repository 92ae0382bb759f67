/*
 * libmoe — routed-expert MLP (grouped GEMM over ragged per-expert token
 * groups), forward and backward, for one NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [FK] "Improving MoE training throughput with advanced fused kernels"
 *        (高度な融合カーネルによる MoE 学習スループットの向上):
 *        "Overcoming training bottlenecks in the MoE block",
 *        "Optimizing GLU activations with fused GEMM epilogues" (Figure 2),
 *        "Eliminating host-device synchronisation and CPU launch overhead",
 *        "Reducing exposed memory overhead by fusing MXFP8 and NVFP4
 *        quantization", "From kernel-level gains to end-to-end pretraining
 *        speedups".
 *   [DL] "Accelerating dropless MoE training with JAX and NVIDIA Transformer
 *        Engine", "Claims and evidence" (grouped GEMM over ragged tensors).
 *
 * Conventions shared by every call
 * --------------------------------
 * Notation: T tokens, E experts, k experts per token, d model width, F GLU
 * half width (FC1: d -> 2F, FC2: F -> d), R = T*k routed rows.
 *
 * Row layout ("ragged tensor", [DL]): routed rows are stored expert after
 * expert.  Expert e's group starts at padded_offsets[e], a multiple of
 * desc->align (128), and holds counts[e] rows in ascending token order; the
 * rows up to padded_offsets[e+1] are padding and every per-row tensor the
 * library writes is zero there.  Per-row buffers hold `capacity` rows, with
 * capacity >= T*k + E*(align-1) (any routing fits; no overflow is possible).
 *
 * FC1 weights are used "repacked" ([FK] GLU section, Figure 2): logical
 * w1 [E,2F,d] (rows 0..F-1 gate, F..2F-1 linear) becomes w1p [E,2F_pad,d]
 * whose row block b (256 rows) holds gate rows 128b..128b+127 then linear
 * rows 128b..128b+127; F_pad = F rounded up to 128, padding rows zero.  So
 * one 256-column output tile carries both halves of 128 GLU features.
 * b1p and every FC1-shaped output (h, dh, dw1p, db1p) use the same packed
 * column order.
 *
 * All tensors are row-major, bf16 unless stated (fp32 throughout with
 * MOE_DTYPE_FP32, see the fp32 / TF32 section).  All pointers are DEVICE
 * pointers (the caller allocates and owns every buffer; the library never
 * allocates, frees or synchronises, and reads no device data on the host),
 * so every call can be captured in a CUDA graph.  Calls are asynchronous on
 * `stream`.
 *
 * Errors: host-detectable problems (null pointer, bad shape, unsupported
 * option, workspace too small, device not sm_103) return a non-zero status
 * and enqueue nothing.  Problems only visible on the device (inconsistent
 * offsets, expert index out of range, an internal wait that ran out) set a
 * sticky device status word and the affected work is skipped; read it with
 * moe_read_device_status() outside any graph.  CUDA launch failures return
 * MOE_ERR_CUDA.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_NULL = 1,         /* a required pointer is NULL */
  MOE_ERR_SHAPE = 2,        /* sizes out of the supported range */
  MOE_ERR_UNSUPPORTED = 3,  /* option not implemented */
  MOE_ERR_WORKSPACE = 4,    /* workspace smaller than moe_workspace_size() */
  MOE_ERR_ARCH = 5,         /* current device is not sm_103 */
  MOE_ERR_CUDA = 6,         /* a CUDA runtime/driver call failed */
  MOE_ERR_DEVICE = 7        /* sticky device status word is set */
} moe_status_t;

/* Device status bits (OR-ed into the sticky word). */
#define MOE_DEV_BAD_OFFSETS 0x1   /* offsets not monotone or past capacity */
#define MOE_DEV_BAD_EXPERT  0x2   /* expert index outside [0,E) */
#define MOE_DEV_TIMEOUT     0x4   /* an in-kernel wait ran past its limit */

/* Operand type of the grouped GEMMs.  BF16: bf16 operands.  MXFP8: the
 * *_mx calls, with E4M3 operands and one E8M0 scale per 32 elements along
 * each GEMM's contraction dimension ([FK] "Reducing exposed memory overhead
 * by fusing MXFP8 and NVFP4 quantization"); requires d and F multiples of 32
 * (recompute_h: see moe_fc1_recompute_h_mx).  Routing, combine and their backward are bf16 in
 * both.  FP32: every activation, weight and gradient tensor is fp32
 * (routing, permutation, combine and their backward included), and the
 * grouped GEMMs run on the TF32 tensor cores (the *_tf32 calls, or
 * moe_mlp_fwd / moe_mlp_bwd with this dtype); fp32 accumulation. */
typedef enum {
  MOE_DTYPE_BF16 = 1,
  MOE_DTYPE_MXFP8 = 2,
  MOE_DTYPE_NVFP4 = 3,
  MOE_DTYPE_FP32 = 4
} moe_dtype_t;
/* NVFP4 (the *_nv calls): E2M1 operands, one UE4M3 scale per 16 elements
 * along each GEMM's contraction dimension and one fp32 encode scale per
 * tensor from its amax; requires d and F multiples of 64 (recompute_h: see
 * moe_fc1_recompute_h_nv). */

/* GLU activations ([FK] "Overcoming training bottlenecks": SwiGLU, GeGLU,
 * sReLU with optional clamp and scaling).  With g the gate half, l the
 * linear half, g' = min(g, limit), l' = clamp(l, -limit, limit):
 *   SWIGLU: A = s * g' * sigmoid(alpha*g') * (l' + linear_offset)
 *   GEGLU:  A = s * 0.5*g'*(1+erf(g'/sqrt2)) * (l' + linear_offset)
 *   SREGLU: A = s * max(g',0)^2 * (l' + linear_offset)   (gated squared ReLU)
 * where s = out_scale.  alpha applies to SWIGLU only. */
typedef enum {
  MOE_ACT_SWIGLU = 0,
  MOE_ACT_GEGLU = 1,
  /* non-gated squared ReLU: FC1 has F outputs (no linear half, no packing:
   * the "packed" FC1 weight is the plain [E,F,d] one and every FC1-shaped
   * tensor is F wide); A = s * max(min(h, limit), 0)^2 */
  MOE_ACT_SRELU = 2,
  MOE_ACT_SREGLU = 3
} moe_act_t;

typedef struct {
  int32_t T;            /* tokens (routing calls; 0 when groups come directly) */
  int32_t E;            /* experts, 1..256 */
  int32_t k;            /* experts per token, 1..min(E,32) */
  int32_t d;            /* model width, multiple of 64 */
  int32_t F;            /* GLU half width, multiple of 32 */
  int32_t dtype;        /* moe_dtype_t */
  int32_t act;          /* moe_act_t */
  float alpha;          /* SwiGLU gate scale (1 = plain SiLU) */
  float limit;          /* clamp limit; +inf disables */
  float linear_offset;  /* added to the linear half (0 = plain GLU) */
  float out_scale;      /* scales the activation output */
  int32_t has_b1;       /* FC1 bias present */
  int32_t has_b2;       /* FC2 bias present */
  int32_t align;        /* group alignment in rows: must be 128 */
  int32_t sm_margin;    /* SMs left free for concurrent kernels ([FK] "From
                           kernel-level gains...": configurable margin) */
  int32_t capacity;     /* rows allocated in every per-row buffer */
  int32_t recompute_h;  /* 1: the forward may skip storing H (h = NULL) and
                           moe_mlp_bwd recomputes it ([FK] "Next steps":
                           activation recompute): inside the dGLU kernel for
                           the GLU activations, into the workspace (which
                           then includes capacity*F bf16) for MOE_ACT_SRELU */
} moe_mlp_desc_t;

/* Optional MXFP8 and NVFP4-preparation outputs of a GEMM epilogue ([FK]
 * "Reducing exposed memory overhead by fusing MXFP8 and NVFP4
 * quantization": the BF16 output is also written as MXFP8 rowwise and as a
 * transposed MXFP8 copy for the backward, and per-tensor amax values are
 * produced in the same pass).  The quantized values are those of the stored
 * bf16 tensor X [capacity, width]; padding rows are zero.  Any member may be
 * NULL to skip that output.
 *   q       rowwise E4M3 codes [capacity, width], blocks of 32 along a row
 *   scale   rowwise E8M0 scales [capacity, width/32]             (with q)
 *   qt      columnwise codes written transposed [width, capacity]; blocks of
 *           32 consecutive rows (never across expert groups)
 *   scale_t columnwise scales [width, capacity/32]               (with qt)
 *   amax    float[2]: max|X| over real rows, and max|H16·s/4| over every
 *           16-row segment s of every column inside each group (the transposed
 *           16x16 Hadamard rotation; segments completed with zeros).  The
 *           call zeroes it first.
 *   layout  where the scales go (moe_mx_layout_t).
 * The same struct describes the MXFP8 inputs of the *_mx GEMM calls, which
 * need the MOE_MX_SCALES_MMA layout. */
typedef enum {
  /* scale of row r, block j at r * (cols/32) + j */
  MOE_MX_SCALES_ROWMAJOR = 0,
  /* the layout the block-scaled tensor-core MMA reads: for a tensor of
   * `rows` rows and `cols` columns (blocks along a row), atoms of 128 rows
   * x 4 blocks, 512 bytes each; the scale of row r, block j is at byte
   *   ((j/4)*RA + r/128)*512 + (r%32)*16 + ((r/32)%4)*4 + j%4,
   * RA = 2*ceil(rows/256).  The buffer holds moe_mx_scale_bytes(rows, cols)
   * bytes; entries past the tensor are read by the GEMMs but never written,
   * so the buffer must be zeroed once when allocated.  For the transposed
   * copy qt [width, capacity], rows = width and cols = capacity. */
  MOE_MX_SCALES_MMA = 1
} moe_mx_layout_t;

typedef struct {
  uint8_t* q;
  uint8_t* scale;
  uint8_t* qt;
  uint8_t* scale_t;
  float* amax;
  int32_t layout;
} moe_mx_out_t;

/* MXFP8 copies of the expert weights for the *_mx calls (each with its
 * MOE_MX_SCALES_MMA scales, per expert moe_mx_scale_bytes(rows, cols) bytes
 * where rows x cols is the per-expert code matrix):
 *   w1  [E, 2F_pad, d]  packed FC1 weight, blocks along d     (FC1)
 *   w1t [E, d, 2F_pad]  its transpose, blocks along 2F_pad   (FC1 dgrad)
 *   w2  [E, d, F]       FC2 weight, blocks along F           (FC2)
 *   w2t [E, F, d]       its transpose, blocks along d        (FC2 dgrad) */
typedef struct {
  uint8_t* w1;
  uint8_t* w1_s;
  uint8_t* w1t;
  uint8_t* w1t_s;
  uint8_t* w2;
  uint8_t* w2_s;
  uint8_t* w2t;
  uint8_t* w2t_s;
} moe_mx_weights_t;

/* F_pad = F rounded up to 128 (packed FC1 width is 2*F_pad). */
int32_t moe_fc1_padded_width(int32_t F);

/* Bytes of scratch `ws` the calls below need for this descriptor. */
moe_status_t moe_workspace_size(const moe_mlp_desc_t* desc, size_t* bytes);

/* FC1 weight repack ([FK] GLU section, Figure 2: input and gate columns
 * interleaved so one thread block owns half a tile of each; done once, e.g.
 * at checkpoint load).  w1 [E,2F,d], b1 [E,2F] or NULL -> w1p [E,2F_pad,d],
 * b1p [E,2F_pad] (NULL allowed iff b1 is NULL).  Bit-exact permutation. */
moe_status_t moe_repack_fc1(const moe_mlp_desc_t* desc, const void* w1, const void* b1,
                            void* w1p, void* b1p, cudaStream_t stream);
/* Inverse of moe_repack_fc1 for a packed [E,2F_pad,d] tensor (e.g. dW1p);
 * also for a packed [E,2F_pad] bias when d is given as 1 in `rows_width`. */
moe_status_t moe_unpack_fc1(const moe_mlp_desc_t* desc, const void* w1p, void* w1,
                            int32_t rows_width, cudaStream_t stream);

/* Routing and permutation ([FK] "Overcoming training bottlenecks": tokens
 * per expert are computed at run time; "Eliminating host-device
 * synchronisation": the group sizes stay in GPU memory; [DL]: ragged groups).
 *   logits fp32 [T,E]; bias fp32 [E] or NULL (selection only);  x [T,d].
 * Selection: the k largest of logits+bias (fp32), equal scores to the lower
 * expert, slots in descending score.  Weights: softmax of the selected raw
 * logits.  Outputs: topk_idx i32 [T,k], topk_w fp32 [T,k], counts i32 [E],
 * offsets i32 [E+1], padded_offsets i32 [E+1], tile_prefix i32 [E+1]
 * (prefix of ceil(counts/128)), row_src i32 [capacity] (token of each row,
 * -1 on padding), row_of i32 [T,k], x_perm [capacity,d].
 * ws: moe_workspace_size() bytes. */
moe_status_t moe_route_permute(const moe_mlp_desc_t* desc, const float* logits,
                               const float* bias, const void* x, int32_t* topk_idx,
                               float* topk_w, int32_t* counts, int32_t* offsets,
                               int32_t* padded_offsets, int32_t* tile_prefix,
                               int32_t* row_src, int32_t* row_of, void* x_perm,
                               void* ws, size_t ws_bytes, cudaStream_t stream);

/* Fused router (the routing work stays on the device with no host step,
 * [FK] "Overcoming training bottlenecks in the MoE block"; fusion of the
 * dispatch side, "Mixture-of-Kittens: MoE Megakernel for NVL72s", Abstract;
 * more fusion patterns, [FK] "Next steps"): logits = x W_r^T on the
 * tensor cores (bf16 x [T,d], bf16 w_router [E,d], fp32 accumulation), and in
 * the GEMM epilogue, per token, the top-k of logit + bias (fp32, ties to the
 * lower expert, descending), the softmax of the selected raw logits and the
 * expert histogram -- the logits never go through HBM unless `logits`
 * (fp32 [T,E]) is given; then, in the same launch, the scan, counting-sort
 * assignment and gather of moe_route_permute (a cooperative launch: after
 * the GEMM every CTA meets at grid-wide barriers whose waits end after a
 * time limit with MOE_DEV_TIMEOUT; MOE_ERR_CUDA if the grid cannot be
 * resident at once).  Outputs as in moe_route_permute; ws:
 * moe_workspace_size() bytes (the histogram and the barrier counter).  The
 * selection is decided on the kernel's fp32 logits. */
moe_status_t moe_route_permute_fused(const moe_mlp_desc_t* desc, const void* x,
                                     const void* w_router, const float* bias, float* logits,
                                     int32_t* topk_idx, float* topk_w, int32_t* counts,
                                     int32_t* offsets, int32_t* padded_offsets,
                                     int32_t* tile_prefix, int32_t* row_src, int32_t* row_of,
                                     void* x_perm, void* ws, size_t ws_bytes,
                                     cudaStream_t stream);

/* Offsets for groups whose sizes are given directly (no router): counts i32
 * [E] -> offsets, padded_offsets, tile_prefix i32 [E+1]. */
moe_status_t moe_group_offsets(const moe_mlp_desc_t* desc, const int32_t* counts,
                               int32_t* offsets, int32_t* padded_offsets,
                               int32_t* tile_prefix, cudaStream_t stream);

/* Expert MLP forward: FC1 grouped GEMM with the GLU epilogue (bias, clamp,
 * scale fused; [FK] GLU section) then FC2 grouped GEMM (+b2).
 *   x_perm [capacity,d]; counts [E]; padded_offsets [E+1];
 *   w1p [E,2F_pad,d]; b1p [E,2F_pad] or NULL; w2 [E,d,F]; b2 [E,d] or NULL.
 * Outputs: h [capacity,2F_pad] (FC1 output incl. bias, packed; saved for the
 * backward; NULL = not stored, to be recomputed), a [capacity,F] (GLU
 * output), y [capacity,d].  a_mx / y_mx
 * (NULL = none): MXFP8 / amax outputs of A (width F) and Y (width d).
 * Persistent tcgen05 kernels read the group sizes from device memory. */
moe_status_t moe_mlp_fwd(const moe_mlp_desc_t* desc, const void* x_perm,
                         const int32_t* counts, const int32_t* padded_offsets,
                         const void* w1p, const void* b1p, const void* w2, const void* b2,
                         void* h, void* a, void* y, const moe_mx_out_t* a_mx,
                         const moe_mx_out_t* y_mx, void* ws, size_t ws_bytes,
                         cudaStream_t stream);

/* The grouped GEMMs one at a time (moe_mlp_fwd / moe_mlp_bwd call exactly
 * these, in this order).  Buffers and layouts as in those two calls.
 *   moe_fc1_glu_fwd    h, a  <- x_perm, w1p, b1p      (FC1 + GLU epilogue [+ MX of A])
 *   moe_fc2_fwd        y     <- a, w2, b2             (FC2 "GroupGemm" [+ MX of Y])
 *   moe_fc2_dgrad_dglu dh    <- dy, w2, h             (dGLU epilogue [+ MX of dH])
 *   moe_fc2_wgrad      dw2   <- dy, a                 (K = group rows)
 *   moe_fc1_dgrad      dx_perm <- dh, w1p
 *   moe_fc1_wgrad      dw1p  <- dh, x_perm            (K = group rows)
 *   moe_bias_grads     db1p, db2 <- dh, dy            (per-group column sums;
 *                      either output may be NULL to skip it) */
moe_status_t moe_fc1_glu_fwd(const moe_mlp_desc_t* desc, const void* x_perm,
                             const int32_t* counts, const int32_t* padded_offsets,
                             const void* w1p, const void* b1p, void* h, void* a,
                             const moe_mx_out_t* a_mx, cudaStream_t stream);
moe_status_t moe_fc2_fwd(const moe_mlp_desc_t* desc, const void* a, const int32_t* counts,
                         const int32_t* padded_offsets, const void* w2, const void* b2, void* y,
                         const moe_mx_out_t* y_mx, cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu(const moe_mlp_desc_t* desc, const void* dy, const void* h,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const void* w2, void* dh, const moe_mx_out_t* dh_mx,
                                cudaStream_t stream);
moe_status_t moe_fc2_wgrad(const moe_mlp_desc_t* desc, const void* dy, const void* a,
                           const int32_t* counts, const int32_t* padded_offsets, void* dw2,
                           cudaStream_t stream);
moe_status_t moe_fc1_dgrad(const moe_mlp_desc_t* desc, const void* dh, const int32_t* counts,
                           const int32_t* padded_offsets, const void* w1p, void* dx_perm,
                           cudaStream_t stream);
moe_status_t moe_fc1_wgrad(const moe_mlp_desc_t* desc, const void* dh, const void* x_perm,
                           const int32_t* counts, const int32_t* padded_offsets, void* dw1p,
                           cudaStream_t stream);
moe_status_t moe_bias_grads(const moe_mlp_desc_t* desc, const void* dy, const void* dh,
                            const int32_t* counts, const int32_t* padded_offsets, void* db1p,
                            void* db2, cudaStream_t stream);

/* Unfused comparison path (for measuring the fusion gain; [FK] "Overcoming
 * training bottlenecks": activations usually run as separate memory-bound
 * kernels; "From kernel-level gains...": fused vs unfused up to 1.3x forward,
 * 2.1x backward).  Same results as the fused calls, computed as a plain
 * grouped GEMM followed by a separate elementwise pass:
 *   moe_fc1_glu_fwd_unfused:    H = X W1p^T (+b1), then A = GLU(H) from the
 *                               stored bf16 H.
 *   moe_fc2_dgrad_dglu_unfused: dA = dY W2 into `da` [capacity, F] (bf16,
 *                               caller scratch), then dH = dGLU(dA, H). */
moe_status_t moe_fc1_glu_fwd_unfused(const moe_mlp_desc_t* desc, const void* x_perm,
                                     const int32_t* counts, const int32_t* padded_offsets,
                                     const void* w1p, const void* b1p, void* h, void* a,
                                     cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu_unfused(const moe_mlp_desc_t* desc, const void* dy,
                                        const void* h, const int32_t* counts,
                                        const int32_t* padded_offsets, const void* w2, void* da,
                                        void* dh, cudaStream_t stream);

/* Activation recompute ([FK] "Next steps" lists it): H = X W1p^T (+b1) as a
 * plain grouped GEMM, the FC1 output the backward needs when the forward did
 * not keep it.  h [capacity, 2F_pad] packed, padding rows zero. */
moe_status_t moe_fc1_recompute_h(const moe_mlp_desc_t* desc, const void* x_perm,
                                 const int32_t* counts, const int32_t* padded_offsets,
                                 const void* w1p, const void* b1p, void* h, cudaStream_t stream);

/* Weighted combine: out[t] = sum_s topk_w[t,s] * y[row_of[t,s]] (fp32 sum in
 * slot order, then bf16).  out [T,d]. */
moe_status_t moe_unpermute_combine(const moe_mlp_desc_t* desc, const void* y,
                                   const int32_t* row_of, const float* topk_w, void* out,
                                   cudaStream_t stream);

/* Backward of the combine: dy[row_of[t,s]] = topk_w[t,s]*dout[t] (bf16,
 * padding rows zero) and dw[t,s] = <dout[t], y[row_of[t,s]]> (fp32).
 * row_src/padded_offsets locate the padding rows. */
moe_status_t moe_unpermute_combine_bwd(const moe_mlp_desc_t* desc, const void* dout,
                                       const void* y, const int32_t* row_of,
                                       const float* topk_w, const int32_t* row_src,
                                       const int32_t* padded_offsets, void* dy, float* dw,
                                       cudaStream_t stream);

/* The permutation and the combine backward with the rowwise MXFP8 copy of
 * the rows they write fused in ([FK] "Reducing exposed memory overhead by
 * fusing MXFP8 and NVFP4 quantization": the quantization happens in the
 * kernel that produces the tensor): moe_route_permute_mx also writes x_mx
 * (q [capacity,d] E4M3 codes, scale in the MMA layout) of x_perm, and
 * moe_unpermute_combine_bwd_mx the same of dy, quantized from its stored
 * bf16 values; padding rows get zero codes and scales.  Codes and scales are
 * bit for bit those of moe_quantize_act_mx (same rule, same conversions).
 * Rowwise only (x_mx / dy_mx: q and scale given, qt NULL, no amax, MMA
 * layout): the transposed copies need 32-row column blocks and stay with
 * moe_quantize_act_mx given only qt / scale_t.  Other arguments, results and
 * errors as moe_route_permute / moe_unpermute_combine_bwd. */
moe_status_t moe_route_permute_mx(const moe_mlp_desc_t* desc, const float* logits,
                                  const float* bias, const void* x, int32_t* topk_idx,
                                  float* topk_w, int32_t* counts, int32_t* offsets,
                                  int32_t* padded_offsets, int32_t* tile_prefix,
                                  int32_t* row_src, int32_t* row_of, void* x_perm,
                                  const moe_mx_out_t* x_mx, void* ws, size_t ws_bytes,
                                  cudaStream_t stream);
moe_status_t moe_unpermute_combine_bwd_mx(const moe_mlp_desc_t* desc, const void* dout,
                                          const void* y, const int32_t* row_of,
                                          const float* topk_w, const int32_t* row_src,
                                          const int32_t* padded_offsets, void* dy,
                                          const moe_mx_out_t* dy_mx, float* dw,
                                          cudaStream_t stream);

/* Expert MLP backward: FC2 dgrad with the dGLU epilogue ([FK] GLU section:
 * the epilogue reads the GEMM output and computes dSwiGLU) -> dh
 * [capacity,2F_pad] packed; FC2 wgrad dw2 [E,d,F] = sum over the group's
 * rows of dy^T a; FC1 dgrad dx_perm [capacity,d] = dh w1p; FC1 wgrad
 * dw1p [E,2F_pad,d] = dh^T x_perm (packed); db1p [E,2F_pad] and db2 [E,d]
 * (NULL when the bias is absent).  Experts with no rows get zero gradients.
 * dh_mx (NULL = none): MXFP8 / amax outputs of dH (width 2*F_pad, packed).
 * h = NULL (needs desc->recompute_h = 1): H is recomputed from x_perm, w1p
 * and b1p (b1p is used only then) -- for the GLU activations inside the
 * dGLU kernel (moe_fc2_dgrad_dglu_recompute: H never reaches HBM), for
 * MOE_ACT_SRELU by a plain FC1 grouped GEMM into the workspace first (a
 * workspace of moe_workspace_size() bytes). */
moe_status_t moe_mlp_bwd(const moe_mlp_desc_t* desc, const void* dy, const void* x_perm,
                         const void* h, const void* a, const int32_t* counts,
                         const int32_t* padded_offsets, const void* w1p, const void* b1p,
                         const void* w2, void* dh, void* dx_perm, void* dw1p, void* db1p,
                         void* dw2, void* db2, const moe_mx_out_t* dh_mx, void* ws,
                         size_t ws_bytes, cudaStream_t stream);

/* Backward of the permutation: dx[t] = sum_s dx_perm[row_of[t,s]] (fp32 in
 * slot order, then bf16).  dx [T,d]. */
moe_status_t moe_permute_bwd(const moe_mlp_desc_t* desc, const void* dx_perm,
                             const int32_t* row_of, void* dx, cudaStream_t stream);

/* Backward of the routing softmax: dlogits fp32 [T,E] with
 * dlogits[t,idx[t,s]] = w[t,s]*(dw[t,s] - sum_s' w[t,s']*dw[t,s']), 0 elsewhere. */
moe_status_t moe_route_bwd(const moe_mlp_desc_t* desc, const float* dw, const float* topk_w,
                           const int32_t* topk_idx, float* dlogits, cudaStream_t stream);

/* MXFP8 quantization of fp32 values in [rows, cols] (row-major), with the
 * device quantizer the fused epilogues use ([FK] "Reducing exposed memory
 * overhead by fusing MXFP8 and NVFP4 quantization"; format: OCP MX E4M3
 * payload, one E8M0 scale per 32 elements, scale 2^(floor(log2 amax)-8),
 * round-to-nearest-even with saturation to +-448).
 *   colwise = 0: blocks run along each row; q [rows, cols], scales
 *                [rows, cols/32]; cols % 32 == 0.
 *   colwise = 1: blocks run down each column; q is written transposed
 *                [cols, rows], scales [cols, rows/32]; rows % 32 == 0.
 * in and q 16-byte aligned. */
moe_status_t moe_quantize_mx(const float* in, int32_t rows, int32_t cols, int32_t colwise,
                             uint8_t* q, uint8_t* scales, cudaStream_t stream);

/* ------------------------------------------------------------- MXFP8 path
 * [FK] "Reducing exposed memory overhead by fusing MXFP8 and NVFP4
 * quantization": the MoE GEMMs read MXFP8 operands; the FC1 epilogue writes
 * the activation both rowwise (next GEMM) and transposed (its weight
 * gradient); the dSwiGLU epilogue does the same for dH.  Every GEMM operand
 * is quantized along that GEMM's contraction dimension; weight gradients
 * contract over an expert group's rows, in 32-row blocks from the group's
 * start.  Accumulation is fp32; H, A, Y, dH, dX_perm and dW are stored bf16. */

/* Bytes of a MOE_MX_SCALES_MMA scale buffer of a [rows, cols] tensor (0 for
 * an empty one). */
size_t moe_mx_scale_bytes(int64_t rows, int64_t cols);

/* bf16 in [batch, rows, cols] -> MXFP8 (rows, cols multiples of 32): q
 * [batch, rows, cols] with blocks along a row and/or qt [batch, cols, rows]
 * with blocks down a column; scales in out->layout, per batch entry
 * moe_mx_scale_bytes(rows, cols) resp. (cols, rows) bytes in the MMA layout.
 * out->amax must be NULL.  Same quantizer as the fused epilogues. */
moe_status_t moe_quantize_mx_bf16(const void* in, int64_t batch, int64_t rows, int64_t cols,
                                  const moe_mx_out_t* out, cudaStream_t stream);

/* An activation [capacity, width] (x_perm or dY) in MXFP8, rowwise and/or
 * transposed, MOE_MX_SCALES_MMA; only rows below padded_offsets[E] (read on
 * the device) are converted. */
moe_status_t moe_quantize_act_mx(const moe_mlp_desc_t* desc, const void* in, int32_t width,
                                 const int32_t* padded_offsets, const moe_mx_out_t* out,
                                 cudaStream_t stream);

/* Weight preparation, once per optimizer step: w1p [E,2F_pad,d] and w2
 * [E,d,F] (bf16) -> the four MXFP8 copies of moe_mx_weights_t. */
moe_status_t moe_quantize_weights_mx(const moe_mlp_desc_t* desc, const void* w1p,
                                     const void* w2, const moe_mx_weights_t* out,
                                     cudaStream_t stream);

/* MXFP8 forward (desc->dtype = MOE_DTYPE_MXFP8):
 *   x_mx  x_perm rowwise (q, scale)                      [input]
 *   h     H bf16 [capacity, 2F_pad] (kept for the dGLU)  [output]
 *   a     A bf16 [capacity, F] or NULL to skip it        [output]
 *   a_mx  A rowwise (q, scale: FC2's operand) and, when qt is given, the
 *         transposed copy (qt, scale_t: FC2 weight gradient); amax optional
 *   y     Y bf16 [capacity, d]
 * Biases as in moe_mlp_fwd.  Same groups, padding and errors as moe_mlp_fwd. */
moe_status_t moe_mlp_fwd_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                            const int32_t* counts, const int32_t* padded_offsets,
                            const moe_mx_weights_t* w, const void* b1p, const void* b2, void* h,
                            void* a, const moe_mx_out_t* a_mx, void* y, cudaStream_t stream);

/* The MXFP8 grouped GEMMs one at a time (moe_mlp_fwd_mx / moe_mlp_bwd_mx
 * call exactly these, in this order); arguments as in those two calls.
 *   moe_fc1_glu_fwd_mx    h, a, a_mx <- x_mx (rowwise), w1
 *   moe_fc2_fwd_mx        y          <- a_mx (rowwise), w2
 *   moe_fc2_dgrad_dglu_mx dh, dh_mx  <- dy_mx (rowwise), w2t, h
 *                         (dh, the bf16 dH, may be NULL: only the MXFP8
 *                         copies the later GEMMs read are then written; the
 *                         FC1 bias gradient needs dh)
 *   moe_fc2_wgrad_mx      dw2        <- dy_mx, a_mx (transposed copies)
 *   moe_fc1_dgrad_mx      dx_perm    <- dh_mx (rowwise), w1t
 *   moe_fc1_wgrad_mx      dw1p       <- dh_mx, x_mx (transposed copies) */
moe_status_t moe_fc1_glu_fwd_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const moe_mx_weights_t* w, const void* b1p, void* h, void* a,
                                const moe_mx_out_t* a_mx, cudaStream_t stream);
moe_status_t moe_fc2_fwd_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* a_mx,
                            const int32_t* counts, const int32_t* padded_offsets,
                            const moe_mx_weights_t* w, const void* b2, void* y,
                            cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_mx,
                                   const void* h, const int32_t* counts,
                                   const int32_t* padded_offsets, const moe_mx_weights_t* w,
                                   void* dh, const moe_mx_out_t* dh_mx, cudaStream_t stream);
moe_status_t moe_fc2_wgrad_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_mx,
                              const moe_mx_out_t* a_mx, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw2, cudaStream_t stream);
moe_status_t moe_fc1_dgrad_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_mx,
                              const int32_t* counts, const int32_t* padded_offsets,
                              const moe_mx_weights_t* w, void* dx_perm, cudaStream_t stream);
moe_status_t moe_fc1_wgrad_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_mx,
                              const moe_mx_out_t* x_mx, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw1p, cudaStream_t stream);

/* Activation recompute on the MXFP8 path (desc->recompute_h = 1): the
 * forward may pass h = NULL to moe_fc1_glu_fwd_mx / moe_mlp_fwd_mx; before
 * the backward, this call regenerates H [capacity, W1] bf16 into a buffer
 * of the caller's from the forward's x_mx (rowwise) and w->w1 with the same
 * MMAs in the same order (bitwise the H the forward would have stored), to
 * be passed as h to moe_fc2_dgrad_dglu_mx / moe_mlp_bwd_mx. */
moe_status_t moe_fc1_recompute_h_mx(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                                    const int32_t* counts, const int32_t* padded_offsets,
                                    const moe_mx_weights_t* w, const void* b1p, void* h,
                                    cudaStream_t stream);

/* MXFP8 backward:
 *   dy     dY bf16 [capacity, d] (bias gradient)   dy_mx  its rowwise and
 *          transposed MXFP8 copies                  x_mx   x_perm transposed
 *          (qt, scale_t)                            a_mx   A transposed
 *   h      the forward's H;  dh: dH bf16 [capacity, 2F_pad] (output)
 *   dh_mx  receives dH rowwise and transposed (q, scale, qt, scale_t)
 *   dx_perm, dw1p, db1p, dw2, db2 as in moe_mlp_bwd (db1p / db2 NULL to skip). */
moe_status_t moe_mlp_bwd_mx(const moe_mlp_desc_t* desc, const void* dy,
                            const moe_mx_out_t* dy_mx, const moe_mx_out_t* x_mx, const void* h,
                            const moe_mx_out_t* a_mx, const int32_t* counts,
                            const int32_t* padded_offsets, const moe_mx_weights_t* w, void* dh,
                            const moe_mx_out_t* dh_mx, void* dx_perm, void* dw1p, void* db1p,
                            void* dw2, void* db2, cudaStream_t stream);

/* ------------------------------------------------------------- NVFP4 path
 * [FK] "Reducing exposed memory overhead by fusing MXFP8 and NVFP4
 * quantization": for NVFP4 the GEMM epilogues emit the BF16 output with its
 * per-tensor amax and the amax of its transposed Hadamard rotation, and the
 * tensor is then quantized for the next NVFP4 GEMMs with the per-tensor
 * scale those amax values give.  Readings: E2M1 values (+-{0, .5, 1, 1.5, 2,
 * 3, 4, 6}, round to nearest even, saturating) in blocks of 16 along the
 * contraction axis; per block a UE4M3 scale s = E4M3((amax_block / 6) * g)
 * (round to nearest even, saturating at 448); per tensor g = 2688 / amax
 * (1 for amax 0); a value is code * s / g; every step in fp32.  The copies
 * that the weight gradients contract over tokens are rotated first by H16/4
 * (Sylvester Hadamard) in 16-row segments inside each group and use the
 * rotated tensor's amax.
 *
 * NVFP4 tensors are described by moe_mx_out_t with layout MOE_MX_SCALES_MMA:
 *   q       packed E2M1 [rows, cols/2] (two values per byte, element 2i in
 *           the low nibble), 16-byte aligned; scale: UE4M3 codes in the MMA
 *           layout of MXFP8 with 16-element blocks (moe_nvfp4_scale_bytes).
 *   qt      the transposed copy [cols, rows/2], scale_t its scales.
 *   amax    float[2]: [0] the amax that encodes q (the tensor's), [1] the
 *           one that encodes qt (the rotated tensor's).  Weights use
 *           moe_nv_weights_t below instead.
 * The GEMMs divide the encode scales out of the accumulator (factor
 * 1 / (g_a g_b)) before bias, activation and output. */

/* Bytes of the NVFP4 scale buffer of a [rows, cols] operand (0 for empty):
 * ceil(cols/64) * 2*ceil(rows/256) atoms of 512 bytes. */
size_t moe_nvfp4_scale_bytes(int64_t rows, int64_t cols);

/* amax[0] = max |x|, amax[1] = max |H16 x / 4| (each column rotated along
 * the rows in 16-row segments) of bf16 [batch, rows, cols], rows % 16 == 0,
 * cols % 8 == 0, in 16-byte aligned, over the rows below *row_limit (device
 * int; NULL = all rows).  amax is overwritten. */
moe_status_t moe_amax_nvfp4(const void* in, int64_t batch, int64_t rows, int64_t cols,
                            const int32_t* row_limit, float* amax, cudaStream_t stream);

/* bf16 [batch, rows, cols] (rows, cols multiples of 32) -> NVFP4 with the
 * encode amax values in out->amax (device float[2], read on the device):
 * rowwise (out->q) and/or transposed (out->qt, rotated by H16/4 along the
 * rows when rotate_t != 0).  Scales per batch entry: moe_nvfp4_scale_bytes
 * (rows, cols) resp. (cols, rows). */
moe_status_t moe_quantize_nvfp4_bf16(const void* in, int64_t batch, int64_t rows, int64_t cols,
                                     const moe_mx_out_t* out, int32_t rotate_t,
                                     cudaStream_t stream);

/* An activation [capacity, width] (x_perm, A, dY or dH) in NVFP4: rowwise
 * and/or the rotated transposed copy, only rows below padded_offsets[E].
 * compute_amax != 0: out->amax is first computed from the tensor (x_perm,
 * dY); 0: out->amax already holds it (A, dH: written by the GEMM epilogue). */
moe_status_t moe_quantize_act_nvfp4(const moe_mlp_desc_t* desc, const void* in, int32_t width,
                                    const int32_t* padded_offsets, const moe_mx_out_t* out,
                                    int32_t compute_amax, cudaStream_t stream);

/* NVFP4 copies of the expert weights: as moe_mx_weights_t (w1 [E, W1, d/2]
 * rowwise along d, w1t [E, d, W1/2], w2 [E, d, F/2], w2t [E, F, d/2], scales
 * per expert moe_nvfp4_scale_bytes) plus amax: device float[4], written by
 * moe_quantize_weights_nvfp4: [0] = max|W1p| (encodes w1 and w1t), [2] =
 * max|W2| (w2, w2t); [1] and [3] hold the rotated amax, which is unused. */
typedef struct {
  moe_mx_weights_t q;
  float* amax;
} moe_nv_weights_t;

moe_status_t moe_quantize_weights_nvfp4(const moe_mlp_desc_t* desc, const void* w1p,
                                        const void* w2, const moe_nv_weights_t* out,
                                        cudaStream_t stream);

/* The NVFP4 grouped GEMMs (desc->dtype = MOE_DTYPE_NVFP4), as the *_mx
 * calls, with NVFP4 operands:
 *   moe_fc1_glu_fwd_nv    h, a, a_amax  <- x_nv (q), w1      a_amax: float[2]
 *   moe_fc2_fwd_nv        y             <- a_nv (q), w2
 *   moe_fc2_dgrad_dglu_nv dh, dh_amax   <- dy_nv (q), w2t, h dh_amax: float[2]
 *   moe_fc2_wgrad_nv      dw2           <- dy_nv, a_nv (qt: rotated copies)
 *   moe_fc1_dgrad_nv      dx_perm       <- dh_nv (q), w1t
 *   moe_fc1_wgrad_nv      dw1p          <- dh_nv, x_nv (qt: rotated copies)
 * a_amax / dh_amax receive the plain and rotated amax of the bf16 A / dH
 * (over real rows), which moe_quantize_act_nvfp4 then uses. */
moe_status_t moe_fc1_glu_fwd_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_nv,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const moe_nv_weights_t* w, const void* b1p, void* h, void* a,
                                float* a_amax, cudaStream_t stream);
moe_status_t moe_fc2_fwd_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* a_nv,
                            const int32_t* counts, const int32_t* padded_offsets,
                            const moe_nv_weights_t* w, const void* b2, void* y,
                            cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_nv,
                                   const void* h, const int32_t* counts,
                                   const int32_t* padded_offsets, const moe_nv_weights_t* w,
                                   void* dh, float* dh_amax, cudaStream_t stream);
moe_status_t moe_fc2_wgrad_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dy_nv,
                              const moe_mx_out_t* a_nv, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw2, cudaStream_t stream);
moe_status_t moe_fc1_dgrad_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_nv,
                              const int32_t* counts, const int32_t* padded_offsets,
                              const moe_nv_weights_t* w, void* dx_perm, cudaStream_t stream);
moe_status_t moe_fc1_wgrad_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* dh_nv,
                              const moe_mx_out_t* x_nv, const int32_t* counts,
                              const int32_t* padded_offsets, void* dw1p, cudaStream_t stream);

/* Activation recompute on the NVFP4 path (desc->recompute_h = 1): the
 * forward may pass h = NULL; this call regenerates H [capacity, W1] bf16
 * into a caller buffer from the forward's x_nv (rowwise) and w->q.w1 with
 * the same MMAs and encode factors (bitwise the H the forward would have
 * stored), to be passed as h to the dGLU call. */
moe_status_t moe_fc1_recompute_h_nv(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_nv,
                                    const int32_t* counts, const int32_t* padded_offsets,
                                    const moe_nv_weights_t* w, const void* b1p, void* h,
                                    cudaStream_t stream);

/* NVFP4 forward (desc->dtype = MOE_DTYPE_NVFP4) in one call:
 *   x_perm bf16 [capacity, d] -> x_nv (amax computed, rowwise + rotated
 *   transposed copies) -> FC1 + GLU (h, a bf16; a_nv->amax) -> a_nv (rowwise
 *   + rotated transposed copies) -> FC2 (y).
 * x_nv / a_nv: NVFP4 buffers (q, scale, qt, scale_t, amax[2]) as described
 * above, widths d and F. */
moe_status_t moe_mlp_fwd_nv(const moe_mlp_desc_t* desc, const void* x_perm,
                            const moe_mx_out_t* x_nv, const int32_t* counts,
                            const int32_t* padded_offsets, const moe_nv_weights_t* w,
                            const void* b1p, const void* b2, void* h, void* a,
                            const moe_mx_out_t* a_nv, void* y, cudaStream_t stream);

/* NVFP4 backward in one call: dY bf16 [capacity, d] -> dy_nv -> FC2 dgrad +
 * dGLU (dh bf16, dh_nv->amax) -> dh_nv -> FC2 wgrad (dw2, from dy_nv and
 * a_nv's transposed copies), FC1 dgrad (dx_perm), FC1 wgrad (dw1p, from
 * dh_nv and x_nv's transposed copies), bias gradients (db1p / db2, NULL to
 * skip).  x_nv and a_nv are the forward's buffers. */
moe_status_t moe_mlp_bwd_nv(const moe_mlp_desc_t* desc, const void* dy,
                            const moe_mx_out_t* dy_nv, const moe_mx_out_t* x_nv, const void* h,
                            const moe_mx_out_t* a_nv, const int32_t* counts,
                            const int32_t* padded_offsets, const moe_nv_weights_t* w, void* dh,
                            const moe_mx_out_t* dh_nv, void* dx_perm, void* dw1p, void* db1p,
                            void* dw2, void* db2, cudaStream_t stream);

/* FC2 dgrad + dGLU with activation recompute inside the kernel ([FK] "Next
 * steps" names activation recompute as future work): for each tile of 128
 * rows x 128 GLU features the kernel computes H = X W1p^T (+b1) for the
 * tile's packed block (128 gate + 128 linear columns) and dA = dY W2, both
 * over K = d, into tensor memory, rounds H to bf16 (as the stored H is) and
 * applies the dGLU from there: H never reaches HBM, and the forward need not
 * keep it (moe_fc1_glu_fwd with h = NULL when desc->recompute_h).  dh as in
 * moe_fc2_dgrad_dglu (bf16, packed), plus the optional MXFP8 / amax outputs
 * of dh_mx.  H's MMAs are the forward's, so dH equals the stored-H path's.
 * GLU activations only (MOE_ERR_UNSUPPORTED for MOE_ACT_SRELU).
 *   moe_fc2_dgrad_dglu_recompute:    bf16 operands x_perm, dy, w1p, w2.
 *   moe_fc2_dgrad_dglu_recompute_mx: the forward's MXFP8 x_mx (rowwise),
 *                                    dY's dy_mx (rowwise), the weights' w1
 *                                    and w2t copies; dh_mx receives dH's
 *                                    MXFP8 rowwise and transposed copies. */
moe_status_t moe_fc2_dgrad_dglu_recompute(const moe_mlp_desc_t* desc, const void* x_perm,
                                          const void* dy, const int32_t* counts,
                                          const int32_t* padded_offsets, const void* w1p,
                                          const void* b1p, const void* w2, void* dh,
                                          const moe_mx_out_t* dh_mx, cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu_recompute_mx(const moe_mlp_desc_t* desc,
                                             const moe_mx_out_t* x_mx,
                                             const moe_mx_out_t* dy_mx, const int32_t* counts,
                                             const int32_t* padded_offsets,
                                             const moe_mx_weights_t* w, const void* b1p,
                                             void* dh, const moe_mx_out_t* dh_mx,
                                             cudaStream_t stream);

/* The unfused MXFP8 arrangement the fused epilogues replace ([FK]
 * "Overcoming training bottlenecks in the MoE block": activation and
 * quantization as separate memory-bound kernels; "From kernel-level gains
 * to end-to-end pretraining speedups" measures the fused kernels against
 * it).  Each call runs three kernels one after another:
 *   moe_fc1_glu_fwd_mx_unfused:    H = X W1p^T (+b1) as a plain grouped GEMM
 *                                  on the MXFP8 operands (h, bf16 [capacity,
 *                                  2F_pad], packed), then A = GLU(H) from the
 *                                  stored bf16 H (a, bf16 [capacity, F]),
 *                                  then MXFP8 quantization of A rowwise and
 *                                  transposed into a_mx (MMA scale layout).
 *   moe_fc2_dgrad_dglu_mx_unfused: dA = dY W2 as a plain grouped GEMM on the
 *                                  MXFP8 operands (da, bf16 [capacity, F],
 *                                  caller scratch), then dH = dGLU(dA, H)
 *                                  (dh, bf16, packed), then MXFP8 quantization
 *                                  of dH rowwise and transposed into dh_mx.
 * GLU activations only (MOE_ERR_UNSUPPORTED for MOE_ACT_SRELU).  A is
 * computed from the bf16-rounded H here (the fused epilogue uses the fp32
 * accumulator), so results agree with the fused calls to bf16 rounding, not
 * bit for bit. */
moe_status_t moe_fc1_glu_fwd_mx_unfused(const moe_mlp_desc_t* desc, const moe_mx_out_t* x_mx,
                                        const int32_t* counts, const int32_t* padded_offsets,
                                        const moe_mx_weights_t* w, const void* b1p, void* h,
                                        void* a, const moe_mx_out_t* a_mx, cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu_mx_unfused(const moe_mlp_desc_t* desc,
                                           const moe_mx_out_t* dy_mx, const void* h,
                                           const int32_t* counts, const int32_t* padded_offsets,
                                           const moe_mx_weights_t* w, void* da, void* dh,
                                           const moe_mx_out_t* dh_mx, cudaStream_t stream);

/* ------------------------------------------------------- fp32 / TF32 path
 * The same routed-expert MLP ([FK] "Overcoming training bottlenecks in the
 * MoE block": grouped GEMM + activation and + dActivation; "Optimizing GLU
 * activations with fused GEMM epilogues", Figure 2: the repacked FC1 tile
 * and its GLU epilogue; [DL] "Claims and evidence": ragged groups) on fp32
 * tensors.
 * desc->dtype == MOE_DTYPE_FP32: the tensors of every call are fp32 (same
 * shapes, layouts, padding and packing as the bf16 path).  The routing,
 * permutation, combine and bias-gradient calls (moe_route_permute,
 * moe_route_permute_noalloc, moe_unpermute_combine[_bwd], moe_permute_bwd,
 * moe_bias_grads, moe_repack_fc1, moe_unpack_fc1) follow the descriptor's
 * dtype; their sums are fp32.  The grouped GEMMs run on the TF32 tensor cores
 * (tcgen05 kind::tf32: operands rounded to TF32's 10-bit mantissa by the
 * tensor core, fp32 accumulation) with the same fused epilogues as the bf16
 * calls, and store fp32 results.  Every operand is read K-major, so the
 * backward reads transposed copies:
 *   moe_transpose_weights_tf32  w1t [E, d, W1] = w1p^T, w2t [E, F, d] = w2^T
 *                               (once per weight update)
 *   moe_transpose_rows_f32      out [width, capacity] = in^T for the rows
 *                               below padded_offsets[E] (x_perm, dY, A)
 *   moe_fc1_glu_fwd_tf32        h, a (+ a_t = A^T [F, capacity], optional)
 *                               <- x_perm, w1p, b1p
 *   moe_fc2_fwd_tf32            y <- a, w2, b2
 *   moe_fc2_dgrad_dglu_tf32     dh and/or dh_t = dH^T [W1, capacity]
 *                               <- dy, h, w2t
 *   moe_fc2_wgrad_tf32          dw2 [E, d, F] <- dy_t [d, capacity],
 *                               a_t [F, capacity]   (K = group rows)
 *   moe_fc1_dgrad_tf32          dx_perm <- dh, w1t
 *   moe_fc1_wgrad_tf32          dw1p [E, W1, d] <- dh_t [W1, capacity],
 *                               x_t [d, capacity]   (K = group rows)
 * W1 = 2*F_pad for the GLU activations, F for MOE_ACT_SRELU.  The transposed
 * copies hold zeros in the padding rows' columns (the row tensors are zero
 * there).  moe_mlp_fwd with MOE_DTYPE_FP32 runs the two forward GEMMs (a_mx,
 * y_mx must be NULL); moe_mlp_bwd makes the transposed weights and
 * activations in its workspace (moe_workspace_size includes them), then runs
 * the four backward GEMMs and the bias gradients (dh_mx NULL).
 * recompute_h is not supported with fp32 tensors.  Output pointers (h, a,
 * a_t, y, dh, dh_t, dw1p, dw2, dx_perm) must be 16-byte aligned (else
 * MOE_ERR_SHAPE); other errors as for the bf16 calls. */
moe_status_t moe_transpose_weights_tf32(const moe_mlp_desc_t* desc, const void* w1p,
                                        const void* w2, void* w1t, void* w2t,
                                        cudaStream_t stream);
moe_status_t moe_transpose_rows_f32(const moe_mlp_desc_t* desc, const void* in, int32_t width,
                                    const int32_t* padded_offsets, void* out,
                                    cudaStream_t stream);
moe_status_t moe_fc1_glu_fwd_tf32(const moe_mlp_desc_t* desc, const void* x_perm,
                                  const int32_t* counts, const int32_t* padded_offsets,
                                  const void* w1p, const void* b1p, void* h, void* a, void* a_t,
                                  cudaStream_t stream);
moe_status_t moe_fc2_fwd_tf32(const moe_mlp_desc_t* desc, const void* a, const int32_t* counts,
                              const int32_t* padded_offsets, const void* w2, const void* b2,
                              void* y, cudaStream_t stream);
moe_status_t moe_fc2_dgrad_dglu_tf32(const moe_mlp_desc_t* desc, const void* dy, const void* h,
                                     const int32_t* counts, const int32_t* padded_offsets,
                                     const void* w2t, void* dh, void* dh_t, cudaStream_t stream);
moe_status_t moe_fc2_wgrad_tf32(const moe_mlp_desc_t* desc, const void* dy_t, const void* a_t,
                                const int32_t* counts, const int32_t* padded_offsets, void* dw2,
                                cudaStream_t stream);
moe_status_t moe_fc1_dgrad_tf32(const moe_mlp_desc_t* desc, const void* dh,
                                const int32_t* counts, const int32_t* padded_offsets,
                                const void* w1t, void* dx_perm, cudaStream_t stream);
moe_status_t moe_fc1_wgrad_tf32(const moe_mlp_desc_t* desc, const void* dh_t, const void* x_t,
                                const int32_t* counts, const int32_t* padded_offsets,
                                void* dw1p, cudaStream_t stream);

/* moe_route_permute for callers that cannot allocate device memory (for
 * example a host program whose device memory is all handed to its own fixed
 * pool, or a runtime that allows no allocation after start-up).  The pages
 * have no counterpart to this call; it exists only for such callers.
 * Same arguments and results as moe_route_permute minus ws/ws_bytes: the
 * scratch histogram lives in a static device array of this library
 * (256 KiB, reserved on every GPU that loads the library until the process
 * exits).  Requires ceil(T/256)*E*4 <= 262144 bytes, else returns
 * MOE_ERR_WORKSPACE and enqueues nothing.  It allocates nothing.  The first
 * call on a device looks up the array's device address (with that device
 * current) and should happen before any stream capture; the address is kept
 * until the process exits, so a device reset (cudaDeviceReset) after that
 * first call is not supported (the same holds for every call of this
 * library, which keeps the address of its status word).  All calls share
 * the array: calls whose GPU work may overlap (unordered streams) race;
 * calls ordered on one stream are safe because each call zeroes the
 * histogram before use. */
moe_status_t moe_route_permute_noalloc(const moe_mlp_desc_t* desc, const float* logits,
                                       const float* bias, const void* x, int32_t* topk_idx,
                                       float* topk_w, int32_t* counts, int32_t* offsets,
                                       int32_t* padded_offsets, int32_t* tile_prefix,
                                       int32_t* row_src, int32_t* row_of, void* x_perm,
                                       cudaStream_t stream);

/* Failure-detection self test (the pages have no counterpart): one CTA waits,
 * through the bounded mbarrier wait the GEMM pipelines use, on a phase that
 * nothing completes; after limit_us microseconds (1..5e6) the wait gives up,
 * sets MOE_DEV_TIMEOUT in the status word and the kernel returns, leaving
 * the context usable. */
moe_status_t moe_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/* The same for the grid-wide barrier of the fused router's cooperative
 * launch: one CTA arrives at a barrier that expects a second arrival nobody
 * makes; after limit_us microseconds (1..5e6) the wait gives up, sets
 * MOE_DEV_TIMEOUT and the kernel returns. */
moe_status_t moe_selftest_grid_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/* Read (and optionally clear) the sticky device status word of the current
 * device.  Synchronises the device; call outside stream capture. */
moe_status_t moe_read_device_status(int32_t* host_status, int32_t clear);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
