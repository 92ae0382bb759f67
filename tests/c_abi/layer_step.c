/*
 * One forward + backward step of a routed-expert MLP layer through libmoe's
 * C ABI from plain C: the caller owns every device buffer (cudaMalloc), the
 * library gets pointers, sizes and a stream.  Used by the tests to show the
 * boundary needs nothing but C and the CUDA runtime.
 *
 *   layer_step IN OUT
 *
 * IN  (little endian): int32 T, E, k, d, F; then fp32 logits [T,E], bf16 x
 *     [T,d], bf16 w1 [E,2F,d] (gate rows then linear rows), bf16 w2 [E,d,F],
 *     bf16 dout [T,d] (bf16 as raw 16-bit words).
 * OUT: bf16 out [T,d], bf16 dx [T,d], fp32 dlogits [T,E], bf16 dw1 [E,2F,d]
 *     (logical order), bf16 dw2 [E,d,F], int32 counts [E].
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe.h"

#define CHECK_CUDA(call)                                                      \
  do {                                                                        \
    cudaError_t e_ = (call);                                                  \
    if (e_ != cudaSuccess) {                                                  \
      fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));      \
      return 1;                                                               \
    }                                                                         \
  } while (0)

#define CHECK_MOE(call)                                                       \
  do {                                                                        \
    moe_status_t s_ = (call);                                                 \
    if (s_ != MOE_OK) {                                                       \
      fprintf(stderr, "%s failed: %s\n", #call, moe_status_string(s_));       \
      return 1;                                                               \
    }                                                                         \
  } while (0)

static int read_exact(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n ? 0 : 1; }
static int write_exact(FILE* f, const void* p, size_t n) { return fwrite(p, 1, n, f) == n ? 0 : 1; }

/* device buffer of n bytes, zeroed */
static void* dev_zeros(size_t n) {
  void* p = NULL;
  if (cudaMalloc(&p, n ? n : 16) != cudaSuccess) return NULL;
  if (cudaMemset(p, 0, n ? n : 16) != cudaSuccess) return NULL;
  return p;
}

/* device copy of a host array */
static void* dev_from(const void* h, size_t n) {
  void* p = dev_zeros(n);
  if (p && cudaMemcpy(p, h, n, cudaMemcpyHostToDevice) != cudaSuccess) return NULL;
  return p;
}

int main(int argc, char** argv) {
  if (argc != 3) {
    fprintf(stderr, "usage: %s IN OUT\n", argv[0]);
    return 2;
  }
  FILE* fi = fopen(argv[1], "rb");
  if (!fi) {
    fprintf(stderr, "cannot open %s\n", argv[1]);
    return 1;
  }
  int32_t hdr[5];
  if (read_exact(fi, hdr, sizeof(hdr))) return 1;
  const int32_t T = hdr[0], E = hdr[1], k = hdr[2], d = hdr[3], F = hdr[4];
  const size_t n_logits = (size_t)T * E, n_x = (size_t)T * d, n_w1 = (size_t)E * 2 * F * d,
               n_w2 = (size_t)E * d * F;
  float* h_logits = malloc(n_logits * 4);
  uint16_t* h_x = malloc(n_x * 2);
  uint16_t* h_w1 = malloc(n_w1 * 2);
  uint16_t* h_w2 = malloc(n_w2 * 2);
  uint16_t* h_dout = malloc(n_x * 2);
  if (!h_logits || !h_x || !h_w1 || !h_w2 || !h_dout) return 1;
  if (read_exact(fi, h_logits, n_logits * 4) || read_exact(fi, h_x, n_x * 2) ||
      read_exact(fi, h_w1, n_w1 * 2) || read_exact(fi, h_w2, n_w2 * 2) ||
      read_exact(fi, h_dout, n_x * 2)) {
    fprintf(stderr, "short input file\n");
    return 1;
  }
  fclose(fi);

  /* the descriptor: bf16 tensors, SwiGLU, groups aligned to 128 rows, room
   * for any routing (T*k + E*127 rows, rounded up to 128) */
  moe_mlp_desc_t desc;
  memset(&desc, 0, sizeof(desc));
  desc.T = T;
  desc.E = E;
  desc.k = k;
  desc.d = d;
  desc.F = F;
  desc.dtype = MOE_DTYPE_BF16;
  desc.act = MOE_ACT_SWIGLU;
  desc.alpha = 1.0f;
  desc.limit = INFINITY;
  desc.linear_offset = 0.0f;
  desc.out_scale = 1.0f;
  desc.align = 128;
  desc.capacity = (T * k + E * 127 + 127) / 128 * 128;
  const size_t cap = (size_t)desc.capacity;
  const size_t W1 = 2 * (size_t)moe_fc1_padded_width(F);
  size_t ws_bytes = 0;
  CHECK_MOE(moe_workspace_size(&desc, &ws_bytes));

  cudaStream_t stream;
  CHECK_CUDA(cudaStreamCreate(&stream));
  void* d_logits = dev_from(h_logits, n_logits * 4);
  void* d_x = dev_from(h_x, n_x * 2);
  void* d_w1 = dev_from(h_w1, n_w1 * 2);
  void* d_w2 = dev_from(h_w2, n_w2 * 2);
  void* d_dout = dev_from(h_dout, n_x * 2);
  void* d_w1p = dev_zeros((size_t)E * W1 * d * 2);
  void* d_ws = dev_zeros(ws_bytes);
  int32_t* topk_idx = dev_zeros((size_t)T * k * 4);
  float* topk_w = dev_zeros((size_t)T * k * 4);
  int32_t* counts = dev_zeros((size_t)E * 4);
  int32_t* offsets = dev_zeros((size_t)(E + 1) * 4);
  int32_t* padded = dev_zeros((size_t)(E + 1) * 4);
  int32_t* tiles = dev_zeros((size_t)(E + 1) * 4);
  int32_t* row_src = dev_zeros(cap * 4);
  int32_t* row_of = dev_zeros((size_t)T * k * 4);
  void* x_perm = dev_zeros(cap * d * 2);
  void* h = dev_zeros(cap * W1 * 2);
  void* a = dev_zeros(cap * F * 2);
  void* y = dev_zeros(cap * d * 2);
  void* out = dev_zeros(n_x * 2);
  void* dy = dev_zeros(cap * d * 2);
  float* dw = dev_zeros((size_t)T * k * 4);
  void* dh = dev_zeros(cap * W1 * 2);
  void* dx_perm = dev_zeros(cap * d * 2);
  void* dw1p = dev_zeros((size_t)E * W1 * d * 2);
  void* dw2 = dev_zeros(n_w2 * 2);
  void* dx = dev_zeros(n_x * 2);
  float* dlogits = dev_zeros(n_logits * 4);
  void* dw1 = dev_zeros(n_w1 * 2);
  if (!d_logits || !d_x || !d_w1 || !d_w2 || !d_dout || !d_w1p || !d_ws || !topk_idx ||
      !topk_w || !counts || !offsets || !padded || !tiles || !row_src || !row_of || !x_perm ||
      !h || !a || !y || !out || !dy || !dw || !dh || !dx_perm || !dw1p || !dw2 || !dx ||
      !dlogits || !dw1) {
    fprintf(stderr, "device allocation failed\n");
    return 1;
  }

  /* weights: FC1 repacked once */
  CHECK_MOE(moe_repack_fc1(&desc, d_w1, NULL, d_w1p, NULL, stream));
  /* forward: route + permute, the expert MLP, the weighted combine */
  CHECK_MOE(moe_route_permute(&desc, d_logits, NULL, d_x, topk_idx, topk_w, counts, offsets,
                              padded, tiles, row_src, row_of, x_perm, d_ws, ws_bytes, stream));
  CHECK_MOE(moe_mlp_fwd(&desc, x_perm, counts, padded, d_w1p, NULL, d_w2, NULL, h, a, y, NULL,
                        NULL, d_ws, ws_bytes, stream));
  CHECK_MOE(moe_unpermute_combine(&desc, y, row_of, topk_w, out, stream));
  /* backward */
  CHECK_MOE(moe_unpermute_combine_bwd(&desc, d_dout, y, row_of, topk_w, row_src, padded, dy, dw,
                                      stream));
  CHECK_MOE(moe_mlp_bwd(&desc, dy, x_perm, h, a, counts, padded, d_w1p, NULL, d_w2, dh, dx_perm,
                        dw1p, NULL, dw2, NULL, NULL, d_ws, ws_bytes, stream));
  CHECK_MOE(moe_permute_bwd(&desc, dx_perm, row_of, dx, stream));
  CHECK_MOE(moe_route_bwd(&desc, dw, topk_w, topk_idx, dlogits, stream));
  CHECK_MOE(moe_unpack_fc1(&desc, dw1p, dw1, d, stream));
  CHECK_CUDA(cudaStreamSynchronize(stream));
  int32_t status = 0;
  CHECK_MOE(moe_read_device_status(&status, 1));
  if (status != 0) {
    fprintf(stderr, "device status word 0x%x\n", (unsigned)status);
    return 1;
  }

  /* results to the host */
  uint16_t* h_out = malloc(n_x * 2);
  uint16_t* h_dx = malloc(n_x * 2);
  float* h_dlogits = malloc(n_logits * 4);
  uint16_t* h_dw1 = malloc(n_w1 * 2);
  uint16_t* h_dw2 = malloc(n_w2 * 2);
  int32_t* h_counts = malloc((size_t)E * 4);
  if (!h_out || !h_dx || !h_dlogits || !h_dw1 || !h_dw2 || !h_counts) return 1;
  CHECK_CUDA(cudaMemcpy(h_out, out, n_x * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_dx, dx, n_x * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_dlogits, dlogits, n_logits * 4, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_dw1, dw1, n_w1 * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_dw2, dw2, n_w2 * 2, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(h_counts, counts, (size_t)E * 4, cudaMemcpyDeviceToHost));
  FILE* fo = fopen(argv[2], "wb");
  if (!fo) {
    fprintf(stderr, "cannot open %s\n", argv[2]);
    return 1;
  }
  if (write_exact(fo, h_out, n_x * 2) || write_exact(fo, h_dx, n_x * 2) ||
      write_exact(fo, h_dlogits, n_logits * 4) || write_exact(fo, h_dw1, n_w1 * 2) ||
      write_exact(fo, h_dw2, n_w2 * 2) || write_exact(fo, h_counts, (size_t)E * 4)) {
    fprintf(stderr, "write failed\n");
    return 1;
  }
  fclose(fo);
  printf("layer step ok: T=%d E=%d k=%d d=%d F=%d\n", T, E, k, d, F);
  return 0;
}
