// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05) for
// the routed-expert MLP, forward and backward, with the fused epilogues.
//
// Sources: "Improving MoE training throughput with advanced fused kernels":
//   - "Overcoming training bottlenecks in the MoE block": the GroupGemm
//     kernel families (GroupGemm + Activation, GroupGemm + dActivation).
//   - "Optimizing GLU activations with fused GEMM epilogues" (Figure 2): with
//     the FC1 weight repacked, one CTA's accumulator tile holds 128 gate and
//     the matching 128 linear features, so the GLU (with bias, clamp and
//     scaling) is applied in the epilogue; the backward epilogue reads the
//     GEMM output and computes dSwiGLU.
//   - "Eliminating host-device synchronisation and CPU launch overhead": the
//     per-group token counts are read from GPU memory by the kernel; the grid
//     is sized from the SM count, never from the routing result.
//   - "From kernel-level gains to end-to-end pretraining speedups": the grid
//     leaves `sm_margin` SMs free.
// "Accelerating dropless MoE training with JAX and NVIDIA Transformer
// Engine", "Claims and evidence": one grouped GEMM call over ragged groups.
//
// Design of the grouped GEMM (one CTA per SM, 10 warps):
//   warp 0   TMA producer: 128B-swizzled operand tiles into a ring of 4
//            stages (3 for NVFP4 and for the async-H dGLU variants).
//   warp 1   TMEM owner and single-thread MMA issuer (M=128, N=256; K=16
//            per bf16 MMA, K=32 per block-scaled MXFP8 MMA, K=64 per NVFP4
//            MMA).
//   warps 2-9 epilogue, two warps per TMEM lane quarter, each taking 16 of
//            every 32 accumulator columns: tcgen05.ld, fused math, bf16
//            (and MXFP8) outputs.  Two 256-column accumulators in TMEM let
//            the epilogue of one tile overlap the MMAs of the next.
// The bf16 weight-gradient kernel on CTA pairs uses the same warp roles.
// Tiles are 128 rows x 256 columns.  Every expert group starts at a
// multiple of 128 rows, so an M tile never straddles two experts; rows past
// the group's count are padding and are written as zeros.  Weight-gradient
// tiles (ragged K) run the K loop over the group's rows only; groups are
// visited largest first for balance.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_act.cuh"
#include "moe_internal.h"
#include "moe_mx.cuh"
#include "moe_ptx.cuh"
#include "moe_route.cuh"

namespace moe {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;                       // 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int B_BYTES = BN * BK * 2;         // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int MN_BOX_BYTES = 64 * BK * 2;    // one 64(MN) x 64(K) box, 8 KB
constexpr int TMEM_COLS = 2 * BN;            // two fp32 accumulators
constexpr int GEMM_THREADS = 320;            // producer, MMA, 8 epilogue warps (both kernels)
constexpr int kGemmEpiThreads = 256;
constexpr int kRing = 4;                     // output staging boxes (shared by the epilogue)
constexpr int BOX_BYTES = 128 * 32 * 2;      // one 128-row x 32-column bf16 output box
constexpr int kEpiBar = 1;                   // named barrier of the epilogue warps
constexpr size_t SMEM_BYTES =
    1024 + static_cast<size_t>(STAGES) * STAGE_BYTES + kRing * BOX_BYTES;
// MXFP8 operands: the same 128-byte rows hold 128 E4M3 values, so a stage
// covers K = 128; its scales (A: one 512-byte atom, B: two) follow the
// operand stages, and the output ring shrinks to 3 boxes to make room.
constexpr int BK_MX = 128;
constexpr int SF_STAGE_BYTES = 1536;
constexpr int kRingMx = 3;
constexpr size_t SMEM_BYTES_MX = 1024 + static_cast<size_t>(STAGES) * STAGE_BYTES +
                                 static_cast<size_t>(STAGES) * SF_STAGE_BYTES +
                                 kRingMx * BOX_BYTES;
// TMEM columns (from the start of the accumulator NOT in use by the current
// tile) that receive one stage's scales: A at +0 (4 columns), B at +32 (8),
// both 32-column aligned.  The epilogue releases them once it has read the
// accumulator's first 64 columns.
constexpr uint32_t kSfaCol = 0, kSfbCol = 32;
// NVFP4 operands: packed E2M1 (two per byte), so a 128-byte row holds 256
// values and a stage covers K = 256, four MMAs of K = 64.  Every MMA takes
// its own scale atoms (A: one 512-byte atom, B: two), 6 KB per stage; with
// three stages the full output ring still fits.
constexpr int BK_NV = 256;
constexpr int STAGES_NV = 3;
constexpr int SF_STAGE_BYTES_NV = 6144;
constexpr size_t SMEM_BYTES_NV = 1024 + static_cast<size_t>(STAGES_NV) *
                                            (STAGE_BYTES + SF_STAGE_BYTES_NV) +
                                 kRing * BOX_BYTES;
// operand formats of k_grouped_gemm.  kOpBf16H / kOpMxH are bf16 / MXFP8
// with the FC2 dgrad + dGLU epilogue reading the saved H (gate and linear
// share of each 32-feature chunk, 64 bytes per thread) through cp.async into
// a shared buffer kHDepth chunks deep, so that several chunks' loads are in
// flight without holding registers; the buffer takes one operand stage.
// That pays where the epilogue, not the operand feed, sets the pace: short K
// (measured, bf16: K = 2048 10 % faster, K = 2880 9 % slower, K = 7168 15 %
// slower; MXFP8, whose epilogue also quantizes dH both ways: K = 2880 14 %
// faster, K = 7168 6 % slower).
constexpr int kOpBf16 = 0, kOpMx = 1, kOpNv = 2, kOpBf16H = 3, kOpMxH = 4;
constexpr int kHAsyncMaxK = 2048, kHAsyncMaxKMx = 4096;
__host__ __device__ constexpr bool op_mx(int op) { return op == kOpMx || op == kOpMxH; }
constexpr int kHDepth = 3;
// dGLU with H recomputed in the kernel: 128 GLU features per tile; TMEM holds
// H for the tile's packed block (128 gate + 128 linear columns) at 0..255,
// dA at 256..383, and the MXFP8 scale slots at 384 (A) and 416 (B), so the
// next tile's scales never wait for an epilogue
constexpr int RC_N = 128;
constexpr uint32_t kRcDa = 256, kRcSfa = 384, kRcSfb = 416;
constexpr int H_BUF_BYTES = kHDepth * 4 * kGemmEpiThreads * 16;
constexpr size_t SMEM_BYTES_HA = 1024 + static_cast<size_t>(STAGES - 1) * STAGE_BYTES +
                                 kRing * BOX_BYTES + H_BUF_BYTES;
constexpr size_t SMEM_BYTES_MXH = 1024 + static_cast<size_t>(STAGES - 1) *
                                             (STAGE_BYTES + SF_STAGE_BYTES) +
                                  kRingMx * BOX_BYTES + H_BUF_BYTES;

struct Tile {
  int e;        // expert
  int m0;       // first output row (ragged M: routed row; ragged K: weight row)
  int n0;       // first output column
  int k_row0;   // ragged K: first routed row of the group
  int num_kb;   // K blocks (64 bf16 or 128 E4M3 per block)
};

// The 16-column share of one chunk (see the grouped GEMM's epilogue).
template <int ACT>
__device__ __forceinline__ void dglu_compute16(const uint32_t (&r)[16], const uint4 (&hg)[2],
                                               const uint4 (&hl)[2], const ActP& ap,
                                               float (&dg)[16], float (&dl)[16]) {
  float g[16], l[16];
  unpack_bf16x16(hg, g);
  unpack_bf16x16(hl, l);
#pragma unroll
  for (int i = 0; i < 16; ++i) glu_bwd<ACT>(__uint_as_float(r[i]), g[i], l[i], ap, dg[i], dl[i]);
}

// Output staging: the epilogue warps share a ring of NR boxes of 128 rows x
// 32 bf16 (64-byte rows, 64-byte swizzle as in the output tensor maps).
// Each thread writes its row's share of a box; after a named barrier one
// thread issues a single TMA bulk tensor store for the whole box and waits
// until at most NR-2 stores are still reading shared memory, so the box the
// next round reuses is free by the time the other threads pass the next
// barrier.  All epilogue threads must stage in the same sequence.
struct StoreRing {
  uint32_t base;   // shared address of the first box
  int slot;
  uint8_t* gbase;  // the same box as a generic pointer
};

// Grouped-GEMM variant: eight epilogue warps, two per TMEM lane quarter;
// the warp of `half` h writes columns 16h .. 16h+15 of its row into the box
// (two 16-byte chunks), all 256 threads meet at the barrier, and one thread
// stores the whole box.  `map` may be null: the box is then only staged.
template <int NR>
__device__ __forceinline__ void ring_store_half(StoreRing& ring, const float (&v)[16], bool live,
                                                const CUtensorMap* map, int x, int y, int z,
                                                int row, int half, bool issuer) {
  const uint32_t buf = ring.base + ring.slot * BOX_BYTES;
  const uint32_t raddr = buf + row * 64;
  const uint32_t sw = (row >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (live) {
      w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    }
    st_shared_v4(raddr + (((2 * half + q) ^ sw) << 4), w);
  }
  fence_proxy_async_smem();
  named_bar_sync(kEpiBar, kGemmEpiThreads);
  if (issuer) {
    if (map != nullptr) {
      tma_store_3d(map, buf, x, y, z);
      bulk_commit();
      bulk_wait_read<NR - 2>();
    } else {
      bulk_wait_read<0>();   // staged only: keep the slot-reuse distance without a new store
    }
  }
  ring.slot = ring.slot == NR - 1 ? 0 : ring.slot + 1;
}

// A whole output tile of zeros (a weight-gradient tile of an empty group):
// one box is zeroed once and stored `nch` times along the tile's columns in
// one bulk group, instead of staging and meeting once per box.
template <int NR>
__device__ __forceinline__ void ring_store_zero_tile(StoreRing& ring, const CUtensorMap* map,
                                                     int x0, int nch, int y, int z, int row,
                                                     int half, bool issuer) {
  const uint32_t buf = ring.base + ring.slot * BOX_BYTES;
  const uint32_t raddr = buf + row * 64;
  const uint4 zero = make_uint4(0, 0, 0, 0);
  st_shared_v4(raddr + (2 * half) * 16, zero);
  st_shared_v4(raddr + (2 * half + 1) * 16, zero);
  fence_proxy_async_smem();
  named_bar_sync(kEpiBar, kGemmEpiThreads);
  if (issuer) {
    for (int j = 0; j < nch; ++j) tma_store_3d(map, buf, x0 + 32 * j, y, z);
    bulk_commit();
    bulk_wait_read<NR - 2>();
  }
  ring.slot = ring.slot == NR - 1 ? 0 : ring.slot + 1;
}

// MXFP8 of a staged 32 x 32 block shared by the two warps of a lane quarter:
// half 0 quantizes its rows, half 1 its columns.
__device__ __forceinline__ void mx_block_half(const MxOut& mx, const uint8_t* box, int row0,
                                              long long r0, int col0, int lane, int half) {
  MxOut m = mx;
  if (half == 0) m.qt = nullptr; else m.q = nullptr;
  mx_block_from_box(m, box, row0, r0, col0, lane);
}

// amax of one warp's 16 columns of a 32-row block held one row per lane in
// v (bf16-rounded values, zero on padding rows): the plain maximum and the
// maximum of the 16-row Walsh-Hadamard rotation (H16 s / 4) of each column
// segment (half warps are the 16-row segments), folded into this lane's
// running maxima m_acc / h_acc (published once per warp by mx_amax_publish).
__device__ __forceinline__ void mx_amax_regs16(const float (&v)[16], int lane, float& m_acc,
                                               float& h_acc) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    m_acc = fmaxf(m_acc, fabsf(v[i]));
    float x = v[i];
#pragma unroll
    for (int b = 1; b < 16; b <<= 1) {
      const float p = __shfl_xor_sync(0xFFFFFFFFu, x, b);
      x = (lane & b) ? (p - x) : (x + p);
    }
    h_acc = fmaxf(h_acc, fabsf(x) * 0.25f);
  }
}

// Warp-reduce the running maxima and fold them into mx.amax (one atomic
// pair per warp per kernel).  Whole warp calls.
__device__ __forceinline__ void mx_amax_publish(const MxOut& mx, float m, float h, int lane) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    h = fmaxf(h, __shfl_xor_sync(0xFFFFFFFFu, h, o));
  }
  if (lane == 0) {
    atomic_max_nonneg(mx.amax, m);
    atomic_max_nonneg(mx.amax + 1, h);
  }
}

// The box the next ring_store stages into (generic pointer to shared memory).
__device__ __forceinline__ const uint8_t* ring_next_box(const StoreRing& ring) {
  return ring.gbase + ring.slot * BOX_BYTES;
}

// Two adjacent 32-column chunks per round, one TMA store for both, through
// a ring of three slot pairs (see ring_store_pair).  map2 views the output as
// [E][W/32][rows][32]; the second chunk of a single-chunk round lies past the
// tensor's end and is clipped.  Each thread stages the 16 columns of its half.
__device__ __forceinline__ void stage_box_half(uint32_t buf, const float (&v)[16], bool live,
                                               int row, int half) {
  const uint32_t raddr = buf + row * 64;
  const uint32_t sw = (row >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (live) {
      w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    }
    st_shared_v4(raddr + (((2 * half + q) ^ sw) << 4), w);
  }
}

template <int NPAIRS>
__device__ __forceinline__ void ring_store_pair(StoreRing& ring, const float (&v0)[16],
                                                const float (&v1)[16], bool two, bool live,
                                                const CUtensorMap* map2, int c0, int y, int z,
                                                int row, int half, bool issuer) {
  // Round r stages into pair r % NPAIRS; each of the eight epilogue warps
  // writes its 16 columns of both chunks.  With 3 pairs the issuer only
  // waits (after issuing) for the store one round older, so a store overlaps
  // the next round's staging; the pair a round writes was stored 3 rounds
  // ago and that store was waited for before the previous round's barrier.
  static_assert(NPAIRS == 3, "three slot pairs");
  const uint32_t buf = ring.base + ring.slot * BOX_BYTES;   // slot 0, 2 or 4
  stage_box_half(buf, v0, live, row, half);
  if (two) stage_box_half(buf + BOX_BYTES, v1, live, row, half);
  fence_proxy_async_smem();
  named_bar_sync(kEpiBar, kGemmEpiThreads);
  if (issuer) {
    tma_store_4d(map2, buf, 0, y, c0 / 32, z);
    bulk_commit();
    bulk_wait_read<1>();
  }
  ring.slot = ring.slot == 2 * (NPAIRS - 1) ? 0 : ring.slot + 2;
}

// The pair kernel's zero tile (an empty group): one staged pair of zero
// boxes stored along the tile's columns in one bulk group.
__device__ __forceinline__ void ring_store_pair_zero_tile(StoreRing& ring, const CUtensorMap* map2,
                                                          int n0, int nch, int y, int z, int row,
                                                          int half, bool issuer) {
  const float zero[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
  const uint32_t buf = ring.base + ring.slot * BOX_BYTES;
  stage_box_half(buf, zero, false, row, half);
  stage_box_half(buf + BOX_BYTES, zero, false, row, half);
  fence_proxy_async_smem();
  named_bar_sync(kEpiBar, kGemmEpiThreads);
  if (issuer) {
    for (int j = 0; j < nch; j += 2) tma_store_4d(map2, buf, 0, y, (n0 + 32 * j) / 32, z);
    bulk_commit();
    bulk_wait_read<1>();
  }
  ring.slot = ring.slot == 2 * (3 - 1) ? 0 : ring.slot + 2;
}

// bf16: the backward reads transposed operands MN-major from the forward's
// buffers.  MXFP8 / NVFP4: every operand is K-major (the transposed copies
// are quantized along the contraction dimension).
template <int MODE, int OP>
struct Traits {
  static constexpr bool kScaled = op_mx(OP) || OP == kOpNv;
  static constexpr bool kRaggedK = (MODE == kWgrad);
  static constexpr bool kAmn = !kScaled && (MODE == kWgrad);
  static constexpr bool kBmn = !kScaled && (MODE == kDgradDglu || MODE == kDgradFc1 ||
                                            MODE == kWgrad || MODE == kDgradAct);
  static constexpr uint32_t kIdesc = idesc_bf16(BM, BN, kAmn, kBmn);
  static constexpr int kBK = OP == kOpNv ? BK_NV : (op_mx(OP) ? BK_MX : BK);
  static constexpr int kNR = op_mx(OP) ? kRingMx : kRing;
  static constexpr bool kHAsync = MODE == kDgradDglu && (OP == kOpBf16H || OP == kOpMxH);
  static constexpr int kStages = OP == kOpNv ? STAGES_NV : (kHAsync ? STAGES - 1 : STAGES);
  static constexpr int kSfStage =
      OP == kOpNv ? SF_STAGE_BYTES_NV : (op_mx(OP) ? SF_STAGE_BYTES : 0);
};

// Accumulator factor of an NVFP4 GEMM: both operands were encoded with
// g = 2688 / amax of their tensor, so the product carries g_a g_b.
__device__ __forceinline__ float nv_encode_scale(float amax) {
  return amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;
}

template <int MODE, int KB>
__device__ __forceinline__ Tile decode_tile(int t, int n_tiles, int m_tiles, const int* s_off,
                                            const int* s_cnt, const int* s_order, int E) {
  Tile ti;
  if (MODE == kWgrad) {
    const int per_e = m_tiles * n_tiles;
    const int slot = t / per_e;
    const int rem = t - slot * per_e;
    const int mb = rem / n_tiles;
    const int nb = rem - mb * n_tiles;
    ti.e = s_order[slot];
    ti.m0 = mb * BM;
    ti.n0 = nb * BN;
    ti.k_row0 = s_off[ti.e];
    ti.num_kb = (s_cnt[ti.e] + KB - 1) / KB;
  } else {
    const int mb = t / n_tiles;
    const int nb = t - mb * n_tiles;
    const int row = mb * BM;
    // last expert whose group starts at or before `row`
    int lo = 0, hi = E;  // answer in [lo, hi)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= row) lo = mid; else hi = mid;
    }
    ti.e = lo;
    ti.m0 = row;
    ti.n0 = nb * (MODE == kDgradDgluRc ? RC_N : BN);
    ti.k_row0 = 0;
    ti.num_kb = 0;  // filled by caller from K
  }
  return ti;
}

// The fused router's permutation, in the same launch as its logits GEMM
// (a cooperative launch, every CTA resident): once all CTAs have written
// their tokens' top-k choices and the per-chunk expert histogram (grid
// barrier 1), each CTA assigns the rows of chunks blockIdx.x,
// blockIdx.x + gridDim.x, ... with the first kTokensPerChunk threads (the
// standalone scan_assign's arithmetic, its scratch in the now idle operand
// stages); once every row source is known (grid barrier 2), all warps of
// the grid gather x_perm row by row.
// Fused router epilogue for one token (this lane's accumulator row at trow):
// the top-k experts of logit + bias, ties to the lower expert, in descending
// score, and the softmax of their raw logits.  The best LIST scores are kept
// sorted in registers (static indices only): experts arrive in ascending
// order and a candidate moves ahead of an entry only with a strictly larger
// score, so equal scores keep the lower expert first; candidates not above
// the current k-th score are skipped.  LIST >= args.topk.
template <int LIST>
__device__ __forceinline__ void router_topk_row(const GemmArgs& args, uint32_t trow, long long gr,
                                                bool valid) {
  const int Ec = args.n_ext, kk = args.topk;
  float sv[LIST], lv[LIST];
  int iv[LIST];
#pragma unroll
  for (int s = 0; s < LIST; ++s) {
    sv[s] = -INFINITY;
    lv[s] = 0.0f;
    iv[s] = kMaxExperts + s;
  }
  float kth = -INFINITY;                      // score of slot kk-1
#pragma unroll 1
  for (int c0 = 0; c0 < Ec; c0 += 32) {
    uint32_t r[32];
    tmem_ld32(trow + c0, r);
    tmem_ld_wait(r);
    // the chunk fully unrolled: the accumulator registers keep static
    // indices (a runtime index would put them in local memory)
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = c0 + i;
      const float l = __uint_as_float(r[i]);
      if (e < Ec && valid && args.r_logits) args.r_logits[gr * Ec + e] = l;
      float cs = l + (args.r_bias && e < Ec ? __ldg(args.r_bias + e) : 0.0f);
      if (!(e < Ec && cs > kth)) continue;     // also drops NaN and -inf
      float cl = l;
      int ci = e;
#pragma unroll
      for (int s = 0; s < LIST; ++s) {
        if (cs > sv[s]) {
          const float ts = sv[s], tl = lv[s];
          const int ti = iv[s];
          sv[s] = cs;
          lv[s] = cl;
          iv[s] = ci;
          cs = ts;
          cl = tl;
          ci = ti;
        }
      }
#pragma unroll
      for (int s = 0; s < LIST; ++s)
        if (s == kk - 1) kth = sv[s];
    }
  }
  if (!valid) return;
  // slots [0, kk); unfilled ones (non-finite scores) keep their sentinel
  float mx_l = -INFINITY;
  bool short_list = false;
#pragma unroll
  for (int s = 0; s < LIST; ++s)
    if (s < kk) {
      if (iv[s] < Ec) mx_l = fmaxf(mx_l, lv[s]);
      else short_list = true;
    }
  if (short_list) set_status(args.status, MOE_DEV_BAD_EXPERT);
  float sum = 0.0f;
#pragma unroll
  for (int s = 0; s < LIST; ++s)
    if (s < kk && iv[s] < Ec) sum += expf(lv[s] - mx_l);
#pragma unroll
  for (int s = 0; s < LIST; ++s) {
    if (s < kk) {
      const bool got = iv[s] < Ec;
      const int e = got ? iv[s] : s;
      args.r_idx[gr * kk + s] = e;
      args.r_w[gr * kk + s] = got ? expf(lv[s] - mx_l) / sum : 0.0f;
      atomicAdd(&args.r_hist[(gr / kTokensPerChunk) * Ec + e], 1);
    }
  }
}

// top-k beyond 8: the long list in a call of its own, so that its
// registers do not weigh on the kernel's common path
__device__ __noinline__ void router_topk_row_long(const GemmArgs& args, uint32_t trow,
                                                  long long gr, bool valid) {
  router_topk_row<kMaxTopK>(args, trow, gr, valid);
}

__device__ __noinline__ void router_permute_tail(const GemmArgs& args, uint8_t* smem) {
  __shared__ int s_gfail;
  if (threadIdx.x == 0) s_gfail = 0;
  if (!grid_sync(args.r_grid, gridDim.x, args.status, &s_gfail)) return;
  AssignSmem& sm = *reinterpret_cast<AssignSmem*>(smem);
  const int E = args.n_ext;
  for (int c = blockIdx.x; c < args.r_nchunks; c += gridDim.x) {
    if (threadIdx.x < kTokensPerChunk)
      scan_assign_chunk(c, static_cast<int>(threadIdx.x), args.r_idx, args.r_tokens, E,
                        args.topk, args.r_hist, args.r_nchunks, args.r_capacity, args.r_counts,
                        args.r_offsets, args.r_padded, args.r_tiles, args.r_row_src,
                        args.r_row_of, args.status, sm,
                        [] { named_bar_sync(2, kTokensPerChunk); });
    __syncthreads();                            // the scratch is reused by the next chunk
  }
  if (!grid_sync(args.r_grid, 2 * gridDim.x, args.status, &s_gfail)) return;
  const int rows = min(__ldcg(args.r_padded + E), args.r_capacity);
  const int warps = GEMM_THREADS / 32;
  const int lane = threadIdx.x & 31;
  for (int j = blockIdx.x * warps + (threadIdx.x >> 5); j < rows; j += gridDim.x * warps)
    gather_row_warp(static_cast<const uint4*>(args.r_x), args.r_row_src, j, args.r_vec_per_row,
                    args.r_tokens, static_cast<uint4*>(args.r_x_perm), lane);
}

template <int MODE, int ACT, int OP>
__global__ void __launch_bounds__(GEMM_THREADS, 1) k_grouped_gemm(const __grid_constant__ GemmArgs args) {
  using Tr = Traits<MODE, OP>;
  constexpr bool MX = op_mx(OP), NV = OP == kOpNv;
  constexpr int NST = Tr::kStages;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[NST];
  __shared__ __align__(8) uint64_t empty_bar[NST];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t tearly_bar[2];   // MX: first chunk of an accumulator read
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_order[kMaxExperts];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;

  // ---- group tables (sizes live in device memory; no host round trip)
  __shared__ int s_dense_cnt;
  const int* __restrict__ s_cnt = args.counts;   // group sizes read through L1
  if (args.dense_rows > 0) {                     // one dense group (router GEMM)
    if (threadIdx.x == 0) {
      s_off[0] = 0;
      s_off[1] = (args.dense_rows + BM - 1) / BM * BM;
      s_dense_cnt = args.dense_rows;
    }
    s_cnt = &s_dense_cnt;
  } else {
    for (int i = threadIdx.x; i <= E; i += GEMM_THREADS) s_off[i] = args.padded_offsets[i];
  }
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 8);
      mbar_init(&tearly_bar[a], 8);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();

  constexpr bool RC = MODE == kDgradDgluRc;
  constexpr int TN = RC ? RC_N : BN;
  const int n_tiles = (args.n_ext + TN - 1) / TN;
  const int m_tiles = Tr::kRaggedK ? (args.m_ext + BM - 1) / BM : 0;
  // validate the offsets and sizes read from device memory (one group per
  // thread: a serial loop would chain one memory round trip per group);
  // skip all work if any is bad
  bool ok_e = true;
  for (int e = threadIdx.x; e < E; e += GEMM_THREADS) {
    const int span = s_off[e + 1] - s_off[e];
    const int c = s_cnt[e];
    ok_e = ok_e && span >= 0 && (span % BM) == 0 && c >= 0 && c <= span;
  }
  if (Tr::kRaggedK) {
    // largest group first; equal sizes keep expert order
    for (int e = threadIdx.x; e < E; e += GEMM_THREADS) {
      int rank = 0;
      for (int j = 0; j < E; ++j)
        rank += (s_cnt[j] > s_cnt[e]) || (s_cnt[j] == s_cnt[e] && j < e);
      s_order[rank] = e;
    }
  }
  const bool ok = __syncthreads_and(ok_e) != 0 && s_off[0] == 0 && s_off[E] <= args.capacity;
  if (!ok && threadIdx.x == 0) set_status(args.status, MOE_DEV_BAD_OFFSETS);
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = !ok ? 0 : (Tr::kRaggedK ? E * m_tiles * n_tiles : (s_off[E] / BM) * n_tiles);
  const int kb_half = (args.K + Tr::kBK - 1) / Tr::kBK;   // K blocks of one GEMM
  const int kb_fixed = Tr::kRaggedK ? 0 : (RC ? 2 * kb_half : kb_half);
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&args.tma_a);
      tma_prefetch_desc(&args.tma_b);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        Tile ti = decode_tile<MODE, Tr::kBK>(t, n_tiles, m_tiles, s_off, s_cnt, s_order, E);
        const int num_kb = Tr::kRaggedK ? ti.num_kb : kb_fixed;
        // boxes that hold at least one in-range column (skip fully-outside boxes)
        const int b_boxes = Tr::kBmn ? (args.b_atoms4d ? 4 : min(4, (args.b_ext - ti.n0 + 63) / 64)) : 1;
        const int a_boxes = Tr::kAmn ? min(2, (args.m_ext - ti.m0 + 63) / 64) : 1;
        // the router's B tile is only as tall as the expert count (rounded to 16)
        const uint32_t b_rows = MODE == kRouter ? (args.n_ext + 15) / 16 * 16 : BN;
        const uint32_t tx = (Tr::kAmn ? a_boxes * MN_BOX_BYTES : A_BYTES) +
                            (Tr::kBmn ? b_boxes * MN_BOX_BYTES : b_rows * BK * 2);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, args.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          uint64_t* fb = &full_bar[stage];
          if constexpr (RC) {
            // K blocks 0 .. kb_half-1: X and the tile's packed W1p block (256
            // rows) for H; then dY and W2's 128 rows of the tile's features
            // for dA.  K = d in both.
            const bool p1 = kb < kb_half;
            const int kq = p1 ? kb : kb - kb_half;
            if constexpr (MX) {
              const int kx = kq * BK_MX;
              const long long kt = kx / BK_MX;
              uint8_t* ssf = smem + NST * STAGE_BYTES + stage * SF_STAGE_BYTES;
              if (p1) {
                mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + SF_STAGE_BYTES);
                tma_load_3d(sa, &args.tma_a, fb, kx, ti.m0, 0);
                tma_load_3d(sb, &args.tma_b, fb, kx, 2 * ti.n0, ti.e);
                bulk_load(ssf, args.sfa + (kt * args.sfa_atoms + (ti.m0 >> 7)) * 512, 512, fb);
                bulk_load(ssf + 512,
                          args.sfb + ti.e * args.sfb_expert_bytes +
                              (kt * args.sfb_atoms + ((2 * ti.n0) >> 7)) * 512,
                          1024, fb);
              } else {
                mbar_arrive_expect_tx(fb, A_BYTES + RC_N * BK_MX + 1024);
                tma_load_3d(sa, &args.tma_a2, fb, kx, ti.m0, 0);
                tma_load_3d(sb, &args.tma_b2, fb, kx, ti.n0, ti.e);
                bulk_load(ssf, args.sfa2 + (kt * args.sfa2_atoms + (ti.m0 >> 7)) * 512, 512, fb);
                bulk_load(ssf + 512,
                          args.sfb2 + ti.e * args.sfb2_expert_bytes +
                              (kt * args.sfb2_atoms + (ti.n0 >> 7)) * 512,
                          512, fb);
              }
            } else {
              const int kk = kq * BK;
              if (p1) {
                mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
                tma_load_3d(sa, &args.tma_a, fb, kk, ti.m0, 0);
                tma_load_3d(sb, &args.tma_b, fb, kk, 2 * ti.n0, ti.e);
              } else {
                // W2 read MN-major: two 64-feature atoms (4-D box), or one
                // box per atom that holds an in-range feature
                const int nb2 = args.b2_atoms4d ? 2 : min(2, (args.b_ext - ti.n0 + 63) / 64);
                mbar_arrive_expect_tx(fb, A_BYTES + nb2 * MN_BOX_BYTES);
                tma_load_3d(sa, &args.tma_a2, fb, kk, ti.m0, 0);
                if (args.b2_atoms4d)
                  tma_load_4d(sb, &args.tma_b2, fb, 0, kk, ti.n0 / 64, ti.e);
                else
                  for (int i = 0; i < nb2; ++i)
                    tma_load_3d(sb + i * MN_BOX_BYTES, &args.tma_b2, fb, ti.n0 + 64 * i, kk,
                                ti.e);
              }
            }
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if constexpr (NV) {
            // packed E2M1 tiles (K-major, 256 K per 128-byte row; the TMA
            // coordinate is in bytes) and the scale atoms of each K = 64
            // step that lies inside K (the last stage of a group or of an
            // odd K may hold fewer than four)
            const int kx = (Tr::kRaggedK ? ti.k_row0 : 0) + kb * BK_NV;
            const int krem = (Tr::kRaggedK ? s_cnt[ti.e] : args.K) - kb * BK_NV;
            const int nk = min(4, (krem + 63) / 64);
            mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + nk * 1536);
            uint8_t* ssf = smem + NST * STAGE_BYTES + stage * SF_STAGE_BYTES_NV;
            tma_load_3d(sa, &args.tma_a, fb, kx / 2, ti.m0, 0);
            tma_load_3d(sb, &args.tma_b, fb, kx / 2, ti.n0, Tr::kRaggedK ? 0 : ti.e);
            const uint8_t* sfb_e = args.sfb + (Tr::kRaggedK ? 0 : ti.e * args.sfb_expert_bytes);
            for (int k = 0; k < nk; ++k) {
              const long long kt = kx / 64 + k;        // atom column of this K = 64 step
              bulk_load(ssf + k * 512, args.sfa + (kt * args.sfa_atoms + (ti.m0 >> 7)) * 512,
                        512, fb);
              bulk_load(ssf + 2048 + k * 1024,
                        sfb_e + (kt * args.sfb_atoms + (ti.n0 >> 7)) * 512, 1024, fb);
            }
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if constexpr (MX) {
            // E4M3 tiles (K-major, 128 K per row) and their scale atoms
            mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES + SF_STAGE_BYTES);
            const int kx = (Tr::kRaggedK ? ti.k_row0 : 0) + kb * BK_MX;
            const long long kt = kx / BK_MX;
            uint8_t* ssf = smem + NST * STAGE_BYTES + stage * SF_STAGE_BYTES;
            tma_load_3d(sa, &args.tma_a, fb, kx, ti.m0, 0);
            tma_load_3d(sb, &args.tma_b, fb, kx, ti.n0, Tr::kRaggedK ? 0 : ti.e);
            bulk_load(ssf, args.sfa + (kt * args.sfa_atoms + (ti.m0 >> 7)) * 512, 512, fb);
            bulk_load(ssf + 512,
                      args.sfb + (Tr::kRaggedK ? 0 : ti.e * args.sfb_expert_bytes) +
                          (kt * args.sfb_atoms + (ti.n0 >> 7)) * 512,
                      1024, fb);
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          mbar_arrive_expect_tx(fb, tx);
          const int kk = kb * BK;
          // ---- A operand
          if (Tr::kAmn) {
            for (int i = 0; i < a_boxes; ++i)
              tma_load_3d(sa + i * MN_BOX_BYTES, &args.tma_a, fb, ti.m0 + 64 * i, ti.k_row0 + kk, 0);
          } else {
            tma_load_3d(sa, &args.tma_a, fb, kk, ti.m0, 0);
          }
          // ---- B operand
          if (MODE == kFc1Glu || MODE == kFc2 || MODE == kFc1Act || MODE == kRouter) {
            tma_load_3d(sb, &args.tma_b, fb, kk, ti.n0, ti.e);
          } else if (MODE == kDgradDglu || MODE == kDgradFc1 || MODE == kDgradAct) {
            if (args.b_atoms4d)
              tma_load_4d(sb, &args.tma_b, fb, 0, kk, ti.n0 / 64, ti.e);
            else
              for (int i = 0; i < b_boxes; ++i)
                tma_load_3d(sb + i * MN_BOX_BYTES, &args.tma_b, fb, ti.n0 + 64 * i, kk, ti.e);
          } else {
            for (int i = 0; i < b_boxes; ++i)
              tma_load_3d(sb + i * MN_BOX_BYTES, &args.tma_b, fb, ti.n0 + 64 * i, ti.k_row0 + kk, 0);
          }
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        Tile ti = decode_tile<MODE, Tr::kBK>(t, n_tiles, m_tiles, s_off, s_cnt, s_order, E);
        const int num_kb = Tr::kRaggedK ? ti.num_kb : kb_fixed;
        // the recompute mode holds one tile in TMEM (H, dA, scales): one
        // accumulator set, its phase flips every tile
        const int acc = RC ? 0 : (it & 1);
        const uint32_t acc_par = RC ? (it & 1) : ((it >> 1) & 1);
        if (!mbar_wait(&tempty_bar[acc], acc_par ^ 1u, args.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        // MMA width: 256, or for the router the expert count rounded to 16
        const uint32_t idesc =
            MODE == kRouter ? idesc_bf16(BM, (args.n_ext + 15) / 16 * 16, false, false) : Tr::kIdesc;
        // MX: this tile's scales go to the first columns of the other
        // accumulator, which the previous tile's epilogue must have read.
        const uint32_t sf_tmem = tmem_base + (acc ^ 1) * BN;
        if constexpr ((MX || NV) && !RC) {
          if (it > 0) {
            if (!mbar_wait(&tearly_bar[acc ^ 1], ((it - 1) >> 1) & 1, args.status, abort_flag))
              break;
            tc_fence_after();
          }
        }
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, args.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t b_base = a_base + A_BYTES;
          if constexpr (RC) {
            // H (N = 256, K-major B) into columns 0..255, then dA (N = 128)
            // into kRcDa..; each GEMM starts its own accumulation
            const bool p1 = kb < kb_half;
            const bool first = (p1 ? kb : kb - kb_half) == 0;
            const uint32_t dst = tmem_base + (p1 ? 0u : kRcDa);
            if constexpr (MX) {
              const uint32_t sf = smem_u32(smem + NST * STAGE_BYTES + stage * SF_STAGE_BYTES);
              tmem_cp_32x128_x4(tmem_base + kRcSfa, sdesc_noswz(sf, 128, 128));
              tmem_cp_32x128_x4(tmem_base + kRcSfb, sdesc_noswz(sf + 512, 128, 128));
              if (p1)
                tmem_cp_32x128_x4(tmem_base + kRcSfb + 4, sdesc_noswz(sf + 1024, 128, 128));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_mx(dst, sdesc_sw128(a_base + k * 32, 16, 1024),
                        sdesc_sw128(b_base + k * 32, 16, 1024),
                        idesc_mx(BM, p1 ? BN : RC_N, k, k), tmem_base + kRcSfa,
                        tmem_base + kRcSfb, (!first || k > 0) ? 1u : 0u);
            } else {
#pragma unroll
              for (int k = 0; k < BK / 16; ++k) {
                const uint64_t ad = sdesc_sw128(a_base + k * 32, 16, 1024);
                const uint64_t bd = p1 ? sdesc_sw128(b_base + k * 32, 16, 1024)
                                       : sdesc_sw128(b_base + k * 2048, MN_BOX_BYTES, 1024);
                umma_bf16(dst, ad, bd,
                          p1 ? idesc_bf16(BM, BN, false, false)
                             : idesc_bf16(BM, RC_N, false, true),
                          (!first || k > 0) ? 1u : 0u);
              }
            }
            umma_commit(&empty_bar[stage]);
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if constexpr (NV) {
            // per K = 64 step (32 bytes along the swizzled rows): its scale
            // atoms to TMEM -- one 32-bit cell per row holding the four
            // 16-element block scales -- then its MMA.  tcgen05.cp and
            // tcgen05.mma from this thread run in issue order.
            const int krem = (Tr::kRaggedK ? s_cnt[ti.e] : args.K) - kb * BK_NV;
            const int nk = min(4, (krem + 63) / 64);
            const uint32_t sf = smem_u32(smem + NST * STAGE_BYTES + stage * SF_STAGE_BYTES_NV);
            for (int k = 0; k < nk; ++k) {
              tmem_cp_32x128_x4(sf_tmem + kSfaCol, sdesc_noswz(sf + k * 512, 128, 128));
              tmem_cp_32x128_x4(sf_tmem + kSfbCol, sdesc_noswz(sf + 2048 + k * 1024, 128, 128));
              tmem_cp_32x128_x4(sf_tmem + kSfbCol + 4,
                                sdesc_noswz(sf + 2048 + k * 1024 + 512, 128, 128));
              umma_nvf4(d_tmem, sdesc_sw128(a_base + k * 32, 16, 1024),
                        sdesc_sw128(b_base + k * 32, 16, 1024), idesc_nvf4(BM, BN),
                        sf_tmem + kSfaCol, sf_tmem + kSfbCol, (kb > 0 || k > 0) ? 1u : 0u);
            }
            umma_commit(&empty_bar[stage]);
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if constexpr (MX) {
            // scales smem -> TMEM, then 4 MMAs of K = 32 (32 bytes apart in
            // the swizzled rows); MMA k takes byte k of each scale column.
            // tcgen05.cp and tcgen05.mma from this thread run in issue order.
            const uint32_t sf = smem_u32(smem + NST * STAGE_BYTES + stage * SF_STAGE_BYTES);
            tmem_cp_32x128_x4(sf_tmem + kSfaCol, sdesc_noswz(sf, 128, 128));
            tmem_cp_32x128_x4(sf_tmem + kSfbCol, sdesc_noswz(sf + 512, 128, 128));
            tmem_cp_32x128_x4(sf_tmem + kSfbCol + 4, sdesc_noswz(sf + 1024, 128, 128));
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_mx(d_tmem, sdesc_sw128(a_base + k * 32, 16, 1024),
                      sdesc_sw128(b_base + k * 32, 16, 1024), idesc_mx(BM, BN, k, k),
                      sf_tmem + kSfaCol, sf_tmem + kSfbCol, (kb > 0 || k > 0) ? 1u : 0u);
            umma_commit(&empty_bar[stage]);
            if (++stage == NST) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // K-major: +32 B per K=16 step inside the 128-B swizzle row.
            // MN-major: +16 K-rows of 128 B = 2048 B; atoms 8 KB apart along MN.
            const uint64_t ad = Tr::kAmn ? sdesc_sw128(a_base + k * 2048, MN_BOX_BYTES, 1024)
                                         : sdesc_sw128(a_base + k * 32, 16, 1024);
            const uint64_t bd = Tr::kBmn ? sdesc_sw128(b_base + k * 2048, MN_BOX_BYTES, 1024)
                                         : sdesc_sw128(b_base + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);
      }
    }
  } else {
    // ============================ epilogue ================================
    // Eight warps, two per TMEM lane quarter: the warp of `half` h owns
    // columns 16h .. 16h+15 of every 32-column chunk of its 32 rows.  All
    // eight stage each chunk into one shared box and meet at its barrier.
    const int quarter = warp & 3;             // TMEM lanes this warp may read
    const int half = (warp - 2) >> 2;         // warps 2-5: 0, warps 6-9: 1
    const int hc = 16 * half;                 // first column of this warp's share
    const int row_local = quarter * 32 + lane;
    const ActP ap{args.act, args.alpha, args.limit, args.lin_off, args.out_scale};
    uint8_t* const ring_mem = smem + NST * STAGE_BYTES + NST * Tr::kSfStage;
    const uint32_t h_buf = smem_u32(ring_mem + Tr::kNR * BOX_BYTES);   // async H (bf16 dGLU)
    const uint8_t* const h_gen = ring_mem + Tr::kNR * BOX_BYTES;
    StoreRing ring{smem_u32(ring_mem), 0, ring_mem};
    const bool issuer = threadIdx.x == 64;   // first epilogue thread issues the stores
    const MxOut mx{args.mx_q, args.mx_s, args.mx_qt, args.mx_st, args.mx_amax, args.mx_width,
                   args.capacity, args.mx_mma_layout};
    // MX: tell the MMA warp that the accumulator's first 64 columns have
    // been read (the next tile stages its scales there).  Once per tile.
    auto early_release = [&](int acc_id) {
      if constexpr (MX || NV) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tearly_bar[acc_id]);
      }
    };
    const bool want_mx = mx.q != nullptr || mx.qt != nullptr || mx.amax != nullptr;
    // dGLU: the bf16 dH store is optional (the MXFP8 path may need only the
    // quantized copies, which are made from the staged boxes)
    const CUtensorMap* const dh_map = args.out0 != nullptr ? &args.tma_out0 : nullptr;
    // NVFP4: undo the two operands' encode scales on the accumulator
    float nv_alpha = 1.0f;
    if constexpr (NV)
      nv_alpha = __fdiv_rn(1.0f, __fmul_rn(nv_encode_scale(__ldg(args.nv_amax_a)),
                                           nv_encode_scale(__ldg(args.nv_amax_b))));
    float am_m = 0.0f, am_h = 0.0f;           // running amax (plain, Hadamard) of this lane
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      Tile ti = decode_tile<MODE, Tr::kBK>(t, n_tiles, m_tiles, s_off, s_cnt, s_order, E);
      const int acc = RC ? 0 : (it & 1);
      const uint32_t acc_par = RC ? (it & 1) : ((it >> 1) & 1);
      const long long gr = ti.m0 + row_local;
      const bool valid = !Tr::kRaggedK && (gr - s_off[ti.e]) < s_cnt[ti.e];
      const int y0 = ti.m0;                     // first output row of the tile's boxes

      // dGLU: the saved FC1 output H does not depend on the accumulator, so
      // the first chunk's share is fetched before waiting for the MMAs.
      uint4 hg[2][2], hl[2][2];
      const __nv_bfloat16* Hrow = nullptr;
      // async H: chunk jn's share into buffer slot jn % kHDepth (an empty
      // group past the tile's chunks keeps the group count uniform)
      const int nch_h = MODE == kDgradDglu ? min(BN / 32, (args.f_pad - ti.n0) / 32) : 0;
      auto h_issue = [&](int jn) {
        if constexpr (Tr::kHAsync) {
          const int f = ti.n0 + 32 * jn;
          if (jn < nch_h && valid && f < args.f_real) {
            const __nv_bfloat16* src =
                Hrow + (f / kGluHalf) * 2 * kGluHalf + (f % kGluHalf) + hc;
            const uint32_t dst =
                h_buf + ((jn % kHDepth) * 4 * kGemmEpiThreads + (threadIdx.x - 64)) * 16;
            cp_async16(dst, src);
            cp_async16(dst + kGemmEpiThreads * 16, src + 8);
            cp_async16(dst + 2 * kGemmEpiThreads * 16, src + kGluHalf);
            cp_async16(dst + 3 * kGemmEpiThreads * 16, src + kGluHalf + 8);
          }
          cp_async_commit();
        }
      };
      if (MODE == kDgradDglu && Tr::kHAsync) {
        Hrow = static_cast<const __nv_bfloat16*>(args.aux) + gr * args.ld_aux;
        for (int jn = 0; jn < kHDepth - 1; ++jn) h_issue(jn);
      } else if (MODE == kDgradDglu) {
        Hrow = static_cast<const __nv_bfloat16*>(args.aux) + gr * args.ld_aux;
        if (valid && ti.n0 < args.f_real) {
          const long long cg = static_cast<long long>(ti.n0 / kGluHalf) * 2 * kGluHalf +
                               (ti.n0 % kGluHalf) + hc;
          load_raw32(Hrow + cg, hg[0]);
          load_raw32(Hrow + cg + kGluHalf, hl[0]);
        }
      }

      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull_bar[acc], acc_par, args.status, abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      // leave together: the store barriers below need all epilogue warps
      if (named_bar_any(kEpiBar, kGemmEpiThreads, !ok)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN + hc;

      if (MODE == kRouter) {
        // one token per lane (rows of this quarter): top-k of logit + bias
        // over the E accumulator columns, ties to the lower expert, read 32
        // columns at a time; softmax of the selected raw logits
        if (half == 0) {
          const uint32_t trow = tbase - hc;
          if (args.topk <= 8)
            router_topk_row<8>(args, trow, gr, valid);
          else
            router_topk_row_long(args, trow, gr, valid);
        }
      } else if (MODE == kFc1Glu) {
        const __nv_bfloat16* b1 =
            args.bias ? static_cast<const __nv_bfloat16*>(args.bias) + ti.e * args.bias_ld + ti.n0 + hc
                      : nullptr;
        uint32_t rg[16], rl[16];
        tmem_ld16(tbase, rg);
        tmem_ld16(tbase + kGluHalf, rl);
#pragma unroll 1
        for (int j = 0; j < kGluHalf / 32; ++j) {
          tmem_ld_wait16(rg);
          reg_fence16(rl);
          float g[16], l[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            g[i] = __uint_as_float(rg[i]);
            l[i] = __uint_as_float(rl[i]);
            if constexpr (NV) {
              g[i] *= nv_alpha;
              l[i] *= nv_alpha;
            }
          }
          if (j + 1 < kGluHalf / 32) {        // next chunk's accumulator in flight
            tmem_ld16(tbase + 32 * (j + 1), rg);
            tmem_ld16(tbase + kGluHalf + 32 * (j + 1), rl);
          }
          if (j == 0) {                       // columns 0-63 read: the next tile may stage
            tmem_ld_wait16(rg);               // its scales there before this chunk's work
            reg_fence16(rl);
            early_release(acc);
          }
          if (b1) {
            float bg[16], bl[16];
            load_bf16x16(b1 + 32 * j, bg);
            load_bf16x16(b1 + kGluHalf + 32 * j, bl);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              g[i] += bg[i];
              l[i] += bl[i];
            }
          }
          if (args.out0 != nullptr) {           // H kept for the backward (else recomputed)
            ring_store_half<Tr::kNR>(ring, g, valid, &args.tma_out0, ti.n0 + 32 * j, y0, 0,
                                     row_local, half, issuer);
            ring_store_half<Tr::kNR>(ring, l, valid, &args.tma_out0, ti.n0 + kGluHalf + 32 * j,
                                     y0, 0, row_local, half, issuer);
          }
          const int f0 = ti.n0 / 2 + 32 * j;
          if (f0 < args.f_real) {
            float a[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) a[i] = glu_fwd<ACT>(g[i], l[i], ap);
            const uint8_t* box = ring_next_box(ring);
            if (args.out1 != nullptr || want_mx)
              ring_store_half<Tr::kNR>(ring, a, valid, args.out1 ? &args.tma_out1 : nullptr, f0,
                                       y0, 0, row_local, half, issuer);
            if (want_mx) {                      // MXFP8 / amax of the staged bf16 A
              mx_block_half(mx, box, quarter * 32, y0 + quarter * 32, f0, lane, half);
              if (mx.amax) {
#pragma unroll
                for (int i = 0; i < 16; ++i) a[i] = valid ? bf16_round(a[i]) : 0.0f;
                mx_amax_regs16(a, lane, am_m, am_h);
              }
            }
          }
        }
      } else if (MODE == kDgradDglu && Tr::kHAsync) {
        // tile columns are GLU features n0 .. n0+255; dH in packed layout;
        // H arrives kHDepth - 1 chunks ahead through the async buffer
        uint32_t r[16];
        tmem_ld16(tbase, r);
#pragma unroll 1
        for (int j = 0; j < nch_h; ++j) {
          h_issue(j + kHDepth - 1);
          cp_async_wait<kHDepth - 1>();             // this thread's chunk j landed
          const uint8_t* hs =
              h_gen + ((j % kHDepth) * 4 * kGemmEpiThreads + (threadIdx.x - 64)) * 16;
          const uint4 hgv[2] = {*reinterpret_cast<const uint4*>(hs),
                                *reinterpret_cast<const uint4*>(hs + kGemmEpiThreads * 16)};
          const uint4 hlv[2] = {*reinterpret_cast<const uint4*>(hs + 2 * kGemmEpiThreads * 16),
                                *reinterpret_cast<const uint4*>(hs + 3 * kGemmEpiThreads * 16)};
          uint32_t ra[16];
          tmem_ld_wait16(r);
#pragma unroll
          for (int i = 0; i < 16; ++i) ra[i] = r[i];
          if (j + 1 < nch_h) tmem_ld16(tbase + 32 * (j + 1), r);
          if (j == 0) {                       // columns 0-63 read (chunk 1 waited for early)
            tmem_ld_wait16(r);
            early_release(acc);
          }
          const int f0 = ti.n0 + 32 * j;
          const int c0 = (f0 / kGluHalf) * 2 * kGluHalf + (f0 % kGluHalf);
          const bool live = valid && f0 < args.f_real;
          float dg[16], dl[16];
          if (live) dglu_compute16<ACT>(ra, hgv, hlv, ap, dg, dl);
          const uint8_t* box_g = ring_next_box(ring);
          ring_store_half<Tr::kNR>(ring, dg, live, dh_map, c0, y0, 0, row_local, half,
                                   issuer);
          if (want_mx) mx_block_half(mx, box_g, quarter * 32, y0 + quarter * 32, c0, lane, half);
          const uint8_t* box_l = ring_next_box(ring);
          ring_store_half<Tr::kNR>(ring, dl, live, dh_map, c0 + kGluHalf, y0, 0,
                                   row_local, half, issuer);
          if (want_mx)
            mx_block_half(mx, box_l, quarter * 32, y0 + quarter * 32, c0 + kGluHalf, lane, half);
          if (want_mx && mx.amax) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              dg[i] = live ? bf16_round(dg[i]) : 0.0f;
              dl[i] = live ? bf16_round(dl[i]) : 0.0f;
            }
            mx_amax_regs16(dg, lane, am_m, am_h);
            mx_amax_regs16(dl, lane, am_m, am_h);
          }
        }
      } else if (MODE == kDgradDglu) {
        // tile columns are GLU features n0 .. n0+255; dH in packed layout.
        // Chunks go in pairs so the two H prefetch buffers stay static.
        const int nch = min(BN / 32, (args.f_pad - ti.n0) / 32);   // 4 or 8
        uint32_t r[16];
        tmem_ld16(tbase, r);
#pragma unroll 1
        for (int j = 0; j < nch; j += 2) {
          const int f0 = ti.n0 + 32 * j, f1 = f0 + 32, f2 = f0 + 64;
          const int c0 = (f0 / kGluHalf) * 2 * kGluHalf + (f0 % kGluHalf);
          const int c1 = (f1 / kGluHalf) * 2 * kGluHalf + (f1 % kGluHalf);
          const int c2 = (f2 / kGluHalf) * 2 * kGluHalf + (f2 % kGluHalf);
          float dg[16], dl[16];
          uint32_t ra[16];
          // chunk j (buffer 0); prefetch chunk j+1 into buffer 1
          if (valid && f1 < args.f_real) {
            load_raw32(Hrow + c1 + hc, hg[1]);
            load_raw32(Hrow + c1 + hc + kGluHalf, hl[1]);
          }
          tmem_ld_wait16(r);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            ra[i] = NV ? __float_as_uint(__uint_as_float(r[i]) * nv_alpha) : r[i];
          tmem_ld16(tbase + 32 * (j + 1), r);
          if (j == 0) {                       // columns 0-63 read (chunk 1 waited for early)
            tmem_ld_wait16(r);
            early_release(acc);
          }
          const bool live0 = valid && f0 < args.f_real;
          if (live0) dglu_compute16<ACT>(ra, hg[0], hl[0], ap, dg, dl);
          {
            const uint8_t* box_g = ring_next_box(ring);
            ring_store_half<Tr::kNR>(ring, dg, live0, dh_map, c0, y0, 0, row_local, half,
                                     issuer);
            if (want_mx) mx_block_half(mx, box_g, quarter * 32, y0 + quarter * 32, c0, lane, half);
            const uint8_t* box_l = ring_next_box(ring);
            ring_store_half<Tr::kNR>(ring, dl, live0, dh_map, c0 + kGluHalf, y0, 0,
                                     row_local, half, issuer);
            if (want_mx)
              mx_block_half(mx, box_l, quarter * 32, y0 + quarter * 32, c0 + kGluHalf, lane, half);
          }
          if (want_mx && mx.amax) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              dg[i] = live0 ? bf16_round(dg[i]) : 0.0f;
              dl[i] = live0 ? bf16_round(dl[i]) : 0.0f;
            }
            mx_amax_regs16(dg, lane, am_m, am_h);
            mx_amax_regs16(dl, lane, am_m, am_h);
          }
          // chunk j+1 (buffer 1); prefetch chunk j+2 into buffer 0
          if (j + 2 < nch && valid && f2 < args.f_real) {
            load_raw32(Hrow + c2 + hc, hg[0]);
            load_raw32(Hrow + c2 + hc + kGluHalf, hl[0]);
          }
          tmem_ld_wait16(r);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            ra[i] = NV ? __float_as_uint(__uint_as_float(r[i]) * nv_alpha) : r[i];
          if (j + 2 < nch) tmem_ld16(tbase + 32 * (j + 2), r);
          const bool live1 = valid && f1 < args.f_real;
          if (live1) dglu_compute16<ACT>(ra, hg[1], hl[1], ap, dg, dl);
          {
            const uint8_t* box_g = ring_next_box(ring);
            ring_store_half<Tr::kNR>(ring, dg, live1, dh_map, c1, y0, 0, row_local, half,
                                     issuer);
            if (want_mx) mx_block_half(mx, box_g, quarter * 32, y0 + quarter * 32, c1, lane, half);
            const uint8_t* box_l = ring_next_box(ring);
            ring_store_half<Tr::kNR>(ring, dl, live1, dh_map, c1 + kGluHalf, y0, 0,
                                     row_local, half, issuer);
            if (want_mx)
              mx_block_half(mx, box_l, quarter * 32, y0 + quarter * 32, c1 + kGluHalf, lane, half);
          }
          if (want_mx && mx.amax) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              dg[i] = live1 ? bf16_round(dg[i]) : 0.0f;
              dl[i] = live1 ? bf16_round(dl[i]) : 0.0f;
            }
            mx_amax_regs16(dg, lane, am_m, am_h);
            mx_amax_regs16(dl, lane, am_m, am_h);
          }
        }
      } else if (MODE == kDgradDgluRc) {
        // tile columns are GLU features n0 .. n0+127: dA from TMEM columns
        // kRcDa.., the recomputed gate and linear halves of H from columns
        // 0.. and 128.. (bias added, then rounded to bf16 as the stored H
        // is); dH in packed layout (the tile's block starts at column 2*n0)
        const __nv_bfloat16* b1 =
            args.bias ? static_cast<const __nv_bfloat16*>(args.bias) + ti.e * args.bias_ld +
                            2 * ti.n0 + hc
                      : nullptr;
        uint32_t rda[16], rg[16], rl[16];
        tmem_ld16(tbase + kRcDa, rda);
        tmem_ld16(tbase, rg);
        tmem_ld16(tbase + kGluHalf, rl);
#pragma unroll 1
        for (int j = 0; j < RC_N / 32; ++j) {
          tmem_ld_wait16(rda);
          reg_fence16(rg);
          reg_fence16(rl);
          float da[16], g[16], l[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            da[i] = __uint_as_float(rda[i]);
            g[i] = __uint_as_float(rg[i]);
            l[i] = __uint_as_float(rl[i]);
          }
          if (j + 1 < RC_N / 32) {              // next chunk in flight
            tmem_ld16(tbase + kRcDa + 32 * (j + 1), rda);
            tmem_ld16(tbase + 32 * (j + 1), rg);
            tmem_ld16(tbase + kGluHalf + 32 * (j + 1), rl);
          }
          if (b1) {
            float bg[16], bl[16];
            load_bf16x16(b1 + 32 * j, bg);
            load_bf16x16(b1 + kGluHalf + 32 * j, bl);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              g[i] += bg[i];
              l[i] += bl[i];
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            g[i] = bf16_round(g[i]);
            l[i] = bf16_round(l[i]);
          }
          const int f0 = ti.n0 + 32 * j;
          const int c0 = 2 * ti.n0 + 32 * j;
          const bool live = valid && f0 < args.f_real;
          float dg[16], dl[16];
          if (live) {
#pragma unroll
            for (int i = 0; i < 16; ++i) glu_bwd<ACT>(da[i], g[i], l[i], ap, dg[i], dl[i]);
          }
          const uint8_t* box_g = ring_next_box(ring);
          ring_store_half<Tr::kNR>(ring, dg, live, dh_map, c0, y0, 0, row_local, half,
                                   issuer);
          if (want_mx) mx_block_half(mx, box_g, quarter * 32, y0 + quarter * 32, c0, lane, half);
          const uint8_t* box_l = ring_next_box(ring);
          ring_store_half<Tr::kNR>(ring, dl, live, dh_map, c0 + kGluHalf, y0, 0,
                                   row_local, half, issuer);
          if (want_mx)
            mx_block_half(mx, box_l, quarter * 32, y0 + quarter * 32, c0 + kGluHalf, lane, half);
          if (want_mx && mx.amax) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              dg[i] = live ? bf16_round(dg[i]) : 0.0f;
              dl[i] = live ? bf16_round(dl[i]) : 0.0f;
            }
            mx_amax_regs16(dg, lane, am_m, am_h);
            mx_amax_regs16(dl, lane, am_m, am_h);
          }
        }
      } else {
        // kFc2 (+b2), kDgradFc1 and kWgrad: plain row-major bf16 output
        const bool has_acc = !Tr::kRaggedK || ti.num_kb > 0;
        const bool write = !Tr::kRaggedK || y0 < args.m_ext;   // CTA-uniform
        const __nv_bfloat16* bias =
            ((MODE == kFc2 || MODE == kFc1Act) && args.bias)
                ? static_cast<const __nv_bfloat16*>(args.bias) + ti.e * args.bias_ld + hc
                : nullptr;
        const int nch = min(BN / 32, (args.n_ext - ti.n0 + 31) / 32);
        // TMEM is read two 32-column chunks per wait; the next pair is in
        // flight while the current one is staged and stored.
        uint32_t ra[16], rb[16];
        if (has_acc) {
          tmem_ld16(tbase, ra);
          if (nch > 1) tmem_ld16(tbase + 32, rb);
        } else {
          early_release(acc);
          if (write && MODE == kWgrad)
            ring_store_zero_tile<Tr::kNR>(ring, &args.tma_out0, ti.n0, nch, y0, ti.e, row_local,
                                          half, issuer);
        }
#pragma unroll 1
        for (int j = 0; j < nch && (has_acc || MODE != kWgrad); j += 2) {
          const bool two = j + 1 < nch;
          const int c0 = ti.n0 + 32 * j;
          float v0[16], v1[16];
          if (has_acc) {
            tmem_ld_wait16(ra);
            reg_fence16(rb);
            if (j == 0) early_release(acc);           // columns 0-63 read (or all there are)
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              v0[i] = __uint_as_float(ra[i]);
              v1[i] = __uint_as_float(rb[i]);
              if constexpr (NV) {
                v0[i] *= nv_alpha;
                v1[i] *= nv_alpha;
              }
            }
            if (j + 2 < nch) tmem_ld16(tbase + 32 * (j + 2), ra);
            if (j + 3 < nch) tmem_ld16(tbase + 32 * (j + 3), rb);
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v0[i] = v1[i] = 0.0f;
          }
          if (bias && valid) {
            float b[16];
            load_bf16x16(bias + c0, b);
#pragma unroll
            for (int i = 0; i < 16; ++i) v0[i] += b[i];
            if (two) {
              load_bf16x16(bias + c0 + 32, b);
#pragma unroll
              for (int i = 0; i < 16; ++i) v1[i] += b[i];
            }
          }
          if constexpr (MODE == kFc1Act || MODE == kDgradAct) {
            // non-gated activation: FC1 writes H and A = act(H); the dgrad
            // turns dA into dH = act'(H) dA from the saved H
            if (MODE == kDgradAct && valid) {
              const __nv_bfloat16* Hrow =
                  static_cast<const __nv_bfloat16*>(args.aux) + gr * args.ld_aux + c0 + hc;
              float h0[16], h1[16];
              load_bf16x16(Hrow, h0);
              if (two) load_bf16x16(Hrow + 32, h1);
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                v0[i] = srelu_bwd(v0[i], h0[i], ap);
                v1[i] = two ? srelu_bwd(v1[i], h1[i], ap) : 0.0f;
              }
            }
            const uint8_t* bx0 = ring_next_box(ring);
            const uint8_t* bx1 = bx0;
            if (args.out0 != nullptr) {           // H (FC1; skipped when recomputed) / dH
              ring_store_half<Tr::kNR>(ring, v0, valid, &args.tma_out0, c0, y0, 0, row_local,
                                       half, issuer);
              bx1 = ring_next_box(ring);
              if (two)
                ring_store_half<Tr::kNR>(ring, v1, valid, &args.tma_out0, c0 + 32, y0, 0,
                                         row_local, half, issuer);
            }
            if (MODE == kFc1Act) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                v0[i] = srelu_fwd(v0[i], ap);
                v1[i] = srelu_fwd(v1[i], ap);
              }
              bx0 = ring_next_box(ring);
              bx1 = bx0;
              if (args.out1 != nullptr || want_mx) {
                ring_store_half<Tr::kNR>(ring, v0, valid, args.out1 ? &args.tma_out1 : nullptr,
                                         c0, y0, 0, row_local, half, issuer);
                bx1 = ring_next_box(ring);
                if (two)
                  ring_store_half<Tr::kNR>(ring, v1, valid, args.out1 ? &args.tma_out1 : nullptr,
                                           c0 + 32, y0, 0, row_local, half, issuer);
              }
            }
            if (want_mx) {                      // MXFP8 / amax of the staged A (FC1) or dH
              mx_block_half(mx, bx0, quarter * 32, y0 + quarter * 32, c0, lane, half);
              if (two) mx_block_half(mx, bx1, quarter * 32, y0 + quarter * 32, c0 + 32, lane, half);
              if (mx.amax) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  v0[i] = valid ? bf16_round(v0[i]) : 0.0f;
                  v1[i] = valid && two ? bf16_round(v1[i]) : 0.0f;
                }
                mx_amax_regs16(v0, lane, am_m, am_h);
                if (two) mx_amax_regs16(v1, lane, am_m, am_h);
              }
            }
            continue;
          }
          const uint8_t* box0 = ring_next_box(ring);
          const uint8_t* box1 = box0;
          if (write) {
            ring_store_half<Tr::kNR>(ring, v0, Tr::kRaggedK || valid, &args.tma_out0, c0, y0,
                                     Tr::kRaggedK ? ti.e : 0, row_local, half, issuer);
            box1 = ring_next_box(ring);
            if (two)
              ring_store_half<Tr::kNR>(ring, v1, Tr::kRaggedK || valid, &args.tma_out0, c0 + 32,
                                       y0, Tr::kRaggedK ? ti.e : 0, row_local, half, issuer);
          }
          if (MODE == kFc2 && want_mx) {        // MXFP8 / amax of the staged bf16 Y
            mx_block_half(mx, box0, quarter * 32, y0 + quarter * 32, c0, lane, half);
            if (two) mx_block_half(mx, box1, quarter * 32, y0 + quarter * 32, c0 + 32, lane, half);
            if (mx.amax) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                v0[i] = valid ? bf16_round(v0[i]) : 0.0f;
                v1[i] = valid && two ? bf16_round(v1[i]) : 0.0f;
              }
              mx_amax_regs16(v0, lane, am_m, am_h);
              if (two) mx_amax_regs16(v1, lane, am_m, am_h);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
    if (mx.amax) mx_amax_publish(mx, am_m, am_h, lane);
    if (issuer) bulk_wait_all();              // stores done before the CTA exits
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if constexpr (MODE == kRouter) {
    if (args.r_grid != nullptr) router_permute_tail(args, smem);
  }
}

// ---------------------------------------------------------------------------
// Weight gradients on CTA pairs (2-SM MMA).  dW[e] (m_ext x n_ext) = sum over
// the rows of group e of P^T Q, with P [rows, m_ext] and Q [rows, n_ext] both
// read MN-major.  A pair owns a 256 x 256 output tile: CTA r stages rows
// m0+128r.. of P and columns n0+128r.. of Q (16 KB + 16 KB per 64-row K step,
// 5 stages) and keeps output rows m0+128r.. in its TMEM.  The lead CTA issues
// the MMAs (M=256, N=256) and its commits arrive on both CTAs' barriers;
// both CTAs' TMA loads complete on the lead CTA's "full" barriers.  Per SM
// this halves the operand bytes per MMA relative to the single-CTA tile.
constexpr int PAIR_STAGES = 5;
constexpr int PAIR_HALF = 128 * BK * 2;               // 16 KB
constexpr int PAIR_STAGE_BYTES = 2 * PAIR_HALF;       // A half + B half
constexpr int kPairRing = 6;                          // three pairs of output boxes
constexpr size_t PAIR_SMEM_BYTES =
    1024 + static_cast<size_t>(PAIR_STAGES) * PAIR_STAGE_BYTES + kPairRing * BOX_BYTES;
constexpr uint32_t kPairIdesc = idesc_bf16(256, BN, true, true);

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    k_wgrad_pair(const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[PAIR_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[PAIR_STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_total;
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_cnt[kMaxExperts];
  __shared__ int s_order[kMaxExperts];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int E = args.E;

  for (int i = threadIdx.x; i <= E; i += GEMM_THREADS) s_off[i] = args.padded_offsets[i];
  for (int i = threadIdx.x; i < E; i += GEMM_THREADS) s_cnt[i] = args.counts[i];
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < PAIR_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 16);        // 8 epilogue warps x 2 CTAs
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem_base, TMEM_COLS);
    tmem_relinquish_pair();
    tc_fence_before();
  }
  __syncthreads();
  const int m_tiles = (args.m_ext + 255) / 256;
  const int n_tiles = (args.n_ext + BN - 1) / BN;
  if (threadIdx.x == 0) {
    bool ok = s_off[0] == 0 && s_off[E] <= args.capacity;
    for (int e = 0; e < E && ok; ++e) {
      const int span = s_off[e + 1] - s_off[e];
      ok = span >= 0 && (span % BM) == 0 && s_cnt[e] >= 0 && s_cnt[e] <= span;
    }
    if (!ok) set_status(args.status, MOE_DEV_BAD_OFFSETS);
    s_total = ok ? E * m_tiles * n_tiles : 0;
  }
  for (int e = threadIdx.x; e < E; e += GEMM_THREADS) {
    int r = 0;
    for (int j = 0; j < E; ++j) r += (s_cnt[j] > s_cnt[e]) || (s_cnt[j] == s_cnt[e] && j < e);
    s_order[r] = e;
  }
  __syncthreads();
  cluster_sync();                            // peer barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = s_total;
  volatile int* abort_flag = &s_abort;
  const int per_e = m_tiles * n_tiles;

  if (warp == 0) {
    // ====================== TMA producer (both CTAs) ======================
    if (lane == 0) {
      tma_prefetch_desc(&args.tma_a);
      tma_prefetch_desc(&args.tma_b);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs) {
        const int slot = t / per_e, rem = t - slot * per_e;
        const int mb = rem / n_tiles, nb = rem - mb * n_tiles;
        const int e = s_order[slot];
        const int m0 = mb * 256, n0 = nb * BN;
        const int k_row0 = s_off[e];
        const int num_kb = (s_cnt[e] + BK - 1) / BK;
        int nbox[2][2];                      // [cta][A,B] boxes holding in-range data
        for (int r = 0; r < 2; ++r) {
          nbox[r][0] = max(0, min(2, (args.m_ext - (m0 + 128 * r) + 63) / 64));
          nbox[r][1] = max(0, min(2, (args.b_ext - (n0 + 128 * r) + 63) / 64));
          // a 4-D atom load always moves both atoms (out-of-range ones zero-filled)
          if (args.a_atoms4d && nbox[r][0] > 0) nbox[r][0] = 2;
          if (args.b_atoms4d && nbox[r][1] > 0) nbox[r][1] = 2;
        }
        const uint32_t tx = (nbox[0][0] + nbox[0][1] + nbox[1][0] + nbox[1][1]) * MN_BOX_BYTES;
        const int my_a = nbox[rank][0], my_b = nbox[rank][1];
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, args.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * PAIR_STAGE_BYTES;
          uint8_t* sb = sa + PAIR_HALF;
          const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], tx);
          const int kr = k_row0 + kb * BK;
          if (args.a_atoms4d) {
            if (my_a) tma_load_4d_pair(sa, &args.tma_a, fb, 0, kr, (m0 + 128 * rank) / 64, 0);
          } else {
            for (int i = 0; i < my_a; ++i)
              tma_load_3d_pair(sa + i * MN_BOX_BYTES, &args.tma_a, fb, m0 + 128 * rank + 64 * i, kr, 0);
          }
          if (args.b_atoms4d) {
            if (my_b) tma_load_4d_pair(sb, &args.tma_b, fb, 0, kr, (n0 + 128 * rank) / 64, 0);
          } else {
            for (int i = 0; i < my_b; ++i)
              tma_load_3d_pair(sb + i * MN_BOX_BYTES, &args.tma_b, fb, n0 + 128 * rank + 64 * i, kr, 0);
          }
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ====================== MMA issuer (lead CTA only) ====================
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = pair; t < total && ok; t += npairs, ++it) {
        const int slot = t / per_e;
        const int e = s_order[slot];
        const int num_kb = (s_cnt[e] + BK - 1) / BK;
        const int acc = it & 1;
        const uint32_t acc_par = (it >> 1) & 1;
        if (!mbar_wait(&tempty_bar[acc], acc_par ^ 1u, args.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, args.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * PAIR_STAGE_BYTES);
          const uint32_t b_base = a_base + PAIR_HALF;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t ad = sdesc_sw128(a_base + k * 2048, MN_BOX_BYTES, 1024);
            const uint64_t bd = sdesc_sw128(b_base + k * 2048, MN_BOX_BYTES, 1024);
            umma_bf16_pair(d_tmem, ad, bd, kPairIdesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          umma_commit_pair(&empty_bar[stage]);
          if (++stage == PAIR_STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&tfull_bar[acc]);
      }
    }
  } else {
    // ====================== epilogue (both CTAs) ==========================
    // eight warps, two per TMEM lane quarter, 16 of every 32 columns each
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int hc = 16 * half;
    StoreRing ring{smem_u32(smem + PAIR_STAGES * PAIR_STAGE_BYTES), 0, nullptr};
    const bool issuer = threadIdx.x == 64;
    const int row_local = quarter * 32 + lane;
    int it = 0;
    for (int t = pair; t < total; t += npairs, ++it) {
      const int slot = t / per_e, rem = t - slot * per_e;
      const int mb = rem / n_tiles, nb = rem - mb * n_tiles;
      const int e = s_order[slot];
      const int n0 = nb * BN;
      const int y0 = mb * 256 + 128 * static_cast<int>(rank);
      const bool has_acc = s_cnt[e] > 0;
      const int acc = it & 1;
      const uint32_t acc_par = (it >> 1) & 1;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull_bar[acc], acc_par, args.status, abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      // leave together: the store barriers below need all epilogue warps
      if (named_bar_any(kEpiBar, kGemmEpiThreads, !ok)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN + hc;
      const bool write = y0 < args.m_ext;
      const int nch = min(BN / 32, (args.n_ext - n0 + 31) / 32);
      uint32_t ra[16], rb[16];
      if (has_acc) {
        tmem_ld16(tbase, ra);
        if (nch > 1) tmem_ld16(tbase + 32, rb);
      } else if (write) {
        ring_store_pair_zero_tile(ring, &args.tma_out2, n0, nch, y0, e, row_local, half, issuer);
      }
#pragma unroll 1
      for (int j = 0; j < nch && has_acc; j += 2) {
        const bool two = j + 1 < nch;
        float v0[16], v1[16];
        if (has_acc) {
          tmem_ld_wait16(ra);
          reg_fence16(rb);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            v0[i] = __uint_as_float(ra[i]);
            v1[i] = __uint_as_float(rb[i]);
          }
          if (j + 2 < nch) tmem_ld16(tbase + 32 * (j + 2), ra);
          if (j + 3 < nch) tmem_ld16(tbase + 32 * (j + 3), rb);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) v0[i] = v1[i] = 0.0f;
        }
        if (write)
          ring_store_pair<3>(ring, v0, v1, two, true, &args.tma_out2, n0 + 32 * j, y0, e,
                             row_local, half, issuer);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[acc]), 0));
    }
    if (issuer) bulk_wait_all();
  }

  __syncthreads();
  cluster_sync();                            // no remote arrivals after this point
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

cudaError_t launch_wgrad_pair(const GemmArgs& args, int grid, cudaStream_t s) {
  cudaError_t err = cudaFuncSetAttribute(k_wgrad_pair, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(PAIR_SMEM_BYTES));
  if (err != cudaSuccess) return err;
  const int g = grid & ~1;
  k_wgrad_pair<<<g < 2 ? 2 : g, GEMM_THREADS, PAIR_SMEM_BYTES, s>>>(args);
  return cudaGetLastError();
}

template <int MODE, int ACT, int OP>
cudaError_t launch_mode(const GemmArgs& args, int grid, cudaStream_t s) {
  constexpr size_t smem = OP == kOpNv    ? SMEM_BYTES_NV
                         : OP == kOpMxH ? SMEM_BYTES_MXH
                         : OP == kOpMx  ? SMEM_BYTES_MX
                         : Traits<MODE, OP>::kHAsync ? SMEM_BYTES_HA
                                                     : SMEM_BYTES;
  static_assert(smem <= 232448, "shared memory per CTA");
  cudaError_t err = cudaFuncSetAttribute(k_grouped_gemm<MODE, ACT, OP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  if (MODE == kRouter && args.r_grid != nullptr) {
    // the routing tail waits on every CTA: all of them must be resident
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_grouped_gemm<MODE, ACT, OP>,
                                                        GEMM_THREADS, smem);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return err;
    if (grid > per_sm * sms) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_grouped_gemm<MODE, ACT, OP>, args);
  }
  k_grouped_gemm<MODE, ACT, OP><<<grid, GEMM_THREADS, smem, s>>>(args);
  return cudaGetLastError();
}

template <int MODE, int OP>
cudaError_t launch_act(const GemmArgs& args, int grid, cudaStream_t s) {
  switch (args.act) {
    case MOE_ACT_SWIGLU: return launch_mode<MODE, MOE_ACT_SWIGLU, OP>(args, grid, s);
    case MOE_ACT_GEGLU: return launch_mode<MODE, MOE_ACT_GEGLU, OP>(args, grid, s);
    case MOE_ACT_SREGLU: return launch_mode<MODE, MOE_ACT_SREGLU, OP>(args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t grouped_gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_grouped_gemm(int mode, const GemmArgs& args, int grid, cudaStream_t s) {
  switch (mode) {
    case kFc1Glu: return launch_act<kFc1Glu, kOpBf16>(args, grid, s);
    case kFc2: return launch_mode<kFc2, 0, kOpBf16>(args, grid, s);
    case kDgradDglu:
      return args.K <= kHAsyncMaxK ? launch_act<kDgradDglu, kOpBf16H>(args, grid, s)
                                   : launch_act<kDgradDglu, kOpBf16>(args, grid, s);
    case kDgradFc1: return launch_mode<kDgradFc1, 0, kOpBf16>(args, grid, s);
    case kWgradPair: return launch_wgrad_pair(args, grid, s);
    case kFc1Act: return launch_mode<kFc1Act, MOE_ACT_SRELU, kOpBf16>(args, grid, s);
    case kDgradAct: return launch_mode<kDgradAct, MOE_ACT_SRELU, kOpBf16>(args, grid, s);
    case kRouter: return launch_mode<kRouter, 0, kOpBf16>(args, grid, s);
    case kDgradDgluRc: return launch_act<kDgradDgluRc, kOpBf16>(args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_grouped_gemm_mx(int mode, const GemmArgs& args, int grid, cudaStream_t s) {
  switch (mode) {
    case kFc1Glu: return launch_act<kFc1Glu, kOpMx>(args, grid, s);
    case kFc2: return launch_mode<kFc2, 0, kOpMx>(args, grid, s);
    case kDgradDglu:
      return args.K <= kHAsyncMaxKMx ? launch_act<kDgradDglu, kOpMxH>(args, grid, s)
                                     : launch_act<kDgradDglu, kOpMx>(args, grid, s);
    case kDgradFc1: return launch_mode<kDgradFc1, 0, kOpMx>(args, grid, s);
    case kWgrad: return launch_mode<kWgrad, 0, kOpMx>(args, grid, s);
    case kFc1Act: return launch_mode<kFc1Act, MOE_ACT_SRELU, kOpMx>(args, grid, s);
    case kDgradAct: return launch_mode<kDgradAct, MOE_ACT_SRELU, kOpMx>(args, grid, s);
    case kDgradDgluRc: return launch_act<kDgradDgluRc, kOpMx>(args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_grouped_gemm_nv(int mode, const GemmArgs& args, int grid, cudaStream_t s) {
  switch (mode) {
    case kFc1Glu: return launch_act<kFc1Glu, kOpNv>(args, grid, s);
    case kFc2: return launch_mode<kFc2, 0, kOpNv>(args, grid, s);
    case kDgradDglu: return launch_act<kDgradDglu, kOpNv>(args, grid, s);
    case kDgradFc1: return launch_mode<kDgradFc1, 0, kOpNv>(args, grid, s);
    case kWgrad: return launch_mode<kWgrad, 0, kOpNv>(args, grid, s);
    case kFc1Act: return launch_mode<kFc1Act, MOE_ACT_SRELU, kOpNv>(args, grid, s);
    case kDgradAct: return launch_mode<kDgradAct, MOE_ACT_SRELU, kOpNv>(args, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
