// The routed-expert MLP on fp32 tensors: persistent grouped GEMM on the TF32
// tensor cores (tcgen05 kind::tf32) with the fused GLU / dGLU epilogues, and
// the fp32 memory-bound passes around it (combine, combine backward, bias
// column sums, transposes).
//
// Sources: "Improving MoE training throughput with advanced fused kernels":
//   - "Overcoming training bottlenecks in the MoE block": the GroupGemm +
//     Activation and GroupGemm + dActivation kernels.
//   - "Optimizing GLU activations with fused GEMM epilogues" (Figure 2): the
//     repacked FC1 weight puts 128 gate and the matching 128 linear features
//     in one 256-column accumulator tile, so the GLU runs in the epilogue.
//   - "Eliminating host-device synchronisation and CPU launch overhead":
//     group sizes are read from GPU memory; the grid is sized from the SM
//     count.
// "Accelerating dropless MoE training with JAX and NVIDIA Transformer
// Engine", "Claims and evidence": one grouped GEMM over ragged groups.
//
// Design (one CTA per SM, 10 warps, tiles of 128 rows x 256 columns):
//   warp 0    TMA producer: K-major fp32 operand tiles, 32 values (one
//             128-byte swizzled row) per operand row and stage, into a ring
//             of 4 stages (48 KB each).
//   warp 1    TMEM owner and single-thread MMA issuer: M=128, N=256, K=8 per
//             tcgen05.mma kind::tf32 (the same 32 bytes per row per step as
//             a bf16 K=16 step); two 256-column fp32 accumulators, so the
//             epilogue of one tile overlaps the MMAs of the next.
//   warps 2-9 epilogue, two per TMEM lane quarter, each taking 16 of every
//             32 accumulator columns (tcgen05.ld of 16 columns), the fused
//             math, fp32 stores.  A thread owns one output row and writes
//             its 16 values of a chunk as 64 contiguous bytes; the optional
//             transposed copies are written one column per store, 32
//             consecutive rows = 128 contiguous bytes per warp.
// Every operand is K-major: the backward reads transposed weight copies and
// transposed activations (A and dH transposed by the epilogues that produce
// them, x_perm and dY by k_transpose_f32).  Tiles whose 128 rows are all
// padding issue no MMA; their epilogue writes zeros.  Weight-gradient tiles
// (ragged K) run the K loop over the group's rows only, largest group first.
#include <cuda.h>
#include <math.h>
#include <stdint.h>

#include "moe_act.cuh"
#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {

namespace {

constexpr int TM = 128;
constexpr int TN = 256;
constexpr int TK = 32;                          // fp32 values per 128-byte row
constexpr int T_STAGES = 4;
constexpr int TA_BYTES = TM * TK * 4;           // 16 KB
constexpr int TB_BYTES = TN * TK * 4;           // 32 KB
constexpr int T_STAGE_BYTES = TA_BYTES + TB_BYTES;
constexpr int T_THREADS = 320;                  // producer, MMA, 8 epilogue warps
constexpr int T_EPI_WARPS = 8;
constexpr int T_TMEM_COLS = 2 * TN;
constexpr size_t T_SMEM_BYTES = 1024 + static_cast<size_t>(T_STAGES) * T_STAGE_BYTES;

struct TTile {
  int e;      // expert
  int m0;     // first output row (ragged M: routed row; ragged K: weight row)
  int n0;     // first output column
  int k0;     // ragged K: first routed row of the group
  int nkb;    // K blocks of 32 (0: no MMA, the tile is written as zeros)
};

template <int MODE>
__device__ __forceinline__ TTile tf32_tile(int t, int n_tiles, int m_tiles, const int* s_off,
                                           const int* cnt, const int* s_order, int E,
                                           int kb_full) {
  TTile ti;
  if (MODE == kWgrad) {
    const int per_e = m_tiles * n_tiles;
    const int slot = t / per_e;
    const int rem = t - slot * per_e;
    const int mb = rem / n_tiles;
    ti.e = s_order[slot];
    ti.m0 = mb * TM;
    ti.n0 = (rem - mb * n_tiles) * TN;
    ti.k0 = s_off[ti.e];
    ti.nkb = (cnt[ti.e] + TK - 1) / TK;
  } else {
    const int mb = t / n_tiles;
    const int row = mb * TM;
    int lo = 0, hi = E;   // last expert whose group starts at or before `row`
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= row) lo = mid; else hi = mid;
    }
    ti.e = lo;
    ti.m0 = row;
    ti.n0 = (t - mb * n_tiles) * TN;
    ti.k0 = 0;
    ti.nkb = row < s_off[lo] + cnt[lo] ? kb_full : 0;
  }
  return ti;
}

__device__ __forceinline__ void store_f32x16(float* dst, const float (&v)[16]) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__device__ __forceinline__ void load_f32x16(const float* src, float (&v)[16]) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 w = __ldg(s4 + i);
    v[4 * i] = w.x;
    v[4 * i + 1] = w.y;
    v[4 * i + 2] = w.z;
    v[4 * i + 3] = w.w;
  }
}

// Column c0 + i of this thread's row r, for the 16 values, into the
// transposed copy [width][ld]: lane j of the warp holds row r0 + j, so each
// store instruction writes 32 consecutive floats.
__device__ __forceinline__ void store_t_f32x16(float* dst_t, long long ld, int c0, int r,
                                               const float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) dst_t[static_cast<long long>(c0 + i) * ld + r] = v[i];
}

// The 16 accumulator columns [col, col + 16) of this warp's lane quarter as
// floats (zeros when the tile had no MMA).  Whole warp calls.
__device__ __forceinline__ void acc_load(uint32_t taddr, bool have, float (&v)[16]) {
  uint32_t r[16];
  if (have) {
    tmem_ld16(taddr, r);
    tmem_ld_wait16(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
  }
}

template <int MODE, int ACT>
__global__ void __launch_bounds__(T_THREADS, 1)
    k_grouped_gemm_tf32(const __grid_constant__ GemmArgs args) {
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[T_STAGES];
  __shared__ __align__(8) uint64_t empty_bar[T_STAGES];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;
  __shared__ int s_total;
  __shared__ int s_off[kMaxExperts + 1];
  __shared__ int s_order[kMaxExperts];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;
  const int* __restrict__ cnt = args.counts;   // group sizes, read through L1
  constexpr bool RK = MODE == kWgrad;

  for (int i = threadIdx.x; i <= E; i += T_THREADS) s_off[i] = args.padded_offsets[i];
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < T_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], T_EPI_WARPS);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem_base, T_TMEM_COLS);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();

  const int n_tiles = (args.n_ext + TN - 1) / TN;
  const int m_tiles = RK ? (args.m_ext + TM - 1) / TM : 0;
  if (threadIdx.x == 0) {
    // validate the offsets read from device memory; skip all work if bad
    bool ok = s_off[0] == 0 && s_off[E] <= args.capacity;
    for (int e = 0; e < E && ok; ++e) {
      const int span = s_off[e + 1] - s_off[e];
      ok = span >= 0 && (span % TM) == 0 && cnt[e] >= 0 && cnt[e] <= span;
    }
    if (!ok) {
      set_status(args.status, MOE_DEV_BAD_OFFSETS);
      s_total = 0;
    } else {
      s_total = RK ? E * m_tiles * n_tiles : (s_off[E] / TM) * n_tiles;
    }
  }
  if (RK) {
    // largest group first; equal sizes keep expert order
    for (int e = threadIdx.x; e < E; e += T_THREADS) {
      int rank = 0;
      for (int j = 0; j < E; ++j) rank += (cnt[j] > cnt[e]) || (cnt[j] == cnt[e] && j < e);
      s_order[rank] = e;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem_base;
  const int total = s_total;
  const int kb_full = (args.K + TK - 1) / TK;
  volatile int* abort_flag = &s_abort;

  if (warp == 0) {
    // ============================ TMA producer ============================
    if (lane == 0) {
      tma_prefetch_desc(&args.tma_a);
      tma_prefetch_desc(&args.tma_b);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TTile ti = tf32_tile<MODE>(t, n_tiles, m_tiles, s_off, cnt, s_order, E, kb_full);
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, args.status, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * T_STAGE_BYTES;
          mbar_arrive_expect_tx(&full_bar[stage], T_STAGE_BYTES);
          if (RK) {
            tma_load_3d(sa, &args.tma_a, &full_bar[stage], ti.k0 + kb * TK, ti.m0, 0);
            tma_load_3d(sa + TA_BYTES, &args.tma_b, &full_bar[stage], ti.k0 + kb * TK, ti.n0, 0);
          } else {
            tma_load_3d(sa, &args.tma_a, &full_bar[stage], kb * TK, ti.m0, 0);
            tma_load_3d(sa + TA_BYTES, &args.tma_b, &full_bar[stage], kb * TK, ti.n0, ti.e);
          }
          if (++stage == T_STAGES) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==============================
    if (lane == 0) {
      constexpr uint32_t kIdesc = idesc_tf32(TM, TN);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      int it = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TTile ti = tf32_tile<MODE>(t, n_tiles, m_tiles, s_off, cnt, s_order, E, kb_full);
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(&tempty_bar[acc], (use & 1u) ^ 1u, args.status, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * TN;
        for (int kb = 0; kb < ti.nkb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, args.status, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * T_STAGE_BYTES);
          const uint32_t b_base = a_base + TA_BYTES;
#pragma unroll
          for (int k = 0; k < TK / 8; ++k)
            umma_tf32(d_tmem, sdesc_sw128(a_base + k * 32, 16, 1024),
                      sdesc_sw128(b_base + k * 32, 16, 1024), kIdesc, (kb | k) != 0);
          umma_commit(&empty_bar[stage]);
          if (++stage == T_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);
      }
    }
  } else {
    // ============================== epilogue ==============================
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int hc = 16 * ((warp - 2) >> 2);      // this warp's 16 of every 32 columns
    const ActP ap{args.act, args.alpha, args.limit, args.lin_off, args.out_scale};
    const long long cap = args.capacity;
    float* out0 = static_cast<float*>(args.out0);
    float* out1 = static_cast<float*>(args.out1);
    const float* aux = static_cast<const float*>(args.aux);
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const TTile ti = tf32_tile<MODE>(t, n_tiles, m_tiles, s_off, cnt, s_order, E, kb_full);
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (!mbar_wait(&tfull_bar[acc], use & 1u, args.status, abort_flag)) break;
      tc_fence_after();
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * TN + hc;
      const bool have = ti.nkb > 0;             // warp-uniform
      const int r = ti.m0 + quarter * 32 + lane;
      const float* bias = static_cast<const float*>(args.bias);
      if (bias) bias += static_cast<long long>(ti.e) * args.bias_ld;

      if (MODE == kWgrad) {
        // dW[e] rows m0.., columns n0..; rows past m_ext are not stored
        float* dst = out0 + (static_cast<long long>(ti.e) * args.m_ext + r) * args.ld0;
        for (int c = 0; c < TN / 32 && ti.n0 + 32 * c < args.n_ext; ++c) {
          float v[16];
          acc_load(tbase + 32 * c, have, v);
          if (r < args.m_ext) store_f32x16(dst + ti.n0 + 32 * c + hc, v);
        }
      } else {
        const bool live = have && (r - s_off[ti.e]) < cnt[ti.e];   // a real row of the group
        if (MODE == kFc1Glu) {
          // columns 0..127 gate, 128..255 linear halves of 128 GLU features
          for (int c = 0; c < 4; ++c) {
            float g[16], l[16], a[16];
            acc_load(tbase + 32 * c, have, g);
            acc_load(tbase + 128 + 32 * c, have, l);
            const int cg = ti.n0 + 32 * c + hc, cl = cg + 128;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              g[i] = live ? g[i] + (bias ? bias[cg + i] : 0.0f) : 0.0f;
              l[i] = live ? l[i] + (bias ? bias[cl + i] : 0.0f) : 0.0f;
              a[i] = live ? glu_fwd<ACT>(g[i], l[i], ap) : 0.0f;
            }
            if (out0) {
              store_f32x16(out0 + r * args.ld0 + cg, g);
              store_f32x16(out0 + r * args.ld0 + cl, l);
            }
            const int f0 = ti.n0 / 2 + 32 * c + hc;   // GLU feature of column cg
            if (f0 < args.f_real) {
              if (out1) store_f32x16(out1 + r * args.ld1 + f0, a);
              if (args.out1_t) store_t_f32x16(args.out1_t, cap, f0, r, a);
            }
          }
        } else if (MODE == kFc1Act || MODE == kFc2 || MODE == kDgradFc1) {
          for (int c = 0; c < TN / 32 && ti.n0 + 32 * c < args.n_ext; ++c) {
            float h[16], a[16];
            acc_load(tbase + 32 * c, have, h);
            const int col = ti.n0 + 32 * c + hc;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              h[i] = live ? h[i] + (bias ? bias[col + i] : 0.0f) : 0.0f;
              if (MODE == kFc1Act) a[i] = live ? srelu_fwd(h[i], ap) : 0.0f;
            }
            if (out0) store_f32x16(out0 + r * args.ld0 + col, h);
            if (MODE == kFc1Act) {
              if (out1) store_f32x16(out1 + r * args.ld1 + col, a);
              if (args.out1_t) store_t_f32x16(args.out1_t, cap, col, r, a);
            }
          }
        } else if (MODE == kDgradDglu) {
          // dA for GLU features n0.. ; dG / dL go to the packed columns of H
          for (int c = 0; c < TN / 32 && ti.n0 + 32 * c < args.n_ext; ++c) {
            float da[16], g[16], l[16], dg[16], dl[16];
            acc_load(tbase + 32 * c, have, da);
            const int f0 = ti.n0 + 32 * c + hc;
            const int cg = (f0 / kGluHalf) * 2 * kGluHalf + f0 % kGluHalf, cl = cg + kGluHalf;
            if (live) {
              load_f32x16(aux + r * args.ld_aux + cg, g);
              load_f32x16(aux + r * args.ld_aux + cl, l);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              if (live) {
                glu_bwd<ACT>(da[i], g[i], l[i], ap, dg[i], dl[i]);
              } else {
                dg[i] = 0.0f;
                dl[i] = 0.0f;
              }
            }
            if (out0) {
              store_f32x16(out0 + r * args.ld0 + cg, dg);
              store_f32x16(out0 + r * args.ld0 + cl, dl);
            }
            if (args.out0_t) {
              store_t_f32x16(args.out0_t, cap, cg, r, dg);
              store_t_f32x16(args.out0_t, cap, cl, r, dl);
            }
          }
        } else if (MODE == kDgradAct) {
          for (int c = 0; c < TN / 32 && ti.n0 + 32 * c < args.n_ext; ++c) {
            float da[16], h[16], dh[16];
            acc_load(tbase + 32 * c, have, da);
            const int col = ti.n0 + 32 * c + hc;
            if (live) load_f32x16(aux + r * args.ld_aux + col, h);
#pragma unroll
            for (int i = 0; i < 16; ++i) dh[i] = live ? srelu_bwd(da[i], h[i], ap) : 0.0f;
            if (out0) store_f32x16(out0 + r * args.ld0 + col, dh);
            if (args.out0_t) store_t_f32x16(args.out0_t, cap, col, r, dh);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, T_TMEM_COLS);
  }
}

template <int MODE, int ACT>
cudaError_t launch_tf32(const GemmArgs& args, int grid, cudaStream_t s) {
  auto kern = k_grouped_gemm_tf32<MODE, ACT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(T_SMEM_BYTES));
  if (e != cudaSuccess) return e;
  kern<<<grid, T_THREADS, T_SMEM_BYTES, s>>>(args);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_tf32_act(const GemmArgs& args, int grid, cudaStream_t s) {
  switch (args.act) {
    case MOE_ACT_SWIGLU: return launch_tf32<MODE, MOE_ACT_SWIGLU>(args, grid, s);
    case MOE_ACT_GEGLU: return launch_tf32<MODE, MOE_ACT_GEGLU>(args, grid, s);
    case MOE_ACT_SREGLU: return launch_tf32<MODE, MOE_ACT_SREGLU>(args, grid, s);
  }
  return cudaErrorInvalidValue;
}

// ------------------------------------------------------------- fp32 passes
// out[t] = sum_s w[t,s] * y[row_of[t,s]] (fp32, slot order); w == nullptr:
// unit weights (permute backward).  One block per token.
__global__ void __launch_bounds__(128) k_combine_f32(const float4* __restrict__ y,
                                                     const int32_t* __restrict__ row_of,
                                                     const float* __restrict__ w, int k, int vec,
                                                     float4* __restrict__ out) {
  const int t = blockIdx.x;
  for (int c = threadIdx.x; c < vec; c += blockDim.x) {
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int s = 0; s < k; ++s) {
      const int r = row_of[static_cast<size_t>(t) * k + s];
      const float ws = w ? w[static_cast<size_t>(t) * k + s] : 1.0f;
      const float4 v = __ldg(y + static_cast<size_t>(r) * vec + c);
      acc.x = fmaf(ws, v.x, acc.x);
      acc.y = fmaf(ws, v.y, acc.y);
      acc.z = fmaf(ws, v.z, acc.z);
      acc.w = fmaf(ws, v.w, acc.w);
    }
    out[static_cast<size_t>(t) * vec + c] = acc;
  }
}

// dy[row_of[t,s]] = w[t,s] * dout[t]; dw[t,s] = <dout[t], y[row_of[t,s]]>
// with a fixed-shape block reduction (deterministic).
__global__ void __launch_bounds__(128) k_combine_bwd_f32(
    const float4* __restrict__ dout, const float4* __restrict__ y,
    const int32_t* __restrict__ row_of, const float* __restrict__ w, int k, int vec,
    float4* __restrict__ dy, float* __restrict__ dw) {
  __shared__ float s_part[4];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int s = 0; s < k; ++s) {
    const int r = row_of[static_cast<size_t>(t) * k + s];
    const float ws = w[static_cast<size_t>(t) * k + s];
    float part = 0.0f;
    for (int c = threadIdx.x; c < vec; c += blockDim.x) {
      const float4 g = __ldg(dout + static_cast<size_t>(t) * vec + c);
      const float4 v = __ldg(y + static_cast<size_t>(r) * vec + c);
      dy[static_cast<size_t>(r) * vec + c] = make_float4(ws * g.x, ws * g.y, ws * g.z, ws * g.w);
      part = fmaf(g.x, v.x, part);
      part = fmaf(g.y, v.y, part);
      part = fmaf(g.z, v.z, part);
      part = fmaf(g.w, v.w, part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, o);
    if (lane == 0) s_part[warp] = part;
    __syncthreads();
    if (threadIdx.x == 0)
      dw[static_cast<size_t>(t) * k + s] = (s_part[0] + s_part[1]) + (s_part[2] + s_part[3]);
    __syncthreads();
  }
}

// db[e, c] = sum over the group's rows of g[r, c] (fp32, fixed order: warp w
// sums rows w, w+8, ... in order, then the eight partial sums in warp order).
__global__ void __launch_bounds__(256) k_group_colsum_f32(const float* __restrict__ g,
                                                          const int32_t* __restrict__ counts,
                                                          const int32_t* __restrict__ padded_offsets,
                                                          int width, float* __restrict__ out) {
  __shared__ float s_part[8][32];
  const int e = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  const int r0 = padded_offsets[e], m = counts[e];
  float a = 0.0f;
  if (c < width)
    for (int r = warp; r < m; r += 8) a += __ldg(g + static_cast<size_t>(r0 + r) * width + c);
  s_part[warp][lane] = a;
  __syncthreads();
  if (warp == 0 && c < width) {
    float b = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) b += s_part[i][lane];
    out[static_cast<size_t>(e) * width + c] = b;
  }
}

// out[b][c][r] = in[b][r][c]: 32 x 32 tiles through shared memory (padded
// rows against bank conflicts); block (32, 8), each thread moves 4 values.
// Rows at or past *row_limit (when given) are neither read nor written.
__global__ void __launch_bounds__(256) k_transpose_f32(const float* __restrict__ in, int rows,
                                                       int cols, float* __restrict__ out,
                                                       const int32_t* __restrict__ row_limit) {
  __shared__ float tile[32][33];
  const int lim = row_limit ? min(rows, *row_limit) : rows;
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  if (r0 >= lim) return;
  const size_t plane = static_cast<size_t>(rows) * cols;
  const float* src = in + blockIdx.z * plane;
  float* dst = out + blockIdx.z * plane;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int r = r0 + threadIdx.y + 8 * j, c = c0 + threadIdx.x;
    if (r < lim && c < cols) tile[threadIdx.y + 8 * j][threadIdx.x] = __ldg(src + static_cast<size_t>(r) * cols + c);
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int c = c0 + threadIdx.y + 8 * j, r = r0 + threadIdx.x;
    if (r < lim && c < cols) dst[static_cast<size_t>(c) * rows + r] = tile[threadIdx.x][threadIdx.y + 8 * j];
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_tf32(int mode, const GemmArgs& args, int grid, cudaStream_t s) {
  switch (mode) {
    case kFc1Glu: return launch_tf32_act<kFc1Glu>(args, grid, s);
    case kFc1Act: return launch_tf32<kFc1Act, MOE_ACT_SRELU>(args, grid, s);
    case kFc2: return launch_tf32<kFc2, 0>(args, grid, s);
    case kDgradDglu: return launch_tf32_act<kDgradDglu>(args, grid, s);
    case kDgradAct: return launch_tf32<kDgradAct, MOE_ACT_SRELU>(args, grid, s);
    case kDgradFc1: return launch_tf32<kDgradFc1, 0>(args, grid, s);
    case kWgrad: return launch_tf32<kWgrad, 0>(args, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine_f32(const void* y, const int32_t* row_of, const float* w, int T, int k,
                               int d, void* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_combine_f32<<<T, 128, 0, s>>>(static_cast<const float4*>(y), row_of, w, k, d / 4,
                                  static_cast<float4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_combine_bwd_f32(const void* dout, const void* y, const int32_t* row_of,
                                   const float* w, int T, int k, int d, void* dy, float* dw,
                                   cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  k_combine_bwd_f32<<<T, 128, 0, s>>>(static_cast<const float4*>(dout),
                                      static_cast<const float4*>(y), row_of, w, k, d / 4,
                                      static_cast<float4*>(dy), dw);
  return cudaGetLastError();
}

cudaError_t launch_group_colsum_f32(const void* g, const int32_t* counts,
                                    const int32_t* padded_offsets, int E, int width, void* out,
                                    cudaStream_t s) {
  dim3 grid((width + 31) / 32, E);
  k_group_colsum_f32<<<grid, 256, 0, s>>>(static_cast<const float*>(g), counts, padded_offsets,
                                          width, static_cast<float*>(out));
  return cudaGetLastError();
}

cudaError_t launch_transpose_f32(const void* in, long long batch, long long rows, long long cols,
                                 void* out, const int32_t* row_limit, cudaStream_t s) {
  if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
  if (rows > (1LL << 30) || cols > (1LL << 30) || batch > 65535 || (rows + 31) / 32 > 65535)
    return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>((cols + 31) / 32), static_cast<unsigned>((rows + 31) / 32),
            static_cast<unsigned>(batch));
  k_transpose_f32<<<grid, dim3(32, 8), 0, s>>>(static_cast<const float*>(in),
                                               static_cast<int>(rows), static_cast<int>(cols),
                                               static_cast<float*>(out), row_limit);
  return cudaGetLastError();
}

}  // namespace moe
