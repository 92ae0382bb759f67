// Unfused comparison path: the activation runs as its own memory-bound pass
// between plain grouped GEMMs, instead of inside the GEMM epilogue.
//
// "Improving MoE training throughput with advanced fused kernels",
// "Overcoming training bottlenecks in the MoE block": activation functions
// usually run as memory-bound kernels that read and write large tensors while
// the tensor cores idle; "From kernel-level gains to end-to-end pretraining
// speedups" reports the fused kernels against such an unfused path (up to 1.3x
// forward, 2.1x backward).  These kernels rebuild that unfused path from this
// library's own GEMMs so the fusion gain can be measured on the same GPU:
//   forward:  FC1 GEMM -> H (bf16) -> k_glu_rows -> A -> FC2 GEMM
//   backward: FC2 dgrad GEMM -> dA (bf16) -> k_dglu_rows (reads H) -> dH
// The activation math is the same as the fused epilogues'.
#include <cuda_bf16.h>
#include <math.h>

#include "moe_internal.h"
#include "moe_ptx.cuh"

namespace moe {
namespace {

struct ActArgs {
  int act;
  float alpha, limit, lin_off, out_scale;
};

__device__ __forceinline__ float sig(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

__device__ __forceinline__ float phi_fwd(int act, float gc, float alpha) {
  if (act == MOE_ACT_SWIGLU) return gc * sig(alpha * gc);
  if (act == MOE_ACT_GEGLU) return 0.5f * gc * (1.0f + erff(gc * 0.70710678118654752f));
  const float r = fmaxf(gc, 0.0f);
  return r * r;
}

// Row r of the packed H [cap, 2F_pad] -> A[r, f] for f < F; padding rows of a
// group (and rows past the last group) are written as zero up to rows_end.
// One thread handles 8 consecutive features.
__global__ void __launch_bounds__(256) k_glu_rows(const __nv_bfloat16* __restrict__ h,
                                                  const int32_t* __restrict__ counts,
                                                  const int32_t* __restrict__ padded_offsets,
                                                  int E, int F, int F_pad,
                                                  __nv_bfloat16* __restrict__ a, ActArgs p) {
  const int rows = padded_offsets[E];
  const int vec = F / 8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       i < static_cast<long long>(rows) * vec; i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / vec);
    const int f0 = static_cast<int>(i - static_cast<long long>(r) * vec) * 8;
    // group of row r (binary search over the padded offsets)
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(padded_offsets + mid) <= r) lo = mid; else hi = mid;
    }
    const bool real = r - __ldg(padded_offsets + lo) < __ldg(counts + lo);
    float out[8];
    if (real) {
      const int cg = (f0 / kGluHalf) * 2 * kGluHalf + (f0 % kGluHalf);
      const uint4 gw = __ldg(reinterpret_cast<const uint4*>(h + static_cast<long long>(r) * 2 * F_pad + cg));
      const uint4 lw = __ldg(reinterpret_cast<const uint4*>(h + static_cast<long long>(r) * 2 * F_pad + cg + kGluHalf));
      const uint32_t g4[4] = {gw.x, gw.y, gw.z, gw.w}, l4[4] = {lw.x, lw.y, lw.z, lw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float gs[2] = {bf16_lo(g4[q]), bf16_hi(g4[q])}, ls[2] = {bf16_lo(l4[q]), bf16_hi(l4[q])};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float gc = fminf(gs[u], p.limit);
          const float lc = fminf(fmaxf(ls[u], -p.limit), p.limit);
          out[2 * q + u] = p.out_scale * phi_fwd(p.act, gc, p.alpha) * (lc + p.lin_off);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) out[u] = 0.0f;
    }
    uint4 w;
    w.x = pack_bf16x2(out[0], out[1]);
    w.y = pack_bf16x2(out[2], out[3]);
    w.z = pack_bf16x2(out[4], out[5]);
    w.w = pack_bf16x2(out[6], out[7]);
    *reinterpret_cast<uint4*>(a + static_cast<long long>(r) * F + f0) = w;
  }
}

// dA [cap, F] and packed H -> packed dH [cap, 2F_pad]; zero on padding rows
// and padding features.
__global__ void __launch_bounds__(256) k_dglu_rows(const __nv_bfloat16* __restrict__ da,
                                                   const __nv_bfloat16* __restrict__ h,
                                                   const int32_t* __restrict__ counts,
                                                   const int32_t* __restrict__ padded_offsets,
                                                   int E, int F, int F_pad,
                                                   __nv_bfloat16* __restrict__ dh, ActArgs p) {
  const int rows = padded_offsets[E];
  const int vec = F_pad / 8;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
       i < static_cast<long long>(rows) * vec; i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(i / vec);
    const int f0 = static_cast<int>(i - static_cast<long long>(r) * vec) * 8;
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(padded_offsets + mid) <= r) lo = mid; else hi = mid;
    }
    const bool real = r - __ldg(padded_offsets + lo) < __ldg(counts + lo) && f0 < F;
    const int cg = (f0 / kGluHalf) * 2 * kGluHalf + (f0 % kGluHalf);
    float dg[8], dl[8];
    if (real) {
      const long long hr = static_cast<long long>(r) * 2 * F_pad;
      const uint4 gw = __ldg(reinterpret_cast<const uint4*>(h + hr + cg));
      const uint4 lw = __ldg(reinterpret_cast<const uint4*>(h + hr + cg + kGluHalf));
      const uint4 aw = __ldg(reinterpret_cast<const uint4*>(da + static_cast<long long>(r) * F + f0));
      const uint32_t g4[4] = {gw.x, gw.y, gw.z, gw.w}, l4[4] = {lw.x, lw.y, lw.z, lw.w},
                     a4[4] = {aw.x, aw.y, aw.z, aw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float gs[2] = {bf16_lo(g4[q]), bf16_hi(g4[q])}, ls[2] = {bf16_lo(l4[q]), bf16_hi(l4[q])},
                    as[2] = {bf16_lo(a4[q]), bf16_hi(a4[q])};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float g = gs[u], l = ls[u];
          const float gc = fminf(g, p.limit);
          const float lc = fminf(fmaxf(l, -p.limit), p.limit);
          float phi, dphi;
          if (p.act == MOE_ACT_SWIGLU) {
            const float s = sig(p.alpha * gc);
            phi = gc * s;
            dphi = s + p.alpha * gc * s * (1.0f - s);
          } else if (p.act == MOE_ACT_GEGLU) {
            const float cdf = 0.5f * (1.0f + erff(gc * 0.70710678118654752f));
            phi = gc * cdf;
            dphi = cdf + gc * 0.39894228040143268f * __expf(-0.5f * gc * gc);
          } else {
            const float rr = fmaxf(gc, 0.0f);
            phi = rr * rr;
            dphi = 2.0f * rr;
          }
          const float das = p.out_scale * as[u];
          dg[2 * q + u] = (g <= p.limit) ? das * (lc + p.lin_off) * dphi : 0.0f;
          dl[2 * q + u] = (l >= -p.limit && l <= p.limit) ? das * phi : 0.0f;
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) dg[u] = dl[u] = 0.0f;
    }
    const long long o = static_cast<long long>(r) * 2 * F_pad + cg;
    uint4 w;
    w.x = pack_bf16x2(dg[0], dg[1]);
    w.y = pack_bf16x2(dg[2], dg[3]);
    w.z = pack_bf16x2(dg[4], dg[5]);
    w.w = pack_bf16x2(dg[6], dg[7]);
    *reinterpret_cast<uint4*>(dh + o) = w;
    w.x = pack_bf16x2(dl[0], dl[1]);
    w.y = pack_bf16x2(dl[2], dl[3]);
    w.z = pack_bf16x2(dl[4], dl[5]);
    w.w = pack_bf16x2(dl[6], dl[7]);
    *reinterpret_cast<uint4*>(dh + o + kGluHalf) = w;
  }
}

}  // namespace

cudaError_t launch_glu_rows(const void* h, const int32_t* counts, const int32_t* padded_offsets,
                            int E, int F, int F_pad, void* a, int act, float alpha, float limit,
                            float lin_off, float out_scale, int num_sms, cudaStream_t s) {
  const ActArgs p{act, alpha, limit, lin_off, out_scale};
  k_glu_rows<<<num_sms * 8, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(h), counts,
                                         padded_offsets, E, F, F_pad,
                                         static_cast<__nv_bfloat16*>(a), p);
  return cudaGetLastError();
}

cudaError_t launch_dglu_rows(const void* da, const void* h, const int32_t* counts,
                             const int32_t* padded_offsets, int E, int F, int F_pad, void* dh,
                             int act, float alpha, float limit, float lin_off, float out_scale,
                             int num_sms, cudaStream_t s) {
  const ActArgs p{act, alpha, limit, lin_off, out_scale};
  k_dglu_rows<<<num_sms * 8, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(da),
                                          static_cast<const __nv_bfloat16*>(h), counts,
                                          padded_offsets, E, F, F_pad,
                                          static_cast<__nv_bfloat16*>(dh), p);
  return cudaGetLastError();
}

}  // namespace moe
