// Activation functions of the GLU epilogues and their derivatives, shared by
// the grouped-GEMM kernels of every operand type.
//
// "Improving MoE training throughput with advanced fused kernels",
// "Overcoming training bottlenecks in the MoE block": SwiGLU, GeGLU and
// squared-ReLU activations with optional clamp and scaling; the forward
// epilogue applies them to the FC1 accumulator, the backward epilogue
// (dGLU) differentiates them.  With g the gate half, l the linear half,
// g' = min(g, limit), l' = clamp(l, -limit, limit):
//   A = s * phi(g') * (l' + linear_offset),  s = out_scale,
// phi(x) = x sigmoid(alpha x) (SwiGLU), x Phi(x) (GeGLU), max(x,0)^2
// (gated squared ReLU); the non-gated squared ReLU is s * max(min(h,limit),0)^2.
#pragma once

#include <math.h>

#include "moe.h"

namespace moe {

struct ActP {
  int act;
  float alpha, limit, lin_off, out_scale;
};

// sigmoid(x) = 1 / (1 + e^-x); the approximate reciprocal is within a few
// ulp and returns 0 when e^-x overflows to +inf.
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

template <int ACT>
__device__ __forceinline__ float glu_fwd(float g, float l, const ActP& p) {
  const float gc = fminf(g, p.limit);
  const float lc = fminf(fmaxf(l, -p.limit), p.limit);
  float phi;
  if (ACT == MOE_ACT_SWIGLU) {
    phi = gc * sigmoid_f(p.alpha * gc);
  } else if (ACT == MOE_ACT_GEGLU) {
    phi = 0.5f * gc * (1.0f + erff(gc * 0.70710678118654752f));
  } else {
    const float r = fmaxf(gc, 0.0f);
    phi = r * r;
  }
  return p.out_scale * phi * (lc + p.lin_off);
}

// Non-gated squared ReLU: A = s * max(min(h, limit), 0)^2 and its gradient
// (the clamp passes the gradient where h <= limit).
__device__ __forceinline__ float srelu_fwd(float h, const ActP& p) {
  const float r = fmaxf(fminf(h, p.limit), 0.0f);
  return p.out_scale * r * r;
}

__device__ __forceinline__ float srelu_bwd(float da, float h, const ActP& p) {
  const float r = fmaxf(fminf(h, p.limit), 0.0f);
  return h <= p.limit ? p.out_scale * da * 2.0f * r : 0.0f;
}

template <int ACT>
__device__ __forceinline__ void glu_bwd(float da, float g, float l, const ActP& p, float& dg,
                                        float& dl) {
  const float gc = fminf(g, p.limit);
  const float lc = fminf(fmaxf(l, -p.limit), p.limit);
  float phi, dphi;
  if (ACT == MOE_ACT_SWIGLU) {
    const float s = sigmoid_f(p.alpha * gc);
    phi = gc * s;
    dphi = s + p.alpha * gc * s * (1.0f - s);
  } else if (ACT == MOE_ACT_GEGLU) {
    const float cdf = 0.5f * (1.0f + erff(gc * 0.70710678118654752f));
    const float pdf = 0.39894228040143268f * __expf(-0.5f * gc * gc);
    phi = gc * cdf;
    dphi = cdf + gc * pdf;
  } else {
    const float r = fmaxf(gc, 0.0f);
    phi = r * r;
    dphi = 2.0f * r;
  }
  const float das = p.out_scale * da;
  dg = (g <= p.limit) ? das * (lc + p.lin_off) * dphi : 0.0f;
  dl = (l >= -p.limit && l <= p.limit) ? das * phi : 0.0f;
}

}  // namespace moe
