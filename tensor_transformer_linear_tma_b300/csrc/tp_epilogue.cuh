// Elementwise operations applied inside GEMM epilogues and combine kernels.
//
// The activations are the local elementwise operations of the "CUDA tensor
// parallel computations" page (section on local elementwise computation):
// ReLU, GELU (exact erf form, the default of the tutorial page's nn.GELU
// sample) and SiLU, plus the SwiGLU gate silu(gate) * up of the tutorial
// page's MLP-block section. They use CUDA's erff / expf.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace tpk {

enum Act : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU = 2, ACT_SILU = 3, ACT_SWIGLU = 4 };

__device__ __forceinline__ float act_relu(float x) { return fmaxf(x, 0.0f); }
__device__ __forceinline__ float act_gelu(float x) {
  return 0.5f * x * (1.0f + erff(x * 0.70710678118654752440f));
}
__device__ __forceinline__ float act_silu(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ float apply_act(int act, float x) {
  switch (act) {
    case ACT_RELU: return act_relu(x);
    case ACT_GELU: return act_gelu(x);
    case ACT_SILU: return act_silu(x);
    default: return x;
  }
}

// Gradient through the local activation (the backward of the tutorial
// page's MLP block step 2): given dh = dL/dH for H = act(g), or H = silu(g) u
// for SwiGLU, returns dg = dL/dg and du = dL/du (0 except for SwiGLU):
// relu'(g) = [g > 0]; gelu'(g) = Phi(g) + g phi(g), the normal CDF and
// density; silu'(g) = s (1 + g (1 - s)), s = 1 / (1 + e^-g).
__device__ __forceinline__ void act_grad(int act, float dh, float g, float u, float& dg, float& du) {
  du = 0.0f;
  switch (act) {
    case ACT_RELU: dg = g > 0.0f ? dh : 0.0f; break;
    case ACT_GELU: {
      const float Phi = 0.5f * (1.0f + erff(g * 0.70710678118654752440f));
      const float phi = 0.39894228040143267794f * expf(-0.5f * g * g);
      dg = dh * (Phi + g * phi);
      break;
    }
    case ACT_SILU:
    case ACT_SWIGLU: {
      // the fast exponential and an IEEE reciprocal: a few ulp of fp32,
      // far inside the bf16 rounding of the gradient that is stored
      const float sg = __frcp_rn(1.0f + __expf(-g));
      const float d = sg * (1.0f + g * (1.0f - sg));
      if (act == ACT_SILU) {
        dg = dh * d;
      } else {
        dg = dh * u * d;
        du = dh * g * sg;
      }
      break;
    }
    default: dg = dh;
  }
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

}  // namespace tpk
