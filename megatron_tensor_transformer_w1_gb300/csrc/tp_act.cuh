// tp_act.cuh -- the activation functions of the FFN and their derivatives,
// in fp32, shared by every kernel that applies them (tensor-core epilogues,
// the SIMT GEMM of fp32 plans, the decode SwiGLU combine), so that all paths
// evaluate them identically.
//
//   gelu_tanh(z)  = z/2 * (1 + tanh(sqrt(2/pi) * (z + 0.044715 z^3)))
//                   (the tanh approximation of GELU, Hendrycks & Gimpel)
//   gelu_tanh'(z) = (1 + t)/2 + z/2 * (1 - t^2) * sqrt(2/pi) * (1 + 3 * 0.044715 z^2),
//                   t = tanh(sqrt(2/pi) * (z + 0.044715 z^3))
//   sigmoid(a)    = 1 / (1 + e^-a);  silu(a) = a * sigmoid(a);
//   silu'(a)      = sigmoid(a) * (1 + a * (1 - sigmoid(a)))
//
// tanhf and expf are CUDA's own; for |z| or |a| large enough that tanh
// saturates or e^-a overflows, these forms give the limits (gelu -> 0 or z,
// gelu' -> 0 or 1, sigmoid -> 0 or 1) without a NaN.
#pragma once

namespace tpffn {

__device__ __forceinline__ float gelu_tanh_f(float z) {
  const float k = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * z * (1.0f + tanhf(k * (z + 0.044715f * z * z * z)));
}
__device__ __forceinline__ float gelu_tanh_grad_f(float z) {
  const float k = 0.7978845608028654f;
  const float t = tanhf(k * (z + 0.044715f * z * z * z));
  return 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * k * (1.0f + 3.0f * 0.044715f * z * z);
}
__device__ __forceinline__ float sigmoid_f(float a) { return 1.0f / (1.0f + expf(-a)); }

}  // namespace tpffn
