// tp_act.cuh -- the activation functions of the FFN and their derivatives,
// in fp32, shared by every kernel that applies them (tensor-core epilogues,
// the SIMT GEMM of fp32 plans, the decode SwiGLU combine), so that all paths
// evaluate them identically.
//
// Both activations reduce to the logistic function:
//   sigmoid(a)    = 1 / (1 + e^-a);  silu(a) = a sigmoid(a);
//   silu'(a)      = s (1 + a (1 - s)),  s = sigmoid(a);
//   gelu_tanh(z)  = z/2 (1 + tanh(u)),  u = sqrt(2/pi) (z + 0.044715 z^3)
//                 = z sigmoid(2u)                        [1 + tanh(u) = 2 sigmoid(2u)]
//   gelu_tanh'(z) = s + 2 z s (1 - s) u',  s = sigmoid(2u),
//                   u' = sqrt(2/pi) (1 + 3 * 0.044715 z^2)  [1 - tanh^2(u) = 4 s (1 - s)]
// The GELU forms take 1 - s as E s with E = e^-x, so neither subtracts two
// nearly equal numbers: the textbook tanh form loses 1 + tanh(u) to
// cancellation for z << 0 (where CUDA's tanhf leaves up to 4.5e-5 relative
// error in gelu and 2.3e-4 in gelu' at values above 1e-3), the logistic form
// does not.
//
// Two evaluations of the logistic function are used, each where it measured
// faster:
//  * GELU (forward and derivative): e^-x as 2^(-x log2 e) with the SFU's
//    ex2.approx.ftz.f32 and the reciprocal with rcp.approx.ftz.f32 (PTX
//    instructions).  Measured on GB300 against float64 over z in [-40, 40]
//    (step 2^-10), relative error where |value| >= 1e-3: gelu 9.3e-7
//    (< 2^-20), gelu' 1.4e-5 (< 2^-16, near its zero crossing), at about
//    half the instruction cost of the tanhf form; Megatron-8.3B-shaped
//    dgrad_h_gelu 0.460 -> 0.431 ms, up_gelu unchanged.
//  * SwiGLU: sigmoid(a) = 1 / (1 + expf(-a)) with CUDA's expf and an IEEE
//    division (relative error 1.6e-7, measured the same way).  The SFU form
//    cut the instructions here too but slowed the Llama-3-8B-shaped SwiGLU
//    GEMMs (up 1622-1629 -> 1480, dh 1429-1431 -> 1361-1364 TFLOP/s, same
//    box, alternating), so these epilogues keep it.
// For large |x|, e^-x overflows to +inf or underflows to 0 and the forms
// reach their limits (sigmoid 0 or 1, gelu 0 or z, derivatives 0 or 1)
// without a NaN.
#pragma once

namespace tpffn {

__device__ __forceinline__ float exp2_sfu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_sfu(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kGeluK = 0.7978845608028654f;  // sqrt(2/pi)
constexpr float kGeluC = 0.044715f;

// SFU logistic: 1 / (1 + 2^(-x log2 e)), and 1 - that = e^-x times it (1
// when e^-x overflows), without a subtraction
__device__ __forceinline__ void sigmoid_sfu_pair(float x, float& s, float& one_minus_s) {
  const float e = exp2_sfu(x * -kLog2e);
  s = rcp_sfu(1.0f + e);
  one_minus_s = fminf(e * s, 1.0f);  // inf * 0 -> NaN -> 1
}
__device__ __forceinline__ float sigmoid_sfu(float x) { return rcp_sfu(1.0f + exp2_sfu(x * -kLog2e)); }

// the logistic of the SwiGLU epilogues
__device__ __forceinline__ float sigmoid_f(float a) { return 1.0f / (1.0f + expf(-a)); }

__device__ __forceinline__ float gelu_tanh_f(float z) {
  const float u = kGeluK * (z + kGeluC * z * z * z);
  return z * sigmoid_sfu(2.0f * u);
}
__device__ __forceinline__ float gelu_tanh_grad_f(float z) {
  const float u = kGeluK * (z + kGeluC * z * z * z);
  float s, om;
  sigmoid_sfu_pair(2.0f * u, s, om);
  return s + 2.0f * z * s * om * kGeluK * (1.0f + 3.0f * kGeluC * z * z);
}

}  // namespace tpffn
