// Device-side helpers shared by the kernels of the MLP training step.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace mlpk {

enum Act : int { ACT_NONE = 0, ACT_RELU = 1, ACT_GELU_TANH = 2 };
// DT_F32X3: fp32 values held as three bf16 planes for the tensor cores
// (internal to the fp32 model's step; never a model dtype).
enum DType : int { DT_F32 = 0, DT_BF16 = 1, DT_F32X3 = 2 };

// Device error word bits (latched in the model's control block).
enum : uint32_t {
  ERRBIT_LABEL_RANGE = 1u << 0,   // a label outside [0, C)
  ERRBIT_NONFINITE = 1u << 1,     // non-finite batch loss
  ERRBIT_TIMEOUT = 1u << 2,       // a bounded device-side wait gave up
  ERRBIT_BAD_LAUNCH = 1u << 3,    // a kernel saw parameters it cannot handle
};

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch: inside the step's CUDA graph each kernel may
// be launched before its predecessor has finished.  Every kernel calls this
// before its first global memory access: it waits until the predecessor grid
// has completed and its writes are visible, then lets the next kernel be
// scheduled (its blocks run their own prologue and wait here in turn).
// Without a programmatic dependency both instructions return at once.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// tanh-form GELU (Hendrycks & Gimpel): gelu(u) = 0.5 u (1 + tanh(a)),
// a = sqrt(2/pi) (u + 0.044715 u^3).  Evaluated through the identities
// 1 + tanh(a) = 2 s and 1 - tanh(a)^2 = 4 s (1 - s), s = 1 / (1 + e^{-2a}),
// 1 - s = 1 / (1 + e^{2a}), which keep fp32 relative accuracy in both tails
// (1 + tanh(a) computed directly cancels to 0 for very negative u).
// The GEMM epilogues evaluate this for every output, so it is written for
// few instructions: with c0 = -2 log2(e) sqrt(2/pi) and c1 = 0.044715 c0,
// e^{-2a} = 2^{u (c0 + c1 u^2)} (a multiply, an FMA, a multiply and the
// ex2.approx instruction), and 1 / (1 + e) by rcp.approx -- each about 2 ulp
// in fp32, far below the bf16 rounding of the stored result.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kGeluC0 = -2.302208198144325f;    // -2 log2(e) sqrt(2/pi)
constexpr float kGeluC1 = -0.1029432395800235f;   // 0.044715 kGeluC0
constexpr float kGeluK0 = 0.7978845608028654f;    // sqrt(2/pi)
constexpr float kGeluK3 = 0.10703222440890038f;   // 3 * 0.044715 sqrt(2/pi)
// u s with s = 1 / (1 + e^{-2a}).  For very negative u, e^{-2a} overflows
// to +inf and s to 0: the result is -0, the value bf16 storage gives anyway.
__device__ __forceinline__ float gelu_tanh(float u) {
  const float e = ex2_fast(u * fmaf(kGeluC1, u * u, kGeluC0));
  return u * rcp_fast(1.0f + e);
}
// s + 2 u s (1 - s) a', a' = sqrt(2/pi) (1 + 3 * 0.044715 u^2), with
// 1 - s = e s; the exponent is clamped so that e stays finite.
__device__ __forceinline__ float gelu_tanh_grad(float u) {
  const float u2 = u * u;
  const float x = fminf(fmaxf(u * fmaf(kGeluC1, u2, kGeluC0), -126.f), 126.f);
  const float e = ex2_fast(x);
  const float s = rcp_fast(1.0f + e);
  const float d = fmaf(kGeluK3, u2, kGeluK0);
  return fmaf(2.0f * u * s * (e * s), d, s);
}
__device__ __forceinline__ float apply_act(float v, int act) {
  if (act == ACT_RELU) return fmaxf(v, 0.0f);
  if (act == ACT_GELU_TANH) return gelu_tanh(v);
  return v;
}
// Derivative factor of the activation, from what the forward stored:
// ReLU: stored h (mask h > 0); GELU: stored pre-activation u.
__device__ __forceinline__ float act_grad_from_stored(float s, int act) {
  if (act == ACT_RELU) return s > 0.0f ? 1.0f : 0.0f;
  if (act == ACT_GELU_TANH) return gelu_tanh_grad(s);
  return 1.0f;
}

// 1 - beta^t in fp32 without cancellation: -expm1(t log1p(beta - 1)) (beta - 1
// is exact for beta in [0.5, 1]); a few ulp.  GB300's fp64 pipe is slow, so
// the step's scalars stay in fp32.
__device__ __forceinline__ float one_minus_pow(float beta, int64_t t) {
  return -expm1f((float)t * log1pf(beta - 1.0f));
}

// Advance the device step counter to t and store AdamW's bias corrections
// for that step, 1/(1 - beta1^t) and 1/sqrt(1 - beta2^t) (one thread, once
// per step).
__device__ __forceinline__ void advance_step(int64_t* counter, float* bias_corr, float beta1, float beta2) {
  const int64_t t = *counter + 1;
  *counter = t;
  if (bias_corr) {
    bias_corr[0] = 1.0f / one_minus_pow(beta1, t);
    bias_corr[1] = 1.0f / sqrtf(one_minus_pow(beta2, t));
  }
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace mlpk
