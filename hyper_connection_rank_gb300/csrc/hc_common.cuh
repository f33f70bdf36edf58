// Device helpers shared by the GPU kernels of the low-rank mix block.
//
// Numerics follow ONNX Runtime PR #33384 "HyperConnectionLowRankMix",
// section "Numerics contract": fp32 arithmetic, one round-to-nearest-even to
// the I/O type T at each listed step, and an accurate expf-based sigmoid.
// Where the contract fixes an unfused order (the prologue add, the norm and
// the pre-mix), the _rn intrinsics below keep the compiler from contracting
// a multiply and an add into one FMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hc {

// ---------------------------------------------------------------- types ----

template <typename T> struct Ty;
template <> struct Ty<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Ty<__half> {
  static __device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};
template <> struct Ty<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

template <typename T> __device__ __forceinline__ float ldf(const T* p) { return Ty<T>::to_f(*p); }
template <typename T> __device__ __forceinline__ void stf(T* p, float v) { *p = Ty<T>::from_f(v); }
// Round an fp32 value to T and back: the contract's single rounding step.
template <typename T> __device__ __forceinline__ float rT(float x) { return Ty<T>::to_f(Ty<T>::from_f(x)); }

// --------------------------------------------------------------- numerics --

// sigmoid(x) = 1 / (1 + exp(-x)): CUDA's accurate expf, IEEE add and divide.
__device__ __forceinline__ float sigmoid_acc(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
}

// Prologue: S = rT(streams + gate * prev), multiply then add, each rounded.
template <typename T> __device__ __forceinline__ float prologue_s(float s, float gate, float prev) {
  return rT<T>(__fadd_rn(s, __fmul_rn(gate, prev)));
}

// RMS statistic: inv = 1 / sqrt(sum / H + eps), correctly rounded steps.
__device__ __forceinline__ float inv_rms(float sumsq, int H, float eps) {
  float mean = __fdiv_rn(sumsq, static_cast<float>(H));
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// hn = rT((S * inv) * norm_scale).
template <typename T> __device__ __forceinline__ float norm_hn(float s, float inv, float ns) {
  return rT<T>(__fmul_rn(__fmul_rn(s, inv), ns));
}

// ScaledSiLU at its three rounding sites: Z = rT(a*x), SG = rT(sigmoid(Z)),
// hidden = rT(x * SG). x is the already-rounded down projection.
template <typename T> __device__ __forceinline__ float scaled_silu(float x, float alpha) {
  float z = rT<T>(__fmul_rn(alpha, x));
  float sg = rT<T>(sigmoid_acc(z));
  return rT<T>(__fmul_rn(x, sg));
}

// post_gate = rT(sigmoid(inject / gate_div) * gate_mul), inject already rounded.
template <typename T> __device__ __forceinline__ float post_gate_of(float inj, float gate_div, float gate_mul) {
  return rT<T>(__fmul_rn(sigmoid_acc(__fdiv_rn(inj, gate_div)), gate_mul));
}

struct Attrs {
  float eps, rho, alpha, gate_div, gate_mul;
};

// ---------------------------------------------- programmatic dependent launch

// Wait until the preceding grid on the stream has completed and its writes are
// visible. Returns at once when the launch has no programmatic dependency.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid on the stream to begin launching.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------- reductions --

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block sum in a fixed order: butterfly inside each warp, then warp results
// added in warp order by every thread. `red` holds >= 32 floats. Ends with a
// barrier, so `red` may be reused right after.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.0f;
  for (int w = 0; w < nw; ++w) t += red[w];
  __syncthreads();
  return t;
}

}  // namespace hc
