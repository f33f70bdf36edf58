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
// Not inlined: the IEEE divide and expf are ~2 KB of code per copy, and the
// kernels that call this are bound by instruction fetch, not by call cost.
static __device__ __noinline__ float sigmoid_acc(float x) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-x)));
}

// g = rT(sigmoid(x)) with exactly the bits of rT(sigmoid_acc(x)), at a
// fraction of the cost. Fast evaluation: 2^t for t = -x*log2(e), with the
// product split as t_hi + t_lo (Cody and Waite's argument reduction: the FMA
// residual of t_hi plus x times the tail of log2(e)), the hardware ex2 and
// reciprocal approximations and one Newton step for the reciprocal. Measured
// over 2^30 points in [-40, 40] it stays within 6 fp32 ulps of sigmoid_acc, so
// rounding it to T gives the same result unless it lies within a few ulps of
// a rounding midpoint of T; there (within kSigWindow = 8 ulps), in T's
// subnormal range, for |x| > 80 (including infinities) and for NaN the
// accurate form is evaluated instead. Its inputs are values of T, so the claim
// is checked on every one of them (hc_debug_sigmoid_exact). The narrower the
// window, the fewer warps take the accurate branch (in the prefill epilogue
// that branch, not the fast form, set the cost of the fp16 gate).
__device__ __forceinline__ float sigmoid_fast_f32(float x) {
  const float kLog2e = 1.44269502f, kLog2eTail = 1.9259630e-08f, kLn2 = 0.69314718f;
  const float nx = -x;
  const float t_hi = __fmul_rn(nx, kLog2e);
  const float t_lo = __fadd_rn(fmaf(nx, kLog2e, -t_hi), __fmul_rn(nx, kLog2eTail));
  float p;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(t_hi));
  const float s = __fadd_rn(1.0f, __fmul_rn(p, fmaf(t_lo, kLn2, 1.0f)));
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return fmaf(r, fmaf(-s, r, 1.0f), r);
}
constexpr int kSigWindow = 8;
template <typename T> struct SigmoidT;
template <> struct SigmoidT<float> {
  static __device__ __forceinline__ float eval(float x) { return sigmoid_acc(x); }
};
template <> struct SigmoidT<__nv_bfloat16> {
  static __device__ __forceinline__ float eval(float x) {
    const float f = sigmoid_fast_f32(x);
    const int lo = static_cast<int>(__float_as_uint(f) & 0xFFFFu) - 0x8000;
    const bool slow = (lo < kSigWindow && lo > -kSigWindow) || !(x >= -80.0f && x <= 80.0f);
    return Ty<__nv_bfloat16>::to_f(Ty<__nv_bfloat16>::from_f(slow ? sigmoid_acc(x) : f));
  }
};
template <> struct SigmoidT<__half> {
  static __device__ __forceinline__ float eval(float x) {
    const float f = sigmoid_fast_f32(x);
    const int lo = static_cast<int>(__float_as_uint(f) & 0x1FFFu) - 0x1000;
    const bool slow = (lo < kSigWindow && lo > -kSigWindow) || !(x >= -80.0f && x <= 80.0f) || f < 6.103515625e-05f;
    return Ty<__half>::to_f(Ty<__half>::from_f(slow ? sigmoid_acc(x) : f));
  }
};
template <typename T> __device__ __forceinline__ float sigmoid_rT(float x) { return SigmoidT<T>::eval(x); }

// Prologue: S = rT(streams + gate * prev), multiply then add, each rounded.
template <typename T> __device__ __forceinline__ float prologue_s(float s, float gate, float prev) {
  return rT<T>(__fadd_rn(s, __fmul_rn(gate, prev)));
}

// RMS statistic: inv = 1 / sqrt(sum / H + eps), correctly rounded steps. The
// last step is the correctly rounded reciprocal, which is the correctly
// rounded quotient 1 / y for every y (infinities, zeros and NaN included),
// with a shorter instruction sequence than the general divide; it sits on
// the decode kernels' critical path.
__device__ __forceinline__ float inv_rms(float sumsq, int H, float eps) {
  const float mean = __fdiv_rn(sumsq, static_cast<float>(H));
  return __frcp_rn(__fsqrt_rn(__fadd_rn(mean, eps)));
}

// hn = rT((S * inv) * norm_scale).
template <typename T> __device__ __forceinline__ float norm_hn(float s, float inv, float ns) {
  return rT<T>(__fmul_rn(__fmul_rn(s, inv), ns));
}

// ScaledSiLU at its three rounding sites: Z = rT(a*x), SG = rT(sigmoid(Z)),
// hidden = rT(x * SG). x is the already-rounded down projection.
template <typename T> __device__ __noinline__ float scaled_silu(float x, float alpha) {
  float z = rT<T>(__fmul_rn(alpha, x));
  float sg = rT<T>(sigmoid_acc(z));
  return rT<T>(__fmul_rn(x, sg));
}

// post_gate = rT(sigmoid(inject / gate_div) * gate_mul), inject already rounded.
template <typename T> __device__ __noinline__ float post_gate_of(float inj, float gate_div, float gate_mul) {
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
