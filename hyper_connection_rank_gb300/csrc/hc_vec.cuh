// 16-byte vector loads and stores of fp16 / bf16 and the ScaledSiLU with the
// fast exact sigmoid, shared by the fp16 / bf16 decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "hc_common.cuh"

namespace hc {

// 16-byte vectors of T <-> 8 floats. bf16 widens by a shift: the value is the
// top half of an fp32 word.
template <typename T> struct V8;
template <> struct V8<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(q[i] << 16);
      f[2 * i + 1] = __uint_as_float(q[i] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
  }
};
template <> struct V8<__half> {
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __half22float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* f) {
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return u;
  }
};

template <typename T> __device__ __forceinline__ uint4 ld16(const T* p) { return *reinterpret_cast<const uint4*>(p); }
template <typename T> __device__ __forceinline__ void st16(T* p, const uint4& u) { *reinterpret_cast<uint4*>(p) = u; }

// ScaledSiLU at its three rounding sites, with the sigmoid evaluated by the
// fast form that reproduces rT(sigmoid_acc(z)) bit for bit (its input z is
// already a value of T).
template <typename T> __device__ __forceinline__ float scaled_silu_t(float x, float alpha) {
  const float z = rT<T>(__fmul_rn(alpha, x));
  const float sg = sigmoid_rT<T>(z);
  return rT<T>(__fmul_rn(x, sg));
}

}  // namespace hc
