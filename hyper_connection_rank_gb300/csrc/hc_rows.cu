// Row-reduction kernels of the two companion operations:
//
//   inv_rms      FreeToken PR #101, "perf(dsv4): compute the hyper-connection
//                pre-norm in one kernel" ("The problem", "The change"):
//                out[r] = 1 / sqrt(mean_i(x[r, i]^2) + eps), read once from
//                the 16-bit (or fp32) source, fp32 accumulation, one fp32
//                scalar per row.
//   engram_gate  com.microsoft.EngramGate (its kernel README, "Description"):
//                per row (b, m) the squares of key and query and the scaled
//                cross term sum((key * key_scale[m]) * (query * query_scale[m]))
//                accumulate in one fp32 pass; then
//                dot  = cross * ik * iq / sqrt(D), ik = 1/sqrt(mean(key^2) + eps),
//                gate = sigmoid(sign(dot) * sqrt(max(|dot|, 1e-6))),
//                out[b, m, :] = gate * value[b, :], narrowed to T at the store.
//
// Both are bound by HBM reads. A group of G threads reduces one row (G = 32:
// one warp, eight rows per CTA, for short rows; G = 256: the whole CTA for
// long rows). Every thread issues eight 16-byte loads before it reduces any of
// them. Sums are pairwise within a vector and across a thread's vectors, then
// a warp-shuffle tree and a tree over the CTA's warps: for a 16384-wide row
// the depth is about 15 additions, so the relative error of a sum of squares
// is below 16 fp32 unit roundoffs. Divides and square roots are the correctly
// rounded ones.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_vec.cuh"

namespace hc {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowUnroll = 8;

// A 16-byte vector of T as floats: 8 elements of a 16-bit type, 4 of fp32.
template <typename T> struct Vec16 {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) { V8<T>::unpack(u, f); }
};
template <> struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void unpack(const uint4& u, float* f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

// Pairwise sum of the squares of n (4 or 8) floats.
template <int N> __device__ __forceinline__ float sumsq(const float* f) {
  float p[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) p[i] = fmaf(f[2 * i], f[2 * i], __fmul_rn(f[2 * i + 1], f[2 * i + 1]));
  if constexpr (N == 8) return __fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3]));
  else return __fadd_rn(p[0], p[1]);
}

// Pairwise sum of a thread's kRowUnroll partials.
__device__ __forceinline__ float tree8(const float* p) {
  return __fadd_rn(__fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3])),
                   __fadd_rn(__fadd_rn(p[4], p[5]), __fadd_rn(p[6], p[7])));
}

// Sum of `v` over the G threads of a group (G = 32 or kRowThreads); every
// thread of the group gets the sum. `red` holds kRowThreads / 32 floats per value.
template <int G, int NV>
__device__ __forceinline__ void group_sum(float (&v)[NV], float (*red)[kRowThreads / 32]) {
#pragma unroll
  for (int j = 0; j < NV; ++j) v[j] = warp_sum(v[j]);
  if (G > 32) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
#pragma unroll
      for (int j = 0; j < NV; ++j) red[j][warp] = v[j];
    __syncthreads();
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      // tree over the eight warps
      const float* r = red[j];
      v[j] = __fadd_rn(__fadd_rn(__fadd_rn(r[0], r[1]), __fadd_rn(r[2], r[3])),
                       __fadd_rn(__fadd_rn(r[4], r[5]), __fadd_rn(r[6], r[7])));
    }
  }
}

// out[0 .. VE) = T(gate * value vector u)
template <typename T> __device__ __forceinline__ void store_gated(T* dst, const uint4& u, float gate) {
  constexpr int VE = Vec16<T>::N;
  float f[VE];
  Vec16<T>::unpack(u, f);
  if constexpr (VE == 8) {
    float o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = __fmul_rn(gate, f[e]);
    st16(dst, V8<T>::pack(o));
  } else {
    st16(dst, make_uint4(__float_as_uint(__fmul_rn(gate, f[0])), __float_as_uint(__fmul_rn(gate, f[1])),
                         __float_as_uint(__fmul_rn(gate, f[2])), __float_as_uint(__fmul_rn(gate, f[3]))));
  }
}

// ---------------------------------------------------------------- inv_rms --

template <typename T, int G>
__global__ void __launch_bounds__(kRowThreads) inv_rms_kernel(const T* __restrict__ x, int64_t rows, int64_t dim,
                                                               float eps, float* __restrict__ out, int vec) {
  __shared__ float red[1][kRowThreads / 32];
  constexpr int VE = Vec16<T>::N;
  const int t = threadIdx.x % G;
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (kRowThreads / G) + threadIdx.x / G;
  float acc[1] = {0.0f};
  if (r < rows) {
    const T* xr = x + r * dim;
    if (vec) {
      const int64_t nv = dim / VE;
      for (int64_t v0 = t; v0 < nv; v0 += kRowUnroll * G) {
        uint4 u[kRowUnroll];
#pragma unroll
        for (int j = 0; j < kRowUnroll; ++j) {
          const int64_t v = v0 + j * G;
          u[j] = v < nv ? ld16(xr + v * VE) : make_uint4(0u, 0u, 0u, 0u);
        }
        float p[kRowUnroll];
#pragma unroll
        for (int j = 0; j < kRowUnroll; ++j) {
          float f[VE];
          Vec16<T>::unpack(u[j], f);
          p[j] = sumsq<VE>(f);
        }
        acc[0] = __fadd_rn(acc[0], tree8(p));
      }
    } else {
      for (int64_t i = t; i < dim; i += G) {
        const float v = ldf(xr + i);
        acc[0] = fmaf(v, v, acc[0]);
      }
    }
  }
  group_sum<G>(acc, red);
  if (t == 0 && r < rows) {
    const float mean = __fdiv_rn(acc[0], static_cast<float>(dim));
    out[r] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
  }
}

// ------------------------------------------------------------ engram_gate --

// Every load a row needs is issued before any is used: U vectors each of
// key, query, the two scale rows and the value row per thread and round, so
// a row costs one memory round trip (the value vectors of the first round
// stay in registers for the output pass; longer rows load the rest again).
template <typename T, int G>
__global__ void __launch_bounds__(kRowThreads)
engram_gate_kernel(const T* __restrict__ key, const T* __restrict__ query, const T* __restrict__ value,
                   const T* __restrict__ kscale, const T* __restrict__ qscale, int64_t nrows, int M, int64_t D,
                   float eps, T* __restrict__ out, int vec) {
  __shared__ float red[3][kRowThreads / 32];
  constexpr int VE = Vec16<T>::N;
  constexpr int U = 2;  // vectors per tensor per thread and round
  const int t = threadIdx.x % G;
  const int64_t rr = static_cast<int64_t>(blockIdx.x) * (kRowThreads / G) + threadIdx.x / G;
  const bool live = rr < nrows;
  const int64_t b = live ? rr / M : 0;
  const int m = live ? static_cast<int>(rr - b * M) : 0;
  const T* vr = value + b * D;
  float acc[3] = {0.0f, 0.0f, 0.0f};  // sum key^2, sum query^2, sum (key ks)(query qs)
  uint4 held[U];                      // value vectors of the first round
  const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
  if (live) {
    const T* kr = key + rr * D;
    const T* qr = query + rr * D;
    const T* ksr = kscale + static_cast<int64_t>(m) * D;
    const T* qsr = qscale + static_cast<int64_t>(m) * D;
    if (vec) {
      const int64_t nv = D / VE;
      for (int64_t v0 = t; v0 < nv; v0 += U * G) {
        uint4 uk[U], uq[U], zk[U], zq[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int64_t v = v0 + j * G;
          const bool in = v < nv;
          uk[j] = in ? ld16(kr + v * VE) : z4;
          uq[j] = in ? ld16(qr + v * VE) : z4;
          zk[j] = in ? ld16(ksr + v * VE) : z4;
          zq[j] = in ? ld16(qsr + v * VE) : z4;
          if (v0 == t) held[j] = in ? ld16(vr + v * VE) : z4;
        }
        float pk[U], pq[U], pc[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
          float fk[VE], fq[VE], sk[VE], sq[VE];
          Vec16<T>::unpack(uk[j], fk);
          Vec16<T>::unpack(uq[j], fq);
          Vec16<T>::unpack(zk[j], sk);
          Vec16<T>::unpack(zq[j], sq);
          pk[j] = sumsq<VE>(fk);
          pq[j] = sumsq<VE>(fq);
          // cross term: (key * ks) * (query * qs), the last product fused into
          // the pairwise sum (two accumulators, added at the end)
          float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
          for (int e = 0; e < VE; e += 2) {
            s0 = fmaf(__fmul_rn(fk[e], sk[e]), __fmul_rn(fq[e], sq[e]), s0);
            s1 = fmaf(__fmul_rn(fk[e + 1], sk[e + 1]), __fmul_rn(fq[e + 1], sq[e + 1]), s1);
          }
          pc[j] = __fadd_rn(s0, s1);
        }
        acc[0] = __fadd_rn(acc[0], __fadd_rn(pk[0], pk[1]));
        acc[1] = __fadd_rn(acc[1], __fadd_rn(pq[0], pq[1]));
        acc[2] = __fadd_rn(acc[2], __fadd_rn(pc[0], pc[1]));
      }
    } else {
      for (int64_t i = t; i < D; i += G) {
        const float k = ldf(kr + i), q = ldf(qr + i);
        acc[0] = fmaf(k, k, acc[0]);
        acc[1] = fmaf(q, q, acc[1]);
        acc[2] = __fadd_rn(acc[2], __fmul_rn(__fmul_rn(k, ldf(ksr + i)), __fmul_rn(q, ldf(qsr + i))));
      }
    }
  }
  group_sum<G>(acc, red);
  if (!live) return;
  const float fd = static_cast<float>(D);
  const float ik = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc[0], fd), eps)));
  const float iq = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc[1], fd), eps)));
  const float dot = __fdiv_rn(__fmul_rn(__fmul_rn(acc[2], ik), iq), __fsqrt_rn(fd));
  // sign(0) = 0: a zero dot product gives exactly sigmoid(0) = 1/2
  const float sgn = dot > 0.0f ? 1.0f : (dot < 0.0f ? -1.0f : 0.0f);
  const float z = __fmul_rn(sgn, __fsqrt_rn(fmaxf(fabsf(dot), 1e-6f)));
  const float gate = sigmoid_acc(z);
  T* orow = out + rr * D;
  if (vec) {
    const int64_t nv = D / VE;
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int64_t v = t + j * G;
      if (v < nv) store_gated<T>(orow + v * VE, held[j], gate);
    }
    for (int64_t v = t + U * G; v < nv; v += G) store_gated<T>(orow + v * VE, ld16(vr + v * VE), gate);
  } else {
    for (int64_t i = t; i < D; i += G) stf(orow + i, __fmul_rn(gate, ldf(vr + i)));
  }
}

template <typename T>
cudaError_t launch_inv_rms_t(const void* x, int64_t rows, int64_t dim, float eps, float* out, bool vec,
                             cudaStream_t s) {
  const T* xp = static_cast<const T*>(x);
  if (dim >= 4096) {
    inv_rms_kernel<T, kRowThreads><<<static_cast<unsigned>(rows), kRowThreads, 0, s>>>(xp, rows, dim, eps, out, vec);
  } else {
    const unsigned grid = static_cast<unsigned>((rows + kRowThreads / 32 - 1) / (kRowThreads / 32));
    inv_rms_kernel<T, 32><<<grid, kRowThreads, 0, s>>>(xp, rows, dim, eps, out, vec);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_engram_t(const EngramProblem& p) {
  const int64_t nrows = p.rows * p.M;
  const T* k = static_cast<const T*>(p.key);
  const T* q = static_cast<const T*>(p.query);
  const T* v = static_cast<const T*>(p.value);
  const T* ks = static_cast<const T*>(p.key_scale);
  const T* qs = static_cast<const T*>(p.query_scale);
  T* o = static_cast<T*>(p.output);
  const int vec = p.vec ? 1 : 0;
  if (p.D >= 2048) {
    engram_gate_kernel<T, kRowThreads><<<static_cast<unsigned>(nrows), kRowThreads, 0, p.stream>>>(
        k, q, v, ks, qs, nrows, p.M, p.D, p.eps, o, vec);
  } else {
    const unsigned grid = static_cast<unsigned>((nrows + kRowThreads / 32 - 1) / (kRowThreads / 32));
    engram_gate_kernel<T, 32><<<grid, kRowThreads, 0, p.stream>>>(k, q, v, ks, qs, nrows, p.M, p.D, p.eps, o, vec);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_inv_rms(const void* x, int64_t rows, int64_t dim, float eps, hc_dtype_t dt, float* out, bool vec,
                           cudaStream_t s) {
  switch (dt) {
    case HC_F32: return launch_inv_rms_t<float>(x, rows, dim, eps, out, vec, s);
    case HC_F16: return launch_inv_rms_t<__half>(x, rows, dim, eps, out, vec, s);
    default: return launch_inv_rms_t<__nv_bfloat16>(x, rows, dim, eps, out, vec, s);
  }
}

cudaError_t launch_engram_gate(const EngramProblem& p) {
  switch (p.dt) {
    case HC_F32: return launch_engram_t<float>(p);
    case HC_F16: return launch_engram_t<__half>(p);
    default: return launch_engram_t<__nv_bfloat16>(p);
  }
}

}  // namespace hc
