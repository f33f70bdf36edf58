// General CUDA-core path of the low-rank mix block: any shape, any number of
// rows, any T, any pointer alignment. It plays the role of the operator's
// "general path" (ONNX Runtime PR #33384, "CUDA implementation": norm kernel
// + three GEMMs + elementwise kernels with the same rounding points), written
// here with our own CUDA-core tiles instead of a library GEMM.
//
// Four kernels, each launched with programmatic dependent launch:
//   1. gen_norm   : prologue S (written to streams_out), branch RMS, hn -> workspace
//   2. gen_gemm   : [down | inject] = hn @ [down_weight | inject_weight], rounded -> workspace
//   3. gen_gemm   : up = ScaledSiLU(down) @ up_weight; g = rT(sigmoid(rT(up))) -> workspace
//   4. gen_premix : pre_output = rT(rho * sum_c hn*g), post_gate = rT(sigmoid(inject/div)*mul)
// Every output element is accumulated by one thread in increasing k, so the
// result is deterministic and a row's bits never depend on the row count.
#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {
namespace {

constexpr int kNormThreads = 256;
constexpr int kTileM = 64, kTileN = 64, kTileK = 16, kGemmThreads = 256;

template <typename T>
__device__ __forceinline__ float s_value(const T* streams, const T* prev_out, const T* prev_gate,
                                         int64_t b, int c, int h, int C, int H) {
  float v = ldf(streams + (b * C + c) * H + h);
  if (prev_out != nullptr) v = prologue_s<T>(v, ldf(prev_gate + b * C + c), ldf(prev_out + b * H + h));
  return v;
}

// One CTA per (row, branch).
template <typename T>
__global__ void __launch_bounds__(kNormThreads)
gen_norm(const T* __restrict__ streams, const T* __restrict__ prev_out, const T* __restrict__ prev_gate,
         const T* __restrict__ norm_scale, int C, int H, float eps, T* __restrict__ streams_out,
         T* __restrict__ hn) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[32];
  const int64_t bc = blockIdx.x;
  const int64_t b = bc / C;
  const int c = static_cast<int>(bc % C);
  float ss = 0.0f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float v = s_value(streams, prev_out, prev_gate, b, c, h, C, H);
    if (streams_out != nullptr) {
      if (prev_out != nullptr) stf(streams_out + bc * H + h, v);
      else streams_out[bc * H + h] = streams[bc * H + h];  // bit copy
    }
    ss = fmaf(v, v, ss);
  }
  ss = block_sum(ss, red);
  const float inv = inv_rms(ss, H, eps);
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const float v = s_value(streams, prev_out, prev_gate, b, c, h, C, H);
    stf(hn + bc * H + h, norm_hn<T>(v, inv, ldf(norm_scale + c * H + h)));
  }
}

// C[m, n] = sum_k A(m, k) * B(k, n) in increasing k, one thread per element
// (4x4 elements per thread), then epi(m, n, acc).
template <class A, class B, class E>
__global__ void __launch_bounds__(kGemmThreads) gen_gemm(int M, int N, int K, A a, B bop, E epi) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[kTileK][kTileM + 4];
  __shared__ float Bs[kTileK][kTileN + 4];
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * kTileM, n0 = blockIdx.x * kTileN;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += kTileK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * kGemmThreads;
      const int mm = idx / kTileK, kk = idx % kTileK, m = m0 + mm, k = k0 + kk;
      As[kk][mm] = (m < M && k < K) ? a(m, k) : 0.0f;
      const int kb = idx / kTileN, nn = idx % kTileN, n = n0 + nn, k2 = k0 + kb;
      Bs[kb][nn] = (n < N && k2 < K) ? bop(k2, n) : 0.0f;
    }
    __syncthreads();
    const int kmax = min(kTileK, K - k0);
    for (int kk = 0; kk < kmax; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (m < M && n < N) epi(m, n, acc[i][j]);
    }
}

template <typename T> struct LoadRows {  // row-major [M, ld] of T
  const T* p; int64_t ld;
  __device__ float operator()(int m, int k) const { return ldf(p + m * ld + k); }
};
template <typename T> struct LoadDownInject {  // virtual [C*H, R + C] = [down_weight | inject_weight]
  const T* wd; const T* wi; int R, C;
  __device__ float operator()(int k, int n) const {
    return n < R ? ldf(wd + static_cast<int64_t>(k) * R + n) : ldf(wi + static_cast<int64_t>(k) * C + (n - R));
  }
};
template <typename T> struct StoreRoundedF32 {  // rT(acc) kept as float
  float* p; int64_t ld;
  __device__ void operator()(int m, int n, float v) const { p[m * ld + n] = rT<T>(v); }
};
template <typename T> struct LoadHidden {  // d = ScaledSiLU(down) from the rounded down values
  const float* dz; int64_t ld; float alpha;
  __device__ float operator()(int m, int k) const { return scaled_silu<T>(dz[m * ld + k], alpha); }
};
template <typename T> struct StoreGate {  // g = rT(sigmoid(rT(up)))
  T* g; int64_t ld;
  __device__ void operator()(int m, int n, float v) const { stf(g + m * ld + n, sigmoid_acc(rT<T>(v))); }
};

template <typename T>
__global__ void __launch_bounds__(256)
gen_premix(const T* __restrict__ hn, const T* __restrict__ g, const float* __restrict__ dz, int64_t rows, int C,
           int H, int R, Attrs at, T* __restrict__ pre, T* __restrict__ post) {
  pdl_wait();
  pdl_trigger();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t npre = rows * H;
  if (i < npre) {
    const int64_t b = i / H;
    const int h = static_cast<int>(i % H);
    float acc = 0.0f;
    for (int c = 0; c < C; ++c) {
      const int64_t o = (b * C + c) * H + h;
      acc = __fadd_rn(acc, __fmul_rn(ldf(hn + o), ldf(g + o)));
    }
    stf(pre + i, __fmul_rn(at.rho, acc));
  } else if (i < npre + rows * C) {
    const int64_t j = i - npre;
    const int64_t b = j / C;
    const int c = static_cast<int>(j % C);
    stf(post + j, post_gate_of<T>(dz[b * (R + C) + R + c], at.gate_div, at.gate_mul));
  }
}

struct GenLayout {
  size_t hn, dz, g, total;
};

GenLayout gen_layout(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  const size_t es = dtype_size(dt), CH = static_cast<size_t>(C) * H;
  GenLayout L;
  L.hn = 0;
  L.dz = align_up(L.hn + rows * CH * es, 256);
  L.g = align_up(L.dz + rows * static_cast<size_t>(R + C) * 4, 256);
  L.total = align_up(L.g + rows * CH * es, 256);
  return L;
}

template <typename T>
cudaError_t run_general(const Problem& p) {
  const GenLayout L = gen_layout(p.rows, p.C, p.H, p.R, p.dt);
  char* ws = static_cast<char*>(p.workspace);
  T* hn = reinterpret_cast<T*>(ws + L.hn);
  float* dz = reinterpret_cast<float*>(ws + L.dz);
  T* g = reinterpret_cast<T*>(ws + L.g);
  const int C = p.C, H = p.H, R = p.R, CH = C * H;
  const int64_t rows = p.rows;
  const T* streams = static_cast<const T*>(p.streams);
  cudaError_t e;

  e = launch_pdl(gen_norm<T>, dim3(static_cast<unsigned>(rows * C)), dim3(kNormThreads), 0, p.stream, 1,
                 streams, static_cast<const T*>(p.prev_out), static_cast<const T*>(p.prev_gate),
                 static_cast<const T*>(p.norm_scale), C, H, p.eps, static_cast<T*>(p.streams_out), hn);
  if (e != cudaSuccess) return e;

  const unsigned gm = static_cast<unsigned>((rows + kTileM - 1) / kTileM);
  e = launch_pdl(gen_gemm<LoadRows<T>, LoadDownInject<T>, StoreRoundedF32<T>>,
                 dim3((R + C + kTileN - 1) / kTileN, gm), dim3(kGemmThreads), 0, p.stream, 1,
                 static_cast<int>(rows), R + C, CH, LoadRows<T>{hn, CH},
                 LoadDownInject<T>{static_cast<const T*>(p.down_w), static_cast<const T*>(p.inject_w), R, C},
                 StoreRoundedF32<T>{dz, R + C});
  if (e != cudaSuccess) return e;

  e = launch_pdl(gen_gemm<LoadHidden<T>, LoadRows<T>, StoreGate<T>>,
                 dim3((CH + kTileN - 1) / kTileN, gm), dim3(kGemmThreads), 0, p.stream, 1,
                 static_cast<int>(rows), CH, R, LoadHidden<T>{dz, R + C, p.alpha},
                 LoadRows<T>{static_cast<const T*>(p.up_w), CH}, StoreGate<T>{g, CH});
  if (e != cudaSuccess) return e;

  const int64_t n = rows * (H + C);
  const Attrs at{p.eps, p.rho, p.alpha, p.gate_div, p.gate_mul};
  return launch_pdl(gen_premix<T>, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, p.stream, 1,
                    static_cast<const T*>(hn), static_cast<const T*>(g), static_cast<const float*>(dz), rows,
                    C, H, R, at, static_cast<T*>(p.pre_output), static_cast<T*>(p.post_gate));
}

}  // namespace

size_t general_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  return gen_layout(rows, C, H, R, dt).total;
}

cudaError_t launch_general(const Problem& p) {
  switch (p.dt) {
    case HC_F32: return run_general<float>(p);
    case HC_F16: return run_general<__half>(p);
    default: return run_general<__nv_bfloat16>(p);
  }
}

}  // namespace hc
