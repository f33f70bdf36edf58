// Decode path of the low-rank mix block (rows <= 8): two weight-streaming
// kernels linked by programmatic dependent launch.
//
// The block at decode sizes is bound by reading its weights once: down_weight
// (C*H x R) and up_weight (R x C*H) are 13.2 MB in bf16 at C=4, H=2560,
// R=320, against ~50 KB of activations per row. The operator's own fused path
// (ONNX Runtime PR #33384, "CUDA implementation": HcDownKernel + HcUpPreKernel,
// K split in slices inside one branch, fp32 partials, fixed-order reduction,
// no atomics, PDL) is the prior art; this design keeps its split but uses
// sm_100-class features for the plumbing:
//
//   dec_down (grid = C*H/KS CTAs, clusters of CL CTAs inside one branch)
//     - bulk-copies its contiguous KS-row slice of down_weight and
//       inject_weight into shared memory (before griddepcontrol.wait when the
//       weights are static, so the stream overlaps the previous kernel);
//     - computes the branch RMS statistic cooperatively: each cluster rank
//       sums S^2 over 1/CL of the branch and the partial sums are exchanged
//       through distributed shared memory, then added in rank order;
//     - forms hn for its slice, writes streams_out for it, runs the split-K
//       GEMV for down and inject, and reduces the CL partial vectors of its
//       cluster through DSMEM in rank order into one fp32 partial per cluster.
//   dec_up (grid = (H/HS)*C CTAs, clusters of C CTAs, one per branch)
//     - bulk-copies its up_weight tile (R rows x HS columns of branch c) and
//       loads S for its tile before griddepcontrol.wait;
//     - reduces the down partials (each rank 1/C of the R columns, partials
//       added in cluster order), applies ScaledSiLU, and broadcasts d to the
//       cluster through DSMEM;
//     - runs the up GEMV, the sigmoid and the hn*g products, and sums the
//       products over the branches in order 0..C-1 through DSMEM for the
//       pre-mix; one CTA also writes post_gate.
//
// All reductions have a fixed order that depends on the shape only, so the
// results are deterministic and a row's bits do not depend on the row count.
#include <cooperative_groups.h>

#include "hc_async.cuh"
#include "hc_common.cuh"
#include "hc_internal.h"

namespace cg = cooperative_groups;

namespace hc {

// Count of bounded waits that gave up (diagnostic; see hc_debug_wait_timeouts).
__device__ unsigned int g_wait_timeouts = 0;

namespace {

constexpr int kUpThreads = 256;

// 16-byte vector of T from shared memory, widened to fp32.
template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const unsigned char* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
};
template <> struct Vec<__half> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const unsigned char* p, float* out) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const unsigned char* p, float* out) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    out[0] = f.x; out[1] = f.y; out[2] = f.z; out[3] = f.w;
  }
};

__host__ __device__ inline uint32_t a16(uint32_t x) { return (x + 15u) & ~15u; }

// Shared-memory layout of dec_down (byte offsets), for MB rows.
struct DownSmem {
  uint32_t bar, wd, wi, hn, wsum, ssq, inv, red, part, total;
};
__host__ __device__ inline DownSmem down_smem(int MB, int KS, int R, int C, int CL, int nwarps, int es) {
  DownSmem L;
  L.bar = 0;
  L.wd = 16;
  L.wi = a16(L.wd + KS * R * es);
  L.hn = a16(L.wi + KS * C * es);
  L.wsum = a16(L.hn + MB * KS * 4);
  L.ssq = a16(L.wsum + nwarps * MB * 4);
  L.inv = a16(L.ssq + CL * MB * 4);
  L.red = a16(L.inv + MB * 4);
  L.part = a16(L.red + MB * R * 4);
  L.total = a16(L.part + MB * (R + C) * 4);
  return L;
}

// Shared-memory layout of dec_up (byte offsets), for MB rows.
struct UpSmem {
  uint32_t bar, wu, s, ns, d, red, mix, total;
};
__host__ __device__ inline UpSmem up_smem(int MB, int HS, int R, int nwarps, int es) {
  UpSmem L;
  L.bar = 0;
  L.wu = 16;
  L.s = a16(L.wu + R * HS * es);
  L.ns = a16(L.s + MB * HS * 4);
  L.d = a16(L.ns + HS * 4);
  L.red = a16(L.d + MB * R * 4);
  L.mix = a16(L.red + nwarps * MB * HS * 4);
  L.total = a16(L.mix + MB * HS * 4);
  return L;
}

template <typename T>
struct DownArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wd, *wi;
  T* sout;
  float* inv_ws;   // (B, C)
  float* part_ws;  // (NCLU, B, R + C)
  int B, C, H, R, KS, CL, KQ;
  float eps;
  int weights_static;
};

template <typename T>
struct UpArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wu;
  const float* inv_ws;
  const float* part_ws;
  T *pre, *post;
  int B, C, H, R, HS, NP;
  Attrs at;
};

// S(b, c, h) of the prologue, recomputed wherever it is needed (same bits).
template <typename T>
__device__ __forceinline__ float s_at(const T* streams, const T* prev_out, const T* prev_gate, int b, int c,
                                      int h, int C, int H) {
  const int64_t CH = static_cast<int64_t>(C) * H;
  float v = ldf(streams + b * CH + static_cast<int64_t>(c) * H + h);
  if (prev_out != nullptr) v = prologue_s<T>(v, ldf(prev_gate + b * C + c), ldf(prev_out + static_cast<int64_t>(b) * H + h));
  return v;
}

template <typename T, int MB>
__global__ void __launch_bounds__(512) dec_down(const DownArgs<T> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int VEC = Vec<T>::N;
  constexpr int es = sizeof(T);
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  const int B = a.B, C = a.C, H = a.H, R = a.R, KS = a.KS, CL = a.CL, NC = R + C;
  const DownSmem L = down_smem(MB, KS, R, C, CL, nwarps, es);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  unsigned char* wd_s = smem + L.wd;
  const T* wi_s = reinterpret_cast<const T*>(smem + L.wi);
  float* hn_s = reinterpret_cast<float*>(smem + L.hn);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  float* ssq_s = reinterpret_cast<float*>(smem + L.ssq);
  float* inv_s = reinterpret_cast<float*>(smem + L.inv);
  float* red_s = reinterpret_cast<float*>(smem + L.red);
  float* part_s = reinterpret_cast<float*>(smem + L.part);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int slice = blockIdx.x;
  const int k0 = slice * KS;
  const int c = k0 / H, hk0 = k0 - c * H;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const uint32_t wbytes = static_cast<uint32_t>(KS * R * es), ibytes = static_cast<uint32_t>(KS * C * es);
  const bool pro = a.prev_out != nullptr;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (a.weights_static && tid == 0) {
    mbar_arrive_expect_tx(bar, wbytes + ibytes);
    bulk_g2s(wd_s, a.wd + static_cast<int64_t>(k0) * R, wbytes, bar);
    bulk_g2s(smem + L.wi, a.wi + static_cast<int64_t>(k0) * C, ibytes, bar);
  }
  pdl_wait();
  if (!a.weights_static && tid == 0) {
    mbar_arrive_expect_tx(bar, wbytes + ibytes);
    bulk_g2s(wd_s, a.wd + static_cast<int64_t>(k0) * R, wbytes, bar);
    bulk_g2s(smem + L.wi, a.wi + static_cast<int64_t>(k0) * C, ibytes, bar);
  }
  pdl_trigger();

  // ---- branch RMS: this rank sums S^2 over its 1/CL of branch c ----
  const int hc = H / CL, hlo = rank * hc;
  float ss[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) ss[b] = 0.0f;
  for (int h = hlo + tid; h < hlo + hc; h += nthr) {
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B) {
        const float v = s_at(a.streams, a.prev_out, a.prev_gate, b, c, h, C, H);
        ss[b] = fmaf(v, v, ss[b]);
      }
  }
#pragma unroll
  for (int b = 0; b < MB; ++b) {
    const float w = warp_sum(ss[b]);
    if (lane == 0) wsum[warp * MB + b] = w;
  }
  __syncthreads();
  if (tid < B) {
    float t = 0.0f;
    for (int w = 0; w < nwarps; ++w) t += wsum[w * MB + tid];
    for (int pr = 0; pr < CL; ++pr) cluster.map_shared_rank(ssq_s, pr)[rank * MB + tid] = t;
  }
  cluster.sync();
  if (tid < B) {
    float t = 0.0f;
    for (int r = 0; r < CL; ++r) t += ssq_s[r * MB + tid];
    const float iv = inv_rms(t, H, a.eps);
    inv_s[tid] = iv;
    if (hk0 == 0) a.inv_ws[tid * C + c] = iv;
  }
  __syncthreads();

  // ---- hn for this slice; streams_out for this slice ----
  for (int i = tid; i < B * KS; i += nthr) {
    const int b = i / KS, kk = i - b * KS;
    const float v = s_at(a.streams, a.prev_out, a.prev_gate, b, c, hk0 + kk, C, H);
    if (a.sout != nullptr) {
      const int64_t o = b * CH + k0 + kk;
      if (pro) stf(a.sout + o, v);
      else a.sout[o] = a.streams[o];
    }
    hn_s[b * KS + kk] = norm_hn<T>(v, inv_s[b], ldf(a.ns + k0 + kk));
  }
  __syncthreads();
  const bool ok = mbar_wait(bar, 0, &g_wait_timeouts);

  // ---- split-K GEMV over the slice: lanes 0..7 of a quarter-warp read one
  // 128-byte run of a weight row (conflict-free); 4 k-groups per warp ----
  const int NV = R / VEC, NVB = (NV + 7) / 8;
  const int vb = warp % NVB, kq = warp / NVB;
  const int v = vb * 8 + (lane & 7);
  const int kg = kq * 4 + (lane >> 3);
  const int rpk = KS / (4 * a.KQ);
  float acc[MB][VEC];
#pragma unroll
  for (int b = 0; b < MB; ++b)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[b][j] = 0.0f;
  if (ok && kq < a.KQ && v < NV) {
    const unsigned char* wrow = wd_s + static_cast<size_t>(kg * rpk) * R * es + v * 16;
    for (int i = 0; i < rpk; ++i) {
      float w[VEC];
      Vec<T>::load(wrow + static_cast<size_t>(i) * R * es, w);
      const int kk = kg * rpk + i;
#pragma unroll
      for (int b = 0; b < MB; ++b)
        if (b < B) {
          const float hv = hn_s[b * KS + kk];
#pragma unroll
          for (int j = 0; j < VEC; ++j) acc[b][j] = fmaf(hv, w[j], acc[b][j]);
        }
    }
  }
#pragma unroll
  for (int b = 0; b < MB; ++b)
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      acc[b][j] += __shfl_xor_sync(0xffffffffu, acc[b][j], 8);
      acc[b][j] += __shfl_xor_sync(0xffffffffu, acc[b][j], 16);
    }
  const bool leader = (lane >> 3) == 0 && v < NV && kq < a.KQ;
  if (a.KQ == 2 && kq == 1 && leader) {
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B)
#pragma unroll
        for (int j = 0; j < VEC; ++j) red_s[b * R + v * VEC + j] = acc[b][j];
  }
  __syncthreads();
  if (kq == 0 && leader) {
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B)
#pragma unroll
        for (int j = 0; j < VEC; ++j) {
          float t = acc[b][j];
          if (a.KQ == 2) t += red_s[b * R + v * VEC + j];
          part_s[b * NC + v * VEC + j] = ok ? t : __int_as_float(0x7fc00000);
        }
  }
  // inject: KS-term dot products, one thread per (row, branch)
  for (int i = tid; i < B * C; i += nthr) {
    const int b = i / C, cc = i - b * C;
    float t = 0.0f;
    if (ok)
      for (int kk = 0; kk < KS; ++kk) t = fmaf(hn_s[b * KS + kk], ldf(wi_s + kk * C + cc), t);
    part_s[b * NC + R + cc] = ok ? t : __int_as_float(0x7fc00000);
  }
  cluster.sync();

  // ---- cluster reduction of the partial vectors, in rank order ----
  const int ncr = (NC + CL - 1) / CL, clo = rank * ncr, chi = min(NC, clo + ncr), nmine = max(0, chi - clo);
  const int cluster_id = slice / CL;
  for (int i = tid; i < B * nmine; i += nthr) {
    const int b = i / nmine, col = clo + (i - b * nmine);
    float t = 0.0f;
    for (int r = 0; r < CL; ++r) t += cluster.map_shared_rank(part_s, r)[b * NC + col];
    a.part_ws[(static_cast<int64_t>(cluster_id) * B + b) * NC + col] = t;
  }
  cluster.sync();  // keep this CTA's shared memory alive until every peer has read it
}

template <typename T, int MB>
__global__ void __launch_bounds__(kUpThreads) dec_up(const UpArgs<T> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int VEC = Vec<T>::N;
  constexpr int es = sizeof(T);
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  const int B = a.B, C = a.C, H = a.H, R = a.R, HS = a.HS, NC = R + C;
  const UpSmem L = up_smem(MB, HS, R, nwarps, es);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  unsigned char* wu_s = smem + L.wu;
  float* s_s = reinterpret_cast<float*>(smem + L.s);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* d_s = reinterpret_cast<float*>(smem + L.d);
  float* red_s = reinterpret_cast<float*>(smem + L.red);
  float* mix_s = reinterpret_cast<float*>(smem + L.mix);

  cg::cluster_group cluster = cg::this_cluster();
  const int c = static_cast<int>(cluster.block_rank());
  const int q = blockIdx.x / C;
  const int h0 = q * HS;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const int64_t col0 = static_cast<int64_t>(c) * H + h0;
  const uint32_t rowbytes = static_cast<uint32_t>(HS * es);

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // The up weights and the block inputs are never written by the preceding
  // dec_down, which triggers its dependents only after its own wait: reading
  // them before griddepcontrol.wait is safe.
  if (tid == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(R) * rowbytes);
  __syncwarp();
  if (warp == 0)
    for (int r = lane; r < R; r += 32) bulk_g2s(wu_s + static_cast<size_t>(r) * rowbytes, a.wu + r * CH + col0, rowbytes, bar);
  for (int i = tid; i < B * HS; i += nthr) {
    const int b = i / HS, h = i - b * HS;
    s_s[i] = s_at(a.streams, a.prev_out, a.prev_gate, b, c, h0 + h, C, H);
  }
  for (int i = tid; i < HS; i += nthr) ns_s[i] = ldf(a.ns + col0 + i);
  pdl_wait();
  pdl_trigger();
  __syncthreads();

  // ---- down partials -> d for this rank's share of R, broadcast to the cluster
  const int rc = (R + C - 1) / C, rlo = c * rc, rhi = min(R, rlo + rc), nr = max(0, rhi - rlo);
  for (int i = tid; i < B * nr; i += nthr) {
    const int b = i / nr, r = rlo + (i - b * nr);
    float t = 0.0f;
    for (int p = 0; p < a.NP; ++p) t += a.part_ws[(static_cast<int64_t>(p) * B + b) * NC + r];
    const float d = scaled_silu<T>(rT<T>(t), a.at.alpha);
    for (int pr = 0; pr < C; ++pr) cluster.map_shared_rank(d_s, pr)[b * R + r] = d;
  }
  if (q == 0 && c == 0) {
    for (int i = tid; i < B * C; i += nthr) {
      const int b = i / C, cc = i - b * C;
      float t = 0.0f;
      for (int p = 0; p < a.NP; ++p) t += a.part_ws[(static_cast<int64_t>(p) * B + b) * NC + R + cc];
      stf(a.post + b * C + cc, post_gate_of<T>(rT<T>(t), a.at.gate_div, a.at.gate_mul));
    }
  }
  // hn of this tile, in place
  for (int i = tid; i < B * HS; i += nthr) {
    const int b = i / HS, h = i - b * HS;
    s_s[i] = norm_hn<T>(s_s[i], a.inv_ws[b * C + c], ns_s[h]);
  }
  cluster.sync();
  const bool ok = mbar_wait(bar, 0, &g_wait_timeouts);

  // ---- up GEMV: NVh lanes cover one row of the tile, rows strided over groups
  const int NVh = HS / VEC;
  const int lv = lane % NVh, rgw = lane / NVh, RGW = 32 / NVh, RG = nwarps * RGW;
  const int rg = warp * RGW + rgw;
  float acc[MB][VEC];
#pragma unroll
  for (int b = 0; b < MB; ++b)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[b][j] = 0.0f;
  if (ok) {
    for (int r = rg; r < R; r += RG) {
      float w[VEC];
      Vec<T>::load(wu_s + static_cast<size_t>(r) * rowbytes + lv * 16, w);
#pragma unroll
      for (int b = 0; b < MB; ++b)
        if (b < B) {
          const float dv = d_s[b * R + r];
#pragma unroll
          for (int j = 0; j < VEC; ++j) acc[b][j] = fmaf(dv, w[j], acc[b][j]);
        }
    }
  }
  for (int o = NVh; o < 32; o <<= 1)
#pragma unroll
    for (int b = 0; b < MB; ++b)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[b][j] += __shfl_xor_sync(0xffffffffu, acc[b][j], o);
  if (rgw == 0) {
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B)
#pragma unroll
        for (int j = 0; j < VEC; ++j) red_s[(warp * MB + b) * HS + lv * VEC + j] = acc[b][j];
  }
  __syncthreads();

  // ---- up -> g -> hn*g, sent to the rank that finalises that feature
  const int HSc = HS / C;
  for (int i = tid; i < B * HS; i += nthr) {
    const int b = i / HS, h = i - b * HS;
    float u = 0.0f;
    for (int w = 0; w < nwarps; ++w) u += red_s[(w * MB + b) * HS + h];
    const float g = rT<T>(sigmoid_acc(rT<T>(u)));
    const float prod = ok ? __fmul_rn(s_s[i], g) : __int_as_float(0x7fc00000);
    const int j = h / HSc, hl = h - j * HSc;
    cluster.map_shared_rank(mix_s, j)[(c * MB + b) * HSc + hl] = prod;
  }
  cluster.sync();
  for (int i = tid; i < B * HSc; i += nthr) {
    const int b = i / HSc, hl = i - b * HSc;
    float acc2 = 0.0f;
    for (int cc = 0; cc < C; ++cc) acc2 = __fadd_rn(acc2, mix_s[(cc * MB + b) * HSc + hl]);
    stf(a.pre + static_cast<int64_t>(b) * H + h0 + c * HSc + hl, __fmul_rn(a.at.rho, acc2));
  }
}

struct DecodeCfg {
  bool ok;
  int KS, NSL, CL, NCLU, KQ, down_threads, HS, up_threads;
};

DecodeCfg decode_cfg(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  DecodeCfg g{};
  g.ok = false;
  const int es = static_cast<int>(dtype_size(dt)), VEC = 16 / es;
  if (rows < 1 || rows > 8) return g;
  if (!(C == 1 || C == 2 || C == 4 || C == 8)) return g;
  if (R < VEC || R % VEC != 0 || R > 512) return g;
  if (H % 16 != 0 || H > 16384) return g;
  const int CH = C * H;
  // down: the largest slice that still gives at least one CTA per SM
  g.KS = 0;
  for (int ks : {64, 32, 16})
    if (H % ks == 0 && CH / ks >= num_sms) { g.KS = ks; break; }
  if (g.KS == 0) g.KS = 16;
  g.NSL = CH / g.KS;
  g.CL = 1;
  for (int cl : {8, 4, 2})
    if ((H / g.KS) % cl == 0) { g.CL = cl; break; }
  g.NCLU = g.NSL / g.CL;
  const int NV = R / VEC, NVB = (NV + 7) / 8;
  g.KQ = (NVB * 64 <= 512) ? 2 : 1;
  g.down_threads = NVB * 32 * g.KQ;
  // up: the widest tile that still gives at least one CTA per SM
  g.HS = 0;
  for (int hs : {64, 32, 16})
    if (H % hs == 0 && hs % C == 0 && (H / hs) * C >= num_sms) { g.HS = hs; break; }
  if (g.HS == 0) g.HS = 16;
  if ((g.HS / VEC) < 2 || 32 % (g.HS / VEC) != 0) return g;
  g.up_threads = kUpThreads;
  g.ok = true;
  return g;
}

struct DecLayout {
  size_t inv, part, total;
};
DecLayout dec_layout(int64_t rows, int C, int R, const DecodeCfg& g) {
  DecLayout L;
  L.inv = 0;
  L.part = align_up(static_cast<size_t>(rows) * C * 4, 256);
  L.total = align_up(L.part + static_cast<size_t>(g.NCLU) * rows * (R + C) * 4, 256);
  return L;
}

template <typename T, int MB>
cudaError_t run_decode_mb(const Problem& p, const DecodeCfg& g) {
  const int es = sizeof(T);
  const DecLayout WL = dec_layout(p.rows, p.C, p.R, g);
  char* ws = static_cast<char*>(p.workspace);
  float* inv_ws = reinterpret_cast<float*>(ws + WL.inv);
  float* part_ws = reinterpret_cast<float*>(ws + WL.part);

  DownArgs<T> da;
  da.streams = static_cast<const T*>(p.streams);
  da.prev_out = static_cast<const T*>(p.prev_out);
  da.prev_gate = static_cast<const T*>(p.prev_gate);
  da.ns = static_cast<const T*>(p.norm_scale);
  da.wd = static_cast<const T*>(p.down_w);
  da.wi = static_cast<const T*>(p.inject_w);
  da.sout = static_cast<T*>(p.streams_out);
  da.inv_ws = inv_ws;
  da.part_ws = part_ws;
  da.B = static_cast<int>(p.rows);
  da.C = p.C; da.H = p.H; da.R = p.R; da.KS = g.KS; da.CL = g.CL; da.KQ = g.KQ;
  da.eps = p.eps;
  da.weights_static = (p.flags & HC_FLAG_WEIGHTS_STATIC) ? 1 : 0;
  const size_t dsm = down_smem(MB, g.KS, p.R, p.C, g.CL, g.down_threads / 32, es).total;
  cudaError_t e = ensure_smem<dec_down<T, MB>>(dsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(dec_down<T, MB>, dim3(g.NSL), dim3(g.down_threads), dsm, p.stream, static_cast<unsigned>(g.CL), da);
  if (e != cudaSuccess) return e;

  UpArgs<T> ua;
  ua.streams = da.streams;
  ua.prev_out = da.prev_out;
  ua.prev_gate = da.prev_gate;
  ua.ns = da.ns;
  ua.wu = static_cast<const T*>(p.up_w);
  ua.inv_ws = inv_ws;
  ua.part_ws = part_ws;
  ua.pre = static_cast<T*>(p.pre_output);
  ua.post = static_cast<T*>(p.post_gate);
  ua.B = da.B; ua.C = p.C; ua.H = p.H; ua.R = p.R; ua.HS = g.HS; ua.NP = g.NCLU;
  ua.at = Attrs{p.eps, p.rho, p.alpha, p.gate_div, p.gate_mul};
  const size_t usm = up_smem(MB, g.HS, p.R, g.up_threads / 32, es).total;
  e = ensure_smem<dec_up<T, MB>>(usm);
  if (e != cudaSuccess) return e;
  return launch_pdl(dec_up<T, MB>, dim3((p.H / g.HS) * p.C), dim3(g.up_threads), usm, p.stream,
                    static_cast<unsigned>(p.C), ua);
}

template <typename T>
cudaError_t run_decode(const Problem& p, const DecodeCfg& g) {
  if (p.rows <= 1) return run_decode_mb<T, 1>(p, g);
  if (p.rows <= 2) return run_decode_mb<T, 2>(p, g);
  if (p.rows <= 4) return run_decode_mb<T, 4>(p, g);
  return run_decode_mb<T, 8>(p, g);
}

}  // namespace

bool decode_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  return decode_cfg(rows, C, H, R, dt, 148).ok;
}

size_t decode_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  const DecodeCfg g = decode_cfg(rows, C, H, R, dt, num_sms);
  return g.ok ? dec_layout(rows, C, R, g).total : 0;
}

cudaError_t launch_decode(const Problem& p) {
  const DecodeCfg g = decode_cfg(p.rows, p.C, p.H, p.R, p.dt, p.num_sms);
  if (!g.ok) return cudaErrorInvalidValue;
  switch (p.dt) {
    case HC_F32: return run_decode<float>(p, g);
    case HC_F16: return run_decode<__half>(p, g);
    default: return run_decode<__nv_bfloat16>(p, g);
  }
}

unsigned int read_wait_timeouts(bool reset) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_wait_timeouts, &z, sizeof(z));
  }
  return v;
}

}  // namespace hc
