// Decode path of the low-rank mix block (rows <= 8): two weight-streaming
// kernels linked by programmatic dependent launch. These CUDA-core kernels
// serve fp32 I/O (and any fp16/bf16 shape the tensor-core pair in
// hc_decode_tc.cu does not take).
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
//     - copies its up_weight tile (R rows x HS columns of branch c) with
//       16-byte cp.async and loads S for its tile before griddepcontrol.wait;
//     - reduces the down partials (each rank 1/C of the R columns, partials
//       added in cluster order), applies ScaledSiLU, and broadcasts d to the
//       cluster through DSMEM;
//     - runs the up GEMV, the sigmoid and the hn*g products, and sums the
//       products over the branches in order 0..C-1 through DSMEM for the
//       pre-mix; one CTA also writes post_gate.
//
// All reductions have a fixed order that depends on the shape only, so the
// results are deterministic and a row's bits do not depend on the row count.
#include <algorithm>
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

// 16-byte vectors of T, widened to fp32 and narrowed back (values that are
// already representable in T pass through exactly).
template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4& u, float* out) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* in) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(in[2 * i], in[2 * i + 1]);
    return u;
  }
};
template <> struct Vec<__half> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void unpack(const uint4& u, float* out) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
  static __device__ __forceinline__ uint4 pack(const float* in) {
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(in[2 * i], in[2 * i + 1]);
    return u;
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void unpack(const uint4& u, float* out) {
    out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
    out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ uint4 pack(const float* in) {
    return make_uint4(__float_as_uint(in[0]), __float_as_uint(in[1]), __float_as_uint(in[2]), __float_as_uint(in[3]));
  }
};

template <typename T> __device__ __forceinline__ uint4 ld16(const T* p) { return *reinterpret_cast<const uint4*>(p); }
template <typename T> __device__ __forceinline__ void st16(T* p, const uint4& u) { *reinterpret_cast<uint4*>(p) = u; }

__host__ __device__ inline uint32_t a16(uint32_t x) { return (x + 15u) & ~15u; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Shared-memory layout of dec_down (byte offsets), for MB rows.
struct DownSmem {
  uint32_t bar, wd, wi, ns, hn, wsum, inv, red, recv, total;
};
// Columns of [down | inject] owned by each cluster rank in the partial-sum
// reduction: a multiple of 4 so a float4 group never straddles two owners.
__host__ __device__ inline int owner_cols(int R, int C, int CL) { return ceil_div(ceil_div(R + C, CL), 4) * 4; }

__host__ __device__ inline DownSmem down_smem(int MB, int KS, int R, int C, int CL, int nwarps, int es) {
  const int ncr = owner_cols(R, C, CL);
  DownSmem L;
  L.bar = 0;
  L.wd = 16;
  L.wi = a16(L.wd + KS * R * es);
  L.ns = a16(L.wi + KS * C * es);
  L.hn = a16(L.ns + KS * 4);
  L.wsum = a16(L.hn + MB * KS * 4);
  L.inv = a16(L.wsum + nwarps * MB * 4);
  L.red = a16(L.inv + MB * 4);
  L.recv = a16(L.red + MB * R * 4);
  L.total = a16(L.recv + CL * MB * ncr * 4);
  return L;
}

// Shared-memory layout of dec_up (byte offsets), for MB rows.
struct UpSmem {
  uint32_t wu, csum, d, hn, ns, red, mix, total;
};
// csum_bytes: the chunk sums of the partial reduction (see dec_up).
__host__ __device__ inline UpSmem up_smem(int MB, int HS, int R, int nwarps, int es, int csum_bytes) {
  UpSmem L;
  L.wu = 0;
  L.csum = a16(L.wu + R * HS * es);
  L.d = a16(L.csum + csum_bytes);
  L.hn = a16(L.d + MB * R * 4);
  L.ns = a16(L.hn + MB * HS * 4);
  L.red = a16(L.ns + HS * 4);
  L.mix = a16(L.red + nwarps * MB * HS * 4);
  L.total = a16(L.mix + MB * HS * 4);
  return L;
}

template <typename T>
struct DownArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wd, *wi;
  T* sout;
  float* inv_ws;   // (B, C)
  float* part_ws;  // (NCLU, B, NCP)
  int B, C, H, R, KS, CL, KQ, NCP;
  float eps;
  int weights_static;
};

template <typename T>
struct UpArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wu;
  const float* inv_ws;
  const float* part_ws;
  T *pre, *post;
  int B, C, H, R, HS, NP, NCP, split_d, nch, csum_bytes;
  Attrs at;
};

template <typename T, int MB>
__global__ void __launch_bounds__(512) dec_down(const DownArgs<T> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int VEC = Vec<T>::N;
  constexpr int es = sizeof(T);
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  const int B = a.B, C = a.C, H = a.H, R = a.R, KS = a.KS, CL = a.CL, NC = R + C;
  const int ncr = owner_cols(R, C, CL);
  const DownSmem L = down_smem(MB, KS, R, C, CL, nwarps, es);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  unsigned char* wd_s = smem + L.wd;
  const T* wi_s = reinterpret_cast<const T*>(smem + L.wi);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* hn_s = reinterpret_cast<float*>(smem + L.hn);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  float* inv_s = reinterpret_cast<float*>(smem + L.inv);
  float* red_s = reinterpret_cast<float*>(smem + L.red);
  float* recv_s = reinterpret_cast<float*>(smem + L.recv);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int slice = blockIdx.x;
  const int k0 = slice * KS;
  const int c = k0 / H, hk0 = k0 - c * H;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const uint32_t wbytes = static_cast<uint32_t>(KS * R * es), ibytes = static_cast<uint32_t>(KS * C * es);
  const bool pro = a.prev_out != nullptr;

  cluster_arrive_relaxed();
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue_weights = [&]() {
    if (tid == 0) {
      mbar_arrive_expect_tx(bar, wbytes + ibytes);
      bulk_g2s(wd_s, a.wd + static_cast<int64_t>(k0) * R, wbytes, bar);
      bulk_g2s(smem + L.wi, a.wi + static_cast<int64_t>(k0) * C, ibytes, bar);
    }
    #pragma unroll 1
    for (int i = tid; i < KS / VEC; i += nthr) {
      float f[VEC];
      Vec<T>::unpack(ld16(a.ns + k0 + i * VEC), f);
#pragma unroll
      for (int j = 0; j < VEC; ++j) ns_s[i * VEC + j] = f[j];
    }
  };
  if (a.weights_static) issue_weights();
  pdl_wait();
  if (!a.weights_static) issue_weights();
  pdl_trigger();

  // ---- one pass over branch c of every row: S, its sum of squares, the
  // slice's S (kept in shared memory) and streams_out for the slice ----
  const int NVr = H / VEC;
  float ss[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) ss[b] = 0.0f;
  #pragma unroll 1
  for (int v = tid; v < NVr; v += nthr) {
    uint4 sv[MB], pv[MB];
    float gt[MB];
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B) {
        sv[b] = ld16(a.streams + b * CH + static_cast<int64_t>(c) * H + v * VEC);
        if (pro) {
          pv[b] = ld16(a.prev_out + static_cast<int64_t>(b) * H + v * VEC);
          gt[b] = ldf(a.prev_gate + b * C + c);
        }
      }
    const int kk = v * VEC - hk0;
    const bool mine = kk >= 0 && kk < KS;
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B) {
        float sf[VEC];
        Vec<T>::unpack(sv[b], sf);
        if (pro) {
          float pf[VEC];
          Vec<T>::unpack(pv[b], pf);
#pragma unroll
          for (int j = 0; j < VEC; ++j) sf[j] = prologue_s<T>(sf[j], gt[b], pf[j]);
        }
#pragma unroll
        for (int j = 0; j < VEC; ++j) ss[b] = fmaf(sf[j], sf[j], ss[b]);
        if (mine) {
#pragma unroll
          for (int j = 0; j < VEC; ++j) hn_s[b * KS + kk + j] = sf[j];
          if (a.sout != nullptr) st16(a.sout + b * CH + k0 + kk, pro ? Vec<T>::pack(sf) : sv[b]);
        }
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
    const float iv = inv_rms(t, H, a.eps);
    inv_s[tid] = iv;
    if (hk0 == 0) a.inv_ws[tid * C + c] = iv;
  }
  __syncthreads();
  #pragma unroll 1
  for (int i = tid; i < B * KS; i += nthr) {
    const int b = i / KS, kk = i - b * KS;
    hn_s[i] = norm_hn<T>(hn_s[i], inv_s[b], ns_s[kk]);
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
    for (int i0 = 0; i0 < rpk; i0 += 8) {
      uint4 wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u < rpk) wv[u] = *reinterpret_cast<const uint4*>(wrow + static_cast<size_t>(i0 + u) * R * es);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (i0 + u < rpk) {
          float w[VEC];
          Vec<T>::unpack(wv[u], w);
          const int kk = kg * rpk + i0 + u;
#pragma unroll
          for (int b = 0; b < MB; ++b)
            if (b < B) {
              const float hv = hn_s[b * KS + kk];
#pragma unroll
              for (int j = 0; j < VEC; ++j) acc[b][j] = fmaf(hv, w[j], acc[b][j]);
            }
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

  // ---- push this CTA's partial sums to the cluster rank that owns each
  // column (rank r owns columns [r*ncr, (r+1)*ncr) of [down | inject]) ----
  cluster_wait();
  auto push = [&](int b, int col, float val) {
    const int ow = col / ncr;
    cluster.map_shared_rank(recv_s, ow)[(rank * MB + b) * ncr + (col - ow * ncr)] = val;
  };
  const float qnan = __int_as_float(0x7fc00000);
  if (kq == 0 && leader) {
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B)
#pragma unroll
        for (int j0 = 0; j0 < VEC; j0 += 4) {
          float t[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            t[j] = acc[b][j0 + j];
            if (a.KQ == 2) t[j] += red_s[b * R + v * VEC + j0 + j];
            if (!ok) t[j] = qnan;
          }
          const int col = v * VEC + j0, ow = col / ncr;
          float* dst = cluster.map_shared_rank(recv_s, ow) + (rank * MB + b) * ncr + (col - ow * ncr);
          *reinterpret_cast<float4*>(dst) = make_float4(t[0], t[1], t[2], t[3]);
        }
  }
  // inject: one warp per (row, branch), lanes over k, butterfly sum
  #pragma unroll 1
  for (int p = warp; p < B * C; p += nwarps) {
    const int b = p / C, cc = p - b * C;
    float t = 0.0f;
    if (ok)
      #pragma unroll 1
      for (int kk = lane; kk < KS; kk += 32) t = fmaf(hn_s[b * KS + kk], ldf(wi_s + kk * C + cc), t);
    t = warp_sum(t);
    if (lane == 0) push(b, R + cc, ok ? t : qnan);
  }
  cluster_sync_all();

  // ---- reduce the received partials of the owned columns in rank order ----
  const int clo = rank * ncr, nmine = max(0, min(NC, clo + ncr) - clo);
  const int cluster_id = slice / CL;
  #pragma unroll 1
  for (int i = tid; i < B * nmine; i += nthr) {
    const int b = i / nmine, lc = i - b * nmine;
    float x[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) x[r] = r < CL ? recv_s[(r * MB + b) * ncr + lc] : 0.0f;
    float t = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < CL) t += x[r];
    a.part_ws[(static_cast<int64_t>(cluster_id) * B + b) * a.NCP + clo + lc] = t;
  }
}

template <typename T, int MB>
__global__ void __launch_bounds__(kUpThreads) dec_up(const UpArgs<T> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int VEC = Vec<T>::N;
  constexpr int es = sizeof(T);
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  const int B = a.B, C = a.C, H = a.H, R = a.R, HS = a.HS;
  const UpSmem L = up_smem(MB, HS, R, nwarps, es, a.csum_bytes);
  unsigned char* wu_s = smem + L.wu;
  float4* csum_s = reinterpret_cast<float4*>(smem + L.csum);
  float* d_s = reinterpret_cast<float*>(smem + L.d);
  float* hn_s = reinterpret_cast<float*>(smem + L.hn);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* red_s = reinterpret_cast<float*>(smem + L.red);
  float* mix_s = reinterpret_cast<float*>(smem + L.mix);

  cg::cluster_group cluster = cg::this_cluster();
  const int c = static_cast<int>(cluster.block_rank());
  const int q = blockIdx.x / C;
  const int h0 = q * HS;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const int64_t col0 = static_cast<int64_t>(c) * H + h0;
  const uint32_t rowbytes = static_cast<uint32_t>(HS * es);
  const bool pro = a.prev_out != nullptr;

  cluster_arrive_relaxed();
  // The up weights and the block inputs are never written by the preceding
  // dec_down, which triggers its dependents only after its own wait: reading
  // them before griddepcontrol.wait is safe. The tile is R rows of HS
  // contiguous elements: 16-byte cp.async chunks, consecutive threads on
  // consecutive chunks of a row.
  {
    const int cpr = static_cast<int>(rowbytes / 16);
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(a.wu + col0);
    #pragma unroll 1
    for (int i = tid; i < R * cpr; i += nthr) {
      const int r = i / cpr, qd = i - r * cpr;
      cp_async16(wu_s + static_cast<size_t>(r) * rowbytes + qd * 16, gsrc + (static_cast<int64_t>(r) * CH) * es + qd * 16);
    }
    cp_async_commit();
  }
  const int nvh = HS / VEC;
  #pragma unroll 1
  for (int i = tid; i < B * nvh; i += nthr) {
    const int b = i / nvh, qv = i - b * nvh;
    float sf[VEC];
    Vec<T>::unpack(ld16(a.streams + b * CH + col0 + qv * VEC), sf);
    if (pro) {
      float pf[VEC];
      Vec<T>::unpack(ld16(a.prev_out + static_cast<int64_t>(b) * H + h0 + qv * VEC), pf);
      const float gt = ldf(a.prev_gate + b * C + c);
#pragma unroll
      for (int j = 0; j < VEC; ++j) sf[j] = prologue_s<T>(sf[j], gt, pf[j]);
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) hn_s[b * HS + qv * VEC + j] = sf[j];
  }
  #pragma unroll 1
  for (int i = tid; i < nvh; i += nthr) {
    float f[VEC];
    Vec<T>::unpack(ld16(a.ns + col0 + i * VEC), f);
#pragma unroll
    for (int j = 0; j < VEC; ++j) ns_s[i * VEC + j] = f[j];
  }
  pdl_wait();
  pdl_trigger();
  cluster_wait();
  __syncthreads();  // S (in hn_s) and ns_s were written by other threads above
  float inv_r[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) inv_r[b] = b < B ? a.inv_ws[b * C + c] : 0.0f;

  // ---- d = ScaledSiLU(rT(sum of the down partials)), in float4 column
  // groups; at most 2 rows every CTA reduces all R columns itself, above
  // that each cluster rank reduces 1/C of them and broadcasts over DSMEM ----
  const int NR4 = R / 4, NP = a.NP;
  const int64_t pstride4 = static_cast<int64_t>(B) * a.NCP / 4;
  int g_lo = 0, g_hi = NR4;
  if (a.split_d) {
    const int per = ceil_div(NR4, C);
    g_lo = min(NR4, c * per);
    g_hi = min(NR4, g_lo + per);
  }
  const int ng = g_hi - g_lo;
  // Work unit = (chunk of the partials, float4 column group of one row): the
  // NP partials are cut into nch chunks; each unit sums its chunk in partial
  // order, loads issued together (two units per thread in flight), and the
  // chunk sums are then added in chunk order. CTA (0, 0) also reduces the
  // inject columns (scalars) the same way for post_gate.
  const int nch = a.nch, cs = ceil_div(NP, nch);
  const bool do_post = (q == 0 && c == 0);
  const int n_items = B * ng, n_units = n_items * nch;
  const int n_post_units = do_post ? B * C * nch : 0;
  float* psum_s = reinterpret_cast<float*>(csum_s + static_cast<size_t>(n_items) * nch);
  #pragma unroll 1
  for (int u0 = tid; u0 < n_units + n_post_units; u0 += 2 * nthr) {
    // address, stride and count of up to two units, then all their loads
    const float* base[2];
    int64_t stride[2];
    int cnt[2], kind[2], slot[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int u = u0 + k * nthr;
      cnt[k] = 0;
      kind[k] = 0;
      slot[k] = 0;
      base[k] = a.part_ws;
      stride[k] = 0;
      if (u < n_units + n_post_units) {
        const bool post_unit = u >= n_units;
        const int uu = post_unit ? u - n_units : u;
        const int nk = post_unit ? B * C : n_items;
        const int ch = uu / nk, item = uu - ch * nk;
        cnt[k] = min(cs, NP - ch * cs);
        kind[k] = post_unit ? 2 : 1;
        slot[k] = ch * nk + item;
        if (!post_unit) {
          const int b = item / ng, g = g_lo + (item - b * ng);
          base[k] = a.part_ws + static_cast<int64_t>(b) * a.NCP + static_cast<int64_t>(ch * cs) * B * a.NCP + 4 * g;
        } else {
          const int b = item / C, cc = item - b * C;
          base[k] = a.part_ws + static_cast<int64_t>(b) * a.NCP + static_cast<int64_t>(ch * cs) * B * a.NCP + R + cc;
        }
        stride[k] = static_cast<int64_t>(B) * a.NCP;
      }
    }
    float4 x[2][8];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        x[k][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < cnt[k]) {
          if (kind[k] == 1) x[k][j] = *reinterpret_cast<const float4*>(base[k] + j * stride[k]);
          else x[k][j].x = base[k][j * stride[k]];
        }
      }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (kind[k] == 0) continue;
      float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < cnt[k]) {
          t.x += x[k][j].x; t.y += x[k][j].y; t.z += x[k][j].z; t.w += x[k][j].w;
        }
#pragma unroll 1
      for (int j = 8; j < cnt[k]; ++j) {  // chunks longer than 8: remaining loads one by one
        if (kind[k] == 1) {
          const float4 z = *reinterpret_cast<const float4*>(base[k] + j * stride[k]);
          t.x += z.x; t.y += z.y; t.z += z.z; t.w += z.w;
        } else {
          t.x += base[k][j * stride[k]];
        }
      }
      if (kind[k] == 2) psum_s[slot[k]] = t.x;
      else csum_s[slot[k]] = t;
    }
  }
  __syncthreads();
  #pragma unroll 1
  for (int i = tid; i < n_items; i += nthr) {
    const int b = i / ng, g = g_lo + (i - b * ng);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int ch = 0; ch < nch; ++ch) {
      const float4 z = csum_s[ch * n_items + i];
      t.x += z.x; t.y += z.y; t.z += z.z; t.w += z.w;
    }
    float dd[4] = {t.x, t.y, t.z, t.w};
#pragma unroll 1
    for (int j = 0; j < 4; ++j) dd[j] = scaled_silu<T>(rT<T>(dd[j]), a.at.alpha);
    const float4 dv = make_float4(dd[0], dd[1], dd[2], dd[3]);
    if (a.split_d) {
      for (int pr = 0; pr < C; ++pr)
        *reinterpret_cast<float4*>(cluster.map_shared_rank(d_s, pr) + b * R + g * 4) = dv;
    } else {
      *reinterpret_cast<float4*>(d_s + b * R + g * 4) = dv;
    }
  }
  if (do_post) {
    #pragma unroll 1
    for (int i = tid; i < B * C; i += nthr) {
      float t = 0.0f;
      for (int ch = 0; ch < nch; ++ch) t += psum_s[ch * (B * C) + i];
      const int b = i / C, cc = i - b * C;
      stf(a.post + b * C + cc, post_gate_of<T>(rT<T>(t), a.at.gate_div, a.at.gate_mul));
    }
  }
  #pragma unroll 1
  for (int i = tid; i < B * HS; i += nthr) {
    const int b = i / HS, h = i - b * HS;
    float iv = inv_r[0];
#pragma unroll
    for (int bb = 1; bb < MB; ++bb)
      if (bb == b) iv = inv_r[bb];
    hn_s[i] = norm_hn<T>(hn_s[i], iv, ns_s[h]);
  }
  if (a.split_d) cluster_sync_all();
  cp_async_wait_all();
  __syncthreads();

  // ---- up GEMV: NVh lanes cover one row of the tile, rows strided over groups
  const int NVh = HS / VEC;
  const int lv = lane % NVh, rgw = lane / NVh, RGW = 32 / NVh, RG = nwarps * RGW;
  const int rg = warp * RGW + rgw;
  float acc[MB][VEC];
#pragma unroll
  for (int b = 0; b < MB; ++b)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[b][j] = 0.0f;
  #pragma unroll 1
  for (int r = rg; r < R; r += RG) {
    float w[VEC];
    Vec<T>::unpack(*reinterpret_cast<const uint4*>(wu_s + static_cast<size_t>(r) * rowbytes + lv * 16), w);
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B) {
        const float dv = d_s[b * R + r];
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[b][j] = fmaf(dv, w[j], acc[b][j]);
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

  // ---- up -> g -> hn*g; the pre-mix sums the products over c = 0..C-1 on
  // the rank that finalises the feature (rank j owns features [j*HSc, ...)) ----
  const int HSc = HS / C;
  #pragma unroll 1
  for (int i = tid; i < B * HS; i += nthr) {
    const int b = i / HS, h = i - b * HS;
    float u = 0.0f;
    for (int w = 0; w < nwarps; ++w) u += red_s[(w * MB + b) * HS + h];
    const float g = rT<T>(sigmoid_acc(rT<T>(u)));
    const float prod = __fmul_rn(hn_s[i], g);
    if (C == 1) {
      stf(a.pre + static_cast<int64_t>(b) * H + h0 + h, __fmul_rn(a.at.rho, __fadd_rn(0.0f, prod)));
    } else {
      const int j = h / HSc, hl = h - j * HSc;
      cluster.map_shared_rank(mix_s, j)[(c * MB + b) * HSc + hl] = prod;
    }
  }
  if (C > 1) {
    cluster_sync_all();
    #pragma unroll 1
    for (int i = tid; i < B * HSc; i += nthr) {
      const int b = i / HSc, hl = i - b * HSc;
      float acc2 = 0.0f;
      for (int cc = 0; cc < C; ++cc) acc2 = __fadd_rn(acc2, mix_s[(cc * MB + b) * HSc + hl]);
      stf(a.pre + static_cast<int64_t>(b) * H + h0 + c * HSc + hl, __fmul_rn(a.at.rho, acc2));
    }
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

// Row stride of the fp32 partials: R + C padded to a multiple of 4 floats so
// the R down columns can be read as float4.
inline int partial_stride(int R, int C) { return (R + C + 3) / 4 * 4; }

struct DecLayout {
  size_t inv, part, total;
};
DecLayout dec_layout(int64_t rows, int C, int R, const DecodeCfg& g) {
  DecLayout L;
  L.inv = 0;
  L.part = align_up(static_cast<size_t>(rows) * C * 4, 256);
  L.total = align_up(L.part + static_cast<size_t>(g.NCLU) * rows * partial_stride(R, C) * 4, 256);
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
  da.NCP = partial_stride(p.R, p.C);
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
  ua.NCP = da.NCP;
  ua.split_d = (p.rows > 2 && p.C > 1) ? 1 : 0;
  {
    const int NR4 = p.R / 4;
    const int ng = ua.split_d ? (NR4 + p.C - 1) / p.C : NR4;
    ua.nch = std::max(1, std::min(8, (g.NCLU + 7) / 8));
    ua.csum_bytes = static_cast<int>(ua.nch * (static_cast<size_t>(p.rows) * ng * 16 + static_cast<size_t>(p.rows) * p.C * 4));
  }
  ua.at = Attrs{p.eps, p.rho, p.alpha, p.gate_div, p.gate_mul};
  const size_t usm = up_smem(MB, g.HS, p.R, g.up_threads / 32, es, ua.csum_bytes).total;
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
  return decode_um_supported(rows, C, H, R, dt) || decode_tc_supported(rows, C, H, R, dt) ||
         decode_cfg(rows, C, H, R, dt, 148).ok;
}

size_t decode_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  if (decode_um_supported(rows, C, H, R, dt)) return decode_um_workspace(rows, C, H, R, dt, num_sms);
  if (decode_tc_supported(rows, C, H, R, dt)) return decode_tc_workspace(rows, C, H, R, dt, num_sms);
  const DecodeCfg g = decode_cfg(rows, C, H, R, dt, num_sms);
  return g.ok ? dec_layout(rows, C, R, g).total : 0;
}

cudaError_t launch_decode(const Problem& p) {
  if (decode_um_supported(p.rows, p.C, p.H, p.R, p.dt)) return launch_decode_um(p);
  if (decode_tc_supported(p.rows, p.C, p.H, p.R, p.dt)) return launch_decode_tc(p);
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
