// Prefill path of the low-rank mix block (many rows, fp16/bf16): the down and
// up projections are dense contractions on the 5th-generation tensor cores
// (tcgen05, fp32 accumulators in tensor memory), fed by TMA tensor copies.
//
//   pf_norm  (one CTA per row, CUDA cores): prologue S -> streams_out, the
//            branch RMS statistic, hn -> workspace. hn is stored in tiles of
//            128 rows x 64 columns, each tile 16 KB of contiguous memory
//            ([row tile][64-column block][row][column]), so that every
//            operand box the tensor-core kernels load is one contiguous read.
//   pf_down  (tcgen05): partial[ks] = hn[:, K_ks] @ [W_d | W_i][K_ks, :] for
//            the K slices ks, 128-row tiles, W_d read in place as an MN-major
//            operand, W_i as 16 extra columns. The slices are branch-sized, or
//            256 wide for batches of up to 512 rows (more CTAs for few tiles);
//            within each regime a row's sums never depend on the row count.
//   pf_mid   : down = rT(sum of the partials in slice order), ScaledSiLU -> d;
//            inject likewise -> post_gate.
//   pf_up    (tcgen05): up = d @ W_u for a tile of 128 rows x (C branches x
//            64 features); the epilogue reads the accumulators from tensor
//            memory and computes g = rT(sigmoid(rT(up))) with exactly the bits
//            of the accurate rounded sigmoid (a table in bf16, the checked
//            fast form in fp16), hn * g, the pre-mix over the branches in
//            order and pre_output, all in registers.
//
// Pipelines: one TMA thread, one MMA thread, four epilogue warps; stage
// hand-off through mbarriers (all waits bounded, see hc_async.cuh).
#include <cuda.h>

#include <algorithm>

#include "hc_async.cuh"
#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_tc.cuh"
#include "hc_vec.cuh"

namespace hc {

// Count of bounded waits in this file's kernels that gave up (diagnostic).
__device__ unsigned int g_pf_wait_timeouts = 0;

namespace {

constexpr int kBM = 128;            // tile rows = tensor-memory lanes
constexpr int kBK = 64;             // K per stage = one 128-byte swizzle row
constexpr int kBoxBytes = 64 * 64 * 2;
constexpr int kATileBytes = kBM * kBK * 2;
constexpr int kTcThreads = 192;     // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2..5 epilogue
constexpr int kNormVec = 4;         // 16-byte vectors per thread in pf_norm
constexpr int kNormMaxThreads = 512; // so C*H <= 512 * 4 * 8 = 16384


// ---------------------------------------------------------------- pf_norm --

// One CTA per row. The row (streams, and prev_out with a prologue) comes into
// shared memory by one bulk copy per tensor, so no register holds load data
// and several CTAs per SM have their rows in flight at once; S goes back to
// shared memory in place of streams for the second pass.
template <typename T, int C>
__global__ void __launch_bounds__(kNormMaxThreads)
pf_norm(const T* __restrict__ streams, const T* __restrict__ prev_out, const T* __restrict__ prev_gate,
        const T* __restrict__ ns, int H, float eps, T* __restrict__ sout, T* __restrict__ hn) {
  extern __shared__ __align__(16) uint8_t row_s[];  // [C*H] streams -> S, then [H] prev_out
  __shared__ uint64_t bar;
  __shared__ float red[C][kNormMaxThreads / 32];
  __shared__ float inv_s[C];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x, nwarps = nthr >> 5;
  const int64_t b = blockIdx.x;
  const int CH = C * H, NV = CH / 8, NVH = H / 8;
  const bool pro = prev_out != nullptr;
  T* srow = reinterpret_cast<T*>(row_s);
  const T* prow = srow + CH;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (tid == 0) {
    const uint32_t sb = static_cast<uint32_t>(CH * sizeof(T)), pb = pro ? static_cast<uint32_t>(H * sizeof(T)) : 0u;
    mbar_arrive_expect_tx(&bar, sb + pb);
    bulk_g2s(row_s, streams + b * CH, sb, &bar);
    if (pro) bulk_g2s(row_s + sb, prev_out + b * H, pb, &bar);
  }
  // branch of each of this thread's vectors, v / NVH without an integer
  // divide: (v + 1/2) / NVH in fp32 is within 1e-6 of a value at least
  // 1/(2 NVH) away from an integer (v < 2^11, quotient <= 8), so truncation
  // is exact
  const float rnvh = 1.0f / static_cast<float>(NVH);
  int cv[kNormVec];
#pragma unroll
  for (int i = 0; i < kNormVec; ++i)
    cv[i] = min(C - 1, static_cast<int>((static_cast<float>(tid + i * nthr) + 0.5f) * rnvh));
  float gt[kNormVec];
  if (pro) {
#pragma unroll
    for (int i = 0; i < kNormVec; ++i) {
      const int v = tid + i * nthr;
      gt[i] = v < NV ? ldf(prev_gate + b * C + cv[i]) : 0.0f;
    }
  }
  const bool ok = mbar_wait(&bar, 0, &g_pf_wait_timeouts);
  float ss[C];
#pragma unroll
  for (int c = 0; c < C; ++c) ss[c] = 0.0f;
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int v = tid + i * nthr;
    if (v < NV) {
      const int c = cv[i], h0 = (v - c * NVH) * 8;
      uint4 sv = *reinterpret_cast<const uint4*>(srow + v * 8);
      // each rounding to T happens once, in the pack that stores the value
      // (S = rT(streams + gate * prev): multiply, add, then the pack rounds)
      if (pro) {
        float s8[8], p8[8];
        V8<T>::unpack(sv, s8);
        V8<T>::unpack(*reinterpret_cast<const uint4*>(prow + h0), p8);
#pragma unroll
        for (int j = 0; j < 8; ++j) s8[j] = __fadd_rn(s8[j], __fmul_rn(gt[i], p8[j]));
        sv = V8<T>::pack(s8);
        *reinterpret_cast<uint4*>(srow + v * 8) = sv;  // this thread's own vector: no race
      }
      if (sout != nullptr) st16(sout + b * CH + v * 8, sv);
      float s8[8];
      V8<T>::unpack(sv, s8);
      float q = 0.0f;
#pragma unroll
      for (int j = 0; j < 8; ++j) q = fmaf(s8[j], s8[j], q);
#pragma unroll
      for (int cc = 0; cc < C; ++cc)
        if (cc == c) ss[cc] += q;
    }
  }
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const float w = warp_sum(ss[c]);
    if (lane == 0) red[c][warp] = w;
  }
  __syncthreads();
  if (tid < C) {
    float t = 0.0f;
    for (int w = 0; w < nwarps; ++w) t += red[tid][w];
    inv_s[tid] = inv_rms(t, H, eps);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kNormVec; ++i) {
    const int v = tid + i * nthr;
    if (v < NV) {
      const float iv = inv_s[cv[i]];
      float s8[8], n8[8], h8[8];
      V8<T>::unpack(*reinterpret_cast<const uint4*>(srow + v * 8), s8);
      V8<T>::unpack(__ldg(reinterpret_cast<const uint4*>(ns + v * 8)), n8);
      // hn = rT((S * inv) * ns): its one rounding is the pack that stores it
#pragma unroll
      for (int j = 0; j < 8; ++j) h8[j] = ok ? __fmul_rn(__fmul_rn(s8[j], iv), n8[j]) : __int_as_float(0x7fc00000);
      // tile (b / 128, v / 8), row b % 128, 16-byte chunk v % 8
      const int64_t tile = (b >> 7) * (CH >> 6) + (v >> 3);
      st16(hn + ((tile << 7) + (b & 127)) * 64 + (v & 7) * 8, V8<T>::pack(h8));
    }
  }
}

// ------------------------------------------------- tensor-core pipelines --

struct PfDownArgs {
  CUtensorMap tm_a;        // hn tiles [row tiles * C*H/64][128][64], box {64 k, 128 rows, 1}
  CUtensorMap tm_b;        // down_w viewed as [R/64 column chunks][C*H rows][64 columns],
                           // box {64 columns, 64 rows, R/64 chunks}
  const uint16_t* wi;      // inject_w [C*H, C] (16-bit codes)
  float* part;             // [ksplit, rows, R + 16] fp32: down columns, then inject
  int rows, R, C, k_per_split, stages;
  int kblocks;             // C*H / 64: hn tiles per row tile
};

template <typename T>
struct PfUpArgs {
  CUtensorMap tm_a;  // d     [rows, R],   box {64 k, 128 rows}
  CUtensorMap tm_b;  // up_w  [R, C*H],    box {64 n, 64 k}
  CUtensorMap tm_hn; // hn tiles [row tiles * C*H/64][128][64], box {64 features, 128 rows, 1}
  const T* hn;       // tiled, as tm_hn
  const uint16_t* sig16;  // fp16: the gate table built by pf_sig16_table (kS16Bytes)
  T* pre;            // [rows, H]
  int rows, C, H, R, stages, nbuf;
  float rho;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_addr(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// Shared state of a pipeline in dynamic shared memory, after the stages.
struct PipeBars {
  uint64_t full[4], empty[4], done, aux;
  uint32_t tmem_base;
};

// The inject projection rides along as 16 extra N columns (chunk R/64 of
// the B operand, C columns used, the rest zero). Its rows are too narrow for
// a TMA copy (C * 2 bytes), so the producer warp writes them into the
// swizzled chunk itself: K-row r of a 128-byte-swizzled MN-major chunk keeps
// columns 0..7 in 16-byte slot (r & 7).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Each CTA loads its own operands: per stage the A tile of its 128 hn rows
// (one 3D copy of a contiguous 16 KB tile) and the W_d slab of the stage's 64
// K rows (one 3D copy of all R/64 column chunks). Row tiles that share a K
// slice read the same slab; L2 serves the repeats.
//
// Shared memory of a stage: the A tile (16 KB), then the B operand as
// [chunk j <= R/64][64 K rows][128 bytes], chunk R/64 being the inject
// columns; each MMA reads its 16 K rows of every chunk with chunk stride 8 KB.
template <bool BF16>
__global__ void __launch_bounds__(kTcThreads, 1) pf_down(const __grid_constant__ PfDownArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int R = a.R, C = a.C, NB = R / 64, S = a.stages, NTOT = R + 16, NP = R + 16;
  const uint32_t chunk_bytes = static_cast<uint32_t>(kBoxBytes);  // 64 K rows x 128 bytes
  const int stage_bytes = kATileBytes + (NB + 1) * kBoxBytes;     // A, then R/64 + 1 chunks of B
  uint8_t* wi_s = smem + S * stage_bytes;                           // this CTA's K rows of inject_weight
  const uint32_t wi_bytes = static_cast<uint32_t>(a.k_per_split * C * 2);
  PipeBars* pb = reinterpret_cast<PipeBars*>(wi_s + ((wi_bytes + 15u) & ~15u));
  const int m0 = blockIdx.x * kBM, ks = blockIdx.y;
  const int k_begin = ks * a.k_per_split, nk = a.k_per_split / kBK;
  const uint32_t ncols = NTOT <= 256 ? 256u : 512u;

  // zero the inject chunk of every stage once; only its first C columns change
  for (int st = 0; st < S; ++st) {
    uint4* z = reinterpret_cast<uint4*>(smem + st * stage_bytes + kATileBytes + NB * chunk_bytes);
    for (uint32_t i = threadIdx.x; i < chunk_bytes / 16; i += blockDim.x) z[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (warp == 0 && lane == 0) {
    for (int st = 0; st < S; ++st) {
      mbar_init(&pb->full[st], 1);
      mbar_init(&pb->empty[st], 1);
    }
    mbar_init(&pb->done, 1);
    mbar_init(&pb->aux, 1);
    fence_mbar_init();
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_b);
  }
  if (warp == 1) {
    tmem_alloc(&pb->tmem_base, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = pb->tmem_base;
  // inject_weight is never written by the preceding kernel (weights): its
  // K slice may be copied before the dependency wait
  if (warp == 0 && lane == 0) {
    mbar_arrive_expect_tx(&pb->aux, wi_bytes);
    bulk_g2s(wi_s, a.wi + static_cast<int64_t>(k_begin) * C, wi_bytes, &pb->aux);
  }
  pdl_wait();
  pdl_trigger();
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) ok = mbar_wait(&pb->aux, 0, &g_pf_wait_timeouts);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int it = 0; it < nk && ok; ++it) {
      const int st = it % S;
      if (lane == 0) ok = mbar_wait(&pb->empty[st], ((it / S) & 1) ^ 1, &g_pf_wait_timeouts);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* sp = smem + st * stage_bytes;
      uint8_t* bsp = sp + kATileBytes;
      const int k = k_begin + it * kBK;
      // the stage's previous MMAs (async proxy) read this inject chunk; order
      // those reads before the generic writes below
      fence_proxy_async_smem();
      for (int kr = lane; kr < kBK; kr += 32) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(wi_s) + static_cast<int64_t>(k - k_begin + kr) * C;
        uint8_t* dst = bsp + NB * chunk_bytes + kr * 128 + ((kr & 7) << 4);
        if (C == 8) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
        else if (C == 4) *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
        else if (C == 2) *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
        else *reinterpret_cast<uint16_t*>(dst) = *src;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&pb->full[st], static_cast<uint32_t>(kATileBytes + NB * kBoxBytes));
        tma_load_3d(sp, &a.tm_a, 0, 0, blockIdx.x * a.kblocks + k / kBK, &pb->full[st]);
        tma_load_3d(bsp, &a.tm_b, 0, k, 0, &pb->full[st]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // One thread issues every MMA, so nothing but the issue itself may sit
      // between two of them: the descriptors of stage 0 are built once and
      // stepped by constants (a descriptor's address field is the shared
      // memory address / 16, linear below 256 KB). N = R + 16 columns go as
      // one MMA of up to 256 columns and one of the rest.
      const int N0 = min(256, NTOT), N1 = NTOT - N0;
      const uint32_t id0 = idesc_f16(BF16, kBM, N0, false, true);
      const uint32_t id1 = idesc_f16(BF16, kBM, N1 > 0 ? N1 : 16, false, true);
      const uint32_t s0 = smem_addr(smem);
      const uint64_t ad0 = smem_desc_sw128(s0, 16, 1024);
      uint64_t bd[kBK / 16];
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk)
        bd[kk] = smem_desc_sw128(s0 + kATileBytes + kk * 16 * 128, chunk_bytes, 1024);
      const uint64_t n1_off = static_cast<uint64_t>((4u * chunk_bytes) >> 4);  // chunk 4 = column 256
      for (int it = 0; it < nk && ok; ++it) {
        const int st = it % S;
        ok = mbar_wait(&pb->full[st], (it / S) & 1, &g_pf_wait_timeouts);
        if (!ok) break;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>((st * stage_bytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint64_t adesc = ad0 + so + static_cast<uint64_t>(kk * 2);  // + 32 bytes per K step
          mma_f16(tmem, adesc, bd[kk] + so, id0, acc);
          if (N1 > 0) mma_f16(tmem + 256, adesc, bd[kk] + so + n1_off, id1, acc);
        }
        mma_commit(&pb->empty[st]);
      }
      mma_commit(&pb->done);
    }
  } else {
    // Epilogue: accumulators -> shared memory (the pipeline stages are idle:
    // every stage has been consumed), then
    // whole rows to global memory with coalesced 16-byte stores.
    ok = mbar_wait(&pb->done, 0, &g_pf_wait_timeouts);
    tc_fence_after();
    const int ew = warp - 2, lq = warp & 3, row = lq * 32 + lane;
    const int NPS = NP + 4;                     // padded row: conflict-free 16-byte writes
    const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16);
    const float qn = __int_as_float(0x7fc00000);
    if (kBM * NPS * 4 > S * stage_bytes) {
      // (too few stages to stage the tile) each thread stores its own row
      const int64_t grow = m0 + row;
      for (int c0 = 0; c0 < NTOT; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
        if (grow < a.rows) {
          float4* dst = reinterpret_cast<float4*>(a.part + (static_cast<int64_t>(ks) * a.rows + grow) * NP + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = ok ? make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]) : make_float4(qn, qn, qn, qn);
        }
      }
    } else {
    fence_proxy_async_smem();
    float* stg = reinterpret_cast<float*>(smem);
    for (int c0 = 0; c0 < NTOT; c0 += 16) {
      float v[16];
      tmem_ld16(taddr + c0, v);
      float4* d4 = reinterpret_cast<float4*>(stg + row * NPS + c0);
#pragma unroll
      for (int q = 0; q < 4; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    named_bar_sync(1, 128);
    for (int r = ew; r < kBM; r += 4) {
      const int64_t grow = m0 + r;
      if (grow >= a.rows) break;
      const float4* s4 = reinterpret_cast<const float4*>(stg + r * NPS);
      float4* dst = reinterpret_cast<float4*>(a.part + (static_cast<int64_t>(ks) * a.rows + grow) * NP);
      for (int c4 = lane; c4 < NP / 4; c4 += 32) dst[c4] = ok ? s4[c4] : make_float4(qn, qn, qn, qn);
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// down = rT(sum of the K-slice partials in slice order) -> ScaledSiLU -> d;
// inject likewise -> post_gate. ScaledSiLU's gate uses the fast sigmoid that
// matches the accurate one bit for bit on T inputs.
//
// pf_mid: one thread per 4 down columns (float4 partial loads, one 8-byte
// store of d) or per inject column: thread x of a block row handles column
// group x of row (blockIdx.x * kMidRows + y), R/4 + C <= kMidCols.
// MANY (more than eight slices: the 256-wide slices of small batches): the
// partials of eight slices are loaded before any is added, so that their
// latencies overlap; they are still added in slice order. With the few
// branch-sized slices of large batches the plain loop, in a variant with
// fewer registers, measured faster.
constexpr int kMidCols = 128, kMidRows = 2;
template <typename T, bool MANY>
__global__ void __launch_bounds__(kMidCols * kMidRows) pf_mid(const float* __restrict__ part, int ksplit,
                                                              int64_t rows, int R, int C, Attrs at, T* __restrict__ d,
                                                              T* __restrict__ post) {
  pdl_wait();
  pdl_trigger();
  const int R4 = R / 4, W = R4 + C, NP = R + 16;
  const int j = threadIdx.x;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kMidRows + threadIdx.y;
  if (row >= rows || j >= W) return;
  if (j < R4) {
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!MANY) {
      for (int ks = 0; ks < ksplit; ++ks) {
        const float4 p = *reinterpret_cast<const float4*>(part + (ks * rows + row) * NP + 4 * j);
        t.x += p.x; t.y += p.y; t.z += p.z; t.w += p.w;
      }
    } else {
      for (int k0 = 0; k0 < ksplit; k0 += 8) {
        float4 p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k0 + i < ksplit) p[i] = *reinterpret_cast<const float4*>(part + ((k0 + i) * rows + row) * NP + 4 * j);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k0 + i < ksplit) {
            t.x += p[i].x; t.y += p[i].y; t.z += p[i].z; t.w += p[i].w;
          }
      }
    }
    T o[4];
    o[0] = Ty<T>::from_f(scaled_silu_t<T>(rT<T>(t.x), at.alpha));
    o[1] = Ty<T>::from_f(scaled_silu_t<T>(rT<T>(t.y), at.alpha));
    o[2] = Ty<T>::from_f(scaled_silu_t<T>(rT<T>(t.z), at.alpha));
    o[3] = Ty<T>::from_f(scaled_silu_t<T>(rT<T>(t.w), at.alpha));
    *reinterpret_cast<uint2*>(d + row * R + 4 * j) = *reinterpret_cast<const uint2*>(o);
  } else {
    const int cc = j - R4;
    float t = 0.0f;
    if (!MANY) {
      for (int ks = 0; ks < ksplit; ++ks) t += part[(ks * rows + row) * NP + R + cc];
    } else {
      for (int k0 = 0; k0 < ksplit; k0 += 8) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k0 + i < ksplit) p[i] = part[((k0 + i) * rows + row) * NP + R + cc];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (k0 + i < ksplit) t += p[i];
      }
    }
    stf(post + row * C + cc, post_gate_of<T>(rT<T>(t), at.gate_div, at.gate_mul));
  }
}

// pf_mid_cols: many slices and few rows (up to kMidColsRows). One thread per
// (row, column) of [down | inject], and up to kMidBatch slices' partials
// loaded before any is added, so that a column's whole sum costs one L2 round
// trip instead of five (a warp's loads of a slice are 32 consecutive floats);
// they are still added in slice order, so the bits are those of pf_mid. No
// shared memory, so its CTAs start beside pf_down's. (Measured in the bench's
// chains: 23.9 -> 22.6 us per block at 16 rows, 26.2 -> 25.1 at 64, but 32.4
// -> 34.1 at 256, where its four times as many load instructions cost more
// than the round trips they save.)
constexpr int kMidBatch = 48;
constexpr int64_t kMidColsRows = 64;
template <typename T>
__global__ void __launch_bounds__(256) pf_mid_cols(const float* __restrict__ part, int ksplit, int64_t rows, int R,
                                                   int C, Attrs at, T* __restrict__ d, T* __restrict__ post) {
  pdl_wait();
  pdl_trigger();
  const int W = R + C, NP = R + 16;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * W) return;
  const int64_t row = idx / W;
  const int col = static_cast<int>(idx - row * W);
  const float* src = part + row * NP + col;
  const int64_t sstride = rows * NP;
  float t = 0.0f;
  for (int k0 = 0; k0 < ksplit; k0 += kMidBatch) {
    float p[kMidBatch];
#pragma unroll
    for (int i = 0; i < kMidBatch; ++i)
      if (k0 + i < ksplit) p[i] = src[(k0 + i) * sstride];
#pragma unroll
    for (int i = 0; i < kMidBatch; ++i)
      if (k0 + i < ksplit) t += p[i];
  }
  if (col < R) stf(d + row * R + col, scaled_silu_t<T>(rT<T>(t), at.alpha));
  else stf(post + row * C + (col - R), post_gate_of<T>(rT<T>(t), at.gate_div, at.gate_mul));
}

// Persistent up projection. A tile is 128 rows x 64 features; its C branches
// are processed in groups of (up to) four, one group per unit of work, so an
// accumulator is at most 4 x 64 = 256 tensor-memory columns and two of them
// (double buffering) always fit. CTA i takes tiles i, i + grid, ..., so the
// CTAs at work at any moment cover a few neighbouring row tiles (their hn
// reads and pre_output writes stay close). Per unit and K block a stage holds
// the d box (128 rows x 64) and, by one 3D copy, the group's W_u columns (a
// view of W_u as [branches][R rows][H columns], box {64, 64, branches}). The
// hn boxes of a unit arrive one branch at a time into a ring of slots, in the
// order the epilogue consumes them, issued by a warp of their own so that they
// run ahead of the epilogue independently of the operand stages. (Keeping a
// row tile's d resident and walking that row tile's feature tiles read fewer
// bytes but spread the concurrent CTAs over all row tiles, and measured slower.)
// The epilogue keeps the pre-mix sum of a tile in registers across its
// groups, adding branches in order 0..C-1. Warps: 0 loads d and W_u, 1 issues
// the MMAs and owns the tensor memory, 2..17 run the epilogue, 18 loads hn.
//
// g = rT(sigmoid(u)) for u = rT(up): in bf16 it is read from a table of the
// accurate sigmoid over every bf16 u whose result is not a constant, built by
// the CTA at start: bit for bit the accurate rounded sigmoid, with neither
// MUFU operation of the formula. Two values are looked up together: the pair
// is rounded by one packed conversion and clamped by packed bf16 minimum and
// maximum (to [-96, 8]: beyond, g is 0 resp. 1), then its magnitude codes
// by packed 16-bit integer minimum and maximum (below 2^-9, g = 1/2; NaN,
// which the clamps turn into the canonical NaN, lands on an entry holding
// NaN); a sign bit moved to bit 11 selects the negative half of the table. The
// table holds bf16 values and hn * g + acc is one mixed-precision fused
// multiply-add (bf16 operands, fp32 addend): no operand is widened first. fp16
// does the same with its own table (kS16*, below), which is too large to
// rebuild in every CTA: pf_sig16_table builds it once per call and each CTA
// copies it in (and runs two operand stages instead of three to make room).
// The exact fast sigmoid on the arithmetic pipes was measured slower in both
// types: it needs two MUFU operations per element.
constexpr int kUpEpiWarps = 16;
constexpr int kUpHnWarp = 2 + kUpEpiWarps;                 // the warp that loads hn
constexpr int kUpThreads = 32 * (kUpHnWarp + 1);
constexpr int kHnBoxBytes = 128 * 64 * 2;   // one branch: 128 rows x 64 features
constexpr int kUpStages = 3;
constexpr int kHnSlotsMax = 6;
constexpr uint32_t kSigLo = 0x3AFFu;        // largest bf16 magnitude code below 2^-9
constexpr uint32_t kSigPosHi = 0x4100u;     // 8.0: positive u are clamped here
constexpr uint32_t kSigNegHi = 0x42C0u;     // 96.0: negative u are clamped at -96
constexpr uint32_t kSigNaN = kSigNegHi + 1; // the magnitude code NaN is moved to
constexpr int kSigHalf = 2048;              // entries per sign; a power of two >= kSigNaN - kSigLo + 1
constexpr int kSigBytes = 2 * kSigHalf * 2; // bf16 entries
static_assert(static_cast<int>(kSigNaN - kSigLo) < kSigHalf, "sigmoid table half too small");

// fp16: the same lookup over fp16 codes. g = rT(sigmoid(u)) is 1/2 below
// 2^-12 (|u|/4 stays under half an ulp of 1/2), 1 from u = 9 on and 0 from
// u = -18 down; the table spans the magnitude codes between (one half per
// sign, 16516 entries each: not a power of two, so the sign selects its half
// by a multiply). Too large to rebuild in every CTA, it is built once per call
// by pf_sig16_table into the workspace and copied into each pf_up CTA.
constexpr uint32_t kS16Lo = 0x0BFFu;          // largest fp16 magnitude code below 2^-12
constexpr uint32_t kS16PosHi = 0x4880u;       // 9.0
constexpr uint32_t kS16NegHi = 0x4C80u;       // 18.0
constexpr uint32_t kS16NaN = kS16NegHi + 1;   // the magnitude code NaN is moved to
constexpr int kS16Half = 16516;               // >= kS16NaN - kS16Lo + 1, even
constexpr int kS16Bytes = 2 * kS16Half * 2;
static_assert(static_cast<int>(kS16NaN - kS16Lo) < kS16Half, "fp16 sigmoid table half too small");

struct UpBars {
  uint64_t full[kUpStages], empty[kUpStages], accf[2], acce[2], hnf[kHnSlotsMax], hne[kHnSlotsMax], tab;
  uint32_t tmem_base;
};

// Tensor-memory allocations are powers of two of at least 32 columns.
__host__ __device__ inline uint32_t tmem_cols_for(int n) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(n)) c <<= 1;
  return c;
}

// Entry i of the table: sign i / kSigHalf, magnitude code kSigLo + i % kSigHalf.
__device__ __forceinline__ uint16_t sig_entry(int i) {
  const uint32_t neg = static_cast<uint32_t>(i) / kSigHalf, m = kSigLo + static_cast<uint32_t>(i) % kSigHalf;
  if (m == kSigNaN) return 0x7FC0u;                      // NaN
  if (m > (neg ? kSigNegHi : kSigPosHi)) return 0;       // never read
  const float u = __uint_as_float(((neg << 15) | m) << 16);
  return __bfloat16_as_ushort(__float2bfloat16_rn(sigmoid_acc(u)));
}

// acc0 += hn0 * g(up0), acc1 += hn1 * g(up1) for a pair of bf16 hn values
// (element 0 in the low half of hn2) and their fp32 up values, with g from
// the table at shared-memory address tab (see above).
__device__ __forceinline__ void sig_pair_fma(const uint16_t* tab, uint32_t hn2, float up0, float up1, float& acc0,
                                             float& acc1) {
  uint32_t v2, m2;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(v2) : "f"(up1), "f"(up0));
  asm("max.NaN.bf16x2 %0, %0, %1;" : "+r"(v2) : "r"(0xC2C0C2C0u));  // -96
  asm("min.NaN.bf16x2 %0, %0, %1;" : "+r"(v2) : "r"(0x41004100u));  // 8
  m2 = v2 & 0x7FFF7FFFu;
  asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(kSigLo * 0x10001u));
  asm("min.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(kSigNaN * 0x10001u));
  const uint32_t idx2 = m2 + ((v2 >> 4) & 0x08000800u) - kSigLo * 0x10001u;
  const uint16_t g0 = tab[idx2 & 0xFFFFu], g1 = tab[idx2 >> 16];
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "fma.rn.f32.bf16 %0, h0, %3, %0;\n\t"
      "fma.rn.f32.bf16 %1, h1, %4, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(hn2), "h"(g0), "h"(g1));
}

// Entry i of the fp16 table: sign i / kS16Half, magnitude code kS16Lo + i % kS16Half.
__device__ __forceinline__ uint16_t sig16_entry(int i) {
  const uint32_t neg = static_cast<uint32_t>(i) >= static_cast<uint32_t>(kS16Half) ? 1u : 0u;
  const uint32_t m = kS16Lo + static_cast<uint32_t>(i) - neg * kS16Half;
  if (m == kS16NaN) return 0x7E00u;                       // NaN
  if (m > (neg ? kS16NegHi : kS16PosHi)) return 0;        // never read
  const float u = __half2float(__ushort_as_half(static_cast<uint16_t>((neg << 15) | m)));
  return __half_as_ushort(__float2half_rn(sigmoid_acc(u)));
}

// The fp16 table, one entry per thread (grid-stride). Launched between
// pf_norm and pf_down when chained: it lets pf_down launch at once and, before
// it ends, waits for pf_norm, so that pf_down's dependency wait still covers
// pf_norm (programmatic dependence reaches only the previous kernel).
__global__ void __launch_bounds__(256) pf_sig16_table(uint16_t* tab, int chained) {
  pdl_trigger();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < 2 * kS16Half; i += gridDim.x * blockDim.x)
    tab[i] = sig16_entry(i);
  if (chained) pdl_wait();
}

// acc0 += hn0 * g(up0), acc1 += hn1 * g(up1) for a pair of fp16 hn values,
// g from the fp16 table (as sig_pair_fma does for bf16).
__device__ __forceinline__ void sig16_pair_fma(const uint16_t* tab, uint32_t hn2, float up0, float up1, float& acc0,
                                               float& acc1) {
  uint32_t v2, m2;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(v2) : "f"(up1), "f"(up0));
  asm("max.NaN.f16x2 %0, %0, %1;" : "+r"(v2) : "r"(0xCC80CC80u));  // -18
  asm("min.NaN.f16x2 %0, %0, %1;" : "+r"(v2) : "r"(0x48804880u));  // 9
  m2 = v2 & 0x7FFF7FFFu;
  asm("max.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(kS16Lo * 0x10001u));
  asm("min.u16x2 %0, %0, %1;" : "+r"(m2) : "r"(kS16NaN * 0x10001u));
  const uint32_t idx2 = m2 + ((v2 >> 15) & 0x00010001u) * static_cast<uint32_t>(kS16Half) - kS16Lo * 0x10001u;
  const uint16_t g0 = tab[idx2 & 0xFFFFu], g1 = tab[idx2 >> 16];
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "fma.rn.f32.f16 %0, h0, %3, %0;\n\t"
      "fma.rn.f32.f16 %1, h1, %4, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(hn2), "h"(g0), "h"(g1));
}

// The fp16 epilogue's gate for every fp16 code (diagnostic for
// hc_debug_sigmoid_table_f16), from a table built by pf_sig16_table: one pair
// of codes per thread, hn = 1, zero sums.
__global__ void __launch_bounds__(256) sigmoid_table16_codes(const uint16_t* table, float* g) {
  extern __shared__ uint16_t tab16[];
  for (int i = threadIdx.x; i < 2 * kS16Half; i += blockDim.x) tab16[i] = table[i];
  __syncthreads();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;  // codes 2p, 2p + 1
  if (p >= 32768) return;
  const float u0 = __half2float(__ushort_as_half(static_cast<uint16_t>(2 * p)));
  const float u1 = __half2float(__ushort_as_half(static_cast<uint16_t>(2 * p + 1)));
  float a0 = 0.0f, a1 = 0.0f;
  sig16_pair_fma(tab16, 0x3C003C00u, u0, u1, a0, a1);  // hn = (1, 1)
  g[2 * p] = a0;
  g[2 * p + 1] = a1;
}

// The epilogue's gate for every bf16 code (diagnostic for
// hc_debug_sigmoid_table): one pair of codes per thread, hn = 1, zero sums.
__global__ void __launch_bounds__(256) sigmoid_table_codes(float* g) {
  __shared__ uint16_t tab[2 * kSigHalf];
  for (int i = threadIdx.x; i < 2 * kSigHalf; i += blockDim.x) tab[i] = sig_entry(i);
  __syncthreads();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;  // codes 2p, 2p + 1
  if (p >= 32768) return;
  const float u0 = __uint_as_float(static_cast<uint32_t>(2 * p) << 16);
  const float u1 = __uint_as_float(static_cast<uint32_t>(2 * p + 1) << 16);
  float a0 = 0.0f, a1 = 0.0f;
  sig_pair_fma(tab, 0x3F803F80u, u0, u1, a0, a1);  // hn = (1, 1)
  g[2 * p] = a0;
  g[2 * p + 1] = a1;
}

template <typename T, bool BF16>
__global__ void __launch_bounds__(kUpThreads, 1) pf_up(const __grid_constant__ PfUpArgs<T> a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = a.C, H = a.H, R = a.R, NH = a.nbuf;
  const int G = (C + 3) / 4, GC = C < 4 ? C : 4;        // groups per tile, branches per group
  const int nk = R / kBK, NG = 64 * GC, S = a.stages;  // S operand stages, at most 3
  const int stage_bytes = kATileBytes + GC * kBoxBytes;  // d box, then W_u of one K block for the group
  uint8_t* st_s = smem;                                  // [S][d box | GC][...]
  uint8_t* hn_s = st_s + S * stage_bytes;                // [NH][128 rows][64] (swizzled)
  uint16_t* sig = reinterpret_cast<uint16_t*>(hn_s + NH * kHnBoxBytes);
  UpBars* pb = reinterpret_cast<UpBars*>(reinterpret_cast<uint8_t*>(sig) + (BF16 ? kSigBytes : kS16Bytes));
  const int n_h = H / 64, n_m = (a.rows + kBM - 1) / kBM, n_tiles = n_m * n_h;
  const uint32_t ncols = tmem_cols_for(2 * NG);

  if (BF16) {
    for (int i = threadIdx.x; i < 2 * kSigHalf; i += blockDim.x) sig[i] = sig_entry(i);
  }
  if (warp == 0 && lane == 0) {
    if (!BF16) {
      // the fp16 table, written by pf_sig16_table three kernels back (pf_up
      // starts only after pf_mid's dependency wait): copied before ours
      mbar_init(&pb->tab, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&pb->tab, static_cast<uint32_t>(kS16Bytes));
      bulk_g2s(sig, a.sig16, static_cast<uint32_t>(kS16Bytes), &pb->tab);
    }
    for (int st = 0; st < S; ++st) {
      mbar_init(&pb->full[st], 1);
      mbar_init(&pb->empty[st], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&pb->accf[b], 1);
      mbar_init(&pb->acce[b], kUpEpiWarps);
    }
    for (int q = 0; q < NH; ++q) {
      mbar_init(&pb->hnf[q], 1);
      mbar_init(&pb->hne[q], kUpEpiWarps);
    }
    fence_mbar_init();
    tma_prefetch_desc(&a.tm_a);
    tma_prefetch_desc(&a.tm_b);
    tma_prefetch_desc(&a.tm_hn);
  }
  if (warp == 1) {
    tmem_alloc(&pb->tmem_base, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = pb->tmem_base;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile / n_h) * kBM, h0 = (tile % n_h) * 64;
        for (int g = 0; g < G && ok; ++g) {
          const int c_lo = g * 4, nc = min(4, C - c_lo);
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int st = it % S;
            ok = mbar_wait(&pb->empty[st], ((it / S) & 1) ^ 1, &g_pf_wait_timeouts);
            if (!ok) break;
            uint8_t* sp = st_s + st * stage_bytes;
            mbar_arrive_expect_tx(&pb->full[st], static_cast<uint32_t>(kATileBytes + nc * kBoxBytes));
            tma_load_2d(sp, &a.tm_a, kb * kBK, m0, &pb->full[st]);
            tma_load_3d(sp + kATileBytes, &a.tm_b, h0, kb * kBK, c_lo, &pb->full[st]);
          }
        }
      }
    }
  } else if (warp == kUpHnWarp) {
    if (lane == 0) {
      int hseq = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        const int mt = tile / n_h, h0 = (tile % n_h) * 64;
        for (int g = 0; g < G && ok; ++g) {
          const int c_lo = g * 4, nc = min(4, C - c_lo);
          for (int cc = 0; cc < nc && ok; ++cc, ++hseq) {
            const int q = hseq % NH;
            ok = mbar_wait(&pb->hne[q], ((hseq / NH) & 1) ^ 1, &g_pf_wait_timeouts);
            if (!ok) break;
            mbar_arrive_expect_tx(&pb->hnf[q], static_cast<uint32_t>(kHnBoxBytes));
            tma_load_3d(hn_s + q * kHnBoxBytes, &a.tm_hn, 0, 0, mt * (C * H / 64) + ((c_lo + cc) * H + h0) / 64,
                        &pb->hnf[q]);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, unit = 0;
      bool ok = true;
      const uint32_t s_b = smem_addr(st_s);
      const uint64_t ad0 = smem_desc_sw128(s_b, 16, 1024);
      const uint64_t bd0 = smem_desc_sw128(s_b + kATileBytes, kBoxBytes, 1024);
      for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
        for (int g = 0; g < G && ok; ++g, ++unit) {
          const int buf = unit & 1, use = unit >> 1, nc = min(4, C - g * 4);
          ok = mbar_wait(&pb->acce[buf], (use & 1) ^ 1, &g_pf_wait_timeouts);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dbase = tmem + static_cast<uint32_t>(buf * NG);
          const uint32_t idn = idesc_f16(BF16, kBM, 64 * nc, false, true);
          for (int kb = 0; kb < nk; ++kb, ++it) {
            const int st = it % S;
            ok = mbar_wait(&pb->full[st], (it / S) & 1, &g_pf_wait_timeouts);
            if (!ok) break;
            tc_fence_after();
            // descriptors stepped by constants, as in pf_down
            const uint64_t so = static_cast<uint64_t>((st * stage_bytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              mma_f16(dbase, ad0 + so + static_cast<uint64_t>(kk * 2), bd0 + so + static_cast<uint64_t>(kk * 128),
                      idn, (kb > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&pb->empty[st]);
          }
          mma_commit(&pb->accf[buf]);
        }
      }
    }
  } else {
    // Epilogue: warp (2 + e) owns tensor-memory lane quarter (warp % 4) and
    // the 16-feature chunk e / 4 of the tile; it loads one branch's 16
    // accumulator columns at a time (few registers, so sixteen warps fit and
    // hide each other's latency).
    const int ew = warp - 2, lq = warp & 3, hc = ew >> 2;
    const int row = lq * 32 + lane;
    int unit = 0, hseq = 0;
    bool ok = true, tab_ready = false;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
      const int m0 = (tile / n_h) * kBM, h0 = (tile % n_h) * 64;
      const int64_t grow = m0 + row;
      const bool live = grow < a.rows;
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
      for (int g = 0; g < G; ++g, ++unit) {
        const int buf = unit & 1, use = unit >> 1, nc = min(4, C - g * 4);
        ok = mbar_wait(&pb->accf[buf], use & 1, &g_pf_wait_timeouts) && ok;
        tc_fence_after();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(buf * NG);
        for (int cc = 0; cc < nc; ++cc, ++hseq) {
          const int q = hseq % NH;
          ok = mbar_wait(&pb->hnf[q], (hseq / NH) & 1, &g_pf_wait_timeouts) && ok;
          // row `row` of this branch's hn box; 16-byte chunk j of a row sits
          // at chunk (j ^ (row & 7)) under the 128-byte swizzle
          const uint8_t* rb = hn_s + q * kHnBoxBytes + row * 128;
          const uint4 v0 = *reinterpret_cast<const uint4*>(rb + (((2 * hc) ^ (row & 7)) << 4));
          const uint4 v1 = *reinterpret_cast<const uint4*>(rb + (((2 * hc + 1) ^ (row & 7)) << 4));
          // the wait names the loaded registers (tmem_ld_wait_r), so no use of
          // them is scheduled above it (a bare wait let the fp16 sigmoid read
          // registers the load had not filled: nondeterministic results)
          uint32_t up[16];
          tmem_ld16_nowait(taddr + cc * 64 + hc * 16, up);
          tmem_ld_wait_r(up);
          if constexpr (BF16) {
            const uint32_t hw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
              sig_pair_fma(sig, hw[i], __uint_as_float(up[2 * i]), __uint_as_float(up[2 * i + 1]), acc[2 * i],
                           acc[2 * i + 1]);
          } else {
            if (!tab_ready) {
              ok = mbar_wait(&pb->tab, 0, &g_pf_wait_timeouts) && ok;
              tab_ready = true;
            }
            const uint32_t hw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
              sig16_pair_fma(sig, hw[i], __uint_as_float(up[2 * i]), __uint_as_float(up[2 * i + 1]), acc[2 * i],
                             acc[2 * i + 1]);
          }
          // the slot is released only after every lane has used what it read
          // from it, and each lane first orders its (generic-proxy) reads
          // before the refill, a TMA write of the async proxy: without the
          // proxy fence the refill could overtake the reads (seen as rows of a
          // 16-feature chunk taking the next box's values)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&pb->hne[q]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pb->acce[buf]);
      }
      if (live) {
        float o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = ok ? __fmul_rn(a.rho, acc[j]) : __int_as_float(0x7fc00000);
        T* dst = a.pre + grow * H + h0 + hc * 16;
        st16(dst, V8<T>::pack(o));
        st16(dst + 8, V8<T>::pack(o + 8));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ------------------------------------------------------------------ host --

bool make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  return make_tmap_2d_sw128(m, base, bf16, inner, outer, box_outer);
}

// 3D map over 16-bit tiles of 128 rows x 64 columns stored contiguously
// ([tile][row][column]), box = one whole tile, 128-byte swizzle.
bool make_tile_map(CUtensorMap* m, const void* base, bool bf16, uint64_t tiles) {
  auto fn = tmap_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(kBM), tiles};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(kBM) * 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBM), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D map viewing a row-major [outer, inner] 16-bit matrix (inner % 64 == 0)
// as [inner/64 column chunks][outer rows][64 columns]; box = all chunks of
// `box_rows` rows, 128-byte swizzle. One copy then lands the chunks one after
// another in shared memory, each a 128-byte-swizzled MN-major block.
bool make_chunk_map(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t outer, uint32_t box_rows) {
  auto fn = tmap_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {64, outer, inner / 64};
  const cuuint64_t strides[2] = {inner * 2, 128};
  const cuuint32_t box[3] = {64, box_rows, static_cast<cuuint32_t>(inner / 64)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D map viewing a row-major [R, C*H] 16-bit matrix as [C branches][R rows]
// [H columns]; box {64 columns, 64 rows, gc branches}, 128-byte swizzle: one
// copy lands a K block of 64 columns of gc consecutive branches, branch after
// branch, each a 128-byte-swizzled MN-major block.
bool make_branch_map(CUtensorMap* m, const void* base, bool bf16, uint64_t H, uint64_t R, uint64_t C, uint32_t gc) {
  auto fn = tmap_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {H, R, C};
  const cuuint64_t strides[2] = {C * H * 2, H * 2};
  const cuuint32_t box[3] = {64, 64, gc};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kSmemBudget = 220 * 1024;

// K split of the down projection. Batches of up to kSmallRows rows have few
// 128-row tiles, so K is cut finer (slices of 256, or the largest of 128/64
// that divides C*H) to give the tensor-core kernel enough CTAs; larger batches
// split by branch. Within each regime the split is fixed, so a row's bits do
// not depend on the batch size; across the boundary the summation order
// differs (as it does between the decode and prefill paths).
constexpr int64_t kSmallRows = 512;
int k_per_split_for(int64_t rows, int C, int H) {
  if (rows > kSmallRows) return H;
  const int CH = C * H;
  for (int ks : {256, 128, 64})
    if (CH % ks == 0) return std::min(ks, H);
  return H;
}

struct PfLayout {
  size_t hn, part, d, sig16, total;
};
PfLayout pf_layout(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  const size_t es = dtype_size(dt), CH = static_cast<size_t>(C) * H;
  const size_t ksplit = CH / k_per_split_for(rows, C, H);
  PfLayout L;
  L.hn = 0;  // whole 128-row tiles
  L.part = align_up(L.hn + static_cast<size_t>((rows + kBM - 1) / kBM) * kBM * CH * es, 256);
  L.d = align_up(L.part + ksplit * rows * (R + 16) * 4, 256);
  L.sig16 = align_up(L.d + rows * static_cast<size_t>(R) * es, 256);  // fp16: the gate table
  L.total = align_up(L.sig16 + (dt == HC_F16 ? static_cast<size_t>(kS16Bytes) : 0), 256);
  return L;
}

template <typename T, bool BF16>
cudaError_t run_prefill(const Problem& p) {
  const PfLayout WL = pf_layout(p.rows, p.C, p.H, p.R, p.dt);
  char* ws = static_cast<char*>(p.workspace);
  T* hn = reinterpret_cast<T*>(ws + WL.hn);
  float* part = reinterpret_cast<float*>(ws + WL.part);
  T* d = reinterpret_cast<T*>(ws + WL.d);
  const int C = p.C, H = p.H, R = p.R, CH = C * H;
  const int64_t rows = p.rows;
  cudaError_t e;

  const size_t nsm = static_cast<size_t>(CH + (p.prev_out != nullptr ? H : 0)) * sizeof(T);
  auto norm = [&](auto kern) {
    const int nv = CH / 8;
    const unsigned nthr = static_cast<unsigned>(std::max(32, (nv + kNormVec - 1) / kNormVec + 31) / 32 * 32);
    return launch_pdl(kern, dim3(static_cast<unsigned>(rows)), dim3(nthr), nsm, p.stream, 1u,
                      static_cast<const T*>(p.streams), static_cast<const T*>(p.prev_out),
                      static_cast<const T*>(p.prev_gate), static_cast<const T*>(p.norm_scale), H, p.eps,
                      static_cast<T*>(p.streams_out), hn);
  };
  switch (C) {
    case 1: e = ensure_smem<pf_norm<T, 1>>(nsm); if (e == cudaSuccess) e = norm(pf_norm<T, 1>); break;
    case 2: e = ensure_smem<pf_norm<T, 2>>(nsm); if (e == cudaSuccess) e = norm(pf_norm<T, 2>); break;
    case 4: e = ensure_smem<pf_norm<T, 4>>(nsm); if (e == cudaSuccess) e = norm(pf_norm<T, 4>); break;
    default: e = ensure_smem<pf_norm<T, 8>>(nsm); if (e == cudaSuccess) e = norm(pf_norm<T, 8>); break;
  }
  if (e != cudaSuccess) return e;
  uint16_t* sig16 = reinterpret_cast<uint16_t*>(ws + WL.sig16);
  if (!BF16) {
    // the fp16 gate table, between pf_norm and pf_down (see pf_sig16_table)
    e = launch_pdl(pf_sig16_table, dim3((2 * kS16Half + 255) / 256), dim3(256), 0, p.stream, 1u, sig16, 1);
    if (e != cudaSuccess) return e;
  }

  const unsigned mtiles = static_cast<unsigned>((rows + kBM - 1) / kBM);
  PfDownArgs da;
  const uint64_t hn_tiles = static_cast<uint64_t>(mtiles) * (CH / 64);
  if (!make_tile_map(&da.tm_a, hn, BF16, hn_tiles) || !make_chunk_map(&da.tm_b, p.down_w, BF16, R, CH, kBK))
    return cudaErrorInvalidValue;
  da.wi = static_cast<const uint16_t*>(p.inject_w);
  da.part = part;
  da.rows = static_cast<int>(rows);
  da.R = R;
  da.C = C;
  da.k_per_split = k_per_split_for(rows, C, H);
  da.kblocks = CH / 64;
  const unsigned ksplit = static_cast<unsigned>(CH / da.k_per_split);
  const int dstage = kATileBytes + (R / 64 + 1) * kBoxBytes;
  const int wi_stage = (da.k_per_split * C * 2 + 15) / 16 * 16;
  da.stages = std::max(1, std::min(4, (kSmemBudget - 1024 - wi_stage - static_cast<int>(sizeof(PipeBars))) / dstage));
  const size_t dsm = 1024 + static_cast<size_t>(da.stages) * dstage + wi_stage + sizeof(PipeBars);
  e = ensure_smem<pf_down<BF16>>(dsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(pf_down<BF16>, dim3(mtiles, ksplit), dim3(kTcThreads), dsm, p.stream, 1u, da);
  if (e != cudaSuccess) return e;

  const Attrs at{p.eps, p.rho, p.alpha, p.gate_div, p.gate_mul};
  if (ksplit > 8 && rows <= kMidColsRows)
    e = launch_pdl(pf_mid_cols<T>, dim3(static_cast<unsigned>((rows * (R + C) + 255) / 256)), dim3(256), 0, p.stream,
                   1u, static_cast<const float*>(part), static_cast<int>(ksplit), rows, R, C, at, d,
                   static_cast<T*>(p.post_gate));
  else
    e = launch_pdl(ksplit > 8 ? pf_mid<T, true> : pf_mid<T, false>,
                   dim3(static_cast<unsigned>((rows + kMidRows - 1) / kMidRows)), dim3(kMidCols, kMidRows), 0,
                   p.stream, 1u, static_cast<const float*>(part), static_cast<int>(ksplit), rows, R, C, at, d,
                   static_cast<T*>(p.post_gate));
  if (e != cudaSuccess) return e;

  PfUpArgs<T> ua;
  const int GC = C < 4 ? C : 4;
  if (!make_map(&ua.tm_a, d, BF16, R, rows, kBM) || !make_branch_map(&ua.tm_b, p.up_w, BF16, H, R, C, GC) ||
      !make_tile_map(&ua.tm_hn, hn, BF16, hn_tiles))
    return cudaErrorInvalidValue;
  ua.hn = hn;
  ua.sig16 = sig16;
  ua.pre = static_cast<T*>(p.pre_output);
  ua.rows = static_cast<int>(rows);
  ua.C = C; ua.H = H; ua.R = R;
  ua.rho = p.rho;
  // shared memory: the operand stages (two in fp16, whose table is larger),
  // the sigmoid table and barriers, then as many hn slots (2..6) as the
  // budget leaves
  ua.stages = BF16 ? kUpStages : 2;
  const size_t fixed = 1024 + static_cast<size_t>(ua.stages) * (kATileBytes + GC * kBoxBytes) +
                       (BF16 ? kSigBytes : kS16Bytes) + sizeof(UpBars);
  const int nh = static_cast<int>(std::min<size_t>(kHnSlotsMax, (kSmemBudget - fixed) / kHnBoxBytes));
  if (nh < 2) return cudaErrorInvalidValue;
  ua.nbuf = nh;
  const size_t usm = fixed + static_cast<size_t>(nh) * kHnBoxBytes;
  e = ensure_smem<pf_up<T, BF16>>(usm);
  if (e != cudaSuccess) return e;
  const int n_tiles = static_cast<int>(mtiles) * (H / 64);
  const int grid = std::max(1, std::min(n_tiles, p.num_sms));
  return launch_pdl(pf_up<T, BF16>, dim3(grid), dim3(kUpThreads), usm, p.stream, 1u, ua);
}

}  // namespace

cudaError_t launch_sigmoid_table_codes(float* g, cudaStream_t s) {
  sigmoid_table_codes<<<128, 256, 0, s>>>(g);
  return cudaGetLastError();
}

size_t sigmoid_table16_bytes() { return kS16Bytes; }

cudaError_t launch_sigmoid_table16_codes(void* table, float* g, cudaStream_t s) {
  pf_sig16_table<<<(2 * kS16Half + 255) / 256, 256, 0, s>>>(static_cast<uint16_t*>(table), 0);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = ensure_smem<sigmoid_table16_codes>(kS16Bytes);
  if (e != cudaSuccess) return e;
  sigmoid_table16_codes<<<128, 256, kS16Bytes, s>>>(static_cast<const uint16_t*>(table), g);
  return cudaGetLastError();
}

bool prefill_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  if (dt != HC_BF16 && dt != HC_F16) return false;
  if (rows < 9 || rows > (int64_t{1} << 24)) return false;
  if (!(C == 1 || C == 2 || C == 4 || C == 8)) return false;
  if (H % 64 != 0 || R % 64 != 0 || R > 448) return false;  // R + 16 inject columns <= 512
  if (static_cast<int64_t>(C) * H > kNormVec * kNormMaxThreads * 8) return false;
  return tmap_encoder() != nullptr;
}

size_t prefill_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  return pf_layout(rows, C, H, R, dt).total;
}

cudaError_t launch_prefill(const Problem& p) {
  return p.dt == HC_BF16 ? run_prefill<__nv_bfloat16, true>(p) : run_prefill<__half, false>(p);
}

unsigned int read_pf_wait_timeouts(bool reset) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_pf_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_pf_wait_timeouts, &z, sizeof(z));
  }
  return v;
}

}  // namespace hc
