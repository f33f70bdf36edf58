// Decode path for fp16 / bf16 I/O (rows <= 8) with both projections on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// Same block and the same two-kernel structure as hc_decode_tc.cu (split-K
// down projection with a per-cluster reduction, then the up projection and
// the pre-mix, linked by programmatic dependent launch); see that file for the
// data flow. What differs is the contraction. Both projections are computed
// transposed, out^T = W^T * act^T, with
//   A = the weight tile, M = 128 output columns x K, MN-major (the weights are
//       row-major K x N in memory), 128-byte swizzle, written into shared
//       memory by 16-byte cp.async chunks at their swizzled positions;
//   B = the activation rows, N = 16 (rows padded with zeros), K-major,
//       128-byte swizzle, written by the threads that compute them;
//   D = fp32 in tensor memory: lane = output column, column = row.
// A thread issuing tcgen05.mma pays a fixed cost per instruction (measured ~76
// cycles, the same for N = 16 and 64), so the MMAs are spread over several
// issuing warps, each committing to a shared mbarrier: one per 128-column tile
// in dec_down, four K ranges into four accumulators (added in a fixed order)
// in dec_up. Each warp then reads 32 output columns x 16 rows per tcgen05.ld.
// This keeps the contraction off the load/store and FMA pipes entirely.
//
//   dec_down_um: the slice's A = [Wd | Wi] widened to MT tiles of 128 columns;
//     the C inject columns sit at columns R..R+C-1 (in the padding of the
//     last tile). Partial sums go to the rank that owns each 32-column group,
//     by st.async into its shared memory, then in rank order to the workspace.
//   dec_up_um: HS = 128 columns of branch c per CTA (one M tile).
#include <algorithm>
#include <cooperative_groups.h>
#include <type_traits>

#include "hc_async.cuh"
#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_tc.cuh"
#include "hc_vec.cuh"

namespace cg = cooperative_groups;

namespace hc {

// Count of bounded waits that gave up (diagnostic; see hc_debug_wait_timeouts).
__device__ unsigned int g_um_wait_timeouts = 0;

namespace {

constexpr int kUmRowsN = 16;    // MMA N: activation rows, padded
constexpr int kUmMaxMT = 4;     // dec_down: at most 4 tiles of 128 columns (R + 8 <= 512)
constexpr int kUpHS = 128;      // dec_up: columns per CTA (one M tile)
constexpr int kUpIssuers = 4;   // dec_up: issuing warps = accumulators
constexpr int kKBlock = 2048;   // one 64-k block of B: 16 rows x 128 bytes
constexpr size_t kUmDownCap = 120 * 1024, kUmUpCap = 150 * 1024;

__host__ __device__ inline uint32_t a16(uint32_t x) { return (x + 15u) & ~15u; }
__host__ __device__ inline uint32_t a1024(uint32_t x) { return (x + 1023u) & ~1023u; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of element (row, col) in a 128-byte-swizzled region of 128-byte
// rows: 16-byte chunk (col / 8) of row `row` is stored at chunk (col / 8) ^ (row % 8).
__host__ __device__ inline uint32_t sw128(int row, int col_in_64) {
  return static_cast<uint32_t>(row * 128 + ((((col_in_64 >> 3) ^ (row & 7)) & 7) << 4) + (col_in_64 & 7) * 2);
}

// B operand (activation rows x K, K-major): k-block kb of 64 holds 16 rows.
__host__ __device__ inline uint32_t b_off(int row, int k) { return static_cast<uint32_t>((k >> 6) * kKBlock) + sw128(row, k & 63); }

// Workspace position of the cluster-summed partial of column `col` (down
// columns 0..R-1, then inject columns R..R+7) for row b of cluster p. With
// one row, (p, b, col) row-major with NCP columns: dec_up_um pulls the whole
// array with one bulk copy. With more rows (split mode, where up rank c
// reduces the `per` down columns c*per.. and rank 0 the inject columns) the
// down columns are grouped by the rank that consumes them, (p, rank, b,
// per), followed by the inject columns as (p, b, 8): each rank pulls one
// contiguous block per cluster and rank 0 one block of inject columns.
__host__ __device__ inline int64_t part_index(bool split, int p, int b, int col, int B, int C, int R, int NCP, int per,
                                              int NCLU) {
  if (!split) return (static_cast<int64_t>(p) * B + b) * NCP + col;
  if (col < R) {
    const int rank = col / per;
    return ((static_cast<int64_t>(p) * C + rank) * B + b) * per + (col - rank * per);
  }
  return static_cast<int64_t>(NCLU) * C * B * per + (static_cast<int64_t>(p) * B + b) * 8 + (col - R);
}

// --------------------------------------------------------------- dec_down --

struct DownSmem {
  uint32_t a, b, wis, ns, ss, wsum, inv, recv, bars, total;
};
// A: 2*MT boxes of 64 columns x KS rows; B: ceil(KS/64) blocks. The region
// starts 1024-aligned (the dynamic shared memory base is aligned by hand).
__host__ __device__ inline DownSmem down_smem(int MB, int KS, int R, int C, int CL, int nwarps) {
  const int MT = ceil_div(R + 8, 128), TPR = ceil_div(MT * 4, CL);
  DownSmem L;
  L.a = 0;
  L.b = a1024(L.a + 2 * MT * KS * 128);
  L.wis = a16(L.b + ceil_div(KS, 64) * kKBlock);
  L.ns = a16(L.wis + KS * C * 2);
  L.ss = a16(L.ns + KS * 4);
  L.wsum = a16(L.ss + MB * KS * 4);
  L.inv = a16(L.wsum + nwarps * MB * 4);
  L.recv = a16(L.inv + MB * 4);
  L.bars = a16(L.recv + CL * MB * TPR * 32 * 4);
  L.total = L.bars + 32 + 1024;  // barriers, TMEM address; slack for aligning the base
  return L;
}

template <typename T>
struct DownArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wd, *wi;
  T* sout;
  float* inv_ws;   // (B, C)
  float* part_ws;  // one row: (NCLU, B, NCP), NCP = R + 8; split: see part_index
  int B, C, H, R, KS, CL, NCP, split, per, NCLU;
  float eps;
  int weights_static;
};

template <typename T>
__device__ __forceinline__ uint32_t idesc_t() {
  return idesc_f16(std::is_same<T, __nv_bfloat16>::value, 128, kUmRowsN, true, false);
}

// 384 threads; registers capped at 64 so that a CTA of dec_up_um keeps fitting
// beside it (measured: without the cap the 2-8 row variants take more
// registers and the two kernels of a block stop overlapping under PDL,
// costing 5-6 us per block).
template <typename T, int MB>
__global__ void __maxnreg__(64) dec_down_um(const DownArgs<T> a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  constexpr int VEC = 8;
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  const int B = a.B, C = a.C, H = a.H, R = a.R, KS = a.KS, CL = a.CL, NCP = a.NCP;
  const int MT = ceil_div(R + 8, 128), TPR = ceil_div(MT * 4, CL), OC = TPR * 32;
  const int boxb = KS * 128;
  const DownSmem L = down_smem(MB, KS, R, C, CL, nwarps);
  uint8_t* sA = smem + L.a;
  uint8_t* sB = smem + L.b;
  const T* wis = reinterpret_cast<const T*>(smem + L.wis);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* ss = reinterpret_cast<float*>(smem + L.ss);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  float* inv_s = reinterpret_cast<float*>(smem + L.inv);
  float* recv_s = reinterpret_cast<float*>(smem + L.recv);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* mma_bar = rbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbar + 2);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int slice = blockIdx.x, k0 = slice * KS;
  const int c = k0 / H, hk0 = k0 - c * H;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const bool pro = a.prev_out != nullptr;
  // 32-column groups (pairs of tile, lane quarter) this rank owns: columns
  // [c_lo, c_lo + ncol) of [down | inject]
  const int c_lo = rank * OC, ncol = max(0, min(NCP, c_lo + OC) - c_lo);
  // inject columns R..R+C-1: box R/64, 16-byte chunk (R%64)/8
  const int ibox = R / 64, ich = (R % 64) / 8;

  if (tid == 0) {
    mbar_init(rbar, 1);
    mbar_init(mma_bar, MT);  // one commit per tile's issuing warp
    mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(CL * ncol * B * 4));
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  cluster_arrive_relaxed();
  // zero B (rows >= B and k >= KS stay zero) and the A chunks no copy writes:
  // box ibox from chunk ich on, and every later box
  #pragma unroll 1
  for (int i = tid; i < ceil_div(KS, 64) * kKBlock / 16; i += nthr) reinterpret_cast<uint4*>(sB)[i] = make_uint4(0, 0, 0, 0);
  #pragma unroll 1
  for (int i = tid; i < (2 * MT - ibox) * KS * 8; i += nthr) {
    const int bx = ibox + i / (KS * 8), rem = i - (bx - ibox) * KS * 8, r = rem >> 3, ch = rem & 7;
    if (bx > ibox || ch >= ich)
      *reinterpret_cast<uint4*>(sA + bx * boxb + r * 128 + ((ch ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // weights: 16-byte chunks of each K row into their swizzled positions; warp
  // 0 also copies the inject slice and, once it lands, places it in column R..
  auto issue_weights = [&]() {
    const int cpr = R / 8;
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(a.wd + static_cast<int64_t>(k0) * R);
    #pragma unroll 1
    for (int i = tid; i < KS * cpr; i += nthr) {
      const int r = i / cpr, q = i - r * cpr;
      cp_async16(sA + (q >> 3) * boxb + r * 128 + (((q & 7) ^ (r & 7)) << 4), gsrc + static_cast<size_t>(r) * R * 2 + q * 16);
    }
    if (warp == 0) {
      const unsigned char* isrc = reinterpret_cast<const unsigned char*>(a.wi + static_cast<int64_t>(k0) * C);
      #pragma unroll 1
      for (int i = lane; i < KS * C * 2 / 16; i += 32) cp_async16(smem + L.wis + i * 16, isrc + i * 16);
    }
    cp_async_commit();
    #pragma unroll 1
    for (int i = tid; i < KS / VEC; i += nthr) {
      float f[VEC];
      V8<T>::unpack(ld16(a.ns + k0 + i * VEC), f);
#pragma unroll
      for (int j = 0; j < VEC; ++j) ns_s[i * VEC + j] = f[j];
    }
  };
  auto place_inject = [&]() {
    cp_async_wait_all();
    __syncwarp();
    #pragma unroll 1
    for (int i = lane; i < KS * C; i += 32) {
      const int r = i / C, cc = i - r * C;
      *reinterpret_cast<T*>(sA + ibox * boxb + r * 128 + ((ich ^ (r & 7)) << 4) + cc * 2) = wis[r * C + cc];
    }
    __syncwarp();
  };
  if (a.weights_static) {
    issue_weights();
    if (warp == 0) place_inject();
  }
  pdl_wait();
  if (!a.weights_static) issue_weights();
  pdl_trigger();

  // ---- one pass over branch c of every row: S, its sum of squares, the
  // slice's S and streams_out for the slice ----
  const int NVr = H / VEC;
  float ssq[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) ssq[b] = 0.0f;
  constexpr int RB = MB < 4 ? MB : 4;  // rows whose loads are in flight together
  #pragma unroll 1
  for (int v = tid; v < NVr; v += nthr) {
    const int kk = v * VEC - hk0;
    const bool mine = kk >= 0 && kk < KS;
#pragma unroll
    for (int b0 = 0; b0 < MB; b0 += RB) {
      uint4 sv[RB], pv[RB];
      float gt[RB];
#pragma unroll
      for (int bi = 0; bi < RB; ++bi)
        if (b0 + bi < B) {
          const int b = b0 + bi;
          sv[bi] = ld16(a.streams + b * CH + static_cast<int64_t>(c) * H + v * VEC);
          if (pro) {
            pv[bi] = ld16(a.prev_out + static_cast<int64_t>(b) * H + v * VEC);
            gt[bi] = ldf(a.prev_gate + b * C + c);
          }
        }
#pragma unroll
      for (int bi = 0; bi < RB; ++bi)
        if (b0 + bi < B) {
          const int b = b0 + bi;
          float sf[VEC];
          V8<T>::unpack(sv[bi], sf);
          if (pro) {
            float pf[VEC];
            V8<T>::unpack(pv[bi], pf);
#pragma unroll
            for (int j = 0; j < VEC; ++j) sf[j] = prologue_s<T>(sf[j], gt[bi], pf[j]);
          }
#pragma unroll
          for (int j = 0; j < VEC; ++j) ssq[b] = fmaf(sf[j], sf[j], ssq[b]);
          if (mine) {
#pragma unroll
            for (int j = 0; j < VEC; ++j) ss[b * KS + kk + j] = sf[j];
            if (a.sout != nullptr) st16(a.sout + b * CH + k0 + kk, pro ? V8<T>::pack(sf) : sv[bi]);
          }
        }
    }
  }
#pragma unroll
  for (int b = 0; b < MB; ++b) {
    const float w = warp_sum(ssq[b]);
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
  // hn of the slice as T, into B at its swizzled position
  #pragma unroll 1
  for (int i = tid; i < B * KS; i += nthr) {
    const int b = i / KS, kk = i - b * KS;
    *reinterpret_cast<T*>(sB + b_off(b, kk)) = Ty<T>::from_f(norm_hn<T>(ss[i], inv_s[b], ns_s[kk]));
  }
  if (!a.weights_static && warp == 0) place_inject();
  cp_async_wait_all();
  fence_proxy_async_smem();  // generic-proxy writes of A and B, visible to the tensor core
  __syncthreads();

  // ---- [down | inject]^T = A * hn^T: tile mt (KS/16 k-steps) issued by
  // lane 0 of warp mt ----
  if (warp < MT && lane == 0) {
    tc_fence_after();
    const int mt = warp;
    const uint32_t abase = smem_addr(sA) + mt * 2 * boxb, bbase = smem_addr(sB);
    for (int kk = 0; kk < KS / 16; ++kk) {
      const uint64_t adesc = smem_desc_sw128(abase + kk * 2048, static_cast<uint32_t>(boxb), 1024);
      const uint64_t bdesc = smem_desc_sw128(bbase + (kk >> 2) * kKBlock + (kk & 3) * 32, 16, 1024);
      mma_f16(tmem + mt * kUmRowsN, adesc, bdesc, idesc_t<T>(), kk > 0 ? 1u : 0u);
    }
    mma_commit(mma_bar);
  }
  const bool ok = mbar_wait(mma_bar, 0, &g_um_wait_timeouts);
  tc_fence_after();

  // ---- each warp reads 32-column groups p = (tile p/4, lane quarter p%4)
  // with p % 4 == warp % 4 (a warp reaches only its own lane quarter) and
  // sends row values to the rank that owns the group ----
  const float qnan = __int_as_float(0x7fc00000);
  cluster_wait();
  #pragma unroll 1
  for (int p = warp; p < MT * 4; p += nwarps) {
    const int q = p & 3, mt = p >> 2;
    uint32_t v[16];
    tmem_ld16_nowait(tmem + (static_cast<uint32_t>(q * 32) << 16) + mt * kUmRowsN, v);
    tmem_ld_wait_r(v);
    const int col = p * 32 + lane;  // = mt * 128 + q * 32 + lane
    if (col < NCP) {
      const int ow = col / OC, lc = col - ow * OC;
      const uint32_t rb = mapa_shared(smem_addr(rbar), ow);
#pragma unroll
      for (int b = 0; b < MB; ++b)
        if (b < B) {
          const uint32_t slot = smem_addr(recv_s + (rank * MB + b) * OC + lc);
          st_async_b32(mapa_shared(slot, ow), ok ? v[b] : __float_as_uint(qnan), rb);
        }
    }
  }
  const bool rok = mbar_wait(rbar, 0, &g_um_wait_timeouts);

  // ---- sum the received partials of the owned columns in rank order ----
  const int cluster_id = slice / CL;
  #pragma unroll 1
  for (int i = tid; i < B * ncol; i += nthr) {
    const int b = i / ncol, lc = i - b * ncol;
    float x[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) x[r] = r < CL ? recv_s[(r * MB + b) * OC + lc] : 0.0f;
    float t = 0.0f;
#pragma unroll
    for (int r = 0; r < 8; ++r)
      if (r < CL) t += x[r];
    a.part_ws[part_index(a.split != 0, cluster_id, b, c_lo + lc, B, C, R, NCP, a.per, a.NCLU)] = rok ? t : qnan;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ----------------------------------------------------------------- dec_up --

struct UpSmem {
  uint32_t a, b, st, hn, ns, mix, bars, total;
};
__host__ __device__ inline UpSmem up_smem(int MB, int R, int C, int st_bytes) {
  const int R16 = (R + 15) / 16 * 16, HSc = kUpHS / C;
  UpSmem L;
  L.a = 0;
  L.b = a1024(L.a + 2 * R16 * 128);
  L.st = a16(L.b + ceil_div(R16, 64) * kKBlock);
  L.hn = a16(L.st + st_bytes);
  L.ns = a16(L.hn + MB * kUpHS * 4);
  L.mix = a16(L.ns + kUpHS * 4);
  L.bars = a16(L.mix + C * MB * HSc * 4);
  L.total = L.bars + 48 + 1024;
  return L;
}

template <typename T>
struct UpArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wu;
  const float* inv_ws;
  const float* part_ws;
  T *pre, *post;
  int B, C, H, R, NCLU, NCP, split, per, st_bytes;
  Attrs at;
};

// post_gate for every row: the inject partials summed in cluster order. One
// CTA runs it; kept out of line so that the others never fetch its code.
template <typename T>
__device__ __noinline__ void dec_post_gate(const float* st, size_t inj_off, bool split, int B, int C, int NCLU, int NCP,
                                           int R, bool ok, T* post, float gate_div, float gate_mul) {
  const float qnan = __int_as_float(0x7fc00000);
  #pragma unroll 1
  for (int i = threadIdx.x; i < B * C; i += blockDim.x) {
    const int b = i / C, cc = i - b * C;
    const float* src = split ? st + inj_off + static_cast<size_t>(b) * 8 + cc : st + static_cast<size_t>(b) * NCP + R + cc;
    const size_t stride = split ? static_cast<size_t>(B) * 8 : static_cast<size_t>(B) * NCP;
    const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
    stf(post + b * C + cc, ok ? post_gate_of<T>(rT<T>(x), gate_div, gate_mul) : qnan);
  }
}

template <typename T, int MB>
__global__ void __launch_bounds__(512) dec_up_um(const UpArgs<T> a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  constexpr int VEC = 8, HS = kUpHS;
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, C = a.C, H = a.H, R = a.R, NCLU = a.NCLU, NCP = a.NCP;
  const int R16 = (R + 15) / 16 * 16, HSc = HS / C, boxb = R16 * 128;
  const UpSmem L = up_smem(MB, R, C, a.st_bytes);
  uint8_t* sA = smem + L.a;
  uint8_t* sB = smem + L.b;
  float* st = reinterpret_cast<float*>(smem + L.st);
  float* hn_s = reinterpret_cast<float*>(smem + L.hn);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* mix_s = reinterpret_cast<float*>(smem + L.mix);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bars);  // partial sums landed
  uint64_t* dbar = bar + 1;                                     // d from every rank landed (split mode)
  uint64_t* mbar = bar + 2;                                     // pre-mix products landed
  uint64_t* mma_bar = bar + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);

  cg::cluster_group cluster = cg::this_cluster();
  const int c = static_cast<int>(cluster.block_rank());
  const int q = blockIdx.x / C;
  const int h0 = q * HS;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const int64_t col0 = static_cast<int64_t>(c) * H + h0;
  const bool pro = a.prev_out != nullptr;
  const bool do_post = (q == 0 && c == 0);
  // one row needs no split (the host never sets it then): the code is left out
  const bool split = MB > 1 && a.split != 0;

  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(dbar, 1);
    mbar_init(mbar, 1);
    mbar_init(mma_bar, min(kUpIssuers, (R + 15) / 16));  // one commit per issuing warp
    mbar_arrive_expect_tx(dbar, split ? static_cast<uint32_t>(R * B * 2) : 0u);
    mbar_arrive_expect_tx(mbar, C > 1 ? static_cast<uint32_t>(C * HSc * B * 4) : 0u);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  cluster_arrive_relaxed();
  // The up weights and the block inputs are never written by the preceding
  // dec_down_um, which triggers its dependents only after its own wait:
  // reading them before griddepcontrol.wait is safe. A: 16 chunks of 16 bytes
  // per K row (two boxes of 64 columns), at their swizzled positions.
  {
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(a.wu + col0);
    #pragma unroll 1
    for (int i = tid; i < R * 16; i += nthr) {
      const int r = i >> 4, qd = i & 15;
      cp_async16(sA + (qd >> 3) * boxb + r * 128 + (((qd & 7) ^ (r & 7)) << 4),
                 gsrc + (static_cast<int64_t>(r) * CH) * 2 + qd * 16);
    }
    cp_async_commit();
    #pragma unroll 1
    for (int i = tid; i < (R16 - R) * 16; i += nthr) {
      const int r = R + (i >> 4), qd = i & 15;
      *reinterpret_cast<uint4*>(sA + (qd >> 3) * boxb + r * 128 + (((qd & 7) ^ (r & 7)) << 4)) = make_uint4(0, 0, 0, 0);
    }
  }
  // B: zero rows >= B, and columns >= R of rows < B (whole 16-byte chunks, R
  // is a multiple of 8). The rest is written with d, possibly by peer CTAs.
  {
    const int nkb = ceil_div(R16, 64);
    #pragma unroll 1
    for (int i = tid; i < nkb * 16 * 8; i += nthr) {
      const int kb = i / 128, rem = i - kb * 128, row = rem >> 3, ch = rem & 7;
      const int kfirst = kb * 64 + ch * 8;
      if (row >= B || kfirst >= R)
        *reinterpret_cast<uint4*>(sB + kb * kKBlock + row * 128 + ((ch ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
    }
  }
  const int nvh = HS / VEC;
  #pragma unroll 1
  for (int i = tid; i < B * nvh; i += nthr) {
    const int b = i / nvh, qv = i - b * nvh;
    float sf[VEC];
    V8<T>::unpack(ld16(a.streams + b * CH + col0 + qv * VEC), sf);
    if (pro) {
      float pf[VEC];
      V8<T>::unpack(ld16(a.prev_out + static_cast<int64_t>(b) * H + h0 + qv * VEC), pf);
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
    V8<T>::unpack(ld16(a.ns + col0 + i * VEC), f);
#pragma unroll
    for (int j = 0; j < VEC; ++j) ns_s[i * VEC + j] = f[j];
  }
  tc_fence_before();
  pdl_wait();
  pdl_trigger();
  cluster_wait();
  __syncthreads();  // barriers, TMEM address, S, ns and the zeroed regions visible CTA-wide
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---- pull the down partials into shared memory ----
  const int ncols = split ? max(0, min(R, (c + 1) * a.per) - c * a.per) : 0;
  const size_t inj_off = static_cast<size_t>(NCLU) * B * a.per;  // floats (split layout)
  if (warp == 0) {
    uint32_t bytes;
    if (!split) bytes = static_cast<uint32_t>(NCLU * B * NCP * 4);
    else bytes = static_cast<uint32_t>(NCLU * B * a.per * 4 + (do_post ? NCLU * B * 32 : 0));
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    if (!split) {
      if (lane == 0) bulk_g2s(st, a.part_ws, bytes, bar);
    } else {
      // one block of B * per partials per cluster for this rank, and (rank 0
      // of the first column tile) one block of every cluster's inject partials
      #pragma unroll 1
      for (int p = lane; p < NCLU; p += 32)
        bulk_g2s(st + static_cast<size_t>(p) * B * a.per,
                 a.part_ws + (static_cast<int64_t>(p) * C + c) * B * a.per, static_cast<uint32_t>(B * a.per * 4), bar);
      if (do_post && lane == 0)
        bulk_g2s(st + inj_off, a.part_ws + static_cast<int64_t>(NCLU) * C * B * a.per,
                 static_cast<uint32_t>(NCLU * B * 32), bar);
    }
  }
  float inv_r[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) inv_r[b] = b < B ? a.inv_ws[b * C + c] : 0.0f;
  const bool ok = mbar_wait(bar, 0, &g_um_wait_timeouts);
  const float qnan = __int_as_float(0x7fc00000);

  // ---- d = ScaledSiLU(rT(sum of the partials in cluster order)) as T, into B ----
  if (!split) {
    const size_t stride = static_cast<size_t>(B) * NCP;
    #pragma unroll 1
    for (int i = tid; i < B * R; i += nthr) {
      const int b = i / R, col = i - b * R;
      const float* src = st + static_cast<size_t>(b) * NCP + col;
      const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
      *reinterpret_cast<T*>(sB + b_off(b, col)) = Ty<T>::from_f(ok ? scaled_silu_t<T>(rT<T>(x), a.at.alpha) : qnan);
    }
  }
  if constexpr (MB > 1) if (split) {
    const int npair = ncols / 2;
    const size_t stride = static_cast<size_t>(B) * a.per;
    #pragma unroll 1
    for (int i = tid; i < B * npair; i += nthr) {
      const int b = i / npair, lc = 2 * (i - b * npair);
      const float* src = st + static_cast<size_t>(b) * a.per + lc;
      const float x0 = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
      const float x1 = ordered_sum(NCLU, [&](int p) { return src[p * stride + 1]; });
      T dv[2];
      dv[0] = Ty<T>::from_f(ok ? scaled_silu_t<T>(rT<T>(x0), a.at.alpha) : qnan);
      dv[1] = Ty<T>::from_f(ok ? scaled_silu_t<T>(rT<T>(x1), a.at.alpha) : qnan);
      const uint32_t packed = *reinterpret_cast<const uint32_t*>(dv);
      const uint32_t slot = smem_addr(sB + b_off(b, c * a.per + lc));  // an even column pair is contiguous
      for (int pr = 0; pr < C; ++pr) st_async_b32(mapa_shared(slot, pr), packed, mapa_shared(smem_addr(dbar), pr));
    }
  }
  if (do_post) dec_post_gate<T>(st, inj_off, split, B, C, NCLU, NCP, R, ok, a.post, a.at.gate_div, a.at.gate_mul);
  #pragma unroll 1
  for (int i = tid; i < B * HS; i += nthr) {
    const int b = i / HS, h = i - b * HS;
    float iv = inv_r[0];
#pragma unroll
    for (int bb = 1; bb < MB; ++bb)
      if (bb == b) iv = inv_r[bb];
    hn_s[i] = norm_hn<T>(hn_s[i], iv, ns_s[h]);
  }
  cp_async_wait_all();
  bool dok = true;
  if (split) dok = mbar_wait(dbar, 0, &g_um_wait_timeouts);
  fence_proxy_async_smem();  // A (cp.async) and B (d) visible to the tensor core
  __syncthreads();

  // ---- up^T = Wu^T * d^T: the R16/16 k-steps in NI contiguous ranges, range
  // j issued by lane 0 of warp j into accumulator j (TMEM columns 16j..) ----
  const int nks = R16 / 16, NI = min(kUpIssuers, nks);
  if (warp < NI && lane == 0) {
    tc_fence_after();
    const uint32_t abase = smem_addr(sA), bbase = smem_addr(sB);
    const int kb = warp * nks / NI, ke = (warp + 1) * nks / NI;
    for (int kk = kb; kk < ke; ++kk) {
      const uint64_t adesc = smem_desc_sw128(abase + kk * 2048, static_cast<uint32_t>(boxb), 1024);
      const uint64_t bdesc = smem_desc_sw128(bbase + (kk >> 2) * kKBlock + (kk & 3) * 32, 16, 1024);
      mma_f16(tmem + warp * kUmRowsN, adesc, bdesc, idesc_t<T>(), kk > kb ? 1u : 0u);
    }
    mma_commit(mma_bar);
  }
  const bool mmok = mbar_wait(mma_bar, 0, &g_um_wait_timeouts);
  tc_fence_after();

  // ---- epilogue: warp w < 4 holds columns 32w..32w+31 (its TMEM lane
  // quarter), rows in TMEM columns: g = rT(sigmoid(rT(up))), hn*g, pre-mix ----
  if (warp < 4) {
    // accumulators 0..NI-1 of this lane quarter, added as ((a0 + a1) + (a2 + a3))
    uint32_t acc[kUpIssuers][16];
    const uint32_t tq = tmem + (static_cast<uint32_t>(warp * 32) << 16);
#pragma unroll
    for (int j = 0; j < kUpIssuers; ++j)
      if (j < NI) tmem_ld16_nowait(tq + j * kUmRowsN, acc[j]);
#pragma unroll
    for (int j = 0; j < kUpIssuers; ++j)
      if (j < NI) tmem_ld_wait_r(acc[j]);
    float v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float x[kUpIssuers];
#pragma unroll
      for (int j = 0; j < kUpIssuers; ++j) x[j] = j < NI ? __uint_as_float(acc[j][r]) : 0.0f;
      v[r] = __fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3]));
    }
    const int h = warp * 32 + lane;
    const int j = h / HSc, hl = h - j * HSc;
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B) {
        const float up = v[b];
        const float gg = sigmoid_rT<T>(rT<T>(up));
        const float prod = (dok && mmok) ? __fmul_rn(hn_s[b * HS + h], gg) : qnan;
        if (C == 1) {
          stf(a.pre + static_cast<int64_t>(b) * H + h0 + h, __fmul_rn(a.at.rho, __fadd_rn(0.0f, prod)));
        } else {
          st_async_b32(mapa_shared(smem_addr(mix_s + (c * MB + b) * HSc + hl), j), __float_as_uint(prod),
                       mapa_shared(smem_addr(mbar), j));
        }
      }
  }
  // ---- pre-mix: rank j sums features [j*HSc, (j+1)*HSc) over c = 0..C-1 ----
  if (C > 1) {
    const bool mok = mbar_wait(mbar, 0, &g_um_wait_timeouts);
    #pragma unroll 1
    for (int i = tid; i < B * HSc; i += nthr) {
      const int b = i / HSc, hl = i - b * HSc;
      float acc2 = 0.0f;
      for (int cc = 0; cc < C; ++cc) acc2 = __fadd_rn(acc2, mix_s[(cc * MB + b) * HSc + hl]);
      stf(a.pre + static_cast<int64_t>(b) * H + h0 + c * HSc + hl, mok ? __fmul_rn(a.at.rho, acc2) : qnan);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ------------------------------------------------------------ configuration

struct UmCfg {
  bool ok;
  int KS, NSL, CL, NCLU, NCP, R, down_threads, up_threads;
};

int cluster_for(int n) {
  for (int cl : {8, 4, 2})
    if (n % cl == 0) return cl;
  return 1;
}

struct Stage {
  int split, per, bytes;
};
Stage stage_for(int64_t rows, int C, int R, int NCLU, int NCP) {
  Stage s;
  // From 2 rows on each rank reduces 1/C of the columns and broadcasts d: the
  // staging stays small enough for a dec_down_um CTA to share the SM.
  s.split = (rows > 1 && C > 1) ? 1 : 0;
  s.per = ceil_div(ceil_div(R, C), 4) * 4;
  s.bytes = s.split ? static_cast<int>(NCLU * rows * s.per * 4 + NCLU * rows * 32)
                    : static_cast<int>(NCLU * rows * NCP * 4);
  return s;
}

UmCfg um_cfg(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  UmCfg g{};
  g.ok = false;
  if (dt != HC_F16 && dt != HC_BF16) return g;
  if (rows < 1 || rows > 8) return g;
  if (!(C == 1 || C == 2 || C == 4 || C == 8)) return g;
  if (R < 16 || R % 8 != 0 || R + 8 > kUmMaxMT * 128) return g;
  if (H % kUpHS != 0 || H > 16384) return g;
  const int CH = C * H;
  g.NCP = R + 8;
  g.R = R;
  g.down_threads = 12 * 32;  // a multiple of 4 warps (TMEM lane quarters)
  g.KS = 0;
  for (int ks = 16; ks <= H; ks += 16) {
    if (H % ks != 0) continue;
    if (down_smem(8, ks, R, C, cluster_for(H / ks), g.down_threads / 32).total > kUmDownCap) break;
    g.KS = ks;
    if (CH / ks <= num_sms) break;
  }
  if (g.KS == 0) return g;
  g.NSL = CH / g.KS;
  g.CL = cluster_for(H / g.KS);
  g.NCLU = g.NSL / g.CL;
  const Stage sg = stage_for(rows, C, R, g.NCLU, g.NCP);
  if (up_smem(8, R, C, sg.bytes).total > kUmUpCap) return g;
  g.up_threads = std::min(16, std::max(4, ceil_div(R, 32))) * 32;
  g.ok = true;
  return g;
}

struct Layout {
  size_t inv, part, total;
};
Layout um_layout(int64_t rows, int C, const UmCfg& g) {
  Layout L;
  L.inv = 0;
  L.part = align_up(static_cast<size_t>(rows) * C * 4, 256);
  const Stage sg = stage_for(rows, C, g.R, g.NCLU, g.NCP);
  const size_t nf = sg.split ? static_cast<size_t>(g.NCLU) * rows * (static_cast<size_t>(C) * sg.per + 8)
                             : static_cast<size_t>(g.NCLU) * rows * g.NCP;
  L.total = align_up(L.part + nf * 4, 256);
  return L;
}

template <typename T, int MB>
cudaError_t run_um_mb(const Problem& p, const UmCfg& g) {
  const Layout WL = um_layout(p.rows, p.C, g);
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
  da.C = p.C; da.H = p.H; da.R = p.R; da.KS = g.KS; da.CL = g.CL; da.NCP = g.NCP; da.NCLU = g.NCLU;
  const Stage sg = stage_for(p.rows, p.C, p.R, g.NCLU, g.NCP);
  da.split = sg.split; da.per = sg.per;
  da.eps = p.eps;
  da.weights_static = (p.flags & HC_FLAG_WEIGHTS_STATIC) ? 1 : 0;
  const size_t dsm = down_smem(MB, g.KS, p.R, p.C, g.CL, g.down_threads / 32).total;
  cudaError_t e = ensure_smem<dec_down_um<T, MB>>(dsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(dec_down_um<T, MB>, dim3(g.NSL), dim3(g.down_threads), dsm, p.stream, static_cast<unsigned>(g.CL), da);
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
  ua.B = da.B; ua.C = p.C; ua.H = p.H; ua.R = p.R; ua.NCLU = g.NCLU; ua.NCP = g.NCP;
  ua.split = sg.split; ua.per = sg.per; ua.st_bytes = sg.bytes;
  ua.at = Attrs{p.eps, p.rho, p.alpha, p.gate_div, p.gate_mul};
  const size_t usm = up_smem(MB, p.R, p.C, sg.bytes).total;
  e = ensure_smem<dec_up_um<T, MB>>(usm);
  if (e != cudaSuccess) return e;
  return launch_pdl(dec_up_um<T, MB>, dim3((p.H / kUpHS) * p.C), dim3(g.up_threads), usm, p.stream,
                    static_cast<unsigned>(p.C), ua);
}

template <typename T>
cudaError_t run_um(const Problem& p, const UmCfg& g) {
  if (p.rows <= 1) return run_um_mb<T, 1>(p, g);
  if (p.rows <= 2) return run_um_mb<T, 2>(p, g);
  if (p.rows <= 4) return run_um_mb<T, 4>(p, g);
  return run_um_mb<T, 8>(p, g);
}

}  // namespace

bool decode_um_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  return um_cfg(rows, C, H, R, dt, 148).ok;
}

size_t decode_um_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  const UmCfg g = um_cfg(rows, C, H, R, dt, num_sms);
  return g.ok ? um_layout(rows, C, g).total : 0;
}

cudaError_t launch_decode_um(const Problem& p) {
  const UmCfg g = um_cfg(p.rows, p.C, p.H, p.R, p.dt, p.num_sms);
  if (!g.ok) return cudaErrorInvalidValue;
  return p.dt == HC_F16 ? run_um<__half>(p, g) : run_um<__nv_bfloat16>(p, g);
}

unsigned int read_um_wait_timeouts(bool reset) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_um_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_um_wait_timeouts, &z, sizeof(z));
  }
  return v;
}

}  // namespace hc
