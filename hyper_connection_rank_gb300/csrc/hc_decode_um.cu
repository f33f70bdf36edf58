// Decode path for fp16 / bf16 I/O (rows <= 16) with both projections on the
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
//   dec_up_um: one M tile of 128 output columns per CTA: F = 128 / C
//     features of every branch, so the pre-mix over the branches sums in the
//     CTA's own shared memory.
#include <algorithm>
#include <atomic>
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
constexpr int kDownClusterMax = 16;  // dec_down: largest cluster (16 is a non-portable size)
constexpr int kDownWarps = 12;  // dec_down: 384 threads, a multiple of 4 warps (TMEM lane quarters)
constexpr int kUpHS = 128;      // dec_up: output columns per CTA (one M tile: C branches x 128/C features)
constexpr int kUpIssuers = 4;   // dec_up: issuing warps = accumulators
constexpr int kKBlock = 2048;   // one 64-k block of B: 16 rows x 128 bytes
constexpr size_t kUmDownCap = 120 * 1024, kUmUpCap = 150 * 1024;
constexpr size_t kUmSmPerSm = 233472;  // shared memory of an SM (228 KB)
constexpr int kUmMaxRows = 16;         // rows of one call: the MMA's N

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
// array with one bulk copy. With more rows (split mode: SR up ranks, rank c
// reducing the `per` down columns c*per.. and rank 0 the inject columns) the
// down columns are grouped by the rank that consumes them, (rank, p, b,
// per), followed by the inject columns as (p, b, 8): each rank pulls one
// contiguous block (every cluster's share of its columns) and rank 0 one
// block of inject columns. SR = 0 means no split.
__host__ __device__ inline int64_t part_index(int SR, int p, int b, int col, int B, int R, int NCP, int per, int NCLU) {
  if (SR == 0) return (static_cast<int64_t>(p) * B + b) * NCP + col;
  if (col < R) {
    const int rank = col / per;
    return ((static_cast<int64_t>(rank) * NCLU + p) * B + b) * per + (col - rank * per);
  }
  return static_cast<int64_t>(NCLU) * SR * B * per + (static_cast<int64_t>(p) * B + b) * 8 + (col - R);
}

// Phase clocks (diagnostic, hc_debug_phase_clocks): in the TIMED variants
// thread 0 of every CTA records (%globaltimer in ns, clock64 in SM cycles) at
// fixed points of the kernel into rec[CTA][point][2]. Thread 0 takes part in
// every CTA-wide barrier and wait, so its stamps mark when the CTA as a whole
// passed each point.
constexpr int kPhasePoints = 10;
constexpr int kPhaseMaxCtas = 256;
__device__ __forceinline__ void phase_stamp(unsigned long long* rec, int point) {
  unsigned long long gt;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(gt)::"memory");
  const unsigned long long ck = static_cast<unsigned long long>(clock64());
  rec[(blockIdx.x * kPhasePoints + point) * 2] = gt;
  rec[(blockIdx.x * kPhasePoints + point) * 2 + 1] = ck;
}
#define HC_PHASE(point)                                        \
  do {                                                         \
    if constexpr (TIMED) {                                     \
      if (threadIdx.x == 0) phase_stamp(a.phase, (point));     \
    }                                                          \
  } while (0)

// --------------------------------------------------------------- dec_down --

struct DownSmem {
  uint32_t a, b, wis, ns, ss, wsum, gs, recv, bars, total;
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
  L.ss = a16(L.ns + KS * 2);       // norm_scale of the slice, T
  L.wsum = a16(L.ss + MB * KS * 2);  // S of the slice, T (already rounded to T: exact)
  L.gs = a16(L.wsum + nwarps * MB * 4);  // 32-vector group sums of squares (several rows)
  L.recv = a16(L.gs + nwarps * MB * 4);
  L.bars = a16(L.recv + CL * MB * TPR * 32 * 4);
  L.total = L.bars + 48 + 1024;  // barriers, TMEM address; slack for aligning the base
  return L;
}

template <typename T>
struct DownArgs {
  CUtensorMap tm_wd;  // down_w [C*H rows, R columns], box {64 columns, KS rows}, 128-byte swizzle
  const T *streams, *prev_out, *prev_gate, *ns, *wd, *wi;
  T* sout;
  float* inv_ws;   // (B, C)
  float* part_ws;  // one row: (NCLU, B, NCP), NCP = R + 8; split: see part_index
  int B, C, H, R, KS, CL, NCP, split, per, NCLU;  // split: the up ranks SR sharing d, 0 = none
  float eps;
  int weights_static;
  const T* wu;                 // up_w: each CTA prefetches wu_prefetch_bytes of it into L2
  uint32_t wu_prefetch_bytes;  // a multiple of 16; 0 = no prefetch
  unsigned long long* phase;  // TIMED variants only: [CTA][kPhasePoints][2]
};

template <typename T>
__device__ __forceinline__ uint32_t idesc_t() {
  return idesc_f16(std::is_same<T, __nv_bfloat16>::value, 128, kUmRowsN, true, false);
}

// 384 threads; registers capped at 64 so that a CTA of dec_up_um keeps fitting
// beside it (measured: without the cap the 2-8 row variants take more
// registers and the two kernels of a block stop overlapping under PDL,
// costing 5-6 us per block).
// Phase points (TIMED): 0 entry, 1 weights issued (before the dependency
// wait), 2 wait returned, 3 S pass done (the branch sums of squares in shared
// memory), 4 inverse RMS stored, 5 weights landed, 6 MMA operands ready, 7 MMA
// done, 8 cluster exchange landed, 9 partial sums written.
template <typename T, int MB, bool TIMED = false>
__global__ void __maxnreg__(MB > 8 ? 72 : 64) dec_down_um(const __grid_constant__ DownArgs<T> a) {
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
  T* ns_s = reinterpret_cast<T*>(smem + L.ns);
  T* ss = reinterpret_cast<T*>(smem + L.ss);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  float* recv_s = reinterpret_cast<float*>(smem + L.recv);
  float* gs = reinterpret_cast<float*>(smem + L.gs);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* mma_bar = rbar + 1;
  uint64_t* wbar = rbar + 2;  // the slice's weights and norm_scale landed
  uint64_t* xbar = rbar + 3;  // every group sum of squares landed (shared statistic)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbar + 4);

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
  const int nbt = ceil_div(R, 64);  // boxes the W_d copies fill (a ragged last one with zeros)
  // Shared statistic (three or more rows): the branch's sum of squares of a row
  // is, at every row count, the sum in group order of G butterfly sums over
  // 32 consecutive vectors (the warps' sums of the one-pass form, where
  // thread v takes vector v). With several rows the eight ranks of a cluster
  // (eight slices of the branch) split the (group, row) pairs, each loading
  // only its groups' vectors, and send the group sums to every rank: the
  // same additions in the same order, a fraction of the loads.
  const int NVr = H / VEC, G = ceil_div(NVr, 32);
  // (Both forms give the same bits; at two rows the exchange costs more than
  // the loads it saves, measured 9.75 vs 9.5 us per block.)
  const bool xmode = MB >= 4 && CL >= 8 && NVr <= nthr && G * B <= nwarps * CL;
  HC_PHASE(0);

  if (tid == 0) {
    mbar_init(rbar, 1);
    mbar_init(mma_bar, MT);  // one commit per tile's issuing warp
    mbar_init(wbar, 1);
    mbar_init(xbar, 1);
    mbar_arrive_expect_tx(xbar, xmode ? static_cast<uint32_t>(G * B * 4) : 0u);
    tma_prefetch_desc(&a.tm_wd);
    mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(CL * ncol * B * 4));
    fence_mbar_init();
  }
  // the last warp owns the tensor memory: it frees it as soon as every warp
  // has read its accumulators, off the path of the warps that still work
  const int tm_warp = nwarps - 1;
  if (warp == tm_warp) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  cluster_arrive_relaxed();
  // zero B (rows >= B and k >= KS stay zero) and the A boxes no copy writes
  // (every box from nbt on; the copies fill the columns of a ragged last box
  // past R with zeros)
  #pragma unroll 1
  for (int i = tid; i < ceil_div(KS, 64) * kKBlock / 16; i += nthr) reinterpret_cast<uint4*>(sB)[i] = make_uint4(0, 0, 0, 0);
  #pragma unroll 1
  for (int i = tid; i < (2 * MT - nbt) * KS * 8; i += nthr)
    reinterpret_cast<uint4*>(sA + nbt * boxb)[i] = make_uint4(0, 0, 0, 0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // weights, by one thread: the slice's KS rows of W_d as nbt tensor copies of
  // 64 columns (each lands as one 128-byte-swizzled box of A), its rows of
  // W_i and of norm_scale as two bulk copies, all completing on wbar; once
  // they land warp 0 places the inject values in column R.. of A
  auto issue_weights = [&]() {
    if (tid == 0) {
      const uint32_t ib = static_cast<uint32_t>(KS * C * 2), nb = static_cast<uint32_t>(KS * 2);
      mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(nbt * boxb) + ib + nb);
      for (int j = 0; j < nbt; ++j) tma_load_2d(sA + j * boxb, &a.tm_wd, j * 64, k0, wbar);
      bulk_g2s(smem + L.wis, a.wi + static_cast<int64_t>(k0) * C, ib, wbar);
      bulk_g2s(ns_s, a.ns + k0, nb, wbar);
      // this CTA's share of the up weights into L2, for dec_up_um, whose
      // CTAs start only after this kernel's dependency wait: the up weights
      // then stream from HBM while this kernel runs, and dec_up_um's copies
      // hit L2 (a prefetch changes no data; L2 is the point of coherence)
      if (a.wu_prefetch_bytes != 0)
        l2_prefetch(reinterpret_cast<const uint8_t*>(a.wu) + static_cast<size_t>(slice) * a.wu_prefetch_bytes,
                    a.wu_prefetch_bytes);
    }
  };
  // one thread per K row copies the row's C inject values (C * 2 bytes, at
  // the start of a 16-byte chunk since R % 8 == 0) into column R.. of A
  auto place_inject = [&]() {
    if (tid < KS) {
      const int r = tid;
      uint8_t* dst = sA + ibox * boxb + r * 128 + ((ich ^ (r & 7)) << 4);
      const T* src = wis + r * C;
      if (C == 8) *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
      else if (C == 4) *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
      else if (C == 2) *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
      else *reinterpret_cast<T*>(dst) = *src;
    }
  };
  // With static weights the copies start before the dependency wait.
  if (a.weights_static) issue_weights();
  HC_PHASE(1);
  pdl_wait();
  HC_PHASE(2);
  if (!a.weights_static) issue_weights();
  pdl_trigger();

  bool xok = true;
  if (xmode) {
    // ---- shared statistic: (group, row) pair t goes to rank t % CL, warp
    // t / CL; thread i < B * KS/8 also loads vector i of the slice ----
    const int NS = KS / VEC, npair = G * B;
    const int t = warp * CL + rank;
    const bool task = t < npair;
    const int tw = task ? t / B : 0, tb = task ? t - (t / B) * B : 0, tv = tw * 32 + lane;
    const bool tload = task && tv < NVr;
    const bool sl = tid < B * NS;
    const int sb = sl ? tid / NS : 0, sv = sl ? tid - (tid / NS) * NS : 0;
    uint4 qv = make_uint4(0, 0, 0, 0), qp = make_uint4(0, 0, 0, 0), lv = make_uint4(0, 0, 0, 0),
          lp = make_uint4(0, 0, 0, 0);
    float qg = 0.0f, lg = 0.0f;
    if (tload) {
      qv = ld16(a.streams + tb * CH + static_cast<int64_t>(c) * H + tv * VEC);
      if (pro) {
        qp = ld16(a.prev_out + static_cast<int64_t>(tb) * H + tv * VEC);
        qg = ldf(a.prev_gate + tb * C + c);
      }
    }
    if (sl) {
      lv = ld16(a.streams + sb * CH + k0 + sv * VEC);
      if (pro) {
        lp = ld16(a.prev_out + static_cast<int64_t>(sb) * H + hk0 + sv * VEC);
        lg = ldf(a.prev_gate + sb * C + c);
      }
    }
    float q = 0.0f;
    if (tload) {
      float sf[VEC];
      V8<T>::unpack(qv, sf);
      if (pro) {
        float pf[VEC];
        V8<T>::unpack(qp, pf);
#pragma unroll
        for (int j = 0; j < VEC; ++j) sf[j] = prologue_s<T>(sf[j], qg, pf[j]);
      }
#pragma unroll
      for (int j = 0; j < VEC; ++j) q = fmaf(sf[j], sf[j], q);
    }
    if (sl) {
      float sf[VEC];
      V8<T>::unpack(lv, sf);
      if (pro) {
        float pf[VEC];
        V8<T>::unpack(lp, pf);
#pragma unroll
        for (int j = 0; j < VEC; ++j) sf[j] = prologue_s<T>(sf[j], lg, pf[j]);
      }
      const uint4 sv_t = pro ? V8<T>::pack(sf) : lv;  // S as T (each value already rounded)
      *reinterpret_cast<uint4*>(ss + sb * KS + sv * VEC) = sv_t;
      if (a.sout != nullptr) st16(a.sout + sb * CH + k0 + sv * VEC, sv_t);
    }
    const float gsum = warp_sum(q);  // the one-pass form's warp sum for group tw
    cluster_wait();                  // every rank has started: its gs and xbar exist
    if (task && lane < CL) {
      const uint32_t slot = smem_addr(gs + tw * MB + tb);
      st_async_b32(mapa_shared(slot, lane), __float_as_uint(gsum), mapa_shared(smem_addr(xbar), lane));
    }
    xok = mbar_wait(xbar, 0, &g_um_wait_timeouts);
    // each row's inverse RMS, once, from the group sums in group order (the
    // barrier below publishes it with the slice's S)
    if (tid < B) {
      float tsum = 0.0f;
      for (int w = 0; w < G; ++w) tsum += gs[w * MB + tid];
      wsum[tid] = inv_rms(tsum, H, a.eps);
    }
    __syncthreads();  // the slice's S (ss) and the inverse RMS written by other threads
  } else {
  // ---- one pass over branch c of every row: S, its sum of squares, the
  // slice's S and streams_out for the slice ----
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
            const uint4 sv_t = pro ? V8<T>::pack(sf) : sv[bi];  // S as T (each value already rounded)
            *reinterpret_cast<uint4*>(ss + b * KS + kk) = sv_t;
            if (a.sout != nullptr) st16(a.sout + b * CH + k0 + kk, sv_t);
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
  }
  HC_PHASE(3);
  // One row: every thread forms the inverse RMS itself from the warps' sums
  // (the same sum in the same order in every thread, so the same bits; no
  // second CTA barrier on the critical path). The shared statistic's sum runs
  // over the G groups only: the one-pass form's warps past the last group
  // hold +0, and adding them changes nothing.
  // (With several rows the statistic of row b is already in wsum[b].)
  auto inv_of = [&](int b) {
    if (xmode) return wsum[b];
    float t = 0.0f;
    if constexpr (MB <= 2) {
      float x[kDownWarps];  // blockDim.x == kDownWarps * 32
#pragma unroll
      for (int w = 0; w < kDownWarps; ++w) x[w] = wsum[w * MB + b];  // all loads in flight, then the sum in order
#pragma unroll
      for (int w = 0; w < kDownWarps; ++w) t += x[w];
    } else {
      #pragma unroll 1
      for (int w = 0; w < nwarps; ++w) t += wsum[w * MB + b];
    }
    return inv_rms(t, H, a.eps);
  };
  // One or two rows: the inverse RMS once per thread, before the weights are
  // waited for, and one thread per K row of the slice for hn (no division)
  float inv2[2] = {0.0f, 0.0f};
  if constexpr (MB == 1) {
    inv2[0] = inv_of(0);
  } else if constexpr (MB == 2) {
    if (xmode) {
      inv2[0] = wsum[0];
      inv2[1] = wsum[1];
    } else {
      // both rows at once: the 24 warp sums loaded together (wsum is
      // [warp][row]), the two sums added in warp order side by side
      float2 x[kDownWarps];
#pragma unroll
      for (int w = 0; w < kDownWarps; ++w) x[w] = reinterpret_cast<const float2*>(wsum)[w];
      float t0 = 0.0f, t1 = 0.0f;
#pragma unroll
      for (int w = 0; w < kDownWarps; ++w) {
        t0 += x[w].x;
        t1 += x[w].y;
      }
      inv2[0] = inv_rms(t0, H, a.eps);
      inv2[1] = inv_rms(t1, H, a.eps);
    }
  }
  if (hk0 == 0 && tid < B) a.inv_ws[tid * C + c] = MB <= 2 ? (tid == 0 ? inv2[0] : inv2[1]) : inv_of(tid);
  HC_PHASE(4);
  const bool wok = mbar_wait(wbar, 0, &g_um_wait_timeouts);
  HC_PHASE(5);
  // hn of the slice as T, into B at its swizzled position
  if constexpr (MB <= 2) {
    if (tid < KS) {
      const float nsv = Ty<T>::to_f(ns_s[tid]);
#pragma unroll
      for (int b = 0; b < MB; ++b)
        if (b < B)
          *reinterpret_cast<T*>(sB + b_off(b, tid)) =
              Ty<T>::from_f(norm_hn<T>(Ty<T>::to_f(ss[b * KS + tid]), inv2[b], nsv));
    }
  } else {
    int b_inv = -1;
    float iv = 0.0f;
    #pragma unroll 1
    for (int i = tid; i < B * KS; i += nthr) {
      const int b = i / KS, kk = i - b * KS;
      if (b != b_inv) {
        iv = inv_of(b);
        b_inv = b;
      }
      *reinterpret_cast<T*>(sB + b_off(b, kk)) =
          Ty<T>::from_f(norm_hn<T>(Ty<T>::to_f(ss[i]), iv, Ty<T>::to_f(ns_s[kk])));
    }
  }
  place_inject();
  fence_proxy_async_smem();  // generic-proxy writes of A and B, visible to the tensor core
  __syncthreads();
  HC_PHASE(6);

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
  const bool ok = mbar_wait(mma_bar, 0, &g_um_wait_timeouts) && wok && xok;
  tc_fence_after();
  HC_PHASE(7);

  // ---- each warp reads 32-column groups p = (tile p/4, lane quarter p%4)
  // with p % 4 == warp % 4 (a warp reaches only its own lane quarter) and
  // sends row values to the rank that owns the group ----
  const float qnan = __int_as_float(0x7fc00000);
  if (!xmode) cluster_wait();
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
  tc_fence_before();
  if (warp == tm_warp) {
    named_bar_sync(1, static_cast<uint32_t>(nthr));  // every warp's tensor-memory loads are done
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  } else {
    named_bar_arrive(1, static_cast<uint32_t>(nthr));
  }
  const bool rok = mbar_wait(rbar, 0, &g_um_wait_timeouts);
  HC_PHASE(8);

  // ---- sum the received partials of the owned columns in rank order ----
  const int cluster_id = slice / CL;
  #pragma unroll 1
  for (int i = tid; i < B * ncol; i += nthr) {
    const int b = i / ncol, lc = i - b * ncol;
    float x[kDownClusterMax];
#pragma unroll
    for (int r = 0; r < kDownClusterMax; ++r) x[r] = r < CL ? recv_s[(r * MB + b) * OC + lc] : 0.0f;
    float t = 0.0f;
#pragma unroll
    for (int r = 0; r < kDownClusterMax; ++r)
      if (r < CL) t += x[r];
    a.part_ws[part_index(a.split, cluster_id, b, c_lo + lc, B, R, NCP, a.per, a.NCLU)] = rok ? t : qnan;
  }
  if constexpr (TIMED) {
    __syncthreads();
    HC_PHASE(9);
  }
}

// ----------------------------------------------------------------- dec_up --

struct UpSmem {
  uint32_t a, b, st, hn, ns, inv, mix, bars, total;
};
__host__ __device__ inline UpSmem up_smem(int MB, int R, int C, int st_bytes) {
  const int R16 = (R + 15) / 16 * 16;
  UpSmem L;
  L.a = 0;
  L.b = a1024(L.a + 2 * R16 * 128);
  L.st = a16(L.b + ceil_div(R16, 64) * kKBlock);
  L.hn = a16(L.st + st_bytes);        // S, then hn, of the tile: T (both already rounded to T)
  L.ns = a16(L.hn + MB * kUpHS * 2);  // norm_scale of the tile, T
  L.inv = a16(L.ns + kUpHS * 2);      // inverse RMS of every (row, branch)
  L.mix = a16(L.inv + MB * C * 4);    // hn * g of every (row, tile column)
  L.bars = a16(L.mix + MB * kUpHS * 4);
  L.total = L.bars + 48 + 1024;
  return L;
}

template <typename T>
struct UpArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wu;
  const float* inv_ws;
  const float* part_ws;
  T *pre, *post;
  int B, C, H, R, NCLU, NCP, split, per, st_bytes;  // split: the cluster size SR, 0 = none
  Attrs at;
  unsigned long long* phase;  // TIMED variants only: [CTA][kPhasePoints][2]
};

// post_gate for every row: the inject partials summed in cluster order. One
// CTA runs it, on its last warp (the one with the least of the d work, none
// at one row), so that it stays off the path of the threads that feed the
// MMA; kept out of line so that the other CTAs never fetch its code.
template <typename T>
__device__ __noinline__ void dec_post_gate(const float* st, size_t inj_off, bool split, int B, int C, int NCLU, int NCP,
                                           int R, bool ok, T* post, float gate_div, float gate_mul) {
  const float qnan = __int_as_float(0x7fc00000);
  #pragma unroll 1
  for (int i = static_cast<int>(threadIdx.x) - static_cast<int>(blockDim.x - 32); i >= 0 && i < B * C; i += 32) {
    const int b = i / C, cc = i - b * C;
    const float* src = split ? st + inj_off + static_cast<size_t>(b) * 8 + cc : st + static_cast<size_t>(b) * NCP + R + cc;
    const size_t stride = split ? static_cast<size_t>(B) * 8 : static_cast<size_t>(B) * NCP;
    const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
    stf(post + b * C + cc, ok ? post_gate_of<T>(rT<T>(x), gate_div, gate_mul) : qnan);
  }
}

// The same at 9-16 rows, where no CTA stages the inject partials: they are
// read from the workspace (inj: row 0 of cluster 0, rows 8 and clusters
// 8 * B floats apart). (One function serving both, with its source pointer
// chosen by the caller, measured 0.1-0.2 us per block slower at 2-8 rows.)
template <typename T>
__device__ __noinline__ void dec_post_gate_ws(const float* inj, int B, int C, int NCLU, bool ok, T* post,
                                              float gate_div, float gate_mul) {
  const float qnan = __int_as_float(0x7fc00000);
  #pragma unroll 1
  for (int i = static_cast<int>(threadIdx.x) - static_cast<int>(blockDim.x - 32); i >= 0 && i < B * C; i += 32) {
    const int b = i / C, cc = i - b * C;
    const float* src = inj + static_cast<size_t>(b) * 8 + cc;
    const size_t stride = static_cast<size_t>(B) * 8;
    const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
    stf(post + b * C + cc, ok ? post_gate_of<T>(rT<T>(x), gate_div, gate_mul) : qnan);
  }
}

// Phase points (TIMED): 0 entry, 1 prefetches issued (before the dependency
// wait), 2 wait returned, 3 partial sums landed, 4 MMA operands ready, 5 MMA
// done, 6 pre-mix products landed, 7 pre_output written.
template <typename T, int MB, bool TIMED = false>
__global__ void __launch_bounds__(512, (MB > 8 ? 1 : 2)) dec_up_um(const UpArgs<T> a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  constexpr int VEC = 8, HS = kUpHS;
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, C = a.C, H = a.H, R = a.R, NCLU = a.NCLU, NCP = a.NCP;
  const int R16 = (R + 15) / 16 * 16, F = HS / C, boxb = R16 * 128;
  const int lgF = 31 - __clz(F);  // F = 128 / C is a power of two
  const UpSmem L = up_smem(MB, R, C, a.st_bytes);
  uint8_t* sA = smem + L.a;
  uint8_t* sB = smem + L.b;
  float* st = reinterpret_cast<float*>(smem + L.st);
  T* hn_s = reinterpret_cast<T*>(smem + L.hn);
  T* ns_s = reinterpret_cast<T*>(smem + L.ns);
  float* inv_s = reinterpret_cast<float*>(smem + L.inv);
  float* mix_s = reinterpret_cast<float*>(smem + L.mix);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bars);  // partial sums landed
  uint64_t* dbar = bar + 1;                                     // d from every rank landed (split mode)
  uint64_t* mma_bar = bar + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 4);

  // Tile column m (= TMEM lane, = row of A) is feature f0 + m % F of branch
  // m / F, f0 = blockIdx.x * F. With two or more rows, SR consecutive CTAs
  // form a cluster in which rank p reduces share p of the down columns and
  // broadcasts its part of d (split mode; d is the same for every tile); one
  // row needs no cluster.
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int f0 = blockIdx.x * F;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const bool pro = a.prev_out != nullptr;
  const bool do_post = blockIdx.x == 0;
  // one row needs no split (the host never sets it then): the code is left out
  const bool split = MB > 1 && a.split != 0;
  const int SR = a.split;
  HC_PHASE(0);
  // The next block's dec_down_um reads nothing before its own dependency wait
  // but static weights (HC_FLAG_WEIGHTS_STATIC), and writes nothing before it:
  // it may launch now and stream its weights during this kernel.
  pdl_trigger();

  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(dbar, 1);
    mbar_init(mma_bar, min(kUpIssuers, (R + 15) / 16));  // one commit per issuing warp
    mbar_arrive_expect_tx(dbar, split ? static_cast<uint32_t>(R * B * 2) : 0u);
    fence_mbar_init();
  }
  // a warp with no epilogue work owns the tensor memory and frees it once the
  // four epilogue warps have read their accumulators
  const int tm_warp = (nthr >> 5) - 2;
  if (warp == tm_warp) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  cluster_arrive_relaxed();
  // The up weights and the block inputs are never written by the preceding
  // dec_down_um, which triggers its dependents only after its own wait:
  // reading them before griddepcontrol.wait is safe. norm_scale of the tile
  // first, in a copy group of its own (the hn step waits for it alone); then
  // A: 16 chunks of 16 bytes per K row (two boxes of 64 columns), at their
  // swizzled positions; chunk qd holds tile columns 8 qd .. 8 qd + 7, i.e.
  // features of branch 8 qd / F.
  #pragma unroll 1
  for (int i = tid; i < HS / VEC; i += nthr) {
    const int m0 = i * VEC, cb = m0 >> lgF;
    cp_async16(ns_s + m0, a.ns + static_cast<int64_t>(cb) * H + f0 + (m0 - (cb << lgF)));
  }
  cp_async_commit();
  {
    #pragma unroll 1
    for (int i = tid; i < R * 16; i += nthr) {
      const int r = i >> 4, qd = i & 15, m0 = qd * 8, cb = m0 >> lgF;
      cp_async16(sA + (qd >> 3) * boxb + r * 128 + (((qd & 7) ^ (r & 7)) << 4),
                 a.wu + static_cast<int64_t>(r) * CH + static_cast<int64_t>(cb) * H + f0 + (m0 - (cb << lgF)));
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
    const int b = i / nvh, m0 = (i - b * nvh) * VEC, cb = m0 >> lgF, f = f0 + (m0 - (cb << lgF));
    uint4 sv = ld16(a.streams + b * CH + static_cast<int64_t>(cb) * H + f);
    if (pro) {
      float sf[VEC], pf[VEC];
      V8<T>::unpack(sv, sf);
      V8<T>::unpack(ld16(a.prev_out + static_cast<int64_t>(b) * H + f), pf);
      const float gt = ldf(a.prev_gate + b * C + cb);
#pragma unroll
      for (int j = 0; j < VEC; ++j) sf[j] = prologue_s<T>(sf[j], gt, pf[j]);
      sv = V8<T>::pack(sf);
    }
    *reinterpret_cast<uint4*>(hn_s + b * HS + m0) = sv;
  }
  tc_fence_before();
  HC_PHASE(1);
  pdl_wait();
  cluster_wait();
  __syncthreads();  // barriers, TMEM address, S, ns and the zeroed regions visible CTA-wide
  tc_fence_after();
  HC_PHASE(2);
  const uint32_t tmem = *tmem_slot;

  // ---- pull the down partials into shared memory ----
  const int ncols = split ? max(0, min(R, (rank + 1) * a.per) - rank * a.per) : 0;
  // up to 8 rows, CTA 0 also stages every cluster's inject partials for the
  // post gate; at 9-16 rows they stay in the workspace (the post gate reads
  // them there) to leave room for a dec_down_um CTA beside this one
  constexpr bool kStageInj = MB <= 8;
  const size_t inj_off = static_cast<size_t>(NCLU) * B * a.per;  // floats (split layout)
  if (warp == 0) {
    uint32_t bytes;
    if (!split) bytes = static_cast<uint32_t>(NCLU * B * NCP * 4);
    else bytes = static_cast<uint32_t>(NCLU * B * a.per * 4 + (kStageInj && do_post ? NCLU * B * 32 : 0));
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    if (!split) {
      if (lane == 0) bulk_g2s(st, a.part_ws, bytes, bar);
    } else {
      // one block of every cluster's B * per partials for this rank, and
      // (rank 0 of the first column tile, up to 8 rows) one block of every
      // cluster's inject partials
      if (lane == 0)
        bulk_g2s(st, a.part_ws + static_cast<int64_t>(rank) * NCLU * B * a.per,
                 static_cast<uint32_t>(NCLU * B * a.per * 4), bar);
      if (kStageInj && do_post && lane == 0)
        bulk_g2s(st + inj_off, a.part_ws + static_cast<int64_t>(NCLU) * SR * B * a.per,
                 static_cast<uint32_t>(NCLU * B * 32), bar);
    }
  }
  // the inverse RMS of every (row, branch), from dec_down_um: its load is
  // issued before the wait for the partial sums, so the two latencies
  // overlap (B * C <= 64 < nthr)
  const float inv_ld = tid < B * C ? a.inv_ws[tid] : 0.0f;
  const bool ok = mbar_wait(bar, 0, &g_um_wait_timeouts);
  if (tid < B * C) inv_s[tid] = inv_ld;
  cp_async_wait_group1();  // this thread's norm_scale chunk landed (the W_u copies may still fly)
  __syncthreads();
  const float qnan = __int_as_float(0x7fc00000);
  HC_PHASE(3);

  // ---- d = ScaledSiLU(rT(sum of the partials in cluster order)) as T, into B,
  // on every warp but the last, which computes the post gate meanwhile ----
  const int nthr_d = nthr - 32;
  const bool d_thread = tid < nthr_d;
  if (!split) {
    const size_t stride = static_cast<size_t>(B) * NCP;
    #pragma unroll 1
    for (int i = d_thread ? tid : B * R; i < B * R; i += nthr_d) {
      const int b = i / R, col = i - b * R;
      const float* src = st + static_cast<size_t>(b) * NCP + col;
      const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
      *reinterpret_cast<T*>(sB + b_off(b, col)) = Ty<T>::from_f(ok ? scaled_silu_t<T>(rT<T>(x), a.at.alpha) : qnan);
    }
  }
  if constexpr (MB > 1) if (split && d_thread) {
    // one column per thread; lanes 2k and 2k + 1 hold columns lc and lc + 1
    // of one row (ncols and nthr_d are even), swap their values to form the
    // contiguous pair and send it to half of the ranks each
    const int total = B * ncols;
    const size_t stride = static_cast<size_t>(B) * a.per;
    #pragma unroll 1
    for (int wb = tid - lane; wb < total; wb += nthr_d) {  // warp-uniform: every lane reaches the shuffle
      const int i = wb + lane;
      const bool act = i < total;
      const int b = act ? i / ncols : 0, lc = act ? i - b * ncols : 0;
      float x = 0.0f;
      if (act) {
        const float* src = st + static_cast<size_t>(b) * a.per + lc;
        x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
      }
      const T dv = Ty<T>::from_f(ok ? scaled_silu_t<T>(rT<T>(x), a.at.alpha) : qnan);
      const uint32_t mine = *reinterpret_cast<const uint16_t*>(&dv);
      const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
      if (act) {
        const uint32_t packed = (lane & 1) ? (other | (mine << 16)) : (mine | (other << 16));
        const int lc0 = lc & ~1;
        const uint32_t slot = smem_addr(sB + b_off(b, rank * a.per + lc0));  // an even column pair is contiguous
        const int half = SR / 2, r0 = (lane & 1) ? half : 0, r1 = (lane & 1) ? SR : half;
        for (int pr = r0; pr < r1; ++pr)
          st_async_b32(mapa_shared(slot, pr), packed, mapa_shared(smem_addr(dbar), pr));
      }
    }
  }
  // The MMA may start once the d warps have written d and hn and every
  // thread's W_u copies have landed: the last warp only arrives at that
  // barrier (after its own copies) and then computes the post gate, so the
  // MMA does not wait for it.
  bool dok = true;
  if (d_thread) {
    #pragma unroll 1
    for (int i = tid; i < B * HS; i += nthr_d) {
      const int b = i / HS, m = i - b * HS;
      hn_s[i] = Ty<T>::from_f(norm_hn<T>(Ty<T>::to_f(hn_s[i]), inv_s[b * C + (m >> lgF)], Ty<T>::to_f(ns_s[m])));
    }
    cp_async_wait_all();
    if (split) dok = mbar_wait(dbar, 0, &g_um_wait_timeouts);
    fence_proxy_async_smem();  // A (cp.async) and B (d) visible to the tensor core
    named_bar_sync(2, static_cast<uint32_t>(nthr));
  } else {
    cp_async_wait_all();
    fence_proxy_async_smem();
    named_bar_arrive(2, static_cast<uint32_t>(nthr));
    if constexpr (kStageInj) {
      if (do_post) dec_post_gate<T>(st, inj_off, split, B, C, NCLU, NCP, R, ok, a.post, a.at.gate_div, a.at.gate_mul);
    } else {
      if (do_post)
        dec_post_gate_ws<T>(a.part_ws + static_cast<size_t>(NCLU) * SR * B * a.per, B, C, NCLU, ok, a.post,
                            a.at.gate_div, a.at.gate_mul);
    }
  }
  HC_PHASE(4);

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
  HC_PHASE(5);

  // ---- epilogue: warp w < EW holds tile columns 32(w%4)..+31 (its TMEM
  // lane quarter), rows in TMEM columns; with two rows or more two warps
  // share a lane quarter, each taking every other row (three warps measured
  // slower at eight rows, 11.44 vs 11.38 us per block): g =
  // rT(sigmoid(rT(up))) and hn*g go to shared memory; then each feature's C
  // products are summed in branch order (the pre-mix) and scaled into
  // pre_output ----
  constexpr int EW = MB >= 2 ? 8 : 4, RS = EW / 4;
  if (warp < EW) {
    // accumulators 0..NI-1 of this lane quarter, added as ((a0 + a1) + (a2 + a3))
    uint32_t acc[kUpIssuers][16];
    const uint32_t tq = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
#pragma unroll
    for (int j = 0; j < kUpIssuers; ++j)
      if (j < NI) tmem_ld16_nowait(tq + j * kUmRowsN, acc[j]);
#pragma unroll
    for (int j = 0; j < kUpIssuers; ++j)
      if (j < NI) tmem_ld_wait_r(acc[j]);
    tc_fence_before();
    named_bar_arrive(3, 32 * EW + 32);
    float v[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float x[kUpIssuers];
#pragma unroll
      for (int j = 0; j < kUpIssuers; ++j) x[j] = j < NI ? __uint_as_float(acc[j][r]) : 0.0f;
      v[r] = __fadd_rn(__fadd_rn(x[0], x[1]), __fadd_rn(x[2], x[3]));
    }
    const int m = (warp & 3) * 32 + lane, rh = warp >> 2;
#pragma unroll
    for (int b = 0; b < MB; ++b)
      if (b < B && b % RS == rh) {
        const float gg = sigmoid_rT<T>(rT<T>(v[b]));
        mix_s[b * HS + m] = (dok && mmok) ? __fmul_rn(Ty<T>::to_f(hn_s[b * HS + m]), gg) : qnan;
      }
    named_bar_sync(1, 32 * EW);  // the epilogue warps
    HC_PHASE(6);
    #pragma unroll 1
    for (int i = tid; i < B * F; i += 32 * EW) {
      const int b = i / F, f = i - b * F;
      float acc2 = 0.0f;
      for (int cb = 0; cb < C; ++cb) acc2 = __fadd_rn(acc2, mix_s[b * HS + cb * F + f]);
      stf(a.pre + static_cast<int64_t>(b) * H + f0 + f, __fmul_rn(a.at.rho, acc2));
    }
  }
  if (warp == tm_warp) {
    named_bar_sync(3, 32 * EW + 32);  // the epilogue warps' tensor-memory loads are done
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
  if constexpr (TIMED) {
    __syncthreads();
    HC_PHASE(7);
  }
}

// ------------------------------------------------------------ configuration

struct UmCfg {
  bool ok;
  int KS, NSL, CL, NCLU, NCP, H, R, down_threads, up_threads;
};

int cluster_for(int n) {
  for (int cl : {8, 4, 2})
    if (n % cl == 0) return cl;
  return 1;
}

// Whether this device schedules dec_down_um in clusters of 16 CTAs (a
// non-portable size: it needs 16 SMs of one GPC free at once) with the largest
// shared memory the configuration allows; asked once per device and kept, so
// that the workspace query and the launch always agree.
bool down_cluster16_ok() {
  static std::atomic<int> known[64];  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  const int k = known[dev].load(std::memory_order_acquire);
  if (k != 0) return k == 1;
  auto kern = dec_down_um<__nv_bfloat16, 8, false>;
  bool ok = ensure_smem<dec_down_um<__nv_bfloat16, 8, false>>(kUmDownCap) == cudaSuccess &&
            cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(128);
    cfg.blockDim = dim3(kDownWarps * 32);
    cfg.dynamicSmemBytes = kUmDownCap;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 16;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0;
  }
  cudaGetLastError();  // a refused query leaves no error behind
  known[dev].store(ok ? 1 : 2, std::memory_order_release);
  return ok;
}

// dec_down_um's clusters: 16 slices of a branch where they divide it and the
// device schedules such clusters (allowed on the kernel before its launch),
// else as cluster_for. Measured per block against clusters of 8: rows 1
// 7.33 -> 7.03 us, rows 8 11.36 -> 11.22, rows 4 9.74 -> 9.93.
int down_cluster_for(int n) { return (n % 16 == 0 && down_cluster16_ok()) ? 16 : cluster_for(n); }

struct Stage {
  int split, per, bytes;
};
// From 2 rows on, the up CTAs form clusters of SR (8 where the tile count
// allows) in which each rank reduces 1/SR of the down columns and broadcasts
// its part of d: the staging stays small enough for a dec_down_um CTA to
// share the SM, and each CTA pulls 1/SR of the partial sums.
Stage stage_for(int64_t rows, int C, int H, int R, int NCLU, int NCP) {
  Stage s;
  const int SR = cluster_for((H / kUpHS) * C);
  s.split = (rows > 1 && SR > 1) ? SR : 0;
  s.per = s.split ? ceil_div(ceil_div(R, SR), 4) * 4 : 0;
  s.bytes = s.split ? static_cast<int>(NCLU * rows * s.per * 4 + (rows <= 8 ? NCLU * rows * 32 : 0))
                    : static_cast<int>(NCLU * rows * NCP * 4);
  return s;
}

UmCfg um_cfg(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  UmCfg g{};
  g.ok = false;
  if (dt != HC_F16 && dt != HC_BF16) return g;
  if (rows < 1 || rows > kUmMaxRows) return g;
  if (!(C == 1 || C == 2 || C == 4 || C == 8)) return g;
  if (R < 16 || R % 8 != 0 || R + 8 > kUmMaxMT * 128) return g;
  if (H % kUpHS != 0 || H > 16384) return g;
  const int CH = C * H;
  g.NCP = R + 8;
  g.H = H;
  g.R = R;
  g.down_threads = kDownWarps * 32;
  g.KS = 0;
  for (int ks = 16; ks <= std::min(H, 256); ks += 16) {  // KS rows: one tensor-copy box (at most 256)
    if (H % ks != 0) continue;
    if (down_smem(8, ks, R, C, down_cluster_for(H / ks), g.down_threads / 32).total > kUmDownCap) break;
    g.KS = ks;
    if (CH / ks <= num_sms) break;
  }
  if (g.KS == 0) return g;
  g.NSL = CH / g.KS;
  g.CL = down_cluster_for(H / g.KS);
  g.NCLU = g.NSL / g.CL;
  const Stage sg = stage_for(rows, C, H, R, g.NCLU, g.NCP);
  if (up_smem(8, R, C, sg.bytes).total > kUmUpCap) return g;
  if (rows > 8) {
    // 9-16 rows: only where a CTA of each kernel still fits one SM together
    // (1 KB of each CTA's shared memory is reserved), so the next kernel's
    // CTAs start beside the running ones; the K slices are the same as at
    // eight rows, so a row's bits do not depend on the row count
    // (decided at 16 rows, so the decode/prefill switch of a shape is at 8 or 16 rows)
    const size_t dsm = down_smem(16, g.KS, R, C, g.CL, g.down_threads / 32).total;
    const size_t usm = up_smem(16, R, C, stage_for(16, C, H, R, g.NCLU, g.NCP).bytes).total;
    if (dsm > kUmDownCap || usm > kUmUpCap || dsm + usm + 2048 > kUmSmPerSm) return g;
  }
  // warps for the d columns (at least nine: up to eight epilogue warps and
  // the one that owns the tensor memory), plus one more: the post gate's
  // (dec_post_gate)
  g.up_threads = (std::min(15, std::max(9, ceil_div(R, 32))) + 1) * 32;
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
  const Stage sg = stage_for(rows, C, g.H, g.R, g.NCLU, g.NCP);
  const size_t nf = sg.split ? static_cast<size_t>(g.NCLU) * rows * (static_cast<size_t>(sg.split) * sg.per + 8)
                             : static_cast<size_t>(g.NCLU) * rows * g.NCP;
  L.total = align_up(L.part + nf * 4, 256);
  return L;
}

// Phase-clock recording (hc_debug_phase_clocks): a caller-owned device buffer
// of whole slots; each timed call takes the next slot (one per call, so a
// captured chain of calls keeps every block's record).
struct PhaseState {
  unsigned long long* buf = nullptr;
  size_t slots = 0, next = 0;
};
thread_local PhaseState g_phase;
constexpr size_t kPhaseSlotWords = 2 * kPhaseMaxCtas * kPhasePoints * 2;  // dec_down, then dec_up

template <typename T, int MB, bool TIMED>
cudaError_t run_um_mb(const Problem& p, const UmCfg& g, unsigned long long* phase);

template <typename T, int MB>
cudaError_t run_um_mb(const Problem& p, const UmCfg& g) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value && (MB == 1 || MB == 8)) {
    if (g_phase.buf != nullptr && g.NSL <= kPhaseMaxCtas && (p.H / kUpHS) * p.C <= kPhaseMaxCtas) {
      unsigned long long* slot = g_phase.buf + (g_phase.next++ % g_phase.slots) * kPhaseSlotWords;
      return run_um_mb<T, MB, true>(p, g, slot);
    }
  }
  return run_um_mb<T, MB, false>(p, g, nullptr);
}

template <typename T, int MB, bool TIMED>
cudaError_t run_um_mb(const Problem& p, const UmCfg& g, unsigned long long* phase) {
  const Layout WL = um_layout(p.rows, p.C, g);
  char* ws = static_cast<char*>(p.workspace);
  float* inv_ws = reinterpret_cast<float*>(ws + WL.inv);
  float* part_ws = reinterpret_cast<float*>(ws + WL.part);

  DownArgs<T> da;
  if (!make_tmap_2d_sw128(&da.tm_wd, p.down_w, std::is_same<T, __nv_bfloat16>::value, static_cast<uint64_t>(p.R),
                          static_cast<uint64_t>(p.C) * p.H, static_cast<uint32_t>(g.KS)))
    return cudaErrorInvalidValue;
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
  const Stage sg = stage_for(p.rows, p.C, p.H, p.R, g.NCLU, g.NCP);
  da.split = sg.split; da.per = sg.per;
  da.eps = p.eps;
  da.weights_static = (p.flags & HC_FLAG_WEIGHTS_STATIC) ? 1 : 0;
  da.phase = phase;
  // W_u in NSL equal shares of whole 16-byte units (the tail, if any, is
  // left to dec_up_um's own copies)
  da.wu = static_cast<const T*>(p.up_w);
  da.wu_prefetch_bytes = static_cast<uint32_t>((static_cast<size_t>(p.R) * p.C * p.H * sizeof(T) / g.NSL) & ~size_t{15});
  const size_t dsm = down_smem(MB, g.KS, p.R, p.C, g.CL, g.down_threads / 32).total;
  cudaError_t e = ensure_smem<dec_down_um<T, MB, TIMED>>(dsm);
  if (e == cudaSuccess && g.CL > 8)
    e = cudaFuncSetAttribute(dec_down_um<T, MB, TIMED>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  e = launch_pdl(dec_down_um<T, MB, TIMED>, dim3(g.NSL), dim3(g.down_threads), dsm, p.stream,
                 static_cast<unsigned>(g.CL), da);
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
  ua.phase = phase != nullptr ? phase + kPhaseSlotWords / 2 : nullptr;
  const size_t usm = up_smem(MB, p.R, p.C, sg.bytes).total;
  e = ensure_smem<dec_up_um<T, MB, TIMED>>(usm);
  if (e != cudaSuccess) return e;
  // (H / 128) * C tiles of 128 / C features each; clusters of SR CTAs only
  // where d is split across ranks
  return launch_pdl(dec_up_um<T, MB, TIMED>, dim3((p.H / kUpHS) * p.C), dim3(g.up_threads), usm, p.stream,
                    static_cast<unsigned>(sg.split ? sg.split : 1), ua);
}

template <typename T>
cudaError_t run_um(const Problem& p, const UmCfg& g) {
  if (p.rows <= 1) return run_um_mb<T, 1>(p, g);
  if (p.rows <= 2) return run_um_mb<T, 2>(p, g);
  if (p.rows <= 4) return run_um_mb<T, 4>(p, g);
  if (p.rows <= 8) return run_um_mb<T, 8>(p, g);
  return run_um_mb<T, 16>(p, g);
}

}  // namespace

size_t set_phase_clocks(void* buf, size_t bytes) {
  const size_t slot_bytes = kPhaseSlotWords * sizeof(unsigned long long);
  g_phase.buf = (buf != nullptr && bytes >= slot_bytes) ? static_cast<unsigned long long*>(buf) : nullptr;
  g_phase.slots = g_phase.buf != nullptr ? bytes / slot_bytes : 0;
  g_phase.next = 0;
  return slot_bytes;
}

bool decode_um_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  return um_cfg(rows, C, H, R, dt, 148).ok && tmap_encoder() != nullptr;
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

// One CTA waits, through the same bounded wait as the kernels above, on an
// mbarrier that nothing arrives on and no copy completes: the wait must give
// up after `limit` cycles, count itself in the decode kernels' counter, and
// let the kernel write NaN where its result would go and exit normally.
__global__ void __launch_bounds__(32) wait_timeout_probe(float* out, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  bool ok = true;
  if (threadIdx.x == 0) ok = mbar_wait_limit(&bar, 0, &g_um_wait_timeouts, limit);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  out[threadIdx.x] = ok ? 1.0f : __int_as_float(0x7fc00000);
}

cudaError_t launch_wait_timeout_probe(float* out, long long limit_cycles, cudaStream_t s) {
  wait_timeout_probe<<<1, 32, 0, s>>>(out, limit_cycles);
  return cudaGetLastError();
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
