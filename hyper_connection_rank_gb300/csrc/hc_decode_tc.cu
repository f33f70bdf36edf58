// Decode path for fp16 / bf16 I/O (rows <= 8): two weight-streaming kernels
// linked by programmatic dependent launch, with both projections on the
// tensor cores.
//
// The block at decode sizes is bound by reading its weights once (13.2 MB in
// bf16 at C=4, H=2560, R=320) and by the latency of the steps that depend on
// one another. Both projections are reductions over operands that the block's
// numerics contract (ONNX Runtime PR #33384, "HyperConnectionLowRankMix",
// section "Numerics contract") has already rounded to T: hn = rT(...) times
// down_weight, and the ScaledSiLU output d = rT(...) times up_weight. So they
// run as warp-level mma.sync m16n8k16 with T operands and fp32 accumulation,
// computed transposed: A is a 16-column x 16-k tile of the weights (read with
// ldmatrix.trans from its row-major copy in shared memory) and B holds the
// activation rows (N = 8, so up to 8 rows per instruction). Each warp owns
// whole 16-column tiles, so no cross-warp reduction follows the GEMV.
//
//   dec_down_tc (grid = C*H/KS CTAs, clusters of CL consecutive slices of one
//   branch)
//     - copies its KS rows of down_weight into shared memory (16-byte cp.async
//       into rows padded by 16 bytes: conflict-free ldmatrix) and its
//       inject_weight slice; when the weights are static this happens before
//       griddepcontrol.wait, so the stream overlaps the previous kernel;
//     - one pass over branch c of every row: S (prologue), sum of S^2,
//       streams_out and S of the slice; inv_rms; hn of the slice as T;
//     - [down | inject] = hn @ [Wd | Wi] for the slice: ceil(R/16) + 1 column
//       tiles of 16 (the inject columns padded to one tile), K = KS;
//     - the CL partial vectors of a cluster are summed through distributed
//       shared memory in rank order (each rank owns a range of column tiles)
//       into one fp32 partial per cluster.
//   dec_up_tc (grid = (H/HS)*C CTAs, clusters of C CTAs, one per branch)
//     - copies its up_weight tile (R rows x HS columns of branch c) with
//       16-byte cp.async into padded rows, and S for its tile, before the wait;
//     - pulls the cluster partials into shared memory with bulk copies, sums
//       them in cluster order and applies ScaledSiLU (at most 2 rows: every
//       CTA does all R columns; above that each rank does 1/C of them and
//       broadcasts d through DSMEM); CTA (0, 0) also forms post_gate;
//     - up = d @ Wu for its HS columns, one 16-column tile per warp, then
//       g = rT(sigmoid(rT(up))), hn*g, and the pre-mix sum over the branches
//       in order 0..C-1 through DSMEM.
//
// Every reduction has a fixed order that depends on the shape only, so results
// are deterministic, and a row's bits do not depend on the row count (tensor
// core rows are independent).
#include <algorithm>
#include <cooperative_groups.h>

#include "hc_async.cuh"
#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_mma.cuh"
#include "hc_vec.cuh"

namespace cg = cooperative_groups;

namespace hc {

// Count of bounded waits that gave up (diagnostic; see hc_debug_wait_timeouts).
__device__ unsigned int g_tc_wait_timeouts = 0;

namespace {

constexpr int kMaxTilesPerWarp = 3;  // dec_down: column tiles per warp
constexpr int kUpAcc = 4;            // dec_up: independent accumulators per warp
constexpr size_t kDownSmemCap = 100 * 1024, kUpSmemCap = 120 * 1024;
// Register budget. An SM's registers are four separate files of 16384, one per
// sub-partition, and a warp lives in one of them. With PDL a CTA of each
// kernel shares an SM (up to 4 warps of each per sub-partition), so the two
// kernels together must stay within 16384 / 32 / 4 = 128 registers per
// thread; otherwise each waits for the other's CTAs to leave. The fragment
// batch sizes below keep both near or under 64 (checked with -Xptxas -v).
constexpr int kDownKG = 2;  // dec_down: k-steps whose fragments are loaded before their MMAs
constexpr int kUpKG = 4;    // dec_up: same

__host__ __device__ inline uint32_t a16(uint32_t x) { return (x + 15u) & ~15u; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ dec_down_tc --

// Shared-memory layout (byte offsets). Down-weight rows hold R16 = R rounded up
// to 16 columns (the tail zeroed) padded to WP = 2*R16 + 16 bytes, activation
// rows are padded to AP = 2KS + 16 bytes: the eight rows an ldmatrix reads fall
// in distinct bank groups. The inject slice is widened to 16 columns.
struct DownSmem {
  uint32_t bar, rbar, wd, wis, wie, ns, ss, ha, wsum, inv, recv, total;
};
__host__ __device__ inline DownSmem down_smem(int MB, int KS, int R, int C, int CL, int nwarps) {
  const int R16 = (R + 15) / 16 * 16, WP = 2 * R16 + 16, AP = 2 * KS + 16, NT = R16 / 16 + 1;
  const int TPR = ceil_div(NT, CL);
  DownSmem L;
  L.bar = 0;   // unused
  L.rbar = 8;  // partial sums from the cluster landed
  L.wd = 16;
  L.wis = a16(L.wd + KS * WP);
  L.wie = a16(L.wis + KS * C * 2);
  L.ns = a16(L.wie + KS * 32);
  L.ss = a16(L.ns + KS * 4);
  L.ha = a16(L.ss + MB * KS * 4);
  L.wsum = a16(L.ha + 8 * AP);
  L.inv = a16(L.wsum + nwarps * MB * 4);
  L.recv = a16(L.inv + MB * 4);
  L.total = a16(L.recv + CL * MB * TPR * 16 * 4);
  return L;
}

template <typename T>
struct DownArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wd, *wi;
  T* sout;
  float* inv_ws;   // (B, C)
  float* part_ws;  // (NCLU, B, NCP)
  int B, C, H, R, KS, CL, NCP;
  float eps;
  int weights_static;
};

// At most 512 threads; registers capped at 64 so that a CTA of dec_up_tc fits
// beside it (see the register budget above).
template <typename T, int MB>
__global__ void __maxnreg__(64) dec_down_tc(const DownArgs<T> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int VEC = 8;
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  const int B = a.B, C = a.C, H = a.H, R = a.R, KS = a.KS, CL = a.CL;
  const int R16 = (R + 15) / 16 * 16, NT = R16 / 16 + 1, TPR = ceil_div(NT, CL), OC = TPR * 16;
  const int WP = 2 * R16 + 16, AP = 2 * KS + 16;
  const DownSmem L = down_smem(MB, KS, R, C, CL, nwarps);
  uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + L.rbar);
  const T* wis = reinterpret_cast<const T*>(smem + L.wis);
  T* wie = reinterpret_cast<T*>(smem + L.wie);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* ss = reinterpret_cast<float*>(smem + L.ss);
  T* ha = reinterpret_cast<T*>(smem + L.ha);
  float* wsum = reinterpret_cast<float*>(smem + L.wsum);
  float* inv_s = reinterpret_cast<float*>(smem + L.inv);
  float* recv_s = reinterpret_cast<float*>(smem + L.recv);

  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int slice = blockIdx.x, k0 = slice * KS;
  const int c = k0 / H, hk0 = k0 - c * H;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const bool pro = a.prev_out != nullptr;
  // column tiles this rank owns in the cluster reduction: [t_lo, t_lo + nmine)
  const int t_lo = rank * TPR, nmine = max(0, min(NT, t_lo + TPR) - t_lo);

  // Barriers are initialised before the cluster arrive, whose wait (below, by
  // every peer) then orders the initialisation before any remote complete_tx.
  if (tid == 0) {
    mbar_init(rbar, 1);
    // every rank (this one included) sends 16 columns x 4 bytes per owned tile and row
    mbar_arrive_expect_tx(rbar, static_cast<uint32_t>(CL * nmine * B * 64));
    fence_mbar_init();
  }
  cluster_arrive_relaxed();
  // activation rows >= B stay zero (only this CTA writes this buffer), and so
  // do the weight columns R..R16-1 (the bulk copies write columns < R)
  #pragma unroll 1
  for (int i = tid; i < 8 * AP / 16; i += nthr) reinterpret_cast<uint4*>(smem + L.ha)[i] = make_uint4(0, 0, 0, 0);
  if (R16 > R)
    for (int k = tid; k < KS; k += nthr)
      *reinterpret_cast<uint4*>(smem + L.wd + static_cast<size_t>(k) * WP + 2 * R) = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // The weight slice arrives as 16-byte cp.async chunks issued by every
  // thread into the padded rows (cheap to issue; one bulk copy per row costs
  // the issuing warp tens of cycles each). The warp that owns the inject tile
  // copies the inject slice itself.
  const int w_inj = (NT - 1) % nwarps;
  auto issue_weights = [&]() {
    const int cpr = R / 8;  // 16-byte chunks per weight row
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(a.wd + static_cast<int64_t>(k0) * R);
    #pragma unroll 1
    for (int i = tid; i < KS * cpr; i += nthr) {
      const int r = i / cpr, qd = i - r * cpr;
      cp_async16(smem + L.wd + static_cast<size_t>(r) * WP + qd * 16, gsrc + static_cast<size_t>(r) * R * 2 + qd * 16);
    }
    if (warp == w_inj) {
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
  // inject_weight widened to 16 columns (zeros past C), by the inject warp
  auto widen_inject = [&]() {
    cp_async_wait_all();
    __syncwarp();
    #pragma unroll 1
    for (int i = lane; i < KS * 16; i += 32) {
      const int k = i >> 4, j = i & 15;
      wie[i] = j < C ? wis[k * C + j] : Ty<T>::from_f(0.0f);
    }
    __syncwarp();
  };
  if (a.weights_static) {
    issue_weights();
    if (warp == w_inj) widen_inject();  // off the critical path: before the wait
  }
  pdl_wait();
  if (!a.weights_static) issue_weights();
  pdl_trigger();

  // ---- one pass over branch c of every row: S, its sum of squares, the
  // slice's S (kept in shared memory) and streams_out for the slice ----
  const int NVr = H / VEC;
  float ssq[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) ssq[b] = 0.0f;
  constexpr int RB = MB < 2 ? MB : 2;  // rows whose loads are in flight together
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
  #pragma unroll 1
  for (int i = tid; i < B * KS; i += nthr) {
    const int b = i / KS, kk = i - b * KS;
    ha[b * (AP / 2) + kk] = Ty<T>::from_f(norm_hn<T>(ss[i], inv_s[b], ns_s[kk]));
  }
  if (!a.weights_static && warp == w_inj) widen_inject();
  cp_async_wait_all();
  __syncthreads();  // the weight slice (and hn) visible to every warp

  // ---- [down | inject] for the slice, transposed: out^T (16 columns x rows)
  // = W^T tile (16 x 16 k) * hn^T (16 k x 8 rows). Warp w owns column tiles
  // w, w + nwarps, ...; the last tile is the widened inject_weight ----
  const int ntl = warp < NT ? (NT - 1 - warp) / nwarps + 1 : 0;
  float acc[kMaxTilesPerWarp][4];
#pragma unroll
  for (int j = 0; j < kMaxTilesPerWarp; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[j][e] = 0.0f;
  // B (hn): rows lane&7, k block (lane>>3)&1. A (weights, transposed): k row
  // (lane&7) + 8*((lane>>4)&1), column block 8*((lane>>3)&1) of the tile.
  const uint32_t b_base = smem_addr(ha) + static_cast<uint32_t>((lane & 7) * AP + ((lane >> 3) & 1) * 16);
  const int ak = (lane & 7) + ((lane >> 4) & 1) * 8, an = ((lane >> 3) & 1) * 8;
  uint32_t tb[kMaxTilesPerWarp];  // per tile: its A address at k-step 0
#pragma unroll
  for (int j = 0; j < kMaxTilesPerWarp; ++j) {
    const int tile = warp + j * nwarps;
    tb[j] = tile < NT - 1 ? smem_addr(smem + L.wd) + static_cast<uint32_t>(ak * WP + (tile * 16 + an) * 2)
                          : smem_addr(wie) + static_cast<uint32_t>(ak * 32 + an * 2);
  }
  const uint32_t kstep_wd = static_cast<uint32_t>(16 * WP), kstep_wi = 16u * 32u;
  constexpr int KG = kDownKG;
  #pragma unroll 1
  for (int s0 = 0; s0 < KS / 16; s0 += KG) {
    uint32_t bf[KG][2], af[KG][kMaxTilesPerWarp][4];
#pragma unroll
    for (int u = 0; u < KG; ++u)
      if (s0 + u < KS / 16) {
        const int s = s0 + u;
        ldsm_x2(b_base + s * 32, bf[u][0], bf[u][1]);
#pragma unroll
        for (int j = 0; j < kMaxTilesPerWarp; ++j)
          if (j < ntl) {
            const bool inj = warp + j * nwarps == NT - 1;
            ldsm_x4_trans(tb[j] + s * (inj ? kstep_wi : kstep_wd), af[u][j][0], af[u][j][1], af[u][j][2],
                          af[u][j][3]);
          }
      }
#pragma unroll
    for (int u = 0; u < KG; ++u)
      if (s0 + u < KS / 16)
#pragma unroll
        for (int j = 0; j < kMaxTilesPerWarp; ++j)
          if (j < ntl) Mma<T>::run4(acc[j], af[u][j], bf[u][0], bf[u][1]);
  }

  // ---- send each fragment value (column m0 + g [+8], row 2t [+1]) to the
  // rank that owns its tile: rank r owns tiles [r*TPR, (r+1)*TPR) and receives
  // into recv[src rank][row][owned column] ----
  const float qnan = __int_as_float(0x7fc00000);
  const int g = lane >> 2, t4 = lane & 3;
  cluster_wait();
  if (2 * t4 < B) {
    const uint32_t rbar_local = smem_addr(rbar);
#pragma unroll
    for (int j = 0; j < kMaxTilesPerWarp; ++j)
      if (j < ntl) {
        const int tile = warp + j * nwarps, ow = tile / TPR, lt = tile - ow * TPR;
        const uint32_t rb = mapa_shared(rbar_local, ow);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = 2 * t4 + (e & 1), col = lt * 16 + g + (e >> 1) * 8;
          if (row < B) {
            const uint32_t slot = smem_addr(recv_s + (rank * MB + row) * OC + col);
            st_async_b32(mapa_shared(slot, ow), __float_as_uint(acc[j][e]), rb);
          }
        }
      }
  }
  const bool rok = mbar_wait(rbar, 0, &g_tc_wait_timeouts);

  // ---- sum the received partials of the owned tiles in rank order ----
  const int ncol = nmine * 16;
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
    a.part_ws[(static_cast<int64_t>(cluster_id) * B + b) * a.NCP + t_lo * 16 + lc] = rok ? t : qnan;
  }
}

// -------------------------------------------------------------- dec_up_tc --

// Shared-memory layout (byte offsets). Up-weight rows padded to UP = 2HS + 16
// bytes, d rows to DP = 2*R16 + 16 bytes (R16 = R rounded up to 16).
struct UpSmem {
  uint32_t bar, dbar, mbar, wu, st, da, hn, ns, mix, total;
};
__host__ __device__ inline UpSmem up_smem(int MB, int HS, int R, int C, int st_bytes) {
  const int R16 = (R + 15) / 16 * 16, UP = 2 * HS + 16, DP = 2 * R16 + 16, HSc = HS / C;
  UpSmem L;
  L.bar = 0;    // partial sums landed
  L.dbar = 8;   // d from every rank landed (split mode)
  L.mbar = 16;  // pre-mix products from every rank landed
  L.wu = 32;
  L.st = a16(L.wu + R16 * UP);
  L.da = a16(L.st + st_bytes);
  L.hn = a16(L.da + 8 * DP);
  L.ns = a16(L.hn + MB * HS * 4);
  L.mix = a16(L.ns + HS * 4);
  L.total = a16(L.mix + C * MB * HSc * 4);
  return L;
}

template <typename T>
struct UpArgs {
  const T *streams, *prev_out, *prev_gate, *ns, *wu;
  const float* inv_ws;
  const float* part_ws;
  T *pre, *post;
  int B, C, H, R, HS, NCLU, NCP, split, per, st_bytes;
  Attrs at;
};

template <typename T, int MB>
__global__ void __launch_bounds__(512) dec_up_tc(const UpArgs<T> a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int VEC = 8;
  const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.B, C = a.C, H = a.H, R = a.R, HS = a.HS, NCLU = a.NCLU, NCP = a.NCP;
  const int R16 = (R + 15) / 16 * 16, UP = 2 * HS + 16, DP = 2 * R16 + 16, HSc = HS / C;
  const UpSmem L = up_smem(MB, HS, R, C, a.st_bytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* dbar = reinterpret_cast<uint64_t*>(smem + L.dbar);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L.mbar);
  float* st = reinterpret_cast<float*>(smem + L.st);
  T* da = reinterpret_cast<T*>(smem + L.da);
  float* hn_s = reinterpret_cast<float*>(smem + L.hn);
  float* ns_s = reinterpret_cast<float*>(smem + L.ns);
  float* mix_s = reinterpret_cast<float*>(smem + L.mix);

  cg::cluster_group cluster = cg::this_cluster();
  const int c = static_cast<int>(cluster.block_rank());
  const int q = blockIdx.x / C;
  const int h0 = q * HS;
  const int64_t CH = static_cast<int64_t>(C) * H;
  const int64_t col0 = static_cast<int64_t>(c) * H + h0;
  const bool pro = a.prev_out != nullptr;
  const bool do_post = (q == 0 && c == 0);

  // Barriers are initialised before the cluster arrive; every peer waits on
  // that cluster barrier before its first remote store into this CTA.
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(dbar, 1);
    mbar_init(mbar, 1);
    // split mode: all R columns of d arrive as T, from the ranks that own them
    mbar_arrive_expect_tx(dbar, a.split ? static_cast<uint32_t>(R * B * 2) : 0u);
    // pre-mix: every rank sends its product for each owned feature and row
    mbar_arrive_expect_tx(mbar, C > 1 ? static_cast<uint32_t>(C * HSc * B * 4) : 0u);
    fence_mbar_init();
  }
  cluster_arrive_relaxed();
  // The up weights and the block inputs are never written by the preceding
  // dec_down_tc, which triggers its dependents only after its own wait:
  // reading them before griddepcontrol.wait is safe. The tile is R rows of HS
  // contiguous elements, CH apart: 16-byte cp.async chunks, consecutive threads
  // on consecutive chunks of a row (one instruction per 16 bytes is cheaper to
  // issue here than one bulk copy per row).
  {
    const int cpr = HS / 8;  // 16-byte chunks per weight row
    const unsigned char* gsrc = reinterpret_cast<const unsigned char*>(a.wu + col0);
    #pragma unroll 1
    for (int i = tid; i < R * cpr; i += nthr) {
      const int r = i / cpr, qd = i - r * cpr;
      cp_async16(smem + L.wu + static_cast<size_t>(r) * UP + qd * 16, gsrc + (static_cast<int64_t>(r) * CH) * 2 + qd * 16);
    }
    cp_async_commit();
    #pragma unroll 1
    for (int i = tid; i < (R16 - R) * cpr; i += nthr) {
      const int r = R + i / cpr, qd = i % cpr;
      *reinterpret_cast<uint4*>(smem + L.wu + static_cast<size_t>(r) * UP + qd * 16) = make_uint4(0, 0, 0, 0);
    }
  }
  // A operand: zero the rows >= B and the columns >= R. The rest is written
  // with d later, possibly by peer CTAs, so it is not touched here.
  {
    const int rz = (8 - B) * (DP / 16);
    #pragma unroll 1
    for (int i = tid; i < rz; i += nthr)
      reinterpret_cast<uint4*>(smem + L.da + B * DP)[i] = make_uint4(0, 0, 0, 0);
    if (R16 > R)
      for (int b = tid; b < B; b += nthr)
        *reinterpret_cast<uint4*>(smem + L.da + b * DP + 2 * R) = make_uint4(0, 0, 0, 0);
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
  pdl_wait();
  pdl_trigger();
  cluster_wait();
  __syncthreads();  // barrier init, S, ns and the zeroed A rows are visible CTA-wide

  // ---- pull the down partials into shared memory: all of them (<= 2 rows),
  // or this rank's column range of every partial row plus, on CTA (0, 0), the
  // inject tile ----
  const int ncols = a.split ? max(0, min(R, (c + 1) * a.per) - c * a.per) : 0;
  const size_t inj_off = static_cast<size_t>(NCLU) * B * a.per;  // floats (split layout)
  if (warp == 0) {
    uint32_t bytes;
    if (!a.split) bytes = static_cast<uint32_t>(NCLU * B * NCP * 4);
    else bytes = static_cast<uint32_t>(NCLU * B * ncols * 4 + (do_post ? NCLU * B * 32 : 0));
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    if (!a.split) {
      if (lane == 0) bulk_g2s(st, a.part_ws, bytes, bar);
    } else {
      #pragma unroll 1
      for (int i = lane; i < NCLU * B; i += 32) {
        if (ncols > 0)
          bulk_g2s(st + static_cast<size_t>(i) * a.per, a.part_ws + static_cast<int64_t>(i) * NCP + c * a.per,
                   static_cast<uint32_t>(ncols * 4), bar);
        if (do_post)  // inject columns: the last tile, from column R16
          bulk_g2s(st + inj_off + static_cast<size_t>(i) * 8, a.part_ws + static_cast<int64_t>(i) * NCP + R16, 32u, bar);
      }
    }
  }
  float inv_r[MB];
#pragma unroll
  for (int b = 0; b < MB; ++b) inv_r[b] = b < B ? a.inv_ws[b * C + c] : 0.0f;
  const bool ok = mbar_wait(bar, 0, &g_tc_wait_timeouts);
  const float qnan = __int_as_float(0x7fc00000);

  // ---- d = ScaledSiLU(rT(sum of the partials in cluster order)) as T ----
  if (!a.split) {
    #pragma unroll 1
    for (int i = tid; i < B * R; i += nthr) {
      const int b = i / R, col = i - b * R;
      const float* src = st + static_cast<size_t>(b) * NCP + col;
      const size_t stride = static_cast<size_t>(B) * NCP;
      const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
      da[b * (DP / 2) + col] = Ty<T>::from_f(ok ? scaled_silu_t<T>(rT<T>(x), a.at.alpha) : qnan);
    }
  } else {
    // column pairs (ncols is a multiple of 4), packed as two T in 32 bits
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
      const uint32_t slot = smem_addr(da + b * (DP / 2) + c * a.per + lc);
      for (int pr = 0; pr < C; ++pr)
        st_async_b32(mapa_shared(slot, pr), packed, mapa_shared(smem_addr(dbar), pr));
    }
  }
  if (do_post) {
    #pragma unroll 1
    for (int i = tid; i < B * C; i += nthr) {
      const int b = i / C, cc = i - b * C;
      const float* src = a.split ? st + inj_off + static_cast<size_t>(b) * 8 + cc : st + static_cast<size_t>(b) * NCP + R16 + cc;
      const size_t stride = a.split ? static_cast<size_t>(B) * 8 : static_cast<size_t>(B) * NCP;
      const float x = ordered_sum(NCLU, [&](int p) { return src[p * stride]; });
      stf(a.post + b * C + cc, ok ? post_gate_of<T>(rT<T>(x), a.at.gate_div, a.at.gate_mul) : qnan);
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
  cp_async_wait_all();
  __syncthreads();
  bool dok = true;
  if (a.split) dok = mbar_wait(dbar, 0, &g_tc_wait_timeouts);

  // ---- up = d @ Wu for 16 columns per warp, transposed: up^T (16 columns x
  // rows) = Wu^T tile (16 x 16 k) * d^T (16 k x 8 rows); k-steps spread over
  // kUpAcc accumulators that are added in a fixed order ----
  const int g = lane >> 2, t4 = lane & 3;
  if (warp < HS / 16) {
    const int m0 = warp * 16;
    float acc[kUpAcc][4];
#pragma unroll
    for (int u = 0; u < kUpAcc; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[u][e] = 0.0f;
    const uint32_t b_base = smem_addr(da) + static_cast<uint32_t>((lane & 7) * DP + ((lane >> 3) & 1) * 16);
    const uint32_t a_base = smem_addr(smem + L.wu) +
                            static_cast<uint32_t>(((lane & 7) + ((lane >> 4) & 1) * 8) * UP + (m0 + ((lane >> 3) & 1) * 8) * 2);
    const int nks = R16 / 16;
    constexpr int KG = kUpKG;
    #pragma unroll 1
    for (int s0 = 0; s0 < nks; s0 += KG) {
      uint32_t af[KG][4], bf[KG][2];
#pragma unroll
      for (int u = 0; u < KG; ++u)
        if (s0 + u < nks) {
          ldsm_x4_trans(a_base + (s0 + u) * 16 * UP, af[u][0], af[u][1], af[u][2], af[u][3]);
          ldsm_x2(b_base + (s0 + u) * 32, bf[u][0], bf[u][1]);
        }
#pragma unroll
      for (int u = 0; u < KG; ++u)
        if (s0 + u < nks) Mma<T>::run4(acc[u % kUpAcc], af[u], bf[u][0], bf[u][1]);
    }
    // fragment value e: column m0 + g (+8 for e >= 2), row 2t (+1 for odd e)
    if (2 * t4 < B) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 2 * t4 + (e & 1), h = m0 + g + (e >> 1) * 8;
        if (row < B) {
          const float up = __fadd_rn(__fadd_rn(acc[0][e], acc[1][e]), __fadd_rn(acc[2][e], acc[3][e]));
          const float gg = sigmoid_rT<T>(rT<T>(up));
          const float prod = dok ? __fmul_rn(hn_s[row * HS + h], gg) : qnan;
          if (C == 1) {
            stf(a.pre + static_cast<int64_t>(row) * H + h0 + h, __fmul_rn(a.at.rho, __fadd_rn(0.0f, prod)));
          } else {
            const int j = h / HSc, hl = h - j * HSc;
            st_async_b32(mapa_shared(smem_addr(mix_s + (c * MB + row) * HSc + hl), j), __float_as_uint(prod),
                         mapa_shared(smem_addr(mbar), j));
          }
        }
      }
    }
  }
  // ---- pre-mix: rank j sums features [j*HSc, (j+1)*HSc) over c = 0..C-1 ----
  if (C > 1) {
    const bool mok = mbar_wait(mbar, 0, &g_tc_wait_timeouts);
    #pragma unroll 1
    for (int i = tid; i < B * HSc; i += nthr) {
      const int b = i / HSc, hl = i - b * HSc;
      float acc2 = 0.0f;
      for (int cc = 0; cc < C; ++cc) acc2 = __fadd_rn(acc2, mix_s[(cc * MB + b) * HSc + hl]);
      stf(a.pre + static_cast<int64_t>(b) * H + h0 + c * HSc + hl, mok ? __fmul_rn(a.at.rho, acc2) : qnan);
    }
  }
}

// ------------------------------------------------------------ configuration

struct TcCfg {
  bool ok;
  int KS, NSL, CL, NCLU, NT, NCP, down_threads, HS, up_threads;
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
  s.split = (rows > 2 && C > 1) ? 1 : 0;
  s.per = ceil_div(ceil_div(R, C), 4) * 4;
  s.bytes = s.split ? static_cast<int>(NCLU * rows * s.per * 4 + NCLU * rows * 32)
                    : static_cast<int>(NCLU * rows * NCP * 4);
  return s;
}

TcCfg tc_cfg(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  TcCfg g{};
  g.ok = false;
  if (dt != HC_F16 && dt != HC_BF16) return g;
  if (rows < 1 || rows > 8) return g;
  if (!(C == 1 || C == 2 || C == 4 || C == 8)) return g;
  if (R < 8 || R % 8 != 0 || R > 512) return g;
  if (H < 16 || H % 16 != 0 || H > 16384) return g;
  const int CH = C * H;
  g.NT = (R + 15) / 16 + 1;
  g.NCP = g.NT * 16;
  const int dw = std::min(16, std::max(4, ceil_div(g.NT, 2)));
  if (ceil_div(g.NT, dw) > kMaxTilesPerWarp) return g;
  g.down_threads = dw * 32;
  // down: the smallest slice (multiple of 16 dividing H) that needs no more
  // CTAs than there are SMs
  g.KS = 0;
  for (int ks = 16; ks <= H; ks += 16) {
    if (H % ks != 0) continue;
    if (down_smem(8, ks, R, C, cluster_for(H / ks), dw).total > kDownSmemCap) break;
    g.KS = ks;
    if (CH / ks <= num_sms) break;
  }
  if (g.KS == 0) return g;
  g.NSL = CH / g.KS;
  g.CL = cluster_for(H / g.KS);
  g.NCLU = g.NSL / g.CL;
  // up: the narrowest tile (multiple of 16 and of C dividing H, at most 16
  // warps of 16 columns) that needs no more CTAs than there are SMs
  const Stage sg = stage_for(rows, C, R, g.NCLU, g.NCP);
  g.HS = 0;
  for (int hs = 16; hs <= std::min(H, 256); hs += 16) {
    if (H % hs != 0 || hs % C != 0) continue;
    if (up_smem(8, hs, R, C, sg.bytes).total > kUpSmemCap) break;
    g.HS = hs;
    if ((H / hs) * C <= num_sms) break;
  }
  if (g.HS == 0) return g;
  g.up_threads = std::min(16, std::max({4, g.HS / 16, ceil_div(R, 32)})) * 32;
  g.ok = true;
  return g;
}

struct Layout {
  size_t inv, part, total;
};
Layout tc_layout(int64_t rows, int C, const TcCfg& g) {
  Layout L;
  L.inv = 0;
  L.part = align_up(static_cast<size_t>(rows) * C * 4, 256);
  L.total = align_up(L.part + static_cast<size_t>(g.NCLU) * rows * g.NCP * 4, 256);
  return L;
}

template <typename T, int MB>
cudaError_t run_tc_mb(const Problem& p, const TcCfg& g) {
  const Layout WL = tc_layout(p.rows, p.C, g);
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
  da.C = p.C; da.H = p.H; da.R = p.R; da.KS = g.KS; da.CL = g.CL; da.NCP = g.NCP;
  da.eps = p.eps;
  da.weights_static = (p.flags & HC_FLAG_WEIGHTS_STATIC) ? 1 : 0;
  const size_t dsm = down_smem(MB, g.KS, p.R, p.C, g.CL, g.down_threads / 32).total;
  cudaError_t e = ensure_smem<dec_down_tc<T, MB>>(dsm);
  if (e != cudaSuccess) return e;
  e = launch_pdl(dec_down_tc<T, MB>, dim3(g.NSL), dim3(g.down_threads), dsm, p.stream, static_cast<unsigned>(g.CL), da);
  if (e != cudaSuccess) return e;

  const Stage sg = stage_for(p.rows, p.C, p.R, g.NCLU, g.NCP);
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
  ua.B = da.B; ua.C = p.C; ua.H = p.H; ua.R = p.R; ua.HS = g.HS; ua.NCLU = g.NCLU; ua.NCP = g.NCP;
  ua.split = sg.split; ua.per = sg.per; ua.st_bytes = sg.bytes;
  ua.at = Attrs{p.eps, p.rho, p.alpha, p.gate_div, p.gate_mul};
  const size_t usm = up_smem(MB, g.HS, p.R, p.C, sg.bytes).total;
  e = ensure_smem<dec_up_tc<T, MB>>(usm);
  if (e != cudaSuccess) return e;
  return launch_pdl(dec_up_tc<T, MB>, dim3((p.H / g.HS) * p.C), dim3(g.up_threads), usm, p.stream,
                    static_cast<unsigned>(p.C), ua);
}

template <typename T>
cudaError_t run_tc(const Problem& p, const TcCfg& g) {
  if (p.rows <= 1) return run_tc_mb<T, 1>(p, g);
  if (p.rows <= 2) return run_tc_mb<T, 2>(p, g);
  if (p.rows <= 4) return run_tc_mb<T, 4>(p, g);
  return run_tc_mb<T, 8>(p, g);
}

// Every input code of T through the fast rounded sigmoid and through the
// accurate one (diagnostic for hc_debug_sigmoid_exact).
template <typename T> struct Code;
template <> struct Code<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(uint16_t c) { return __bfloat162float(__ushort_as_bfloat16(c)); }
  static __device__ __forceinline__ uint16_t of(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
};
template <> struct Code<__half> {
  static __device__ __forceinline__ float to_f(uint16_t c) { return __half2float(__ushort_as_half(c)); }
  static __device__ __forceinline__ uint16_t of(float x) { return __half_as_ushort(__float2half_rn(x)); }
};
template <typename T>
__global__ void sigmoid_codes(uint16_t* fast, uint16_t* acc) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= 65536) return;
  const float x = Code<T>::to_f(static_cast<uint16_t>(i));
  fast[i] = Code<T>::of(sigmoid_rT<T>(x));
  acc[i] = Code<T>::of(sigmoid_acc(x));
}

}  // namespace

bool decode_tc_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt) {
  return tc_cfg(rows, C, H, R, dt, 148).ok;
}

size_t decode_tc_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  const TcCfg g = tc_cfg(rows, C, H, R, dt, num_sms);
  return g.ok ? tc_layout(rows, C, g).total : 0;
}

cudaError_t launch_decode_tc(const Problem& p) {
  const TcCfg g = tc_cfg(p.rows, p.C, p.H, p.R, p.dt, p.num_sms);
  if (!g.ok) return cudaErrorInvalidValue;
  return p.dt == HC_F16 ? run_tc<__half>(p, g) : run_tc<__nv_bfloat16>(p, g);
}

unsigned int read_tc_wait_timeouts(bool reset) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_wait_timeouts, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (reset) {
    const unsigned int z = 0;
    cudaMemcpyToSymbol(g_tc_wait_timeouts, &z, sizeof(z));
  }
  return v;
}

cudaError_t launch_sigmoid_codes(hc_dtype_t dt, uint16_t* fast, uint16_t* acc, cudaStream_t s) {
  if (dt == HC_F16) sigmoid_codes<__half><<<256, 256, 0, s>>>(fast, acc);
  else sigmoid_codes<__nv_bfloat16><<<256, 256, 0, s>>>(fast, acc);
  return cudaGetLastError();
}

}  // namespace hc
