// Host-side interfaces between the C ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "hc_lowrank_mix.h"

namespace hc {

// One validated call, as the launchers see it.
struct Problem {
  const void *streams, *norm_scale, *down_w, *up_w, *inject_w, *prev_out, *prev_gate;
  int64_t rows;
  int C, H, R;
  float eps, rho, alpha, gate_div, gate_mul;
  uint32_t flags;
  hc_dtype_t dt;
  void *pre_output, *post_gate, *streams_out;
  void* workspace;
  size_t workspace_bytes;
  cudaStream_t stream;
  int num_sms;
};

inline size_t dtype_size(hc_dtype_t dt) { return dt == HC_F32 ? 4 : 2; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// General CUDA-core path: any shape, any rows, any T, any alignment.
size_t general_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt);
cudaError_t launch_general(const Problem& p);

// Decode path: rows <= 8 (16 for the tcgen05 pair), split-K weight streaming (hc_decode.cu).
bool decode_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt);
size_t decode_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms);
cudaError_t launch_decode(const Problem& p);
// Tensor-core decode kernels for fp16/bf16 (hc_decode_tc.cu); launch_decode
// routes the shapes they support to them.
bool decode_tc_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt);
size_t decode_tc_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms);
cudaError_t launch_decode_tc(const Problem& p);
unsigned int read_tc_wait_timeouts(bool reset);
// tcgen05 decode kernels for fp16/bf16 (hc_decode_um.cu), preferred where
// they apply (H a multiple of 128, R + 8 <= 512).
bool decode_um_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt);
size_t decode_um_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms);
cudaError_t launch_decode_um(const Problem& p);
unsigned int read_um_wait_timeouts(bool reset);
// Phase clocks of the tcgen05 decode pair (bf16, 1 or 8 rows): record into
// `buf` (slots of the returned size) from the next call on; NULL stops.
size_t set_phase_clocks(void* buf, size_t bytes);
// Synchronisation cost probe (hc_sync_probe.cu): mode 0 PDL chain, 1 grid
// barrier, 2 all-to-all flags; scratch of 32 + ctas words, zeroed by the caller.
cudaError_t launch_sync_probe(int mode, int ctas, int rounds, size_t smem, unsigned int* scratch, cudaStream_t s);
// One CTA whose bounded wait on an mbarrier that nothing completes runs out.
cudaError_t launch_wait_timeout_probe(float* out, long long limit_cycles, cudaStream_t s);
// Every 16-bit code through the fast rounded sigmoid and the accurate one.
cudaError_t launch_sigmoid_codes(hc_dtype_t dt, uint16_t* fast, uint16_t* acc, cudaStream_t s);
cudaError_t launch_sigmoid_table_codes(float* g, cudaStream_t s);
// The fp16 prefill gate: its table's size, and every fp16 code through it
// (the table built into `table` first).
size_t sigmoid_table16_bytes();
cudaError_t launch_sigmoid_table16_codes(void* table, float* g, cudaStream_t s);
// Row inverse RMS and Engram gate (hc_rows.cu). `vec`: every pointer 16-byte
// aligned and the row length a multiple of 16 bytes (16-byte vector loads).
cudaError_t launch_inv_rms(const void* x, int64_t rows, int64_t dim, float eps, hc_dtype_t dt, float* out, bool vec,
                           cudaStream_t s);
struct EngramProblem {
  const void *key, *query, *value, *key_scale, *query_scale;
  int64_t rows;  // batch * sequence
  int M;         // hc_mult
  int64_t D;     // hidden size
  float eps;
  hc_dtype_t dt;
  void* output;
  bool vec;
  cudaStream_t stream;
};
cudaError_t launch_engram_gate(const EngramProblem& p);
// Prefill path: many rows, fp16/bf16, tcgen05 contractions (hc_prefill.cu).
bool prefill_supported(int64_t rows, int C, int H, int R, hc_dtype_t dt);
size_t prefill_workspace(int64_t rows, int C, int H, int R, hc_dtype_t dt);
cudaError_t launch_prefill(const Problem& p);
unsigned int read_pf_wait_timeouts(bool reset);

// Tensor (TMA) maps (hc_tmap.cu): the driver's encoder (nullptr if the
// driver lacks it), and a map over a row-major [outer, inner] matrix of 16-bit
// elements (inner * 2 bytes a multiple of 16, base 16-byte aligned), box {64,
// box_outer}, 128-byte swizzle: each box lands as box_outer rows of 128 bytes,
// 16-byte chunk j of row r at chunk j ^ (r % 8); columns past `inner` read 0.
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder();
bool make_tmap_2d_sw128(CUtensorMap* m, const void* base, bool bf16, uint64_t inner, uint64_t outer,
                        uint32_t box_outer);

// Record `msg` as this thread's hc_last_error() text and return `s`.
hc_status_t set_error(hc_status_t s, const char* msg);

// Diagnostic counter of bounded device waits that gave up.
unsigned int read_wait_timeouts(bool reset);

// Opt a kernel in to `bytes` of dynamic shared memory on the current device.
// The attribute is set once per kernel and device and remembered, so later
// calls (including calls made while a stream is being captured into a graph)
// issue no further runtime calls.
template <auto Kernel>
cudaError_t ensure_smem(size_t bytes) {
  static std::atomic<size_t> granted[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && granted[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  // Ask for the largest shared-memory carveout: an SM configured for a smaller
  // one cannot take a CTA of another kernel that needs more until it drains,
  // which would stop consecutive kernels of a PDL chain from sharing SMs.
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev >= 0 && dev < 64) {
    size_t cur = granted[dev].load(std::memory_order_acquire);
    while (cur < bytes && !granted[dev].compare_exchange_weak(cur, bytes)) {
    }
  }
  return e;
}

// Launch with programmatic stream serialisation (PDL) and an optional
// cluster shape along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace hc
