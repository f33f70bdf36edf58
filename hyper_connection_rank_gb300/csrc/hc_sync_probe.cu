// Cost of the synchronisation a one-kernel decode block would need, against
// the kernel boundary the two-kernel pair uses (a diagnostic behind
// hc_debug_sync_probe).
//
// The down and up halves of a block meet at an all-to-all dependency: every
// up CTA needs the partial sums of every down CTA. The pair puts a kernel
// boundary there (programmatic dependent launch: the dependent grid is
// resident and waits in griddepcontrol.wait until the primary grid has
// finished and its writes are visible). One kernel would need a grid-wide
// barrier instead. The probe times `rounds` repetitions of each mechanism
// over `ctas` CTAs that each hold shared memory like a decode CTA:
//   mode 0: a chain of `rounds` kernels linked by programmatic dependent
//           launch (each waits, then lets its dependent launch);
//   mode 1: one cooperative kernel that crosses `rounds` software grid
//           barriers (one counter: release add, acquire poll);
//   mode 2: one cooperative kernel whose CTAs, per round, each publish a flag
//           (release store) and poll every CTA's flag (acquire loads spread
//           over a warp): the all-to-all exchange without a shared counter.
// Every round's poll is bounded (about 0.1 s of SM clock); a CTA that gives
// up records it in `err` and every CTA leaves the remaining rounds (the others
// give up within their own bound), so the kernel always ends. Cooperative launches fail, instead of starting, when the CTAs
// cannot all be resident at once.
#include <cuda_runtime.h>

#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {
namespace {

constexpr long long kProbeLimitCycles = 200000000LL;  // ~0.1 s
constexpr int kProbeThreads = 128;

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release(unsigned int* p, unsigned int v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kProbeThreads) probe_pdl_link(unsigned int* sink) {
  extern __shared__ uint8_t hold[];  // reserved only: sizes the CTA like a decode CTA
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) hold[0] = static_cast<uint8_t>(blockIdx.x);
  if (threadIdx.x == 0 && blockIdx.x == 0) sink[0] += 1u + hold[0];
}

__global__ void __launch_bounds__(kProbeThreads) probe_grid_barrier(unsigned int* counter, int rounds,
                                                                    unsigned int* err) {
  extern __shared__ uint8_t hold[];
  __shared__ int give_up;
  if (threadIdx.x == 0) give_up = 0;
  __syncthreads();
  const unsigned int n = gridDim.x;
  for (int r = 0; r < rounds; ++r) {
    if (threadIdx.x == 0) {
      const long long t0 = clock64();
      red_release_add(counter, 1u);
      const unsigned int target = n * static_cast<unsigned int>(r + 1);
      while (ld_acquire(counter) < target) {
        if (clock64() - t0 > kProbeLimitCycles) {
          atomicAdd(err, 1u);
          give_up = 1;
          break;
        }
      }
    }
    // another CTA gave up: leave too (decided once per CTA, through shared
    // memory, so every thread of the CTA takes the same branch)
    if (threadIdx.x == 0 && *reinterpret_cast<volatile unsigned int*>(err) != 0u) give_up = 1;
    __syncthreads();
    if (give_up) break;
  }
  if (threadIdx.x == 0) hold[0] = 0;
}

__global__ void __launch_bounds__(kProbeThreads) probe_flag_exchange(unsigned int* flags, int rounds,
                                                                     unsigned int* err) {
  extern __shared__ uint8_t hold[];
  __shared__ int give_up;
  if (threadIdx.x == 0) give_up = 0;
  __syncthreads();
  const unsigned int n = gridDim.x;
  for (int r = 0; r < rounds; ++r) {
    const unsigned int want = static_cast<unsigned int>(r + 1);
    const long long t0 = clock64();
    if (threadIdx.x == 0) st_release(flags + blockIdx.x, want);
    if (threadIdx.x < 32) {
      bool ok = true;
      for (unsigned int j = threadIdx.x; j < n && ok; j += 32) {
        while (ld_acquire(flags + j) < want) {
          if (clock64() - t0 > kProbeLimitCycles) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) {
        atomicAdd(err, 1u);
        give_up = 1;
      }
    }
    // another CTA gave up: leave too (decided once per CTA, through shared
    // memory, so every thread of the CTA takes the same branch)
    if (threadIdx.x == 0 && *reinterpret_cast<volatile unsigned int*>(err) != 0u) give_up = 1;
    __syncthreads();
    if (give_up) break;
  }
  if (threadIdx.x == 0) hold[0] = 0;
}

}  // namespace

cudaError_t launch_sync_probe(int mode, int ctas, int rounds, size_t smem, unsigned int* scratch, cudaStream_t s) {
  // scratch: [0] error count, [1] sink / counter, [32..32+ctas) flags; the
  // caller zeroes it before the call
  unsigned int* err = scratch;
  if (mode == 0) {
    cudaError_t e = ensure_smem<probe_pdl_link>(smem);
    for (int r = 0; r < rounds && e == cudaSuccess; ++r)
      e = launch_pdl(probe_pdl_link, dim3(ctas), dim3(kProbeThreads), smem, s, 1u, scratch + 1);
    return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kProbeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (mode == 1) {
    cudaError_t e = ensure_smem<probe_grid_barrier>(smem);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, probe_grid_barrier, scratch + 1, rounds, err);
  }
  cudaError_t e = ensure_smem<probe_flag_exchange>(smem);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, probe_flag_exchange, scratch + 32, rounds, err);
}

}  // namespace hc
