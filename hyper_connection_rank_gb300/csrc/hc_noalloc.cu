// hc_lowrank_mix_decode_noalloc: the decode path with its scratch memory in
// a fixed, file-scope device array instead of a caller-supplied workspace.
//
// Why it exists: some callers cannot allocate device memory at the point
// where they run a block. Examples are a host that hands the whole GPU to
// its own memory pool at start-up and refuses later cudaMalloc calls, a
// plug-in interface that passes tensors and a stream but no allocator, and
// code that runs while a stream is being captured in the strict (global)
// mode, where an allocation would break the capture. This entry point needs
// nothing from them but inputs, outputs and a stream.
//
// Limits and sharing:
//   * the scratch is kHcStaticScratchBytes (1 MiB) per GPU, held from the
//     first load of the library until the process exits;
//   * only decode-path problems fit (up to 8 rows, or 16 where the
//     tensor-core pair serves them; hc_lowrank_mix_path says which), all
//     pointers 16-byte aligned, and a partial-sum buffer that fits in 1 MiB
//     (the 4 x 2560, rank-320 block needs well under 200 KB at 16 rows);
//     anything else returns HC_ERR_UNSUPPORTED with a message in
//     hc_last_error();
//   * every call uses the same array, which keeps whatever the last call left
//     there. The decode kernels write every scratch word they read within one
//     call, so nothing needs clearing, but two calls whose kernels can run at
//     the same time on one GPU (for example on two unordered streams) race on
//     the array. Calls on one stream are ordered and do not race.
//   * the first call on each device looks up the array's device address with
//     cudaGetSymbolAddress while that device is current; make that first call
//     before any stream capture that includes this entry point.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "hc_internal.h"

namespace {

constexpr size_t kHcStaticScratchBytes = size_t{1} << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. In host code this name is only a stand-in for the
// device object: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_hc_static_scratch[kHcStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once.
hc_status_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return hc::set_error(HC_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return hc::set_error(HC_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_hc_static_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return hc::set_error(HC_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e) : "null symbol address");
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return HC_OK;
}

}  // namespace

extern "C" hc_status_t hc_lowrank_mix_decode_noalloc(
    const void* streams, const void* norm_scale, const void* down_w, const void* up_w, const void* inject_w,
    const void* prev_out, const void* prev_gate, int64_t rows, int C, int H, int R, const hc_attrs_t* attrs,
    hc_dtype_t dt, void* pre_output, void* post_gate, void* streams_out, struct CUstream_st* stream) {
  if (rows == 0)  // nothing to launch; the general entry point validates the rest
    return hc_lowrank_mix(streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate, rows, C, H, R, attrs,
                          dt, pre_output, post_gate, streams_out, nullptr, 0, stream);
  const uint32_t flags = attrs ? attrs->flags : 0u;
  const int path = hc_lowrank_mix_path(rows, C, H, R, dt, flags);
  if (path < 0) return hc::set_error(HC_ERR_INVALID_ARG, "invalid sizes or dtype, or no usable device");
  const void* const ptrs[] = {streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate, pre_output,
                              post_gate, streams_out};
  bool aligned = true;
  for (const void* q : ptrs)
    if (q != nullptr && (reinterpret_cast<uintptr_t>(q) & 15u) != 0) aligned = false;
  if (path != HC_PATH_DECODE || !aligned)
    return hc::set_error(HC_ERR_UNSUPPORTED,
                         "the allocation-free entry point serves decode-path problems only "
                         "(hc_lowrank_mix_path gives HC_PATH_DECODE: up to 8 rows, or 16 for the tensor-core pair's "
                         "shapes; 16-byte aligned pointers)");
  int dev = 0, num_sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return hc::set_error(HC_ERR_CUDA, cudaGetErrorString(e));
  const size_t need = hc::decode_workspace(rows, C, H, R, dt, num_sms);
  if (need > kHcStaticScratchBytes) {
    char msg[200];
    snprintf(msg, sizeof(msg), "needs %zu bytes of scratch; the static scratch holds %zu", need,
             kHcStaticScratchBytes);
    return hc::set_error(HC_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  const hc_status_t s = scratch_address(&scratch);
  if (s != HC_OK) return s;
  return hc_lowrank_mix(streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate, rows, C, H, R, attrs, dt,
                        pre_output, post_gate, streams_out, scratch, kHcStaticScratchBytes, stream);
}
