// C ABI of the low-rank mix block: argument validation, path selection and
// dispatch (declared in include/hc_lowrank_mix.h).
//
// Validation mirrors the operator's input checks (ONNX Runtime PR #33384,
// "Summary of Changes": the kernel class validates inputs, selects the path
// and takes scratch from the caller): every error is found on the host before
// any launch and returned as a status. The library keeps no state between
// calls apart from a per-thread error string.
#include <cuda_runtime.h>

#include <cstdarg>
#include <atomic>
#include <cstdio>
#include <cstring>

#include "hc_internal.h"
#include "hc_row_ops.h"

namespace {

thread_local char g_err[512] = "";

hc_status_t fail(hc_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

bool sizes_valid(int64_t rows, int C, int H, int R) {
  if (rows < 0 || C < 1 || H < 1 || R < 1) return false;
  if (static_cast<int64_t>(C) * H > (int64_t{1} << 30) || R > (1 << 20) || C > (1 << 16)) return false;
  if (rows > 4000000) return false;                       // grid.y of the general GEMMs
  if (rows * C >= (int64_t{1} << 31)) return false;       // grid.x of the general norm kernel
  if (rows * C * H > (int64_t{1} << 40)) return false;
  return true;
}

bool dtype_valid(hc_dtype_t dt) { return dt == HC_F32 || dt == HC_F16 || dt == HC_BF16; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  const char* name;
  uintptr_t lo, hi;  // [lo, hi)
};

bool overlaps(const Span& a, const Span& b) {
  return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// Device check: the library is built for sm_103 only.
// SM count of the current device, queried once per device (0 = not yet known).
std::atomic<int> g_sms_of_device[64];

hc_status_t device_info(int* num_sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(HC_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev >= 0 && dev < 64) {
    const int cached = g_sms_of_device[dev].load(std::memory_order_relaxed);
    if (cached > 0) {
      *num_sms = cached;
      return HC_OK;
    }
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(HC_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, major, minor);
  cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64 && *num_sms > 0) g_sms_of_device[dev].store(*num_sms, std::memory_order_relaxed);
  return HC_OK;
}

int select_path(int64_t rows, int C, int H, int R, hc_dtype_t dt, uint32_t flags, int num_sms, bool all_aligned) {
  if (rows == 0) return HC_PATH_NONE;
  if (flags & HC_FLAG_FORCE_GENERAL) return HC_PATH_GENERAL;
  if (!all_aligned) return HC_PATH_GENERAL;
  if (hc::decode_supported(rows, C, H, R, dt)) return HC_PATH_DECODE;
  if (hc::prefill_supported(rows, C, H, R, dt)) return HC_PATH_PREFILL;
  (void)num_sms;
  return HC_PATH_GENERAL;
}

size_t workspace_for(int path, int64_t rows, int C, int H, int R, hc_dtype_t dt, int num_sms) {
  switch (path) {
    case HC_PATH_DECODE: return hc::decode_workspace(rows, C, H, R, dt, num_sms);
    case HC_PATH_PREFILL: return hc::prefill_workspace(rows, C, H, R, dt);
    case HC_PATH_GENERAL: return hc::general_workspace(rows, C, H, R, dt);
    default: return 0;
  }
}

}  // namespace

namespace hc {
hc_status_t set_error(hc_status_t s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace hc

extern "C" {

hc_attrs_t hc_attrs_default(void) {
  hc_attrs_t a;
  a.epsilon = 1e-5f;
  a.reduction_scale = 1.0f;
  a.silu_alpha = 1.0f;
  a.gate_div = 1.0f;
  a.gate_mul = 1.0f;
  a.flags = 0u;
  return a;
}

const char* hc_status_string(hc_status_t s) {
  switch (s) {
    case HC_OK: return "HC_OK";
    case HC_ERR_INVALID_ARG: return "HC_ERR_INVALID_ARG";
    case HC_ERR_UNSUPPORTED: return "HC_ERR_UNSUPPORTED";
    case HC_ERR_WORKSPACE: return "HC_ERR_WORKSPACE";
    case HC_ERR_CUDA: return "HC_ERR_CUDA";
    default: return "HC_ERR_UNKNOWN";
  }
}

const char* hc_last_error(void) { return g_err; }

int hc_lowrank_mix_path(int64_t rows, int C, int H, int R, hc_dtype_t dt, uint32_t flags) {
  if (!sizes_valid(rows, C, H, R) || !dtype_valid(dt)) return -1;
  if (rows == 0) return HC_PATH_NONE;
  int num_sms = 0;
  if (device_info(&num_sms) != HC_OK) return -1;
  return select_path(rows, C, H, R, dt, flags, num_sms, true);
}

size_t hc_lowrank_mix_workspace_size(int64_t rows, int C, int H, int R, hc_dtype_t dt, uint32_t flags) {
  if (!sizes_valid(rows, C, H, R) || !dtype_valid(dt) || rows == 0) return 0;
  int num_sms = 0;
  if (device_info(&num_sms) != HC_OK) return 0;
  // The largest requirement over the aligned and the misaligned choice, so a
  // buffer sized here serves either.
  const size_t a = workspace_for(select_path(rows, C, H, R, dt, flags, num_sms, true), rows, C, H, R, dt, num_sms);
  const size_t b = workspace_for(HC_PATH_GENERAL, rows, C, H, R, dt, num_sms);
  return a > b ? a : b;
}

hc_status_t hc_lowrank_mix(const void* streams, const void* norm_scale, const void* down_w, const void* up_w,
                           const void* inject_w, const void* prev_out, const void* prev_gate, int64_t rows,
                           int C, int H, int R, const hc_attrs_t* attrs, hc_dtype_t dt, void* pre_output,
                           void* post_gate, void* streams_out, void* workspace, size_t workspace_bytes,
                           struct CUstream_st* stream) {
  g_err[0] = '\0';
  if (!sizes_valid(rows, C, H, R))
    return fail(HC_ERR_INVALID_ARG, "invalid sizes rows=%lld C=%d H=%d R=%d", static_cast<long long>(rows), C, H, R);
  if (!dtype_valid(dt)) return fail(HC_ERR_INVALID_ARG, "invalid dtype %d", static_cast<int>(dt));
  if (!norm_scale || !down_w || !up_w || !inject_w)
    return fail(HC_ERR_INVALID_ARG, "a weight pointer (norm_scale, down_w, up_w, inject_w) is NULL");
  if ((prev_out == nullptr) != (prev_gate == nullptr))
    return fail(HC_ERR_INVALID_ARG, "prev_out and prev_gate must both be given or both be NULL");
  if (rows == 0) return HC_OK;
  if (!streams || !pre_output || !post_gate)
    return fail(HC_ERR_INVALID_ARG, "streams, pre_output and post_gate must not be NULL");

  const size_t es = hc::dtype_size(dt);
  const uintptr_t CH = static_cast<uintptr_t>(C) * H;
  const uintptr_t nrows = static_cast<uintptr_t>(rows);
  auto span = [](const char* n, const void* p, uintptr_t bytes) {
    return Span{n, reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + (p ? bytes : 0)};
  };
  const Span ins[] = {span("streams", streams, nrows * CH * es), span("norm_scale", norm_scale, CH * es),
                      span("down_w", down_w, CH * R * es), span("up_w", up_w, CH * R * es),
                      span("inject_w", inject_w, CH * C * es), span("prev_out", prev_out, nrows * H * es),
                      span("prev_gate", prev_gate, nrows * C * es)};
  const Span outs[] = {span("pre_output", pre_output, nrows * H * es), span("post_gate", post_gate, nrows * C * es),
                       span("streams_out", streams_out, nrows * CH * es),
                       span("workspace", workspace, workspace_bytes)};
  for (int i = 0; i < 4; ++i) {
    for (const Span& in : ins)
      if (overlaps(outs[i], in)) return fail(HC_ERR_INVALID_ARG, "%s overlaps input %s", outs[i].name, in.name);
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], outs[j])) return fail(HC_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
  }

  const hc_attrs_t at = attrs ? *attrs : hc_attrs_default();
  int num_sms = 0;
  const hc_status_t ds = device_info(&num_sms);
  if (ds != HC_OK) return ds;

  bool all_aligned = true;
  const void* const ptrs[] = {streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate, pre_output,
                              post_gate, streams_out};
  for (const void* q : ptrs)
    if (q != nullptr && !aligned16(q)) all_aligned = false;
  const int path = select_path(rows, C, H, R, dt, at.flags, num_sms, all_aligned);
  const size_t need = workspace_for(path, rows, C, H, R, dt, num_sms);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need)
      return fail(HC_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                  workspace == nullptr ? size_t{0} : workspace_bytes);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(HC_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  }

  hc::Problem p;
  p.streams = streams; p.norm_scale = norm_scale; p.down_w = down_w; p.up_w = up_w; p.inject_w = inject_w;
  p.prev_out = prev_out; p.prev_gate = prev_gate;
  p.rows = rows; p.C = C; p.H = H; p.R = R;
  p.eps = at.epsilon; p.rho = at.reduction_scale; p.alpha = at.silu_alpha;
  p.gate_div = at.gate_div; p.gate_mul = at.gate_mul; p.flags = at.flags;
  p.dt = dt;
  p.pre_output = pre_output; p.post_gate = post_gate; p.streams_out = streams_out;
  p.workspace = workspace; p.workspace_bytes = workspace_bytes;
  p.stream = reinterpret_cast<cudaStream_t>(stream);
  p.num_sms = num_sms;

  cudaError_t e = cudaSuccess;
  switch (path) {
    case HC_PATH_DECODE: e = hc::launch_decode(p); break;
    case HC_PATH_PREFILL: e = hc::launch_prefill(p); break;
    default: e = hc::launch_general(p); break;
  }
  if (e != cudaSuccess) return fail(HC_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
  return HC_OK;
}

/* Diagnostic: number of bounded device waits that gave up since the last
 * reset (normally 0). Synchronises with the device. */
unsigned int hc_debug_wait_timeouts(int reset) {
  return hc::read_wait_timeouts(reset != 0) + hc::read_tc_wait_timeouts(reset != 0) +
         hc::read_um_wait_timeouts(reset != 0) + hc::read_pf_wait_timeouts(reset != 0);
}

hc_status_t hc_debug_sigmoid_exact(hc_dtype_t dtype, void* fast_out, void* acc_out, struct CUstream_st* stream) {
  if (dtype != HC_F16 && dtype != HC_BF16) return hc::set_error(HC_ERR_INVALID_ARG, "dtype must be HC_F16 or HC_BF16");
  if (fast_out == nullptr || acc_out == nullptr) return hc::set_error(HC_ERR_INVALID_ARG, "null output pointer");
  const cudaError_t e = hc::launch_sigmoid_codes(dtype, static_cast<uint16_t*>(fast_out), static_cast<uint16_t*>(acc_out),
                                                 reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return hc::set_error(HC_ERR_CUDA, cudaGetErrorString(e));
  return HC_OK;
}

size_t hc_debug_phase_clocks(void* buf, size_t bytes) { return hc::set_phase_clocks(buf, bytes); }

hc_status_t hc_debug_sync_probe(int mode, int ctas, int rounds, size_t smem_bytes, void* scratch,
                                size_t scratch_bytes, struct CUstream_st* stream) {
  if (mode < 0 || mode > 2) return hc::set_error(HC_ERR_INVALID_ARG, "mode must be 0, 1 or 2");
  if (ctas < 1 || ctas > 1024 || rounds < 1 || rounds > 100000)
    return hc::set_error(HC_ERR_INVALID_ARG, "ctas must lie in [1, 1024] and rounds in [1, 100000]");
  if (smem_bytes > 200 * 1024) return hc::set_error(HC_ERR_INVALID_ARG, "smem_bytes above 200 KB");
  if (scratch == nullptr || scratch_bytes < (32u + static_cast<size_t>(ctas)) * 4u ||
      (reinterpret_cast<uintptr_t>(scratch) & 15u) != 0)
    return hc::set_error(HC_ERR_WORKSPACE, "scratch must hold (32 + ctas) 32-bit words, 16-byte aligned");
  int num_sms = 0;
  const hc_status_t ds = device_info(&num_sms);
  if (ds != HC_OK) return ds;
  const cudaError_t e = hc::launch_sync_probe(mode, ctas, rounds, smem_bytes, static_cast<unsigned int*>(scratch),
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(HC_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return HC_OK;
}

hc_status_t hc_debug_wait_timeout(float* out, long long limit_cycles, struct CUstream_st* stream) {
  if (out == nullptr) return hc::set_error(HC_ERR_INVALID_ARG, "null output pointer");
  if (limit_cycles < 1000 || limit_cycles > 4000000000LL)
    return hc::set_error(HC_ERR_INVALID_ARG, "limit_cycles must lie in [1e3, 4e9]");
  const cudaError_t e = hc::launch_wait_timeout_probe(out, limit_cycles, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return hc::set_error(HC_ERR_CUDA, cudaGetErrorString(e));
  return HC_OK;
}

size_t hc_debug_sigmoid_table_f16_bytes(void) { return hc::sigmoid_table16_bytes(); }

hc_status_t hc_debug_sigmoid_table_f16(float* g_out, void* table, size_t table_bytes, struct CUstream_st* stream) {
  if (g_out == nullptr || table == nullptr) return hc::set_error(HC_ERR_INVALID_ARG, "null pointer");
  if (table_bytes < hc::sigmoid_table16_bytes() || (reinterpret_cast<uintptr_t>(table) & 15u) != 0)
    return hc::set_error(HC_ERR_WORKSPACE, "table buffer too small or not 16-byte aligned");
  const cudaError_t e = hc::launch_sigmoid_table16_codes(table, g_out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return hc::set_error(HC_ERR_CUDA, cudaGetErrorString(e));
  return HC_OK;
}

hc_status_t hc_debug_sigmoid_table(float* g_out, struct CUstream_st* stream) {
  if (g_out == nullptr) return hc::set_error(HC_ERR_INVALID_ARG, "null output pointer");
  const cudaError_t e = hc::launch_sigmoid_table_codes(g_out, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return hc::set_error(HC_ERR_CUDA, cudaGetErrorString(e));
  return HC_OK;
}


// ---------------------------------------------------------------------------
// Row inverse RMS (FreeToken PR #101) and com.microsoft.EngramGate: declared
// in include/hc_row_ops.h.

hc_status_t hc_inv_rms(const void* x, int64_t rows, int64_t dim, float epsilon, hc_dtype_t dtype, float* out,
                       cudaStream_t stream) {
  if (!dtype_valid(dtype)) return fail(HC_ERR_INVALID_ARG, "invalid dtype %d", static_cast<int>(dtype));
  if (rows < 0 || dim < 1) return fail(HC_ERR_INVALID_ARG, "invalid sizes rows=%lld dim=%lld",
                                       static_cast<long long>(rows), static_cast<long long>(dim));
  if (rows >= (int64_t{1} << 31) || rows * dim > (int64_t{1} << 40))
    return fail(HC_ERR_UNSUPPORTED, "sizes beyond the library's limits");
  if (rows == 0) return HC_OK;
  if (x == nullptr || out == nullptr) return fail(HC_ERR_INVALID_ARG, "null pointer");
  const uintptr_t xs = reinterpret_cast<uintptr_t>(x), os = reinterpret_cast<uintptr_t>(out);
  const Span in{"x", xs, xs + static_cast<uintptr_t>(rows * dim) * hc::dtype_size(dtype)};
  const Span o{"out", os, os + static_cast<uintptr_t>(rows) * 4u};
  if (overlaps(in, o)) return fail(HC_ERR_INVALID_ARG, "out overlaps x");
  int num_sms = 0;
  hc_status_t st = device_info(&num_sms);
  if (st != HC_OK) return st;
  const bool vec = aligned16(x) && (dim * static_cast<int64_t>(hc::dtype_size(dtype))) % 16 == 0;
  const cudaError_t e = hc::launch_inv_rms(x, rows, dim, epsilon, dtype, out, vec, stream);
  if (e != cudaSuccess) return fail(HC_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return HC_OK;
}

hc_status_t hc_engram_gate(const void* key, const void* query, const void* value, const void* key_norm_scale,
                           const void* query_norm_scale, int64_t rows, int hc_mult, int64_t hidden, float epsilon,
                           hc_dtype_t dtype, void* output, cudaStream_t stream) {
  if (!dtype_valid(dtype)) return fail(HC_ERR_INVALID_ARG, "invalid dtype %d", static_cast<int>(dtype));
  if (rows < 0 || hc_mult < 1 || hidden < 1)
    return fail(HC_ERR_INVALID_ARG, "invalid sizes rows=%lld hc_mult=%d hidden=%lld", static_cast<long long>(rows),
                hc_mult, static_cast<long long>(hidden));
  if (rows * hc_mult >= (int64_t{1} << 31) || rows * hc_mult * hidden > (int64_t{1} << 40))
    return fail(HC_ERR_UNSUPPORTED, "sizes beyond the library's limits");
  if (rows == 0) return HC_OK;
  if (!key || !query || !value || !key_norm_scale || !query_norm_scale || !output)
    return fail(HC_ERR_INVALID_ARG, "null pointer");
  const size_t es = hc::dtype_size(dtype);
  auto span = [](const char* n, const void* p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{n, a, a + bytes};
  };
  const size_t row_bytes = static_cast<size_t>(rows) * hc_mult * hidden * es;
  const Span ins[5] = {span("key", key, row_bytes), span("query", query, row_bytes),
                       span("value", value, static_cast<size_t>(rows) * hidden * es),
                       span("key_norm_scale", key_norm_scale, static_cast<size_t>(hc_mult) * hidden * es),
                       span("query_norm_scale", query_norm_scale, static_cast<size_t>(hc_mult) * hidden * es)};
  const Span o = span("output", output, row_bytes);
  for (const Span& in : ins)
    if (overlaps(o, in)) return fail(HC_ERR_INVALID_ARG, "output overlaps input %s", in.name);
  int num_sms = 0;
  hc_status_t st = device_info(&num_sms);
  if (st != HC_OK) return st;
  hc::EngramProblem p{key, query, value, key_norm_scale, query_norm_scale, rows, hc_mult, hidden, epsilon, dtype,
                      output, false, stream};
  p.vec = (hidden * static_cast<int64_t>(es)) % 16 == 0 && aligned16(key) && aligned16(query) && aligned16(value) &&
          aligned16(key_norm_scale) && aligned16(query_norm_scale) && aligned16(output);
  const cudaError_t e = hc::launch_engram_gate(p);
  if (e != cudaSuccess) return fail(HC_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
  return HC_OK;
}

}  // extern "C"
