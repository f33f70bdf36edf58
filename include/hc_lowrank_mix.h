/* hc_lowrank_mix.h -- C ABI of the GB300 (sm_103a) hyper-connection low-rank mix block.
 *
 * The operation is the fused block defined in ONNX Runtime pull request #33384,
 * "com.microsoft.HyperConnectionLowRankMix", sections "Schema summary" and
 * "Numerics contract":
 *
 *   S          = streams + prev_post_gate * prev_block_output   (optional prologue; else S = streams)
 *   hn         = S / sqrt(mean_h(S^2) + epsilon) * norm_scale    (per branch c, over its H features)
 *   down       = hn @ down_weight                                (K = C*H, N = R)
 *   d          = ScaledSiLU(down, silu_alpha) = down * sigmoid(silu_alpha * down)
 *   g          = sigmoid(d @ up_weight)                          (per stream and feature)
 *   pre_output = reduction_scale * sum_c (hn * g)                (shape (..., H))
 *   post_gate  = sigmoid((hn @ inject_weight) / gate_div) * gate_mul   (shape (..., C))
 *   streams_out = S
 *
 * Numerics: products and reductions accumulate in fp32; every step is rounded
 * once to T at S, hn, down, Z (= silu_alpha*down), SG (= sigmoid(Z)), hidden
 * (= down*SG = d), up, g, pre_output, inject, post_gate; the sigmoid is
 * 1/(1+expf(-x)) in fp32 with an IEEE divide. Accumulation order is fixed for a
 * given shape and path: results are bitwise deterministic, and a row's bits do
 * not depend on the number of rows within one path (see hc_lowrank_mix_path);
 * the prefill path splits its down projection differently up to 512 rows and
 * beyond, so there the invariance holds within each of the two ranges. Across
 * paths or ranges a row stays within the stated tolerance of the exact result
 * but may differ in its last bits.
 *
 * Memory: every tensor argument is a DEVICE pointer to contiguous row-major
 * data of element type T (all tensors share T). The caller owns all memory;
 * the library never allocates, never synchronises the host, and keeps no
 * state between calls, so a call can be captured in a CUDA graph.
 */
#ifndef HC_LOWRANK_MIX_H
#define HC_LOWRANK_MIX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is struct CUstream_st* */

typedef enum {
  HC_OK = 0,
  HC_ERR_INVALID_ARG = 1, /* null required pointer, bad size, half a prologue, aliasing outputs */
  HC_ERR_UNSUPPORTED = 2, /* device is not sm_103, or a size beyond the library's limits */
  HC_ERR_WORKSPACE = 3,   /* workspace missing, too small, or not 256-byte aligned */
  HC_ERR_CUDA = 4         /* a CUDA runtime call failed (hc_last_error() has the text) */
} hc_status_t;

/* Element type T of every tensor ("T = float / float16 / bfloat16"). */
typedef enum { HC_F32 = 0, HC_F16 = 1, HC_BF16 = 2 } hc_dtype_t;

/* Operator attributes ("Schema summary", Attributes). num_branches is the C
 * argument of the calls below. */
typedef struct {
  float epsilon;          /* default 1e-5 */
  float reduction_scale;  /* default 1 */
  float silu_alpha;       /* default 1 */
  float gate_div;         /* default 1 */
  float gate_mul;         /* default 1 */
  uint32_t flags;         /* HC_FLAG_* below */
} hc_attrs_t;

/* The weights (norm_scale, down, up, inject) are not written by any kernel
 * still running on the stream when this call is made. The first kernel may
 * then stream its weights before waiting for the previous kernel (programmatic
 * dependent launch). Without the flag it waits first. */
#define HC_FLAG_WEIGHTS_STATIC 1u
/* Run the general CUDA-core path even where a specialised path applies
 * (for cross-path checks). */
#define HC_FLAG_FORCE_GENERAL 2u

/* Path selected for a call (hc_lowrank_mix_path). */
#define HC_PATH_NONE 0    /* rows == 0: nothing is launched */
#define HC_PATH_DECODE 1  /* rows <= 8 (16 for the bf16/fp16 tensor-core pair): split-K weight-streaming pair */
#define HC_PATH_PREFILL 2 /* many rows, fp16/bf16: tcgen05 tensor-core contractions */
#define HC_PATH_GENERAL 3 /* any shape, any rows, any T: CUDA-core kernels */

/* Attribute defaults of the schema: {1e-5, 1, 1, 1, 1, flags 0}. */
hc_attrs_t hc_attrs_default(void);

/* Which path hc_lowrank_mix takes for these sizes on the current device, given
 * that every pointer is 16-byte aligned (misaligned pointers select
 * HC_PATH_GENERAL). Returns a HC_PATH_* value, or -1 for invalid sizes. */
int hc_lowrank_mix_path(int64_t rows, int C, int H, int R, hc_dtype_t dt, uint32_t flags);

/* Bytes of device workspace hc_lowrank_mix needs for these sizes and flags
 * (0 if none). The workspace is scratch: it may hold anything on entry and
 * holds nothing useful on return. */
size_t hc_lowrank_mix_workspace_size(int64_t rows, int C, int H, int R, hc_dtype_t dt, uint32_t flags);

/* Enqueue one block on `stream` (NULL = the legacy default stream).
 *
 * Inputs (device, type T, contiguous):
 *   streams     (rows, C*H): element (b, c, h) at b*C*H + c*H + h
 *   norm_scale  (C*H)
 *   down_w      (C*H, R) row-major [K, N]
 *   up_w        (R, C*H) row-major [K, N]
 *   inject_w    (C*H, C) row-major [K, N]
 *   prev_out    (rows, H)  prev_block_output, or NULL
 *   prev_gate   (rows, C)  prev_post_gate, or NULL; both prologue inputs or neither
 * Outputs (device, type T, contiguous, written in full):
 *   pre_output  (rows, H)
 *   post_gate   (rows, C)
 *   streams_out (rows, C*H) or NULL: S after the prologue (a copy of streams without one)
 * Outputs must not overlap each other, any input, or the workspace.
 * attrs: NULL means hc_attrs_default().
 * workspace: device buffer of at least hc_lowrank_mix_workspace_size(...) bytes,
 *   256-byte aligned; may be NULL when that size is 0.
 * rows == 0 returns HC_OK and launches nothing; row pointers may then be NULL.
 *
 * Errors are detected on the host before anything is launched and returned as a
 * status; hc_last_error() gives a description (per calling thread). Faults
 * during execution surface on the stream, as for any CUDA kernel. */
hc_status_t hc_lowrank_mix(const void* streams, const void* norm_scale, const void* down_w,
                           const void* up_w, const void* inject_w, const void* prev_out,
                           const void* prev_gate, int64_t rows, int C, int H, int R,
                           const hc_attrs_t* attrs, hc_dtype_t dt, void* pre_output,
                           void* post_gate, void* streams_out, void* workspace,
                           size_t workspace_bytes, struct CUstream_st* stream);

/* hc_lowrank_mix for callers that cannot allocate device memory.
 *
 * The page that defines the block has no counterpart to this entry point.
 * Some callers cannot provide a workspace: a host whose memory pool owns the
 * whole GPU and refuses later allocations, a plug-in interface that passes
 * tensors and a stream but no allocator, or code running inside a strict
 * (global-mode) stream capture, where an allocation would break the capture.
 * This variant runs the decode path with its scratch in a fixed 1 MiB device
 * array inside the library (per GPU, held until the process exits) and
 * allocates nothing.
 *
 * Arguments and outputs are those of hc_lowrank_mix without the workspace.
 * Only decode-path problems fit (hc_lowrank_mix_path gives HC_PATH_DECODE:
 * up to 8 rows, or 16 for the bf16/fp16 tensor-core pair's shapes), every
 * pointer 16-byte aligned, partial sums within 1 MiB (the 4 x 2560, rank-320
 * block uses well under 200 KB at 16 rows); anything else returns
 * HC_ERR_UNSUPPORTED with the reason in hc_last_error().
 * All calls share the one array and it keeps the last call's contents (the
 * kernels need no cleared scratch); calls whose kernels may run at the same
 * time on one GPU, such as calls on two unordered streams, race on it.
 * The first call on each device looks up the array's address (with that
 * device current); make that call before capturing a stream that uses it. */
hc_status_t hc_lowrank_mix_decode_noalloc(const void* streams, const void* norm_scale, const void* down_w,
                                          const void* up_w, const void* inject_w, const void* prev_out,
                                          const void* prev_gate, int64_t rows, int C, int H, int R,
                                          const hc_attrs_t* attrs, hc_dtype_t dt, void* pre_output,
                                          void* post_gate, void* streams_out, struct CUstream_st* stream);

/* Static name of a status code. */
const char* hc_status_string(hc_status_t status);

/* Description of the last error returned on the calling thread ("" if none). */
const char* hc_last_error(void);

/* Diagnostic: how many bounded device-side waits (on asynchronous copies) gave
 * up since the last reset; 0 in normal operation. A wait gives up after about
 * one second, writes NaN into the affected outputs and lets the kernel finish.
 * Synchronises with the current device; reset != 0 clears the count. */
unsigned int hc_debug_wait_timeouts(int reset);

/* Diagnostic, with no counterpart on the page that defines the block (it
 * backs the choice of two kernels per decode block over one; the page's
 * research one-kernel variant, "Benchmark", used a grid barrier): enqueues
 * `rounds` repetitions of one synchronisation mechanism over `ctas` CTAs of
 * 128 threads that each reserve smem_bytes of shared memory, for the caller
 * to time with events around the call:
 *   mode 0: a chain of `rounds` kernels linked by programmatic dependent
 *           launch, as between the decode pair's two kernels;
 *   mode 1: one cooperative kernel crossing `rounds` grid barriers (one
 *           counter, release add and acquire poll);
 *   mode 2: one cooperative kernel in which, per round, every CTA publishes
 *           a flag and polls every other CTA's flag.
 * scratch: device buffer owned by the caller, at least (32 + ctas) 32-bit
 * words, 16-byte aligned, ZEROED by the caller before each call; word 0
 * counts polls that gave up (every poll is bounded, about 0.1 s in all, so
 * the kernel always ends; 0 in a valid run). Limits: ctas 1..1024, rounds
 * 1..100000, smem_bytes <= 200 KB. Modes 1 and 2 fail with HC_ERR_CUDA
 * (cooperative launch too large) rather than start when the CTAs cannot all
 * be resident at once. */
hc_status_t hc_debug_sync_probe(int mode, int ctas, int rounds, size_t smem_bytes, void* scratch,
                                size_t scratch_bytes, struct CUstream_st* stream);

/* Diagnostic, with no counterpart on the page that defines the block: phase
 * clocks of the decode path's two tensor-core kernels, to attribute the time
 * of a block to its steps. From the next hc_lowrank_mix call on the calling
 * thread that runs them in bf16 with 1 or 8 rows, each such call writes one
 * slot of `buf` (device memory owned by the caller; consecutive calls take
 * consecutive slots, wrapping after bytes / slot size of them, so every call
 * of a captured chain keeps its own). A slot holds, for the down kernel and
 * then the up kernel, 256 CTAs x 10 points x {globaltimer ns, SM clock64}
 * (unsigned 64-bit), written by thread 0 of each CTA at the points:
 *   down: 0 entry, 1 weights issued, 2 dependency wait returned, 3 S pass
 *         done, 4 inverse RMS stored, 5 weights landed, 6 MMA operands ready,
 *         7 MMA done, 8 cluster exchange landed, 9 partial sums written;
 *   up:   0 entry, 1 prefetches issued, 2 dependency wait returned, 3 partial
 *         sums landed, 4 MMA operands ready, 5 MMA done, 6 pre-mix products
 *         landed, 7 pre_output written.
 * Entries of CTAs beyond the grid and of unused points are left untouched.
 * buf == NULL (or bytes below one slot) stops the recording. Returns the slot
 * size in bytes. The timed kernels compute the same results; they are slower
 * only by the stamps. */
size_t hc_debug_phase_clocks(void* buf, size_t bytes);

/* Diagnostic, with no counterpart on the page that defines the block: makes
 * one bounded device wait run out on purpose, so that the give-up path can be
 * checked without faulting or hanging the GPU. One CTA of 32 threads waits,
 * through the same bounded mbarrier wait the kernels use, on an mbarrier that
 * nothing arrives on and no copy completes, for at most limit_cycles SM clock
 * cycles (1e3 .. 4e9; about 2e6 per millisecond); the wait then gives up,
 * adds one to the count hc_debug_wait_timeouts reports, and the kernel writes
 * NaN to out[0..31] (1.0f where the wait had succeeded) and exits normally.
 * out: device buffer of 32 floats, owned by the caller. Asynchronous on
 * `stream`. HC_ERR_INVALID_ARG for a null pointer or a limit outside the
 * range, HC_ERR_CUDA if the launch fails. */
hc_status_t hc_debug_wait_timeout(float* out, long long limit_cycles, struct CUstream_st* stream);

/* Diagnostic, with no counterpart on the page that defines the block: check of
 * the fast sigmoid the fp16/bf16 kernels use where the contract rounds
 * sigmoid(z) to T for a z that is itself a value of T (the ScaledSiLU gate and
 * g). For each of the 65536 codes x of the 16-bit type `dtype` (HC_F16 or
 * HC_BF16) it writes the T code of that fast rounded sigmoid to fast_out[x]
 * and the T code of rT(1 / (1 + expf(-x))), evaluated with CUDA's accurate
 * expf and an IEEE divide, to acc_out[x]; the two arrays must be identical.
 * fast_out, acc_out: device buffers of 65536 uint16 each, owned by the caller.
 * Asynchronous on `stream`. HC_ERR_INVALID_ARG for another dtype or a null
 * pointer, HC_ERR_CUDA if the launch fails. */
hc_status_t hc_debug_sigmoid_exact(hc_dtype_t dtype, void* fast_out, void* acc_out, struct CUstream_st* stream);

/* Diagnostic, with no counterpart on the page that defines the block: the
 * gate g = rT(sigmoid(rT(up))) exactly as the bf16 prefill epilogue forms it
 * (a shared-memory table of the accurate rounded sigmoid, reached through
 * packed clamps of a pair of values, and the mixed-precision multiply-add of
 * hn * g into an fp32 sum), evaluated with hn = 1 and a zero sum for the up
 * value of each of the 65536 bf16 codes x, so that g_out[x] (fp32) holds g
 * itself; it must equal the accurate rounded sigmoid of x for every code
 * (NaN for NaN). g_out: device buffer of 65536 floats, owned by the caller.
 * Asynchronous on `stream`. HC_ERR_INVALID_ARG for a null pointer,
 * HC_ERR_CUDA if the launch fails. */
hc_status_t hc_debug_sigmoid_table(float* g_out, struct CUstream_st* stream);

/* Diagnostic, with no counterpart on the page that defines the block: the
 * same check for the fp16 prefill epilogue, whose gate table is built per call
 * by a kernel of its own (into the workspace) and copied into each CTA. The
 * table is built into `table` (device scratch owned by the caller, at least
 * hc_debug_sigmoid_table_f16_bytes() bytes, 16-byte aligned), then the gate
 * is formed from it as the epilogue forms it (packed clamps, lookup, the
 * mixed-precision multiply-add of hn * g with hn = 1 and a zero sum) for the up
 * value of each of the 65536 fp16 codes x: g_out[x] (fp32, 65536 floats,
 * caller-owned) must equal the accurate rounded sigmoid of x for every code
 * (NaN for NaN). Asynchronous on `stream`. HC_ERR_INVALID_ARG for a null
 * pointer, HC_ERR_WORKSPACE for a short or misaligned table buffer,
 * HC_ERR_CUDA if a launch fails. */
size_t hc_debug_sigmoid_table_f16_bytes(void);
hc_status_t hc_debug_sigmoid_table_f16(float* g_out, void* table, size_t table_bytes, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* HC_LOWRANK_MIX_H */
