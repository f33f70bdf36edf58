/* hc_row_ops.h -- C ABI of two row-reduction operations that sit beside the
 * hyper-connection low-rank mix block (GB300, sm_103a).
 *
 * hc_inv_rms: the hyper-connection pre-norm scalar of FreeToken pull request
 * #101, "perf(dsv4): compute the hyper-connection pre-norm in one kernel"
 * ("The problem", "The change"):
 *
 *   out[r] = 1 / sqrt( (1/dim) * sum_i x[r, i]^2 + epsilon )
 *
 * read once from the T source (the float32 upcast of a 16-bit value is exact,
 * so the squares do not change), accumulated in fp32, one fp32 value per row.
 * The page judges such a kernel by its distance from a float64 evaluation
 * ("Accuracy"); here the sum of squares is reduced pairwise (within 16-byte
 * vectors, across a thread's vectors, a warp tree, a tree over the CTA's
 * warps), and the divides and the square root are correctly rounded, so
 * out[r] is within 2e-6 relative of the float64 value for rows up to 65536
 * wide (the bound the tests hold it to), as long as the squares and their sum
 * are normal fp32 numbers (|x| between about 2^-60 and 2^60 / sqrt(dim)):
 * beyond that fp32 accumulation underflows or overflows (the sum becomes inf
 * and out[r] = 0), as the page's fp32 kernel does.
 *
 * hc_engram_gate: com.microsoft.EngramGate (its kernel README,
 * "Description", "Inputs", "Outputs", "Attributes"). For every row (b, m):
 *
 *   k^   = key[b, m, :]   / sqrt(mean(key[b, m, :]^2)   + epsilon) * key_norm_scale[m, :]
 *   q^   = query[b, m, :] / sqrt(mean(query[b, m, :]^2) + epsilon) * query_norm_scale[m, :]
 *   dot  = sum(k^ * q^) / sqrt(hidden)
 *   gate = sigmoid(sign(dot) * sqrt(max(|dot|, 1e-6)))      (1e-6 is fixed, not epsilon)
 *   output[b, m, :] = gate * value[b, :]                     (value shared by the hc_mult streams)
 *
 * The two sums of squares and the scaled cross term accumulate in one fp32
 * pass; only the store narrows to T. A zero dot product gives a gate of
 * exactly 1/2. The page's kernels implement float32 and float16; this library
 * also accepts bfloat16.
 *
 * Memory: every tensor argument is a DEVICE pointer to contiguous row-major
 * data owned by the caller; the calls allocate nothing, never synchronise the
 * host and keep no state, so they can be captured in a CUDA graph. Both are
 * asynchronous on `stream`. Results are bitwise deterministic for the same
 * inputs, sizes and device, and a row's result does not depend on the other
 * rows of the call.
 *
 * Errors (checked on the host before any launch): HC_ERR_INVALID_ARG for a bad
 * dtype, negative rows, a zero-sized row, a null pointer (when rows > 0) or an
 * output overlapping an input; HC_ERR_UNSUPPORTED for sizes beyond the
 * library's limits (rows * hc_mult >= 2^31 or more than 2^40 elements) or a
 * device other than sm_103; HC_ERR_CUDA if the launch fails. rows == 0
 * returns HC_OK and launches nothing. hc_last_error() has the message.
 */
#ifndef HC_ROW_OPS_H
#define HC_ROW_OPS_H

#include <stdint.h>

#include "hc_lowrank_mix.h"

#ifdef __cplusplus
extern "C" {
#endif

/* x: (rows, dim) of type dtype. out: rows fp32 values. Any alignment (16-byte
 * aligned x with 16-byte multiple rows takes the vectorised loads). */
hc_status_t hc_inv_rms(const void* x, int64_t rows, int64_t dim, float epsilon, hc_dtype_t dtype, float* out,
                       struct CUstream_st* stream);

/* key, query, output: (rows, hc_mult, hidden); value: (rows, hidden);
 * key_norm_scale, query_norm_scale: (hc_mult, hidden); all of type dtype.
 * rows = batch_size * sequence_length. epsilon: the README's attribute
 * (default 1e-5). */
hc_status_t hc_engram_gate(const void* key, const void* query, const void* value, const void* key_norm_scale,
                           const void* query_norm_scale, int64_t rows, int hc_mult, int64_t hidden, float epsilon,
                           hc_dtype_t dtype, void* output, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* HC_ROW_OPS_H */
