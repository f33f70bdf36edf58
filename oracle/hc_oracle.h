/* CPU oracle of the hyper-connection low-rank mix block (test infrastructure).
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use
 * this library. It is independent of the GPU library: no shared source, no
 * shared header, no shared constants.
 *
 * Definition: ONNX Runtime pull request #33384, "Schema summary" and
 * "Numerics contract" (HyperConnectionLowRankMix). See hc_oracle.cpp for the
 * formulas and the readings taken where the page is silent.
 *
 * Tensors are host arrays, contiguous, row-major, element type T:
 *   dtype 0 = float32, 1 = float16 (raw 16-bit codes), 2 = bfloat16 (raw codes).
 *   streams (rows, C*H), norm_scale (C*H), down_w (C*H, R), up_w (R, C*H),
 *   inject_w (C*H, C), prev_out (rows, H) and prev_gate (rows, C) both or
 *   neither; pre_output (rows, H), post_gate (rows, C), streams_out (rows, C*H)
 *   or NULL.
 * trace, if not NULL, receives per row (hc_oracle_trace_floats_per_row floats):
 *   S[C*H], inv[C], hn[C*H], down[R], inject[C], Z[R], SG[R], hidden[R],
 *   up[C*H], g[C*H] -- each already rounded to T where the contract rounds.
 * Returns 0 on success, 1 on an invalid argument.
 */
#ifndef HC_ORACLE_H
#define HC_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int hc_oracle_abi_version(void);
int64_t hc_oracle_trace_floats_per_row(int C, int H, int R);
int hc_oracle_lowrank_mix(const void* streams, const void* norm_scale, const void* down_w,
                          const void* up_w, const void* inject_w, const void* prev_out,
                          const void* prev_gate, int64_t rows, int C, int H, int R,
                          float epsilon, float reduction_scale, float silu_alpha, float gate_div,
                          float gate_mul, int dtype, void* pre_output, void* post_gate,
                          void* streams_out, float* trace, int nthreads);
/* Row inverse RMS (FreeToken PR #101): out[r] = 1/sqrt(mean_i(x[r,i]^2) + eps)
 * in double, for x (rows, dim) of type dtype. Returns 0, or 1 on a bad argument. */
int hc_oracle_inv_rms(const void* x, int64_t rows, int64_t dim, double eps, int dtype, double* out);
/* com.microsoft.EngramGate: key, query (rows, M, D); value (rows, D); key_scale,
 * query_scale (M, D); output (rows, M, D), all of type dtype; gate_out (rows*M)
 * doubles or NULL. Evaluated in double, output rounded to T. */
int hc_oracle_engram_gate(const void* key, const void* query, const void* value, const void* key_scale,
                          const void* query_scale, int64_t rows, int M, int64_t D, double eps, int dtype,
                          void* output, double* gate_out);
/* The oracle's own rounding to T (identity for float32) and sigmoid, exposed
 * so the tests can pin them against independent library conversions. */
float hc_oracle_round(float x, int dtype);
float hc_oracle_sigmoid(float x);
void hc_oracle_to_float(const void* src, int dtype, int64_t n, float* dst);
void hc_oracle_from_float(const float* src, int dtype, int64_t n, void* dst);

#ifdef __cplusplus
}
#endif

#endif /* HC_ORACLE_H */
