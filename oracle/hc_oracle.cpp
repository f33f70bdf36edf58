// CPU oracle for the hyper-connection low-rank mix block.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously-correct
// statement of what the block computes. Only the test suite, the smoke check
// and the benchmark's CPU-baseline leg load it. The GPU library never links,
// includes or calls it, and it shares no source with the GPU library.
//
// Source of the definition: ONNX Runtime pull request #33384,
// "com.microsoft.HyperConnectionLowRankMix":
//   * "Schema summary": inputs, outputs, layouts and the six formulas
//       S          = streams + prev_post_gate * prev_block_output  (prologue)
//       hn         = S / sqrt(mean_h(S^2) + epsilon) * norm_scale   (per branch)
//       d          = ScaledSiLU(hn @ down_weight, silu_alpha)
//       g          = sigmoid(d @ up_weight)
//       pre_output = reduction_scale * sum_c(hn * g)
//       post_gate  = sigmoid((hn @ inject_weight) / gate_div) * gate_mul
//   * "Numerics contract": fp32 accumulation; one rounding to the I/O type T
//     at S, hn, down, Z, SG, hidden, up, g, pre_output, inject, post_gate;
//     an accurate expf-based fp32 sigmoid rounded once; fixed order, so a row
//     gives the same bits at any batch size.
//
// Readings taken where the page is silent (each is listed with its reason in
// the design notes):
//   * ScaledSiLU(x, a) = x * sigmoid(a * x), with Z = a*x, SG = sigmoid(Z),
//     hidden = x * SG. (Definition not printed; parity with the upstream
//     operator at silu_alpha != 1 is unpinned.)
//   * streams is (..., C, H) flattened, element (c, h) at c*H + h.
//   * norm_scale has C*H entries, indexed like streams.
//   * the prologue adds prev_post_gate[c] * prev_block_output[h] to S[c, h].
//   * mean = sum / H (IEEE divide); inv = 1 / sqrt(mean + eps) (correctly
//     rounded divide and square root); hn = round_T((S * inv) * norm_scale).
//   * reductions are sequential in increasing index; the pre-mix sums the
//     products hn*g over c = 0..C-1 and multiplies by reduction_scale after.
//   * post_gate is rounded once, after the gate_mul multiply.
//   * no multiply-add contraction anywhere (build with -ffp-contract=off).
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fPIC -shared (no fast-math).

#include "hc_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

// ---- IEEE-754 conversions, written from the binary16 / bfloat16 formats ----

inline uint32_t bits_of(float x) { uint32_t u; std::memcpy(&u, &x, 4); return u; }
inline float float_of(uint32_t u) { float x; std::memcpy(&x, &u, 4); return x; }

// bfloat16 is the top half of a binary32; round-to-nearest-even on the
// discarded 16 bits. NaN stays NaN (quiet bit forced).
uint16_t f32_to_bf16(float x) {
  uint32_t u = bits_of(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t keep = u >> 16;
  uint32_t rest = u & 0xffffu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1;  // may carry into exponent: correct
  return static_cast<uint16_t>(keep);
}

float bf16_to_f32(uint16_t h) { return float_of(static_cast<uint32_t>(h) << 16); }

// binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits; round to nearest
// even, overflow to infinity, gradual underflow.
uint16_t f32_to_f16(float x) {
  uint32_t u = bits_of(x);
  uint32_t sign = (u >> 16) & 0x8000u;
  uint32_t a = u & 0x7fffffffu;
  if (a > 0x7f800000u) return static_cast<uint16_t>(sign | 0x7e00u);          // NaN
  if (a >= 0x477ff000u) return static_cast<uint16_t>(sign | 0x7c00u);         // >= 65520 -> inf
  uint32_t e = a >> 23;                 // biased binary32 exponent
  if (e < 113) {                        // below 2^-14: binary16 subnormal (or zero)
    if (e == 0) return static_cast<uint16_t>(sign);                             // binary32 subnormal: < 2^-126
    uint32_t m = (a & 0x7fffffu) | 0x800000u;                                   // value = m * 2^(e-150)
    uint32_t shift = 126 - e;                                                   // value / 2^-24 = m >> shift
    if (shift > 24) return static_cast<uint16_t>(sign);                         // < 2^-25 (half of min subnormal)
    uint32_t r = m >> shift;
    uint32_t rem = m & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (r & 1u))) r += 1;
    return static_cast<uint16_t>(sign | r);
  }
  uint32_t r = ((e - 112) << 10) | ((a & 0x7fffffu) >> 13);
  uint32_t rem = a & 0x1fffu;
  if (rem > 0x1000u || (rem == 0x1000u && (r & 1u))) r += 1;
  return static_cast<uint16_t>(sign | r);
}

float f16_to_f32(uint16_t h) {
  uint32_t sign = (static_cast<uint32_t>(h) & 0x8000u) << 16;
  uint32_t e = (h >> 10) & 0x1fu;
  uint32_t f = h & 0x3ffu;
  if (e == 0x1f) return float_of(sign | 0x7f800000u | (f << 13));             // inf / NaN
  if (e == 0) {                                                               // zero / subnormal: f * 2^-24
    float v = static_cast<float>(f) * float_of(0x33800000u);                  // exact
    return sign ? -v : v;
  }
  return float_of(sign | ((e + 112) << 23) | (f << 13));
}

// round_T: the single rounding step of the numerics contract.
inline float round_t(float x, int dt) {
  if (dt == DT_BF16) return bf16_to_f32(f32_to_bf16(x));
  if (dt == DT_F16) return f16_to_f32(f32_to_f16(x));
  return x;
}

inline float load_t(const void* p, int64_t i, int dt) {
  if (dt == DT_F32) return static_cast<const float*>(p)[i];
  uint16_t h = static_cast<const uint16_t*>(p)[i];
  return dt == DT_BF16 ? bf16_to_f32(h) : f16_to_f32(h);
}

inline void store_t(void* p, int64_t i, float v, int dt) {
  if (dt == DT_F32) { static_cast<float*>(p)[i] = v; return; }
  static_cast<uint16_t*>(p)[i] = dt == DT_BF16 ? f32_to_bf16(v) : f32_to_f16(v);
}

// The accurate sigmoid of the numerics contract: 1 / (1 + exp(-x)) in fp32,
// with the host libm expf and an IEEE divide.
inline float sigmoid(float x) { return 1.0f / (1.0f + std::exp(-x)); }

struct Problem {
  const void *streams, *norm_scale, *down_w, *up_w, *inject_w, *prev_out, *prev_gate;
  int64_t C, H, R;
  float eps, rho, alpha, gate_div, gate_mul;
  int dt;
  void *pre_output, *post_gate, *streams_out;
  float* trace;
};

// One row, start to finish, in the order of the schema formulas.
void one_row(const Problem& p, int64_t b, std::vector<float>& scratch) {
  const int64_t C = p.C, H = p.H, R = p.R, CH = C * H;
  const int dt = p.dt;
  scratch.resize(static_cast<size_t>(4 * CH + 4 * R + 2 * C + 2 * CH));
  float* S = scratch.data();          // CH
  float* hn = S + CH;                 // CH
  float* up = hn + CH;                // CH
  float* g = up + CH;                 // CH
  float* down = g + CH;               // R
  float* Z = down + R;                // R
  float* SG = Z + R;                  // R
  float* d = SG + R;                  // R
  float* inv = d + R;                 // C
  float* inj = inv + C;               // C

  // Prologue: S = streams + prev_post_gate * prev_block_output, rounded to T.
  for (int64_t c = 0; c < C; ++c) {
    for (int64_t h = 0; h < H; ++h) {
      const int64_t k = c * H + h;
      float s = load_t(p.streams, b * CH + k, dt);
      if (p.prev_out != nullptr) {
        float prod = load_t(p.prev_gate, b * C + c, dt) * load_t(p.prev_out, b * H + h, dt);
        s = round_t(s + prod, dt);
      }
      S[k] = s;
    }
  }

  // Branchwise RMS statistic: inv[c] = 1 / sqrt(sum_h S^2 / H + eps).
  for (int64_t c = 0; c < C; ++c) {
    float ss = 0.0f;
    for (int64_t h = 0; h < H; ++h) {
      float s = S[c * H + h];
      ss = ss + s * s;
    }
    float mean = ss / static_cast<float>(H);
    inv[c] = 1.0f / std::sqrt(mean + p.eps);
  }

  // hn = (S * inv) * norm_scale, rounded to T.
  for (int64_t c = 0; c < C; ++c)
    for (int64_t h = 0; h < H; ++h) {
      const int64_t k = c * H + h;
      hn[k] = round_t((S[k] * inv[c]) * load_t(p.norm_scale, k, dt), dt);
    }

  // down = hn @ down_weight (K = C*H, N = R) and inject = hn @ inject_weight
  // (N = C): fp32 sums in increasing k, rounded to T once.
  for (int64_t r = 0; r < R; ++r) down[r] = 0.0f;
  for (int64_t c = 0; c < C; ++c) inj[c] = 0.0f;
  for (int64_t k = 0; k < CH; ++k) {
    const float a = hn[k];
    for (int64_t r = 0; r < R; ++r) down[r] = down[r] + a * load_t(p.down_w, k * R + r, dt);
    for (int64_t c = 0; c < C; ++c) inj[c] = inj[c] + a * load_t(p.inject_w, k * C + c, dt);
  }
  for (int64_t r = 0; r < R; ++r) down[r] = round_t(down[r], dt);
  for (int64_t c = 0; c < C; ++c) inj[c] = round_t(inj[c], dt);

  // ScaledSiLU(down, alpha) = down * sigmoid(alpha * down), rounded at Z, SG, hidden.
  for (int64_t r = 0; r < R; ++r) {
    Z[r] = round_t(p.alpha * down[r], dt);
    SG[r] = round_t(sigmoid(Z[r]), dt);
    d[r] = round_t(down[r] * SG[r], dt);
  }

  // up = d @ up_weight (K = R, N = C*H), rounded; g = sigmoid(up), rounded.
  for (int64_t n = 0; n < CH; ++n) up[n] = 0.0f;
  for (int64_t r = 0; r < R; ++r) {
    const float a = d[r];
    for (int64_t n = 0; n < CH; ++n) up[n] = up[n] + a * load_t(p.up_w, r * CH + n, dt);
  }
  for (int64_t n = 0; n < CH; ++n) {
    up[n] = round_t(up[n], dt);
    g[n] = round_t(sigmoid(up[n]), dt);
  }

  // pre_output[h] = reduction_scale * sum_{c=0..C-1} hn[c,h] * g[c,h], rounded.
  for (int64_t h = 0; h < H; ++h) {
    float acc = 0.0f;
    for (int64_t c = 0; c < C; ++c) acc = acc + hn[c * H + h] * g[c * H + h];
    store_t(p.pre_output, b * H + h, p.rho * acc, dt);
  }

  // post_gate[c] = sigmoid(inject[c] / gate_div) * gate_mul, rounded once.
  for (int64_t c = 0; c < C; ++c)
    store_t(p.post_gate, b * C + c, sigmoid(inj[c] / p.gate_div) * p.gate_mul, dt);

  // streams_out = S (a bit copy of streams when there is no prologue).
  if (p.streams_out != nullptr)
    for (int64_t k = 0; k < CH; ++k) store_t(p.streams_out, b * CH + k, S[k], dt);

  if (p.trace != nullptr) {
    float* t = p.trace + b * hc_oracle_trace_floats_per_row(static_cast<int>(C), static_cast<int>(H),
                                                            static_cast<int>(R));
    auto put = [&t](const float* src, int64_t n) { std::memcpy(t, src, static_cast<size_t>(n) * 4); t += n; };
    put(S, CH); put(inv, C); put(hn, CH); put(down, R); put(inj, C);
    put(Z, R); put(SG, R); put(d, R); put(up, CH); put(g, CH);
  }
}

}  // namespace

extern "C" {

int hc_oracle_abi_version(void) { return 2; }

int64_t hc_oracle_trace_floats_per_row(int C, int H, int R) {
  const int64_t CH = static_cast<int64_t>(C) * H;
  return 4 * CH + 2 * static_cast<int64_t>(C) + 4 * static_cast<int64_t>(R);
}

int hc_oracle_lowrank_mix(const void* streams, const void* norm_scale, const void* down_w,
                          const void* up_w, const void* inject_w, const void* prev_out,
                          const void* prev_gate, int64_t rows, int C, int H, int R,
                          float epsilon, float reduction_scale, float silu_alpha, float gate_div,
                          float gate_mul, int dtype, void* pre_output, void* post_gate,
                          void* streams_out, float* trace, int nthreads) {
  if (rows < 0 || C < 1 || H < 1 || R < 1) return 1;
  if (dtype < DT_F32 || dtype > DT_BF16) return 1;
  if ((prev_out == nullptr) != (prev_gate == nullptr)) return 1;
  if (rows == 0) return 0;
  if (!streams || !norm_scale || !down_w || !up_w || !inject_w || !pre_output || !post_gate) return 1;

  Problem p{streams, norm_scale, down_w, up_w, inject_w, prev_out, prev_gate,
            C, H, R, epsilon, reduction_scale, silu_alpha, gate_div, gate_mul,
            dtype, pre_output, post_gate, streams_out, trace};

  int nt = nthreads > 0 ? nthreads : static_cast<int>(std::thread::hardware_concurrency());
  nt = std::max(1, std::min<int>(nt, static_cast<int>(std::min<int64_t>(rows, 1024))));
  if (nt == 1) {
    std::vector<float> scratch;
    for (int64_t b = 0; b < rows; ++b) one_row(p, b, scratch);
    return 0;
  }
  // Rows are independent; each thread takes a strided subset of them.
  std::vector<std::thread> pool;
  for (int t = 0; t < nt; ++t)
    pool.emplace_back([&p, rows, nt, t]() {
      std::vector<float> scratch;
      for (int64_t b = t; b < rows; b += nt) one_row(p, b, scratch);
    });
  for (auto& th : pool) th.join();
  return 0;
}

// ---- Second workload: the row inverse RMS of FreeToken PR #101 ("perf(dsv4):
// compute the hyper-connection pre-norm in one kernel", sections "The
// problem" and "Accuracy"): inv[r] = 1 / sqrt(mean_i(x[r, i]^2) + eps), the
// scalar the hyper-connection pre-norm multiplies into its mix. The page
// judges a kernel against a float64 evaluation, so that is what this is: the
// squares and their sequential sum in double, the mean by an IEEE divide, the
// square root and the reciprocal correctly rounded in double.
int hc_oracle_inv_rms(const void* x, int64_t rows, int64_t dim, double eps, int dtype, double* out) {
  if (rows < 0 || dim < 1 || dtype < DT_F32 || dtype > DT_BF16) return 1;
  if (rows == 0) return 0;
  if (!x || !out) return 1;
  for (int64_t r = 0; r < rows; ++r) {
    double ss = 0.0;
    for (int64_t i = 0; i < dim; ++i) {
      const double v = load_t(x, r * dim + i, dtype);
      ss += v * v;
    }
    out[r] = 1.0 / std::sqrt(ss / static_cast<double>(dim) + eps);
  }
  return 0;
}

// ---- Third workload: com.microsoft.EngramGate (its kernel README,
// "Description", "Inputs", "Outputs", "Attributes"). For every row
// (batch*sequence index b, stream m) of key and query (rows, M, D):
//   k^ = key / sqrt(mean(key^2) + eps) * key_norm_scale[m]   (likewise q^)
//   dot = sum_i k^_i * q^_i / sqrt(D)
//   gate = sigmoid(sign(dot) * sqrt(max(|dot|, 1e-6)))        (fixed floor)
//   output[b, m, :] = gate * value[b, :]                       (value shared by the M streams)
// Evaluated in double (the README fixes float32 accumulation for its kernels;
// the exact value of the definition is the reference the tests hold a float32
// kernel to). sign(0) = 0, so a zero dot gives a gate of exactly 0.5. The
// output is rounded to T through float32 (a double rounding that can move a
// result by one unit of T only at an exact midpoint). gate_out, if not NULL,
// receives the double gate of each of the rows * M rows.
int hc_oracle_engram_gate(const void* key, const void* query, const void* value, const void* key_scale,
                          const void* query_scale, int64_t rows, int M, int64_t D, double eps, int dtype,
                          void* output, double* gate_out) {
  if (rows < 0 || M < 1 || D < 1 || dtype < DT_F32 || dtype > DT_BF16) return 1;
  if (rows == 0) return 0;
  if (!key || !query || !value || !key_scale || !query_scale || !output) return 1;
  for (int64_t b = 0; b < rows; ++b)
    for (int m = 0; m < M; ++m) {
      const int64_t row = b * M + m;
      double ssk = 0.0, ssq = 0.0;
      for (int64_t i = 0; i < D; ++i) {
        const double k = load_t(key, row * D + i, dtype), q = load_t(query, row * D + i, dtype);
        ssk += k * k;
        ssq += q * q;
      }
      const double ik = 1.0 / std::sqrt(ssk / static_cast<double>(D) + eps);
      const double iq = 1.0 / std::sqrt(ssq / static_cast<double>(D) + eps);
      double dot = 0.0;
      for (int64_t i = 0; i < D; ++i) {
        const double kh = load_t(key, row * D + i, dtype) * ik * load_t(key_scale, m * D + i, dtype);
        const double qh = load_t(query, row * D + i, dtype) * iq * load_t(query_scale, m * D + i, dtype);
        dot += kh * qh;
      }
      dot /= std::sqrt(static_cast<double>(D));
      const double sgn = dot > 0.0 ? 1.0 : (dot < 0.0 ? -1.0 : 0.0);
      const double z = sgn * std::sqrt(std::max(std::fabs(dot), 1e-6));
      const double g = 1.0 / (1.0 + std::exp(-z));
      if (gate_out) gate_out[row] = g;
      for (int64_t i = 0; i < D; ++i)
        store_t(output, row * D + i, static_cast<float>(g * load_t(value, b * D + i, dtype)), dtype);
    }
  return 0;
}

float hc_oracle_round(float x, int dtype) { return round_t(x, dtype); }

float hc_oracle_sigmoid(float x) { return sigmoid(x); }

void hc_oracle_to_float(const void* src, int dtype, int64_t n, float* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = load_t(src, i, dtype);
}

void hc_oracle_from_float(const float* src, int dtype, int64_t n, void* dst) {
  for (int64_t i = 0; i < n; ++i) store_t(dst, i, src[i], dtype);
}

}  // extern "C"
