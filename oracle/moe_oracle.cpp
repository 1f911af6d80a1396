// Oracle for the MoE expert layer: a plain, slow CPU definition in C++17 +
// OpenMP (TEST INFRASTRUCTURE).
//
// Only the tests, the package smoke check and the benchmark's CPU-baseline leg
// load this library.  The CUDA library never links or calls it and shares no
// code, header or table with it.
//
// What it computes
// ----------------
// "Supercharging Olmo-core for Efficient and Scalable MoE Training" (Abstract)
// states the problem: a router sends every token to a few experts, a rowwise
// dispatch writes each token row into its expert's contiguous buffer with no
// permutation pass, routing counts and offsets stay on the device, a grouped GEMM
// runs the uneven per-expert shapes, and the results are combined.  Section 24.1
// adds that keeping the metadata on the device does not change the routing
// calculation.  The article "Olmo-core 3: an open training stack for
// trillion-parameter MoE" (section "Olmo-core 3's answer: experts resident,
// data routed") adds that no expert is padded to a common capacity and that
// MXFP8 is an 8-bit format with shared block scales; Section 24, Evidence 10 of
// the report gives the 33/32-byte MXFP8 payload (one 1-byte scale per 32 one-byte
// values) and the two weight caches.  The pages never write the arithmetic out;
// the readings used (the plainest ones the pages support) are:
//   router      logits = x . W_r^T + bias
//   routing     softmax over all E experts; top-k by logit (descending, equal
//               logits to the lower expert id); gates = the selected softmax
//               probabilities renormalised to sum to one
//   expert      bias-free SwiGLU: y = (silu(x Wg^T) * (x Wu^T)) Wd^T,
//               silu(h) = h / (1 + e^-h)
//   combine     out[t] = sum_j g_tj * y_{e_tj}(x[t]), the gate applied here
//   buffers     expert e owns rows [BM * tile_offsets[e], BM * tile_offsets[e+1])
//               of the dispatched buffer, its routes first in ascending route
//               order (route r = t * k + j), then zero rows
//   backward    exact gradient for the fixed top-k selection
//   load balance  Switch-style LBL = E * sum_e f_e P_e (Section 24.2, Evidence 9)
//   MXFP8       E4M3 values with one E8M0 scale 2^s per 32 values along the
//               contraction axis; s the smallest integer with amax <= 448 * 2^s
//               (clamped to [-127, 127]; 0 for an all-zero block); values
//               x / 2^s rounded to the nearest E4M3 value, ties to the even
//               code, saturating at 448.
// Precision: bf16 inputs (16-bit patterns) are widened exactly; every
// arithmetic operation is in double.  Loops are the definitions written out;
// OpenMP only splits independent rows (no reordering of any sum).
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

#define MO_API extern "C" __attribute__((visibility("default")))

namespace {

double bf16_value(uint16_t bits) {
  const uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// C[n][m] (+)= A[n][K] . B[K][m]: every C[i][j] is the sum over k = 0, 1, ...
// K - 1 in that order.  The loops visit 8 rows x 128 columns of C at a time
// (so that the piece of C stays in the core's L1 cache while k runs); this
// changes which outputs are computed when, not how any one of them is summed.
void gemm(const double* A, int64_t n, int64_t K, const double* B, int64_t m, double* C,
          bool accumulate) {
  constexpr int64_t RB = 8, CB = 128;
  const int64_t nblk = (n + RB - 1) / RB;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t blk = 0; blk < nblk; ++blk) {
    const int64_t i0 = blk * RB, rb = std::min(RB, n - i0);
    for (int64_t j0 = 0; j0 < m; j0 += CB) {
      const int64_t cb = std::min(CB, m - j0);
      double c[RB][CB];
      for (int64_t r = 0; r < rb; ++r)
        for (int64_t j = 0; j < cb; ++j) c[r][j] = accumulate ? C[(i0 + r) * m + j0 + j] : 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double* b = B + k * m + j0;
        for (int64_t r = 0; r < rb; ++r) {
          const double a = A[(i0 + r) * K + k];
          for (int64_t j = 0; j < cb; ++j) c[r][j] += a * b[j];
        }
      }
      for (int64_t r = 0; r < rb; ++r)
        for (int64_t j = 0; j < cb; ++j) C[(i0 + r) * m + j0 + j] = c[r][j];
    }
  }
}

// T[c][r] = X[r][c], 32 x 32 blocks at a time
std::vector<double> transpose(const double* X, int64_t rows, int64_t cols) {
  std::vector<double> T((size_t)rows * cols);
  const int64_t nb = (rows + 31) / 32;
#pragma omp parallel for schedule(static)
  for (int64_t rb = 0; rb < nb; ++rb)
    for (int64_t c0 = 0; c0 < cols; c0 += 32)
      for (int64_t r = rb * 32; r < std::min(rows, rb * 32 + 32); ++r)
        for (int64_t c = c0; c < std::min(cols, c0 + 32); ++c)
          T[(size_t)c * rows + r] = X[(size_t)r * cols + c];
  return T;
}

// C[n][m] = A[n][K] . B[m][K]^T  (B given row-major [m][K])
void matmul_nt(const double* A, int64_t n, int64_t K, const double* B, int64_t m, double* C) {
  const auto BT = transpose(B, m, K);
  gemm(A, n, K, BT.data(), m, C, false);
}

// C[n][m] (+)= A[n][K] . B[K][m]
void matmul_nn(const double* A, int64_t n, int64_t K, const double* B, int64_t m, double* C,
               bool accumulate) {
  gemm(A, n, K, B, m, C, accumulate);
}

// C[n][m] = A[K][n]^T . B[K][m]   (a weight gradient: K runs over an expert's rows)
void matmul_tn(const double* A, int64_t K, int64_t n, const double* B, int64_t m, double* C) {
  const auto AT = transpose(A, K, n);
  gemm(AT.data(), n, K, B, m, C, false);
}

void widen(const uint16_t* bits, size_t n, double* out) {
  for (size_t i = 0; i < n; ++i) out[i] = bf16_value(bits[i]);
}

double silu(double h) { return h / (1.0 + std::exp(-h)); }
double silu_grad(double h) {
  const double s = 1.0 / (1.0 + std::exp(-h));
  return s * (1.0 + h * (1.0 - s));
}

// ------------------------------------------------------------------ E4M3 / E8M0
// OCP MX E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is
// subnormal (m/8 * 2^-6); S.1111.111 is NaN (no infinities); largest 448.
double e4m3_decode(uint8_t c) {
  const double sg = (c & 0x80) ? -1.0 : 1.0;
  const int e = (c >> 3) & 0xF, m = c & 0x7;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0) return sg * (m / 8.0) * std::ldexp(1.0, -6);
  return sg * (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
}

struct E4m3Table {
  double pos[127];   // codes 0..126: the non-negative finite values, ascending
  E4m3Table() {
    for (int c = 0; c < 127; ++c) pos[c] = e4m3_decode((uint8_t)c);
  }
};
const E4m3Table& table() {
  static const E4m3Table t;
  return t;
}

// nearest E4M3 value, ties to the even code, saturating; the sign copied
uint8_t e4m3_encode(double v) {
  const double* pos = table().pos;
  const double a = std::fabs(v);
  int code;
  if (a == 0.0) {
    code = 0;
  } else if (a >= 448.0) {
    code = 126;
  } else {
    // first code whose value is >= a
    int hi = (int)(std::lower_bound(pos, pos + 127, a) - pos);
    if (hi > 126) hi = 126;
    if (pos[hi] == a) {
      code = hi;
    } else {
      const int lo = hi > 0 ? hi - 1 : 0;
      const double dlo = a - pos[lo], dhi = pos[hi] - a;
      if (dlo < dhi) code = lo;
      else if (dhi < dlo) code = hi;
      else code = (lo % 2 == 0) ? lo : hi;
    }
  }
  return (uint8_t)(code | (std::signbit(v) ? 0x80 : 0));
}

// smallest s with amax <= 448 * 2^s, clamped to [-127, 127]; 0 for amax == 0
int64_t mx_scale_exponent(double amax) {
  if (!(amax > 0.0)) return 0;
  int e;
  std::frexp(amax, &e);                // amax = m * 2^e, m in [0.5, 1)
  int64_t s = (int64_t)e - 10;         // 448 * 2^(e - 10) < amax
  for (int i = 0; i < 3; ++i)
    if (amax > 448.0 * std::ldexp(1.0, (int)s)) ++s;
  return std::min<int64_t>(127, std::max<int64_t>(-127, s));
}

// one row of K values -> K codes and K/32 scale bytes
void quantize_row(const double* a, int64_t K, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < K / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(a[b * 32 + i]));
    const int64_t s = mx_scale_exponent(amax);
    const double inv = std::ldexp(1.0, (int)-s);
    for (int i = 0; i < 32; ++i) codes[b * 32 + i] = e4m3_encode(a[b * 32 + i] * inv);
    scales[b] = (uint8_t)(s + 127);
  }
}

void dequantize_row(const uint8_t* codes, const uint8_t* scales, int64_t K, double* out) {
  for (int64_t b = 0; b < K / 32; ++b) {
    const double sc = std::ldexp(1.0, (int)scales[b] - 127);
    for (int i = 0; i < 32; ++i) out[b * 32 + i] = e4m3_decode(codes[b * 32 + i]) * sc;
  }
}

// quantise and dequantise every row of a [rows, K] matrix in place
void qdq_rows(double* a, int64_t rows, int64_t K) {
#pragma omp parallel
  {
    std::vector<uint8_t> c((size_t)K), s((size_t)(K / 32));
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      quantize_row(a + r * K, K, c.data(), s.data());
      dequantize_row(c.data(), s.data(), K, a + r * K);
    }
  }
}

// W[rows, cols], optionally transposed, optionally quantised-dequantised along
// the last axis of the result
std::vector<double> weight(const double* w, int64_t rows, int64_t cols, bool transposed, bool qdq) {
  if (!transposed) {
    std::vector<double> out(w, w + (size_t)rows * cols);
    if (qdq) qdq_rows(out.data(), rows, cols);
    return out;
  }
  std::vector<double> out = transpose(w, rows, cols);
  if (qdq) qdq_rows(out.data(), cols, rows);
  return out;
}

void softmax_row(const double* l, int E, double* p) {
  double m = l[0];
  for (int e = 1; e < E; ++e) m = std::max(m, l[e]);
  double sum = 0.0;
  for (int e = 0; e < E; ++e) {
    p[e] = std::exp(l[e] - m);
    sum += p[e];
  }
  for (int e = 0; e < E; ++e) p[e] /= sum;
}

}  // namespace

// ======================================================================== C ABI
// Every array is row-major and contiguous.  Floating-point arrays are double
// (bf16 inputs are widened exactly by the caller, or by mo_widen_bf16);
// indices are int64 except the top-k ids (int32).  Return 0 on success, -1 on an invalid argument.

MO_API int mo_num_threads() {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

MO_API int mo_widen_bf16(const uint16_t* bits, int64_t n, double* out) {
  widen(bits, (size_t)n, out);
  return 0;
}

MO_API int mo_silu(const double* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = silu(h[i]);
  return 0;
}

MO_API int mo_silu_grad(const double* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = silu_grad(h[i]);
  return 0;
}

// logits[t, e] = sum_i x[t, i] * W_r[e, i] + bias[t, e]   (bias nullable)
MO_API int mo_router_logits(const double* x, const double* wr, const double* bias, int64_t T,
                            int64_t d, int64_t E, double* logits) {
  matmul_nt(x, T, d, wr, E, logits);
  if (bias != nullptr)
    for (int64_t i = 0; i < T * E; ++i) logits[i] += bias[i];
  return 0;
}

// top-k by logit (descending, equal logits to the lower id) and renormalised
// gates = p_sel / sum(p_sel), p the softmax over all E.  -1 on a non-finite logit.
MO_API int mo_softmax_topk_gates(const double* logits, int64_t T, int E, int k, int32_t* idx,
                                 double* gates) {
  if (k < 1 || k > E) return -1;
  for (int64_t i = 0; i < T * E; ++i)
    if (!std::isfinite(logits[i])) return -1;
#pragma omp parallel
  {
    std::vector<int> order((size_t)E);
    std::vector<double> p((size_t)E);
#pragma omp for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
      const double* l = logits + t * E;
      softmax_row(l, E, p.data());
      std::iota(order.begin(), order.end(), 0);
      std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return l[a] > l[b]; });
      double sel = 0.0;
      for (int j = 0; j < k; ++j) sel += p[order[j]];
      for (int j = 0; j < k; ++j) {
        idx[t * k + j] = order[j];
        gates[t * k + j] = p[order[j]] / sel;
      }
    }
  }
  return 0;
}

// counts[e] = number of routes of expert e
MO_API int mo_expert_counts(const int32_t* idx, int64_t R, int E, int64_t* counts) {
  std::fill(counts, counts + E, 0);
  for (int64_t r = 0; r < R; ++r) {
    if (idx[r] < 0 || idx[r] >= E) return -1;
    ++counts[idx[r]];
  }
  return 0;
}

// out[0] = 0, out[e + 1] = out[e] + counts[e]
MO_API int mo_exclusive_scan(const int64_t* counts, int n, int64_t* out) {
  out[0] = 0;
  for (int e = 0; e < n; ++e) out[e + 1] = out[e] + counts[e];
  return 0;
}

// tile_offsets = scan of ceil(counts / bm); row_offsets = bm * tile_offsets
MO_API int mo_tile_layout(const int64_t* counts, int E, int bm, int64_t* tile_offsets,
                          int64_t* row_offsets) {
  if (bm < 1) return -1;
  tile_offsets[0] = 0;
  for (int e = 0; e < E; ++e) tile_offsets[e + 1] = tile_offsets[e] + (counts[e] + bm - 1) / bm;
  for (int e = 0; e <= E; ++e) row_offsets[e] = (int64_t)bm * tile_offsets[e];
  return 0;
}

// routes in ascending (token, choice) order; route r of expert e gets row
// row_offsets[e] + (earlier routes of e); route_of_slot has row_offsets[E]
// entries, -1 on padding rows
MO_API int mo_assign_slots(const int32_t* idx, int64_t T, int k, int E, const int64_t* row_offsets,
                           int64_t* slot_of_route, int64_t* route_of_slot) {
  std::vector<int64_t> cursor((size_t)E, 0);
  std::fill(route_of_slot, route_of_slot + row_offsets[E], (int64_t)-1);
  for (int64_t r = 0; r < T * k; ++r) {
    const int e = idx[r];
    const int64_t s = row_offsets[e] + cursor[e]++;
    slot_of_route[r] = s;
    route_of_slot[s] = r;
  }
  return 0;
}

// Xd[slot_of_route[t * k + j]] = x[t]; padding rows zero
MO_API int mo_dispatch(const double* x, int64_t T, int64_t d, int k, const int64_t* slot_of_route,
                       int64_t n_rows, double* xd) {
  std::fill(xd, xd + n_rows * d, 0.0);
  for (int64_t r = 0; r < T * k; ++r)
    std::memcpy(xd + slot_of_route[r] * d, x + (r / k) * d, (size_t)d * sizeof(double));
  return 0;
}

// One expert's n rows: H = Xd Wg^T, U = Xd Wu^T, A = silu(H) U, Y = A Wd^T,
// with Wg, Wu [f, d] and Wd [d, f].  mx != 0: the MXFP8 forward (Xd is given
// already quantised-dequantised): Wg, Wu quantised along d, Wd along f, and A
// quantised along f (into Aq) before the second GEMM.
MO_API int mo_expert_forward(const double* xd, int64_t n, int64_t d, int64_t f, const double* wg,
                             const double* wu, const double* wd, int mx, double* H, double* U,
                             double* A, double* Aq, double* Y) {
  const auto Wg = weight(wg, f, d, false, mx != 0);
  const auto Wu = weight(wu, f, d, false, mx != 0);
  const auto Wd = weight(wd, d, f, false, mx != 0);
  matmul_nt(xd, n, d, Wg.data(), f, H);
  matmul_nt(xd, n, d, Wu.data(), f, U);
  for (int64_t i = 0; i < n * f; ++i) A[i] = silu(H[i]) * U[i];
  const double* act = A;
  if (mx) {
    std::memcpy(Aq, A, (size_t)(n * f) * sizeof(double));
    qdq_rows(Aq, n, f);
    act = Aq;
  }
  matmul_nt(act, n, f, Wd.data(), d, Y);
  return 0;
}

// out[t] = sum_j gates[t, j] * Y[slot(t, j)]   (j ascending)
MO_API int mo_combine(const double* Y, int64_t d, const double* gates, const int64_t* slot_of_route,
                      int64_t T, int k, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double* o = out + t * d;
    std::fill(o, o + d, 0.0);
    for (int j = 0; j < k; ++j) {
      const double g = gates[t * k + j];
      const double* y = Y + slot_of_route[t * k + j] * d;
      for (int64_t c = 0; c < d; ++c) o[c] += g * y[c];
    }
  }
  return 0;
}

// d_gates[t, j] = <dOut[t], Y[slot(t, j)]>; dY[slot(t, j)] = gates[t, j] dOut[t]; padding rows 0
MO_API int mo_combine_backward(const double* d_out, const double* Y, int64_t d, const double* gates,
                               const int64_t* slot_of_route, int64_t T, int k, int64_t n_rows,
                               double* d_gates, double* dY) {
  std::fill(dY, dY + n_rows * d, 0.0);
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double* go = d_out + t * d;
    for (int j = 0; j < k; ++j) {
      const int64_t s = slot_of_route[t * k + j];
      const double* y = Y + s * d;
      double acc = 0.0;
      for (int64_t c = 0; c < d; ++c) acc += go[c] * y[c];
      d_gates[t * k + j] = acc;
      const double g = gates[t * k + j];
      for (int64_t c = 0; c < d; ++c) dY[s * d + c] = g * go[c];
    }
  }
  return 0;
}

// One expert's n rows: dA = dY Wd; dH = dA U silu'(H); dU = dA silu(H);
// dXd = dH Wg + dU Wu; dWd = dY^T A; dWg = dH^T Xd; dWu = dU^T Xd.
// mx != 0: the MXFP8 backward: the data-gradient GEMMs quantise dY along d and
// dH, dU along f and use the second weight cache (Wd^T quantised along d, Wg^T
// and Wu^T along f); A is the forward's quantised Aq and Xd the dispatched
// quantised tokens; the weight gradients use the unquantised dY, dH, dU.
MO_API int mo_expert_backward(const double* dY, const double* xd, const double* H, const double* U,
                              const double* A, int64_t n, int64_t d, int64_t f, const double* wg,
                              const double* wu, const double* wd, int mx, double* dH, double* dU,
                              double* dXd, double* dWg, double* dWu, double* dWd) {
  std::vector<double> dA((size_t)n * f);
  if (!mx) {
    matmul_nn(dY, n, d, wd, f, dA.data(), false);                 // Wd [d, f]
  } else {
    std::vector<double> dYq(dY, dY + n * d);
    qdq_rows(dYq.data(), n, d);
    const auto WdT = weight(wd, d, f, true, true);                 // [f, d], along d
    matmul_nt(dYq.data(), n, d, WdT.data(), f, dA.data());
  }
  for (int64_t i = 0; i < n * f; ++i) {
    dH[i] = dA[i] * U[i] * silu_grad(H[i]);
    dU[i] = dA[i] * silu(H[i]);
  }
  if (!mx) {
    matmul_nn(dH, n, f, wg, d, dXd, false);                        // Wg [f, d]
    matmul_nn(dU, n, f, wu, d, dXd, true);
  } else {
    std::vector<double> dHq(dH, dH + n * f), dUq(dU, dU + n * f), t1((size_t)n * d);
    qdq_rows(dHq.data(), n, f);
    qdq_rows(dUq.data(), n, f);
    const auto WgT = weight(wg, f, d, true, true);                 // [d, f], along f
    const auto WuT = weight(wu, f, d, true, true);
    matmul_nt(dHq.data(), n, f, WgT.data(), d, dXd);
    matmul_nt(dUq.data(), n, f, WuT.data(), d, t1.data());
    for (int64_t i = 0; i < n * d; ++i) dXd[i] += t1[i];
  }
  matmul_tn(dY, n, d, A, f, dWd);
  matmul_tn(dH, n, f, xd, d, dWg);
  matmul_tn(dU, n, f, xd, d, dWu);
  return 0;
}

// dx[t] = sum_j dXd[slot(t, j)]
MO_API int mo_dispatch_backward(const double* dxd, int64_t d, const int64_t* slot_of_route, int64_t T,
                                int k, double* dx) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    double* o = dx + t * d;
    std::fill(o, o + d, 0.0);
    for (int j = 0; j < k; ++j) {
      const double* s = dxd + slot_of_route[t * k + j] * d;
      for (int64_t c = 0; c < d; ++c) o[c] += s[c];
    }
  }
  return 0;
}

// dl_j = g_j (dg_j - sum_i g_i dg_i) on the selected experts, 0 elsewhere, plus
// the dense `extra` [T, E] (nullable); with W_r (nullable) also
// dx_router = dlogits W_r and dW_r = dlogits^T x.
MO_API int mo_router_backward(const double* d_gates, const double* gates, const int32_t* idx,
                              int64_t T, int k, int E, const double* extra, const double* x,
                              const double* wr, int64_t d, double* dlogits, double* dx_router,
                              double* dw_router) {
  std::fill(dlogits, dlogits + T * E, 0.0);
  for (int64_t t = 0; t < T; ++t) {
    double inner = 0.0;
    for (int j = 0; j < k; ++j) inner += gates[t * k + j] * d_gates[t * k + j];
    for (int j = 0; j < k; ++j)
      dlogits[t * E + idx[t * k + j]] += gates[t * k + j] * (d_gates[t * k + j] - inner);
  }
  if (extra != nullptr)
    for (int64_t i = 0; i < T * E; ++i) dlogits[i] += extra[i];
  if (wr != nullptr) {
    matmul_nn(dlogits, T, E, wr, d, dx_router, false);
    matmul_tn(dlogits, T, E, x, d, dw_router);
  }
  return 0;
}

// LBL = E sum_e f_e P_e, f_e = count_e / (T k), P_e = mean_t softmax(logits[t])_e
MO_API int mo_load_balance(const double* logits, const int32_t* idx, int64_t T, int k, int E,
                           double* lbl, double* P, double* frac) {
  std::vector<double> p((size_t)E);
  std::fill(P, P + E, 0.0);
  std::fill(frac, frac + E, 0.0);
  for (int64_t r = 0; r < T * k; ++r) frac[idx[r]] += 1.0;
  for (int e = 0; e < E; ++e) frac[e] /= (double)(T * k);
  for (int64_t t = 0; t < T; ++t) {
    softmax_row(logits + t * E, E, p.data());
    for (int e = 0; e < E; ++e) P[e] += p[e];
  }
  double s = 0.0;
  for (int e = 0; e < E; ++e) {
    P[e] /= (double)T;
    s += frac[e] * P[e];
  }
  *lbl = E * s;
  return 0;
}

// d(coef * LBL)/dlogits with the counts held fixed:
// coef * E / T * p[t, e] * (f_e - sum_e' f_e' p[t, e'])
MO_API int mo_load_balance_dlogits(const double* logits, const int32_t* idx, int64_t T, int k, int E,
                                   double coef, double* out) {
  std::vector<double> P((size_t)E), frac((size_t)E), p((size_t)E);
  double lbl;
  mo_load_balance(logits, idx, T, k, E, &lbl, P.data(), frac.data());
  for (int64_t t = 0; t < T; ++t) {
    softmax_row(logits + t * E, E, p.data());
    double s = 0.0;
    for (int e = 0; e < E; ++e) s += p[e] * frac[e];
    for (int e = 0; e < E; ++e) out[t * E + e] = coef * E / (double)T * p[e] * (frac[e] - s);
  }
  return 0;
}

// ------------------------------------------------------------------ MXFP8 primitives
MO_API double mo_e4m3_value(int code) { return e4m3_decode((uint8_t)code); }

MO_API int mo_e4m3_encode(const double* v, int64_t n, uint8_t* codes) {
  for (int64_t i = 0; i < n; ++i) codes[i] = e4m3_encode(v[i]);
  return 0;
}

MO_API int mo_mx_scale_exponent(const double* amax, int64_t n, int64_t* s) {
  for (int64_t i = 0; i < n; ++i) s[i] = mx_scale_exponent(amax[i]);
  return 0;
}

// rows of K values (K a multiple of 32) -> codes [rows, K], scales [rows, K/32]
MO_API int mo_quantize_mxfp8(const double* a, int64_t rows, int64_t K, uint8_t* codes,
                             uint8_t* scales) {
  if (K % 32 != 0) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) quantize_row(a + r * K, K, codes + r * K, scales + r * (K / 32));
  return 0;
}

MO_API int mo_dequantize_mxfp8(const uint8_t* codes, const uint8_t* scales, int64_t rows, int64_t K,
                               double* out) {
  if (K % 32 != 0) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) dequantize_row(codes + r * K, scales + r * (K / 32), K, out + r * K);
  return 0;
}

// quantise-dequantise rows in place
MO_API int mo_qdq_rows(double* a, int64_t rows, int64_t K) {
  if (K % 32 != 0) return -1;
  qdq_rows(a, rows, K);
  return 0;
}
