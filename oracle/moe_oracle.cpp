// moe_oracle.cpp -- plain, slow CPU oracle for the routed-expert hot path
// (dispatch -> W13 GEMM -> SwiGLU -> W2 GEMM x score -> combine, and the backward:
// DGRAD, WGRAD, score gradients).  Loops token by token; where OpenMP is
// available the independent outer loops (tokens, gradient rows) are spread over
// host threads, each output element still summed by one thread in index order,
// so results do not depend on the thread count.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls
// this file; only the test suite, the smoke check and the CPU-baseline leg of the
// benchmark do.  It shares no code, header, table or helper with the CUDA path.
//
// Sources (page title, section):
//   [DM]  "Dist-MoE: Meta's Blackwell SM100 MoE Kernels", section "What it is selling":
//         four caller-owned inputs (activations, top-k ids, scores, weights); the
//         pipeline  route on GPU -> W13 -> SwiGLU -> W2 -> combine; FPROP/DGRAD/WGRAD;
//         BF16 operands with FP32 accumulate; MXFP8 E4M3 quantises activations after
//         routing and takes prepared weights; plain or clamped SwiGLU; in-place
//         WGRAD accumulation.
//   [DM-C] same page, section "Caveats": fixed physical token count, padding rows
//         carry zero scores.
//   [NV-G] "nvfp4moe" README, section "Grouped GEMM": contiguous expert-major rows,
//         m_indptr of length E+1, empty experts valid.
//   [NV-M] same README, section "MoE layer": dispatch, FC1 + gated activation, FC2,
//         probability weighting, deterministic combine; distinct int32 ids per row,
//         float32 weights; padded offsets.
//   [NV-D] same README, sections "Dense GEMM" and "Grouped GEMM": the quantiser
//         yields E2M1 codes two to a byte, one E4M3 scale per block and one
//         dequantisation scale per tensor; a GEMM is scaled by the product of its
//         operands' tensor scales.
//   [NV-T] same README, section "Training" and "Supported kernel surface":
//         deterministic dispatch, combine and router gradients; input and weight
//         gradients.
//
// Readings where the pages are silent (each also listed in the design notes):
//   * W13[e] rows [0,I) are the gate projection and rows [I,2I) the up projection
//     (not interleaved; interleaved weights are listed as unsupported in [DM]).
//   * SwiGLU(gate, up) = silu(gate) * up; the clamped variant clips gate and up to
//     [-L, L] first; its gradient passes at exactly +-L and is zero outside.
//   * Rounding to bf16 (round-to-nearest-even) happens at R1..R7 below; every sum
//     is accumulated in the working type in ascending index order.
//   * Rows of one expert are ordered by ascending flat index t*k+j (stable).
//   * The score multiplies the W2 output before its bf16 rounding (R3); the combine
//     sums the k bf16 contributions of a token in column order j = 0..k-1 (R6).
//   * dscores is the gradient w.r.t. the given scores (no softmax behind them).
//   * For WGRAD-W2 the score is folded into h: hs = bf16(s * h) (R7).
//   * MXFP8 (OCP MX): 32-element blocks along K, E8M0 shared exponent
//     X = floor(log2(amax)) - 8, E4M3 elements rounded to nearest even and
//     saturated to +-448; an all-zero block gets scale code 0.
//   * NVFP4 ([DM]: inference only, weights prepared ahead of the call; [NV-D]:
//     E2M1 codes, E4M3 block scales, a per-tensor dequantisation scale; [NV-M]:
//     fixed activation scales): two-level scaling.
//     A tensor with per-tensor dequantisation scale s has encode scale g = 1/s
//     (fp32).  A 16-element block along K with amax A gets the E4M3 scale code
//     E4M3_RNE_satfinite((A / 6) * g), fp32 arithmetic (6 = E2M1's largest
//     value); with S its value, each element becomes E2M1_RNE_satfinite(v * (g / S))
//     (S = 0: all codes 0).  Weights are prepared per expert with
//     s = amax(W[e]) / (6 * 448) (1 for an all-zero expert); activations (x and
//     h) use static scales the caller sets.  A GEMM sums the dequantised block
//     products (code value times block scale) in fp32 and multiplies the sum by
//     alpha = s_activation * s_weight[e] before its rounding point.
//
// Working type: float (the pages' FP32 accumulate) unless built with
// -DORC_DOUBLE, which evaluates every sum and elementwise step in double (used to
// bound the effect of FP32 summation order).
//
// Built with -fopenmp, the token loops of the forward and backward and the
// output rows of WGRAD run on all host cores.  Every sum keeps its order (one
// thread owns each output element and adds in the same index order), so the
// results are bit-identical to the single-threaded build.
//
// bf16 values cross the C interface as raw uint16 bit patterns.

#include <cstdint>
#include <cstring>
#include <cmath>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifdef ORC_DOUBLE
typedef double real;
#else
typedef float real;
#endif

namespace {

// ---- scalar conversions ----------------------------------------------------

float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// float -> bf16, round to nearest, ties to even (the standard bf16 conversion).
uint16_t float_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) {           // inf or nan
    if (u & 0x007fffffu) return static_cast<uint16_t>((u >> 16) | 0x0040u);
    return static_cast<uint16_t>(u >> 16);
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return static_cast<uint16_t>(u >> 16);
}

uint16_t real_to_bf16(real v) { return float_to_bf16(static_cast<float>(v)); }
real bf(uint16_t b) { return static_cast<real>(bf16_to_float(b)); }

real rexp(real v) { return static_cast<real>(std::exp(static_cast<double>(v))); }

// ---- problem description ---------------------------------------------------

struct Problem {
  int T, d, I, E, k;
  float clamp;                 // 0 = plain SwiGLU, L > 0 = clamped to [-L, L]
  const uint16_t* x;           // [T, d]
  const int32_t* ids;          // [T, k]
  const float* scores;         // [T, k]
  const uint16_t* w13;         // [E, 2I, d]
  const uint16_t* w2;          // [E, d, I]
};

// Is routed element (t, j) valid?  Ids must lie in [0, E) and be distinct within
// a token row ([NV-M]).  The first occurrence of a repeated id stays valid.
bool element_valid(const Problem& p, int t, int j) {
  int e = p.ids[(size_t)t * p.k + j];
  if (e < 0 || e >= p.E) return false;
  for (int jj = 0; jj < j; ++jj)
    if (p.ids[(size_t)t * p.k + jj] == e) return false;
  return true;
}

// Forward quantities of one routed row (token t through expert e with score s).
//   a  [2I] bf16 : gate/up pre-activations               (R1)
//   h  [I]  bf16 : SwiGLU output                          (R2)
//   ys [d]  bf16 : score-weighted W2 output               (R3)
void row_forward(const Problem& p, int t, int e, float s,
                 uint16_t* a, uint16_t* h, uint16_t* ys) {
  const int d = p.d, I = p.I;
  const uint16_t* xt = p.x + (size_t)t * d;
  const uint16_t* W13 = p.w13 + (size_t)e * 2 * I * d;
  const uint16_t* W2 = p.w2 + (size_t)e * d * I;
  // W13 GEMM: a_i = sum_c x[t,c] * W13[e,i,c]   (FPROP, [DM])
  for (int i = 0; i < 2 * I; ++i) {
    real acc = 0;
    const uint16_t* wr = W13 + (size_t)i * d;
    for (int c = 0; c < d; ++c) acc += bf(xt[c]) * bf(wr[c]);
    a[i] = real_to_bf16(acc);                                   // R1
  }
  // SwiGLU: h = silu(G) * U with G, U from the rounded gate/up (optionally clipped)
  const real L = p.clamp;
  for (int i = 0; i < I; ++i) {
    real G = bf(a[i]);
    real U = bf(a[I + i]);
    if (L > 0) {
      G = G < -L ? -L : (G > L ? L : G);
      U = U < -L ? -L : (U > L ? L : U);
    }
    real silu = G / (real(1) + rexp(-G));
    h[i] = real_to_bf16(silu * U);                              // R2
  }
  // W2 GEMM and probability weighting: ys_c = s * sum_i h_i * W2[e,c,i]   ([NV-M])
  for (int c = 0; c < d; ++c) {
    real acc = 0;
    const uint16_t* wr = W2 + (size_t)c * I;
    for (int i = 0; i < I; ++i) acc += bf(h[i]) * bf(wr[i]);
    ys[c] = real_to_bf16(static_cast<real>(s) * acc);           // R3
  }
}

// SwiGLU backward of one routed row, given g = dY_t . W2[e] and the forward's a, h:
//   dA [2I] bf16 (R4), hs [I] bf16 (R7)
void swiglu_backward(const Problem& p, float s, const real* g, const uint16_t* a,
                     const uint16_t* h, uint16_t* dA, uint16_t* hs) {
  const int I = p.I;
  const real L = p.clamp;
  for (int i = 0; i < I; ++i) {
    real ag = bf(a[i]), au = bf(a[I + i]);
    real G = ag, U = au, mg = 1, mu = 1;
    if (L > 0) {
      if (G < -L || G > L) mg = 0;
      if (U < -L || U > L) mu = 0;
      G = G < -L ? -L : (G > L ? L : G);
      U = U < -L ? -L : (U > L ? L : U);
    }
    real dh = static_cast<real>(s) * g[i];
    real sig = real(1) / (real(1) + rexp(-G));
    real silu = G * sig;
    real dsilu = sig * (real(1) + G * (real(1) - sig));
    real dgate = dh * U * dsilu * mg;
    real dup = dh * silu * mu;
    dA[i] = real_to_bf16(dgate);                                // R4
    dA[I + i] = real_to_bf16(dup);                              // R4
    hs[i] = real_to_bf16(static_cast<real>(s) * bf(h[i]));      // R7
  }
}

// Backward quantities of one routed row, given its forward a and h.
//   g       [I]  working type : dY_t . W2[e]
//   dscore        working type : sum_i h_i * g_i
//   dA      [2I] bf16 : gradient at the gate/up pre-activations     (R4)
//   dxe     [d]  bf16 : dA . W13[e]                                  (R5)
//   hs      [I]  bf16 : s * h, the WGRAD-W2 operand                  (R7)
void row_backward(const Problem& p, int t, int e, float s, const uint16_t* dy,
                  const uint16_t* a, const uint16_t* h,
                  real* dscore, uint16_t* dA, uint16_t* dxe, uint16_t* hs) {
  const int d = p.d, I = p.I;
  const uint16_t* dyt = dy + (size_t)t * d;
  const uint16_t* W13 = p.w13 + (size_t)e * 2 * I * d;
  const uint16_t* W2 = p.w2 + (size_t)e * d * I;
  std::vector<real> g(I);
  // DGRAD through W2: g_i = sum_c dY[t,c] * W2[e,c,i]
  for (int i = 0; i < I; ++i) {
    real acc = 0;
    for (int c = 0; c < d; ++c) acc += bf(dyt[c]) * bf(W2[(size_t)c * I + i]);
    g[i] = acc;
  }
  // score gradient: y depends on s through s * (h . W2), so dL/ds = sum_i h_i g_i
  real ds = 0;
  for (int i = 0; i < I; ++i) ds += bf(h[i]) * g[i];
  *dscore = ds;
  swiglu_backward(p, s, g.data(), a, h, dA, hs);
  // DGRAD through W13: dxe_c = sum_{i<2I} dA_i * W13[e,i,c]
  for (int c = 0; c < d; ++c) {
    real acc = 0;
    for (int i = 0; i < 2 * I; ++i) acc += bf(dA[i]) * bf(W13[(size_t)i * d + c]);
    dxe[c] = real_to_bf16(acc);                                 // R5
  }
}

Problem make_problem(int T, int d, int I, int E, int k, float clamp,
                     const uint16_t* x, const int32_t* ids, const float* scores,
                     const uint16_t* w13, const uint16_t* w2) {
  Problem p;
  p.T = T; p.d = d; p.I = I; p.E = E; p.k = k; p.clamp = clamp;
  p.x = x; p.ids = ids; p.scores = scores; p.w13 = w13; p.w2 = w2;
  return p;
}

// ---- MXFP8 (E4M3 elements, E8M0 block scales) ------------------------------

// Value of an E4M3 code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
// exponent field 0 is subnormal; 0x7F/0xFF are NaN and never produced here).
double e4m3_value(uint8_t c) {
  int sgn = (c >> 7) & 1, ex = (c >> 3) & 15, man = c & 7;
  double v = ex == 0 ? std::ldexp(man / 8.0, -6) : std::ldexp(1.0 + man / 8.0, ex - 7);
  return sgn ? -v : v;
}

// Nearest E4M3 value to v, ties to the even code, saturating to +-448.  The 127
// non-negative finite codes 0x00..0x7E are monotone in value, so the nearest one
// is found by bisection over that table.
struct E4m3Table {
  double v[127];
  E4m3Table() {
    for (int c = 0; c < 127; ++c) v[c] = e4m3_value(static_cast<uint8_t>(c));
  }
};

uint8_t e4m3_encode(double v) {
  static const E4m3Table tab;                 // built once (thread-safe static init)
  const double* table = tab.v;
  uint8_t sgn = std::signbit(v) ? 0x80 : 0x00;
  double m = std::fabs(v);
  if (m >= table[126]) return sgn | 126;
  int lo = 0, hi = 126;                       // table[lo] <= m < table[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (table[mid] <= m) lo = mid; else hi = mid;
  }
  double dl = m - table[lo], dh = table[hi] - m;
  int c = dl < dh ? lo : (dh < dl ? hi : (lo % 2 == 0 ? lo : hi));
  return sgn | static_cast<uint8_t>(c);
}

// Quantise one 32-element block (bf16 in) to E4M3 codes and an E8M0 code.
void quant_block(const uint16_t* in, int n, uint8_t* codes, uint8_t* scale) {
  float amax = 0;
  for (int i = 0; i < n; ++i) {
    float v = std::fabs(bf16_to_float(in[i]));
    if (v > amax) amax = v;
  }
  if (amax == 0) {
    *scale = 0;
    for (int i = 0; i < n; ++i) codes[i] = 0;
    return;
  }
  int ex;
  std::frexp(static_cast<double>(amax), &ex);       // amax = f * 2^ex, f in [0.5, 1)
  int X = (ex - 1) - 8;                              // floor(log2 amax) - emax(E4M3)
  if (X < -127) X = -127;
  if (X > 127) X = 127;
  *scale = static_cast<uint8_t>(X + 127);
  for (int i = 0; i < n; ++i)
    codes[i] = e4m3_encode(std::ldexp(static_cast<double>(bf16_to_float(in[i])), -X));
}

double e8m0_value(uint8_t s) { return std::ldexp(1.0, static_cast<int>(s) - 127); }

// Dequantised value of prepared element n of a [rows, K] code matrix with
// scales [rows, K/32].
real mx_value(const uint8_t* q, const uint8_t* sc, int K, size_t row, int col) {
  return static_cast<real>(e4m3_value(q[row * K + col]) *
                           e8m0_value(sc[row * (K / 32) + col / 32]));
}

// Quantise n bf16 values in 32-element blocks (the last block may be shorter)
// and return their dequantised values.
void mx_roundtrip(const uint16_t* in, int n, real* out) {
  uint8_t q[32], sc;
  for (int b = 0; b < n; b += 32) {
    const int m = n - b < 32 ? n - b : 32;
    quant_block(in + b, m, q, &sc);
    for (int i = 0; i < m; ++i)
      out[b + i] = static_cast<real>(e4m3_value(q[i]) * e8m0_value(sc));
  }
}

// MXFP8 forward quantities of one routed row ([DM]: activations quantised after
// routing, prepared weights): x row quantised along d, W13 prepared along d,
// a (R1), h (R2), h quantised along I, W2 prepared along I, ys (R3).
void row_forward_mx(const Problem& p, int t, int e, float s, const uint8_t* w13q,
                    const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s, uint16_t* a,
                    uint16_t* h, uint16_t* ys) {
  const int d = p.d, I = p.I;
  std::vector<real> xv(d), hv(I);
  mx_roundtrip(p.x + (size_t)t * d, d, xv.data());
  for (int i = 0; i < 2 * I; ++i) {
    const size_t row = (size_t)e * 2 * I + i;
    real acc = 0;
    for (int c = 0; c < d; ++c) acc += xv[c] * mx_value(w13q, w13s, d, row, c);
    a[i] = real_to_bf16(acc);                                  // R1
  }
  const real L = p.clamp;
  for (int i = 0; i < I; ++i) {
    real G = bf(a[i]), U = bf(a[I + i]);
    if (L > 0) {
      G = G < -L ? -L : (G > L ? L : G);
      U = U < -L ? -L : (U > L ? L : U);
    }
    h[i] = real_to_bf16(G / (real(1) + rexp(-G)) * U);         // R2
  }
  mx_roundtrip(h, I, hv.data());
  for (int c = 0; c < d; ++c) {
    const size_t row = (size_t)e * d + c;
    real acc = 0;
    for (int i = 0; i < I; ++i) acc += hv[i] * mx_value(w2q, w2s, I, row, i);
    ys[c] = real_to_bf16(static_cast<real>(s) * acc);          // R3
  }
}

// MXFP8 backward quantities of one routed row: each GEMM takes its operands
// block-quantised along its own K.
//   g   = Q_d(dY_t) . W2[e]       W2 prepared along d:  w2tq [E, I, d], w2ts [E, I, d/32]
//   dscore, dA (R4), hs (R7)      as in the bf16 backward, from the forward's a, h
//   dxe = Q_2I(dA) . W13[e]       W13 prepared along 2I: w13tq [E, d, 2I], w13ts [E, d, 2I/32]
void row_backward_mx(const Problem& p, int t, int e, float s, const uint16_t* dy,
                     const uint16_t* a, const uint16_t* h, const uint8_t* w13tq,
                     const uint8_t* w13ts, const uint8_t* w2tq, const uint8_t* w2ts,
                     real* dscore, uint16_t* dA, uint16_t* dxe, uint16_t* hs) {
  const int d = p.d, I = p.I;
  std::vector<real> dyv(d), g(I), dav(2 * I);
  mx_roundtrip(dy + (size_t)t * d, d, dyv.data());
  for (int i = 0; i < I; ++i) {
    const size_t row = (size_t)e * I + i;
    real acc = 0;
    for (int c = 0; c < d; ++c) acc += dyv[c] * mx_value(w2tq, w2ts, d, row, c);
    g[i] = acc;
  }
  real ds = 0;
  for (int i = 0; i < I; ++i) ds += bf(h[i]) * g[i];
  *dscore = ds;
  swiglu_backward(p, s, g.data(), a, h, dA, hs);
  mx_roundtrip(dA, 2 * I, dav.data());
  for (int c = 0; c < d; ++c) {
    const size_t row = (size_t)e * d + c;
    real acc = 0;
    for (int i = 0; i < 2 * I; ++i) acc += dav[i] * mx_value(w13tq, w13ts, 2 * I, row, i);
    dxe[c] = real_to_bf16(acc);                                // R5
  }
}

// ---- NVFP4 (E2M1 elements, E4M3 scales per 16 elements, per-tensor scale) ----

// Value of an E2M1 code (1 sign bit, 2 exponent bits with bias 1, 1 mantissa
// bit; exponent field 0 is subnormal): magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
double e2m1_value(uint8_t c) {
  int sgn = (c >> 3) & 1, ex = (c >> 1) & 3, man = c & 1;
  double v = ex == 0 ? man * 0.5 : std::ldexp(1.0 + man / 2.0, ex - 1);
  return sgn ? -v : v;
}

// Nearest E2M1 value to v, ties to the even code (mantissa bit 0), saturating
// to +-6; the sign is kept (negative values that round to zero give code 8).
uint8_t e2m1_encode(double v) {
  const uint8_t sgn = std::signbit(v) ? 8 : 0;
  const double m = std::fabs(v);
  if (m >= 6.0) return sgn | 7;
  int lo = 0;                                   // e2m1_value(lo) <= m < e2m1_value(lo + 1)
  while (lo < 6 && e2m1_value(static_cast<uint8_t>(lo + 1)) <= m) ++lo;
  const double dl = m - e2m1_value(static_cast<uint8_t>(lo));
  const double dh = e2m1_value(static_cast<uint8_t>(lo + 1)) - m;
  const int c = dl < dh ? lo : (dh < dl ? lo + 1 : (lo % 2 == 0 ? lo : lo + 1));
  return sgn | static_cast<uint8_t>(c);
}

// Quantise n (<= 16) bf16 values of one block with encode scale g: E2M1 codes
// (one per byte here) and the E4M3 scale code.
void nv_quant_block(const uint16_t* in, int n, float g, uint8_t* codes, uint8_t* scale) {
  float amax = 0;
  for (int i = 0; i < n; ++i) {
    const float v = std::fabs(bf16_to_float(in[i]));
    if (v > amax) amax = v;
  }
  float t = amax / 6.0f;
  t = t * g;
  const uint8_t sc = e4m3_encode(static_cast<double>(t));
  *scale = sc;
  const float S = static_cast<float>(e4m3_value(sc));
  if (S == 0.0f) {
    for (int i = 0; i < n; ++i) codes[i] = 0;
    return;
  }
  const float r = g / S;
  for (int i = 0; i < n; ++i) {
    const float v = bf16_to_float(in[i]) * r;
    codes[i] = e2m1_encode(static_cast<double>(v));
  }
}

// Dequantised element (row, col) of a packed [rows, K/2] code matrix (element
// 2i in the low nibble of byte i) with E4M3 scales [rows, K/16].
real nv_value(const uint8_t* q, const uint8_t* sc, int K, size_t row, int col) {
  const uint8_t b = q[row * (K / 2) + col / 2];
  const uint8_t c = (col & 1) ? (b >> 4) : (b & 15);
  return static_cast<real>(e2m1_value(c) * e4m3_value(sc[row * (K / 16) + col / 16]));
}

// Quantise n bf16 values (n a multiple of 16) with encode scale g and return
// their dequantised values (code value times block scale; the per-tensor scale
// is applied to the GEMM sum).
void nv_roundtrip(const uint16_t* in, int n, float g, real* out) {
  uint8_t q[16], sc;
  for (int b = 0; b < n; b += 16) {
    nv_quant_block(in + b, 16, g, q, &sc);
    for (int i = 0; i < 16; ++i)
      out[b + i] = static_cast<real>(e2m1_value(q[i]) * e4m3_value(sc));
  }
}

// NVFP4 forward quantities of one routed row ([DM], [NV-M]: BF16 activation
// quantisation, FC1 + gated activation + NVFP4 requantisation, FC2, probability
// weighting): x row quantised along d with the static input scale, W13 and W2
// prepared, a (R1, after alpha), h (R2), h quantised along I with the static
// hidden scale, ys (R3, score times alpha times the W2 sum).
struct NvScales {
  float x_scale, h_scale;            // static activation dequantisation scales
  const float* w13_scale;            // [E] per-expert weight dequantisation scales
  const float* w2_scale;             // [E]
};

void row_forward_nv(const Problem& p, int t, int e, float s, const uint8_t* w13q,
                    const uint8_t* w13s, const uint8_t* w2q, const uint8_t* w2s,
                    const NvScales& sc, uint16_t* a, uint16_t* h, uint16_t* ys) {
  const int d = p.d, I = p.I;
  std::vector<real> xv(d), hv(I);
  const float gx = 1.0f / sc.x_scale, gh = 1.0f / sc.h_scale;
  nv_roundtrip(p.x + (size_t)t * d, d, gx, xv.data());
  const float alpha13 = sc.x_scale * sc.w13_scale[e];
  for (int i = 0; i < 2 * I; ++i) {
    const size_t row = (size_t)e * 2 * I + i;
    real acc = 0;
    for (int c = 0; c < d; ++c) acc += xv[c] * nv_value(w13q, w13s, d, row, c);
    a[i] = real_to_bf16(acc * static_cast<real>(alpha13));     // R1
  }
  const real L = p.clamp;
  for (int i = 0; i < I; ++i) {
    real G = bf(a[i]), U = bf(a[I + i]);
    if (L > 0) {
      G = G < -L ? -L : (G > L ? L : G);
      U = U < -L ? -L : (U > L ? L : U);
    }
    h[i] = real_to_bf16(G / (real(1) + rexp(-G)) * U);         // R2
  }
  nv_roundtrip(h, I, gh, hv.data());
  const float alpha2 = sc.h_scale * sc.w2_scale[e];
  for (int c = 0; c < d; ++c) {
    const size_t row = (size_t)e * d + c;
    real acc = 0;
    for (int i = 0; i < I; ++i) acc += hv[i] * nv_value(w2q, w2s, I, row, i);
    const real v = acc * static_cast<real>(alpha2);
    ys[c] = real_to_bf16(static_cast<real>(s) * v);            // R3
  }
}

}  // namespace

extern "C" {

// Which working type this build uses: 4 (float) or 8 (double).
int orc_real_bytes() { return static_cast<int>(sizeof(real)); }

// Host threads the parallel loops use (1 without OpenMP).
int orc_threads() {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

// Set the number of host threads (ignored without OpenMP); returns orc_threads().
int orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
  return orc_threads();
}

int orc_float_to_bf16(const float* in, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = float_to_bf16(in[i]);
  return 0;
}

// Dispatch ([NV-G], [NV-M], [NV-T]): a stable counting sort of the routed
// elements by expert.  For each valid element (t, j) with e = ids[t,j]:
//   rank_of[t*k+j] = number of valid elements of expert e with smaller flat index
//   row_of[t*k+j]  = off_pad[e] + rank_of[t*k+j]
// invalid elements get rank_of = row_of = -1.
//   counts[e]   = valid elements routed to e
//   m_indptr    = exclusive prefix sum of counts (length E+1)
//   off_pad     = exclusive prefix sum of counts rounded up to a multiple of BM
// Returns the smallest invalid flat index, or -1 if all ids are valid.
long orc_dispatch(int T, int k, int E, int BM, const int32_t* ids,
                  int32_t* counts, int32_t* m_indptr, int32_t* off_pad,
                  int32_t* rank_of, int32_t* row_of) {
  Problem p = make_problem(T, 0, 0, E, k, 0, nullptr, ids, nullptr, nullptr, nullptr);
  long first_bad = -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j) {
      long f = (long)t * k + j;
      if (!element_valid(p, t, j)) {
        if (first_bad < 0) first_bad = f;
        rank_of[f] = -1;
        continue;
      }
      rank_of[f] = counts[ids[f]]++;
    }
  m_indptr[0] = 0;
  off_pad[0] = 0;
  for (int e = 0; e < E; ++e) {
    m_indptr[e + 1] = m_indptr[e] + counts[e];
    off_pad[e + 1] = off_pad[e] + (counts[e] + BM - 1) / BM * BM;
  }
  for (long f = 0; f < (long)T * k; ++f)
    row_of[f] = rank_of[f] < 0 ? -1 : off_pad[ids[f]] + rank_of[f];
  return first_bad;
}

// Gather ([DM] "route on GPU"): xe[r] = x[token_of[r]] for rows r < nrows, zero
// rows where token_of[r] < 0 (padding).
int orc_gather_rows(int nrows, int d, const uint16_t* x, const int32_t* token_of,
                    uint16_t* xe) {
  for (int r = 0; r < nrows; ++r) {
    int t = token_of[r];
    for (int c = 0; c < d; ++c) xe[(size_t)r * d + c] = t < 0 ? 0 : x[(size_t)t * d + c];
  }
  return 0;
}

// Combine ([NV-M], [NV-T] deterministic combine): y[t,c] = bf16(sum_j ys[row_of[t,j], c])
// in column order j = 0..k-1; elements with row_of < 0 are skipped.        (R6)
int orc_combine_rows(int T, int k, int d, const uint16_t* ys, const int32_t* row_of,
                     uint16_t* y) {
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < d; ++c) {
      real acc = 0;
      for (int j = 0; j < k; ++j) {
        int r = row_of[(size_t)t * k + j];
        if (r >= 0) acc += bf(ys[(size_t)r * d + c]);
      }
      y[(size_t)t * d + c] = real_to_bf16(acc);
    }
  return 0;
}

// Forward for the listed tokens (toks == NULL: tokens 0..ntok-1).
//   y  [ntok, d]        bf16 output                               (R6)
//   a  [ntok, k, 2I]    optional, gate/up pre-activations          (R1)
//   h  [ntok, k, I]     optional, SwiGLU outputs                   (R2)
//   ys [ntok, k, d]     optional, score-weighted expert outputs    (R3)
// Invalid elements contribute nothing and leave their optional rows zero.
int orc_forward(int T, int d, int I, int E, int k, float clamp,
                const uint16_t* x, const int32_t* ids, const float* scores,
                const uint16_t* w13, const uint16_t* w2,
                int ntok, const int32_t* toks,
                uint16_t* y, uint16_t* a_out, uint16_t* h_out, uint16_t* ys_out) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, w13, w2);
#pragma omp parallel for schedule(dynamic)
  for (int n = 0; n < ntok; ++n) {
    std::vector<uint16_t> a(2 * I), h(I), ys((size_t)k * d, 0);
    std::vector<char> ok(k);
    int t = toks ? toks[n] : n;
    for (int j = 0; j < k; ++j) {
      ok[j] = element_valid(p, t, j);
      uint16_t* ysj = ys.data() + (size_t)j * d;
      if (!ok[j]) {
        std::memset(ysj, 0, sizeof(uint16_t) * d);
        if (a_out) std::memset(a_out + ((size_t)n * k + j) * 2 * I, 0, sizeof(uint16_t) * 2 * I);
        if (h_out) std::memset(h_out + ((size_t)n * k + j) * I, 0, sizeof(uint16_t) * I);
        continue;
      }
      int e = ids[(size_t)t * k + j];
      float s = scores[(size_t)t * k + j];
      row_forward(p, t, e, s, a.data(), h.data(), ysj);
      if (a_out) std::memcpy(a_out + ((size_t)n * k + j) * 2 * I, a.data(), sizeof(uint16_t) * 2 * I);
      if (h_out) std::memcpy(h_out + ((size_t)n * k + j) * I, h.data(), sizeof(uint16_t) * I);
    }
    if (ys_out) std::memcpy(ys_out + (size_t)n * k * d, ys.data(), sizeof(uint16_t) * k * d);
    for (int c = 0; c < d; ++c) {
      real acc = 0;
      for (int j = 0; j < k; ++j)
        if (ok[j]) acc += bf(ys[(size_t)j * d + c]);
      y[(size_t)n * d + c] = real_to_bf16(acc);                 // R6
    }
  }
  return 0;
}

// Backward for the listed tokens, given the upstream gradient dy [T, d].
//   dx      [ntok, d]      bf16, overwritten                     (R6 of R5)
//   dscores [ntok, k]      float, overwritten (0 for invalid elements)
//   dA      [ntok, k, 2I]  optional                              (R4)
//   hs      [ntok, k, I]   optional                              (R7)
//   g       [ntok, k, I]   optional, float
//   dxe     [ntok, k, d]   optional, per-expert input gradients  (R5)
int orc_backward(int T, int d, int I, int E, int k, float clamp,
                 const uint16_t* x, const int32_t* ids, const float* scores,
                 const uint16_t* w13, const uint16_t* w2, const uint16_t* dy,
                 int ntok, const int32_t* toks,
                 uint16_t* dx, float* dscores,
                 uint16_t* dA_out, uint16_t* hs_out, float* g_out, uint16_t* dxe_out) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, w13, w2);
#pragma omp parallel for schedule(dynamic)
  for (int n = 0; n < ntok; ++n) {
    std::vector<uint16_t> a(2 * I), h(I), ys(d), dA(2 * I), hs(I), dxe((size_t)k * d, 0);
    std::vector<char> ok(k);
    int t = toks ? toks[n] : n;
    for (int j = 0; j < k; ++j) {
      ok[j] = element_valid(p, t, j);
      size_t nj = (size_t)n * k + j;
      if (!ok[j]) {
        dscores[nj] = 0;
        if (dA_out) std::memset(dA_out + nj * 2 * I, 0, sizeof(uint16_t) * 2 * I);
        if (hs_out) std::memset(hs_out + nj * I, 0, sizeof(uint16_t) * I);
        if (g_out) std::memset(g_out + nj * I, 0, sizeof(float) * I);
        continue;
      }
      int e = ids[(size_t)t * k + j];
      float s = scores[(size_t)t * k + j];
      row_forward(p, t, e, s, a.data(), h.data(), ys.data());
      real ds;
      row_backward(p, t, e, s, dy, a.data(), h.data(), &ds, dA.data(),
                   dxe.data() + (size_t)j * d, hs.data());
      dscores[nj] = static_cast<float>(ds);
      if (dA_out) std::memcpy(dA_out + nj * 2 * I, dA.data(), sizeof(uint16_t) * 2 * I);
      if (hs_out) std::memcpy(hs_out + nj * I, hs.data(), sizeof(uint16_t) * I);
      if (g_out) {
        // recompute g in the working type for inspection
        const uint16_t* W2 = w2 + (size_t)e * d * I;
        for (int i = 0; i < I; ++i) {
          real acc = 0;
          for (int c = 0; c < d; ++c) acc += bf(dy[(size_t)t * d + c]) * bf(W2[(size_t)c * I + i]);
          g_out[nj * I + i] = static_cast<float>(acc);
        }
      }
    }
    for (int c = 0; c < d; ++c) {
      real acc = 0;
      for (int j = 0; j < k; ++j)
        if (ok[j]) acc += bf(dxe[(size_t)j * d + c]);
      dx[(size_t)n * d + c] = real_to_bf16(acc);                // R6
    }
    if (dxe_out) {
      for (int j = 0; j < k; ++j)
        for (int c = 0; c < d; ++c)
          dxe_out[((size_t)n * k + j) * d + c] = ok[j] ? dxe[(size_t)j * d + c] : 0;
    }
  }
  return 0;
}

// WGRAD of one expert e ([DM] "in-place WGRAD accumulation"): the increments that
// a backward pass adds to the existing FP32 gradients, summed in FP32 over the
// rows of e in dispatch order (ascending flat index):
//   dw13_delta [2I, d] : sum_rows dA_i * x[t,c]
//   dw2_delta  [d, I]  : sum_rows dY[t,c] * hs_i
// Returns the number of rows of expert e.
int orc_wgrad_expert(int T, int d, int I, int E, int k, float clamp,
                     const uint16_t* x, const int32_t* ids, const float* scores,
                     const uint16_t* w13, const uint16_t* w2, const uint16_t* dy,
                     int e, float* dw13_delta, float* dw2_delta) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, w13, w2);
  // the rows of expert e in dispatch order
  std::vector<int> row_t, row_j;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j)
      if (ids[(size_t)t * k + j] == e && element_valid(p, t, j)) {
        row_t.push_back(t);
        row_j.push_back(j);
      }
  const int rows = static_cast<int>(row_t.size());
  // each row's backward operands dA (R4) and hs (R7)
  std::vector<uint16_t> dA_rows((size_t)rows * 2 * I), hs_rows((size_t)rows * I);
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < rows; ++r) {
    std::vector<uint16_t> a(2 * I), h(I), ys(d), dxe(d);
    const int t = row_t[r];
    const float s = scores[(size_t)t * k + row_j[r]];
    row_forward(p, t, e, s, a.data(), h.data(), ys.data());
    real ds;
    row_backward(p, t, e, s, dy, a.data(), h.data(), &ds, dA_rows.data() + (size_t)r * 2 * I,
                 dxe.data(), hs_rows.data() + (size_t)r * I);
  }
  // dW13 increment: each output row i sums over the rows in dispatch order
#pragma omp parallel for schedule(static)
  for (int i = 0; i < 2 * I; ++i) {
    std::vector<real> acc(d, 0);
    for (int r = 0; r < rows; ++r) {
      const real ai = bf(dA_rows[(size_t)r * 2 * I + i]);
      const uint16_t* xt = x + (size_t)row_t[r] * d;
      for (int c = 0; c < d; ++c) acc[c] += ai * bf(xt[c]);
    }
    for (int c = 0; c < d; ++c) dw13_delta[(size_t)i * d + c] = static_cast<float>(acc[c]);
  }
  // dW2 increment: each output row c sums over the rows in dispatch order
#pragma omp parallel for schedule(static)
  for (int c = 0; c < d; ++c) {
    std::vector<real> acc(I, 0);
    for (int r = 0; r < rows; ++r) {
      const real yc = bf(dy[(size_t)row_t[r] * d + c]);
      const uint16_t* hs = hs_rows.data() + (size_t)r * I;
      for (int i = 0; i < I; ++i) acc[i] += yc * bf(hs[i]);
    }
    for (int i = 0; i < I; ++i) dw2_delta[(size_t)c * I + i] = static_cast<float>(acc[i]);
  }
  return rows;
}

// MXFP8 quantiser ([DM]: MXFP8 E4M3 with prepared weights): quantise a bf16
// matrix [rows, K] along K in 32-element blocks.  codes [rows, K] E4M3 bytes;
// scales [rows, K/32] E8M0 bytes.  K must be a multiple of 32.
int orc_quant_mxfp8(long rows, int K, const uint16_t* in, uint8_t* codes, uint8_t* scales) {
  if (K % 32) return -1;
  for (long r = 0; r < rows; ++r)
    for (int b = 0; b < K / 32; ++b)
      quant_block(in + r * K + b * 32, 32, codes + r * K + b * 32, scales + r * (K / 32) + b);
  return 0;
}

int orc_e4m3_encode(const double* in, uint8_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = e4m3_encode(in[i]);
  return 0;
}

int orc_e4m3_decode(const uint8_t* in, double* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = e4m3_value(in[i]);
  return 0;
}

// MXFP8 forward for the listed tokens.  The routed activation row is quantised
// along d (after routing), the weights arrive prepared (codes + E8M0 scales along
// their K: d for W13, I for W2), gate/up accumulate dequantised products, h is
// rounded to bf16 (R2) and then quantised along I before the W2 GEMM.
//   w13q [E, 2I, d] codes, w13s [E, 2I, d/32];  w2q [E, d, I] codes, w2s [E, d, I/32]
int orc_forward_mxfp8(int T, int d, int I, int E, int k, float clamp,
                      const uint16_t* x, const int32_t* ids, const float* scores,
                      const uint8_t* w13q, const uint8_t* w13s,
                      const uint8_t* w2q, const uint8_t* w2s,
                      int ntok, const int32_t* toks, uint16_t* y, uint16_t* h_out) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, nullptr, nullptr);
#pragma omp parallel for schedule(dynamic)
  for (int n = 0; n < ntok; ++n) {
    std::vector<uint16_t> a(2 * I), h(I), ys((size_t)k * d);
    std::vector<char> ok(k);
    int t = toks ? toks[n] : n;
    for (int j = 0; j < k; ++j) {
      ok[j] = element_valid(p, t, j);
      if (!ok[j]) {
        if (h_out) std::memset(h_out + ((size_t)n * k + j) * I, 0, sizeof(uint16_t) * I);
        continue;
      }
      int e = ids[(size_t)t * k + j];
      float s = scores[(size_t)t * k + j];
      row_forward_mx(p, t, e, s, w13q, w13s, w2q, w2s, a.data(), h.data(),
                     ys.data() + (size_t)j * d);
      if (h_out) std::memcpy(h_out + ((size_t)n * k + j) * I, h.data(), sizeof(uint16_t) * I);
    }
    for (int c = 0; c < d; ++c) {
      real acc = 0;
      for (int j = 0; j < k; ++j)
        if (ok[j]) acc += bf(ys[(size_t)j * d + c]);
      y[(size_t)n * d + c] = real_to_bf16(acc);                 // R6
    }
  }
  return 0;
}

// MXFP8 backward for the listed tokens (training step of an MXFP8 plan; [DM]
// "What it is selling": MXFP8 E4M3 for FPROP/DGRAD/WGRAD with prepared weights).
// The forward quantities are those of orc_forward_mxfp8 (same prepared forward
// weights); the DGRAD GEMMs take dY quantised along d and dA along 2I, with
// weights prepared along the same K:
//   w2tq  [E, I, d]  codes of W2[e]^T,  w2ts  [E, I, d/32]
//   w13tq [E, d, 2I] codes of W13[e]^T, w13ts [E, d, 2I/32]
// Outputs as orc_backward: dx [ntok, d] (R6 of R5), dscores [ntok, k], optional
// dA [ntok, k, 2I] (R4), hs [ntok, k, I] (R7), dxe [ntok, k, d] (R5).
int orc_backward_mxfp8(int T, int d, int I, int E, int k, float clamp,
                       const uint16_t* x, const int32_t* ids, const float* scores,
                       const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q,
                       const uint8_t* w2s, const uint8_t* w13tq, const uint8_t* w13ts,
                       const uint8_t* w2tq, const uint8_t* w2ts, const uint16_t* dy,
                       int ntok, const int32_t* toks, uint16_t* dx, float* dscores,
                       uint16_t* dA_out, uint16_t* hs_out, uint16_t* dxe_out) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, nullptr, nullptr);
#pragma omp parallel for schedule(dynamic)
  for (int n = 0; n < ntok; ++n) {
    std::vector<uint16_t> a(2 * I), h(I), ys(d), dA(2 * I), hs(I), dxe((size_t)k * d, 0);
    std::vector<char> ok(k);
    int t = toks ? toks[n] : n;
    for (int j = 0; j < k; ++j) {
      ok[j] = element_valid(p, t, j);
      const size_t nj = (size_t)n * k + j;
      if (!ok[j]) {
        dscores[nj] = 0;
        if (dA_out) std::memset(dA_out + nj * 2 * I, 0, sizeof(uint16_t) * 2 * I);
        if (hs_out) std::memset(hs_out + nj * I, 0, sizeof(uint16_t) * I);
        continue;
      }
      int e = ids[(size_t)t * k + j];
      float s = scores[(size_t)t * k + j];
      row_forward_mx(p, t, e, s, w13q, w13s, w2q, w2s, a.data(), h.data(), ys.data());
      real ds;
      row_backward_mx(p, t, e, s, dy, a.data(), h.data(), w13tq, w13ts, w2tq, w2ts, &ds,
                      dA.data(), dxe.data() + (size_t)j * d, hs.data());
      dscores[nj] = static_cast<float>(ds);
      if (dA_out) std::memcpy(dA_out + nj * 2 * I, dA.data(), sizeof(uint16_t) * 2 * I);
      if (hs_out) std::memcpy(hs_out + nj * I, hs.data(), sizeof(uint16_t) * I);
    }
    for (int c = 0; c < d; ++c) {
      real acc = 0;
      for (int j = 0; j < k; ++j)
        if (ok[j]) acc += bf(dxe[(size_t)j * d + c]);
      dx[(size_t)n * d + c] = real_to_bf16(acc);                // R6
    }
    if (dxe_out)
      for (int j = 0; j < k; ++j)
        for (int c = 0; c < d; ++c)
          dxe_out[((size_t)n * k + j) * d + c] = ok[j] ? dxe[(size_t)j * d + c] : 0;
  }
  return 0;
}

// MXFP8 WGRAD of one expert e: the WGRAD GEMMs run over the rows of e (dispatch
// order), so their operands are block-quantised along that row dimension: blocks
// of 32 consecutive rows of e, starting at its first row (a shorter last block;
// the zero rows that pad the expert's segment do not change a block's scale).
//   dw2_delta  [d, I]  = sum_rows Q_rows(dY)[r, c] * Q_rows(hs)[r, i]
//   dw13_delta [2I, d] = sum_rows Q_rows(dA)[r, i] * Q_rows(x)[r, c]
// dA and hs come from the MXFP8 backward of each row.  Returns the row count.
int orc_wgrad_expert_mxfp8(int T, int d, int I, int E, int k, float clamp,
                           const uint16_t* x, const int32_t* ids, const float* scores,
                           const uint8_t* w13q, const uint8_t* w13s, const uint8_t* w2q,
                           const uint8_t* w2s, const uint8_t* w13tq, const uint8_t* w13ts,
                           const uint8_t* w2tq, const uint8_t* w2ts, const uint16_t* dy, int e,
                           float* dw13_delta, float* dw2_delta) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, nullptr, nullptr);
  std::vector<int> row_t, row_j;
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < k; ++j)
      if (ids[(size_t)t * k + j] == e && element_valid(p, t, j)) {
        row_t.push_back(t);
        row_j.push_back(j);
      }
  const int rows = static_cast<int>(row_t.size());
  std::vector<uint16_t> dA_rows((size_t)rows * 2 * I), hs_rows((size_t)rows * I);
#pragma omp parallel for schedule(dynamic)
  for (int r = 0; r < rows; ++r) {
    std::vector<uint16_t> a(2 * I), h(I), ys(d), dxe(d);
    const int t = row_t[r];
    const float s = scores[(size_t)t * k + row_j[r]];
    row_forward_mx(p, t, e, s, w13q, w13s, w2q, w2s, a.data(), h.data(), ys.data());
    real ds;
    row_backward_mx(p, t, e, s, dy, a.data(), h.data(), w13tq, w13ts, w2tq, w2ts, &ds,
                    dA_rows.data() + (size_t)r * 2 * I, dxe.data(),
                    hs_rows.data() + (size_t)r * I);
  }
  // dequantised operands, each column quantised along the rows
  auto along_rows = [&](int cols, auto value_of, std::vector<real>& out) {
    out.assign((size_t)rows * cols, 0);
#pragma omp parallel for schedule(static)
    for (int c = 0; c < cols; ++c) {
      std::vector<uint16_t> col(rows);
      std::vector<real> deq(rows);
      for (int r = 0; r < rows; ++r) col[r] = value_of(r, c);
      mx_roundtrip(col.data(), rows, deq.data());
      for (int r = 0; r < rows; ++r) out[(size_t)r * cols + c] = deq[r];
    }
  };
  std::vector<real> qdy, qhs, qdA, qx;
  along_rows(d, [&](int r, int c) { return dy[(size_t)row_t[r] * d + c]; }, qdy);
  along_rows(I, [&](int r, int c) { return hs_rows[(size_t)r * I + c]; }, qhs);
  along_rows(2 * I, [&](int r, int c) { return dA_rows[(size_t)r * 2 * I + c]; }, qdA);
  along_rows(d, [&](int r, int c) { return x[(size_t)row_t[r] * d + c]; }, qx);
#pragma omp parallel for schedule(static)
  for (int i = 0; i < 2 * I; ++i) {
    std::vector<real> acc(d, 0);
    for (int r = 0; r < rows; ++r) {
      const real ai = qdA[(size_t)r * 2 * I + i];
      for (int c = 0; c < d; ++c) acc[c] += ai * qx[(size_t)r * d + c];
    }
    for (int c = 0; c < d; ++c) dw13_delta[(size_t)i * d + c] = static_cast<float>(acc[c]);
  }
#pragma omp parallel for schedule(static)
  for (int c = 0; c < d; ++c) {
    std::vector<real> acc(I, 0);
    for (int r = 0; r < rows; ++r) {
      const real yc = qdy[(size_t)r * d + c];
      for (int i = 0; i < I; ++i) acc[i] += yc * qhs[(size_t)r * I + i];
    }
    for (int i = 0; i < I; ++i) dw2_delta[(size_t)c * I + i] = static_cast<float>(acc[i]);
  }
  return rows;
}

int orc_e2m1_encode(const double* in, uint8_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = e2m1_encode(in[i]);
  return 0;
}

int orc_e2m1_decode(const uint8_t* in, double* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = e2m1_value(in[i]);
  return 0;
}

// NVFP4 quantiser ([NV-D] quantize): a bf16 matrix [rows, K] along K in
// 16-element blocks with the encode scale g (1 / the per-tensor dequantisation
// scale).  codes [rows, K/2] packed E2M1 (element 2i in the low nibble of byte
// i); scales [rows, K/16] E4M3 bytes.  K must be a multiple of 16.
int orc_quant_nvfp4(long rows, int K, const uint16_t* in, float g, uint8_t* codes,
                    uint8_t* scales) {
  if (K % 16) return -1;
  uint8_t q[16];
  for (long r = 0; r < rows; ++r)
    for (int b = 0; b < K / 16; ++b) {
      nv_quant_block(in + r * K + b * 16, 16, g, q, scales + r * (K / 16) + b);
      for (int i = 0; i < 8; ++i)
        codes[r * (K / 2) + b * 8 + i] = static_cast<uint8_t>(q[2 * i] | (q[2 * i + 1] << 4));
    }
  return 0;
}

// Prepared NVFP4 weights ([DM]: weights are prepared ahead of the call): E matrices
// [rows, K] (bf16, consecutive), each with its own dequantisation scale
// scale[e] = amax(W[e]) / (6 * 448) (1 for an all-zero matrix), quantised along
// K with encode scale 1 / scale[e].
int orc_prepare_nvfp4(int E, long rows, int K, const uint16_t* in, uint8_t* codes,
                      uint8_t* scales, float* scale) {
  if (K % 16) return -1;
  for (int e = 0; e < E; ++e) {
    const uint16_t* w = in + (size_t)e * rows * K;
    float amax = 0;
    for (long i = 0; i < rows * K; ++i) {
      const float v = std::fabs(bf16_to_float(w[i]));
      if (v > amax) amax = v;
    }
    const float se = amax > 0 ? amax / 2688.0f : 1.0f;
    scale[e] = se;
    orc_quant_nvfp4(rows, K, w, 1.0f / se, codes + (size_t)e * rows * (K / 2),
                    scales + (size_t)e * rows * (K / 16));
  }
  return 0;
}

// NVFP4 inference forward for the listed tokens ([DM]: NVFP4 is inference-only;
// [NV-M]: static activation scales).  Prepared weights (orc_prepare_nvfp4):
//   w13q [E, 2I, d/2], w13s [E, 2I, d/16], w13_scale [E]
//   w2q  [E, d, I/2],  w2s  [E, d, I/16],  w2_scale  [E]
// x_scale, h_scale: the static dequantisation scales of x and h.
//   y [ntok, d] (R6), optional a [ntok, k, 2I] (R1), h [ntok, k, I] (R2)
int orc_forward_nvfp4(int T, int d, int I, int E, int k, float clamp,
                      const uint16_t* x, const int32_t* ids, const float* scores,
                      const uint8_t* w13q, const uint8_t* w13s, const float* w13_scale,
                      const uint8_t* w2q, const uint8_t* w2s, const float* w2_scale,
                      float x_scale, float h_scale, int ntok, const int32_t* toks, uint16_t* y,
                      uint16_t* a_out, uint16_t* h_out) {
  Problem p = make_problem(T, d, I, E, k, clamp, x, ids, scores, nullptr, nullptr);
  const NvScales sc{x_scale, h_scale, w13_scale, w2_scale};
#pragma omp parallel for schedule(dynamic)
  for (int n = 0; n < ntok; ++n) {
    std::vector<uint16_t> a(2 * I), h(I), ys((size_t)k * d);
    std::vector<char> ok(k);
    int t = toks ? toks[n] : n;
    for (int j = 0; j < k; ++j) {
      ok[j] = element_valid(p, t, j);
      const size_t nj = (size_t)n * k + j;
      if (!ok[j]) {
        if (a_out) std::memset(a_out + nj * 2 * I, 0, sizeof(uint16_t) * 2 * I);
        if (h_out) std::memset(h_out + nj * I, 0, sizeof(uint16_t) * I);
        continue;
      }
      int e = ids[(size_t)t * k + j];
      float s = scores[(size_t)t * k + j];
      row_forward_nv(p, t, e, s, w13q, w13s, w2q, w2s, sc, a.data(), h.data(),
                     ys.data() + (size_t)j * d);
      if (a_out) std::memcpy(a_out + nj * 2 * I, a.data(), sizeof(uint16_t) * 2 * I);
      if (h_out) std::memcpy(h_out + nj * I, h.data(), sizeof(uint16_t) * I);
    }
    for (int c = 0; c < d; ++c) {
      real acc = 0;
      for (int j = 0; j < k; ++j)
        if (ok[j]) acc += bf(ys[(size_t)j * d + c]);
      y[(size_t)n * d + c] = real_to_bf16(acc);                 // R6
    }
  }
  return 0;
}

}  // extern "C"
