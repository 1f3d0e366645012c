// Oracle for the sigmoid-routed top-k MoE FFN layer with a shared expert.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow CPU statement of what
// the layer computes. It exists so that the CUDA library can be checked
// against it. Only the tests, the smoke check and the bench's CPU-baseline leg
// load it. The CUDA library never calls it, and it shares no code, header or
// table with the CUDA library.
//
// Every floating-point step is done in double. Loops are written out plainly,
// with no blocking, fusion or reordering beyond what the definition states.
// OpenMP only splits the independent outer loop over rows/tokens.
//
// Sources. Page titles are abbreviated as:
//   [Hy3]  "腾讯混元 Hy3 在 CANN NPU 上的高性能推理部署与优化实战"
//   [Hy4]  "Hy4-preview（实验性）" (vLLM-Ascend tutorial)
//   [HyI3] "HunyuanImage-3.0 MoE 多流变体实战"
//   [OCP-MX] OCP Microscaling Formats (MX) Specification v1.0 (public spec).
//
// Readings where the pages are silent (listed with reasons in the design notes):
//   - top-k ranks the fp32 logits; equal logits -> lower expert id first;
//     slots are ordered by descending logit.
//   - route_norm: w_k = sigma_k / sum_{j in topK} sigma_j, no epsilon.
//   - router_scaling_factor multiplies the routed weights after route_norm.
//   - expert FFN is SwiGLU: y = W_down (silu(W_gate x) * (W_up x)), no biases.
//   - the shared expert's output is added unweighted.
//   - dropless: every (token, slot) pair is computed; no capacity limit.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// ---------------------------------------------------------------------------
// Scalar helpers.
// ---------------------------------------------------------------------------

// bf16 is the upper 16 bits of an IEEE binary32; widening is exact.
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return (double)f;
}

// Logistic sigmoid, sigma(l) = 1 / (1 + exp(-l)), in double.
// [Hy3] section 一 (模型概览): "top-8 sigmoid routing", moe_router_use_sigmoid=True.
static double sigmoid(double l) { return 1.0 / (1.0 + std::exp(-l)); }

// silu(z) = z * sigma(z), the gate activation of the SwiGLU expert FFN.
static double silu(double z) { return z * sigmoid(z); }

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

// ---------------------------------------------------------------------------
// Gating: the router projection that produces the logits routing ranks.
// [Hy3] section 8.5: the main stream runs Gating first, then the routed path.
// logits[t, e] = sum_c x[t, c] * w_router[e, c], in double.
// x: [T, H] bf16; w_router: [E, H] bf16; logits: [T, E] double out.
// ---------------------------------------------------------------------------
int oracle_gate(int T, int H, int E, const uint16_t* x, const uint16_t* w_router, double* logits) {
  if (T < 0 || H <= 0 || E <= 0) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int c = 0; c < H; ++c)
        acc += bf16_to_double(x[(size_t)t * H + c]) * bf16_to_double(w_router[(size_t)e * H + c]);
      logits[(size_t)t * E + e] = acc;
    }
  return 0;
}

// ---------------------------------------------------------------------------
// Step 1: sigmoid top-k routing with route_norm and router_scaling_factor.
// [Hy3] section 一: 192 routed experts, top-8 sigmoid routing; HYV3Config
// defaults router_scaling_factor=2.826, num_experts_per_tok=8, route_norm=True,
// moe_router_use_sigmoid=True.
//
// For each token t: order all E experts by (logit descending, id ascending),
// keep the first K as topk_idx[t, 0..K-1] in that order. Each kept expert gets
// sigma(logit). With route_norm the K values are divided by their sum. Then
// every weight is multiplied by `scaling`.
//
// logits:   [T, E] fp32, row-major.
// topk_idx: [T, K] int32 out.   topk_w: [T, K] double out.
// Returns 0, or -1 on bad sizes.
// ---------------------------------------------------------------------------
int oracle_route(int T, int E, int K, const float* logits, double scaling,
                 int route_norm, int32_t* topk_idx, double* topk_w) {
  if (T < 0 || E <= 0 || K <= 0 || K > E) return -1;
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    std::vector<int> order(E);
    std::iota(order.begin(), order.end(), 0);
    const float* row = logits + (size_t)t * E;
    std::sort(order.begin(), order.end(), [row](int a, int b) {
      if (row[a] != row[b]) return row[a] > row[b];  // +0 and -0 compare equal
      return a < b;                                   // tie -> lower id first
    });
    double sum = 0.0;
    for (int k = 0; k < K; ++k) sum += sigmoid((double)row[order[k]]);
    for (int k = 0; k < K; ++k) {
      double s = sigmoid((double)row[order[k]]);
      double w = route_norm ? s / sum : s;
      topk_idx[(size_t)t * K + k] = order[k];
      topk_w[(size_t)t * K + k] = w * scaling;
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Step 2: token permutation into expert-contiguous order (the InitRouting step
// of the routed path: [Hy3] section 8.5 "AllGather -> InitRouting -> 分组 GMM
// -> FinalizeRouting"; [Hy3] section 8.1 "通过 InitRouting 完成 token 与专家的
// 路由匹配").
//
// The T*K (token, slot) pairs are numbered by flat index f = t*K + k. They are
// stably sorted by expert id: permuted row r holds flat index perm_src[r];
// rows of expert e are offsets[e] .. offsets[e+1]-1, ascending in f.
// flat_to_perm is the inverse permutation. counts[e] = offsets[e+1]-offsets[e].
// ---------------------------------------------------------------------------
int oracle_permute(int T, int K, int E, const int32_t* topk_idx, int32_t* counts,
                   int32_t* offsets, int32_t* perm_src, int32_t* flat_to_perm) {
  if (T < 0 || K <= 0 || E <= 0) return -1;
  const int TK = T * K;
  for (int f = 0; f < TK; ++f)
    if (topk_idx[f] < 0 || topk_idx[f] >= E) return -1;
  std::vector<int> order(TK);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [topk_idx](int a, int b) { return topk_idx[a] < topk_idx[b]; });
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int f = 0; f < TK; ++f) counts[topk_idx[f]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int r = 0; r < TK; ++r) {
    perm_src[r] = order[r];
    flat_to_perm[order[r]] = r;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Step 3 (one row): the SwiGLU expert FFN applied to one input vector.
//   g = W_gate x, u = W_up x, h = silu(g) * u, y = W_down h.
// [Hy3] section 一: expert FFN intermediate size 1536; the gate/up/down SwiGLU
// form is the reading adopted for the unspecified FFN form.
//
// x: [H] double.  w_gate, w_up: [I, H] bf16 (row i is the i-th output).
// w_down: [H, I] bf16.  y: [H] double out.  h_scratch: [I] double.
// ---------------------------------------------------------------------------
static void swiglu_row(int H, int I, const double* x, const uint16_t* w_gate,
                       const uint16_t* w_up, const uint16_t* w_down,
                       double* h_scratch, double* y) {
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    const uint16_t* wg = w_gate + (size_t)i * H;
    const uint16_t* wu = w_up + (size_t)i * H;
    for (int c = 0; c < H; ++c) {
      g += bf16_to_double(wg[c]) * x[c];
      u += bf16_to_double(wu[c]) * x[c];
    }
    h_scratch[i] = silu(g) * u;
  }
  for (int m = 0; m < H; ++m) {
    double acc = 0.0;
    const uint16_t* wd = w_down + (size_t)m * I;
    for (int i = 0; i < I; ++i) acc += bf16_to_double(wd[i]) * h_scratch[i];
    y[m] = acc;
  }
}

// Dense SwiGLU MLP over rows: y[r] = W_down (silu(W_gate x_r) * W_up x_r).
// x: [R, H] bf16; y: [R, H] double. This is the shared expert of [Hy3]
// section 8.5 / [HyI3] 源码级实现拆解 §1 (shared_mlp = HunyuanMLP(...)).
int oracle_swiglu_mlp(int R, int H, int I, const uint16_t* x, const uint16_t* w_gate,
                      const uint16_t* w_up, const uint16_t* w_down, double* y) {
  if (R < 0 || H <= 0 || I <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < R; ++r) {
    std::vector<double> xv(H), h(I);
    for (int c = 0; c < H; ++c) xv[c] = bf16_to_double(x[(size_t)r * H + c]);
    swiglu_row(H, I, xv.data(), w_gate, w_up, w_down, h.data(), y + (size_t)r * H);
  }
  return 0;
}

// ---------------------------------------------------------------------------
// The whole layer for a subset of tokens, in the pages' order:
//   gating result (logits, given) -> routing (step 1) -> InitRouting (step 2)
//   -> per-expert FFN over each permuted row (step 3) -> FinalizeRouting:
//   out_t = sum_k w[t,k] * y[flat_to_perm[t*K+k]]  (k ascending)
//   -> add the shared expert: out_t += shared(x_t).
// [Hy3] section 8.5 (main stream: Gating, routed path, final combine add;
// shared expert independent of gating). [HyI3] 源码级实现拆解 §3: the output
// is hidden_states_mlp + combined_output.
//
// tokens: n_sel token ids (any order, may repeat). out: [n_sel, H] double.
// topk_idx_out [n_sel, K], topk_w_out [n_sel, K]: the routing of those tokens
// (may be NULL). shared weights may be NULL (no shared expert) if I_shared==0.
// ---------------------------------------------------------------------------
int oracle_layer_forward(int T, int H, int E, int K, int I, int I_shared,
                         double scaling, int route_norm, const uint16_t* x,
                         const float* logits, const uint16_t* w_gate,
                         const uint16_t* w_up, const uint16_t* w_down,
                         const uint16_t* ws_gate, const uint16_t* ws_up,
                         const uint16_t* ws_down, int n_sel, const int32_t* tokens,
                         double* out, int32_t* topk_idx_out, double* topk_w_out) {
  if (T <= 0 || H <= 0 || E <= 0 || K <= 0 || K > E || I <= 0 || I_shared < 0 || n_sel < 0)
    return -1;
  for (int j = 0; j < n_sel; ++j)
    if (tokens[j] < 0 || tokens[j] >= T) return -1;

  // Step 1 on the selected tokens' logit rows.
  std::vector<float> sel_logits((size_t)n_sel * E);
  for (int j = 0; j < n_sel; ++j)
    std::memcpy(&sel_logits[(size_t)j * E], logits + (size_t)tokens[j] * E, sizeof(float) * E);
  std::vector<int32_t> idx((size_t)n_sel * K);
  std::vector<double> w((size_t)n_sel * K);
  if (oracle_route(n_sel, E, K, sel_logits.data(), scaling, route_norm, idx.data(), w.data()))
    return -1;

  // Step 2: expert-contiguous order of the selected (token, slot) pairs.
  std::vector<int32_t> counts(E), offsets(E + 1), perm_src((size_t)n_sel * K),
      flat_to_perm((size_t)n_sel * K);
  if (oracle_permute(n_sel, K, E, idx.data(), counts.data(), offsets.data(),
                     perm_src.data(), flat_to_perm.data()))
    return -1;

  // Step 3: each permuted row through its expert's SwiGLU FFN.
  const int RK = n_sel * K;
  std::vector<double> y_perm((size_t)RK * H);
  std::vector<int> row_expert(RK);
  for (int e = 0; e < E; ++e)
    for (int r = offsets[e]; r < offsets[e + 1]; ++r) row_expert[r] = e;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < RK; ++r) {
    const int e = row_expert[r];
    const int t = tokens[perm_src[r] / K];
    std::vector<double> xv(H), h(I);
    for (int c = 0; c < H; ++c) xv[c] = bf16_to_double(x[(size_t)t * H + c]);
    swiglu_row(H, I, xv.data(), w_gate + (size_t)e * I * H, w_up + (size_t)e * I * H,
               w_down + (size_t)e * H * I, h.data(), &y_perm[(size_t)r * H]);
  }

  // Shared expert on every selected token.
  std::vector<double> s((size_t)n_sel * H, 0.0);
  if (I_shared > 0) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n_sel; ++j) {
      std::vector<double> xv(H), h(I_shared);
      for (int c = 0; c < H; ++c) xv[c] = bf16_to_double(x[(size_t)tokens[j] * H + c]);
      swiglu_row(H, I_shared, xv.data(), ws_gate, ws_up, ws_down, h.data(),
                 &s[(size_t)j * H]);
    }
  }

  // FinalizeRouting (weighted un-permute, k ascending) then the shared add.
  for (int j = 0; j < n_sel; ++j) {
    for (int m = 0; m < H; ++m) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k) {
        const int r = flat_to_perm[(size_t)j * K + k];
        acc += w[(size_t)j * K + k] * y_perm[(size_t)r * H + m];
      }
      out[(size_t)j * H + m] = acc + s[(size_t)j * H + m];
    }
  }
  if (topk_idx_out) std::memcpy(topk_idx_out, idx.data(), sizeof(int32_t) * idx.size());
  if (topk_w_out) std::memcpy(topk_w_out, w.data(), sizeof(double) * w.size());
  return 0;
}

// ---------------------------------------------------------------------------
// MXFP8 (E4M3 elements, one E8M0 scale per 32 consecutive elements).
// [Hy3] section 8.2: W8A8 with W8 and A8 both MXFP8; section 六 mentions
// torch_npu.npu_dynamic_mx_quant producing dynamic MXFP8 values.
// The rule is [OCP-MX]'s conversion of higher-precision values to MX:
//   shared_exp = floor(log2(max_i |v_i|)) - emax_elem, emax_elem = 8 for E4M3;
//   X = 2^shared_exp stored as E8M0 (biased by 127, clamped to [-127, 127]);
//   P_i = v_i / X rounded to nearest-even E4M3, saturating to +-448.
// A block whose amax is 0 gets scale code 0 and all elements +0.
// ---------------------------------------------------------------------------

// Value of an E4M3 (fn variant: no infinities, 0x7F/0xFF are NaN) code, from
// the format definition: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
double oracle_e4m3_value(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
  double mag;
  if (e == 0xF && m == 7) return NAN;
  if (e == 0) mag = std::ldexp((double)m / 8.0, -6);         // subnormal
  else mag = std::ldexp(1.0 + (double)m / 8.0, e - 7);       // normal
  return s ? -mag : mag;
}

// Round |v| (already divided by the scale) to the nearest E4M3 magnitude code
// 0x00..0x7E, ties to the code with even mantissa; values past 448 saturate.
static uint8_t e4m3_round_magnitude(double a) {
  // Codes 0x00..0x7E have increasing values; find the neighbours by bisection.
  int lo = 0, hi = 0x7E;
  if (a >= oracle_e4m3_value(0x7E)) return 0x7E;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (oracle_e4m3_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  const double vlo = oracle_e4m3_value((uint8_t)lo), vhi = oracle_e4m3_value((uint8_t)hi);
  const double dlo = a - vlo, dhi = vhi - a;
  if (dlo < dhi) return (uint8_t)lo;
  if (dhi < dlo) return (uint8_t)hi;
  return (lo & 1) ? (uint8_t)hi : (uint8_t)lo;  // tie -> even mantissa LSB
}

// Sign-magnitude encoding: the sign bit follows the input's sign, also when
// the magnitude rounds to zero (IEEE-style rounding keeps the sign of zero).
uint8_t oracle_e4m3_encode(double v) {
  const uint8_t mag = e4m3_round_magnitude(std::fabs(v));
  return std::signbit(v) ? (uint8_t)(mag | 0x80) : mag;
}

// Quantise one block of n values (n <= 32) in place of the MX rule above.
static void mx_block(const double* v, int n, uint8_t* q, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
  if (amax == 0.0) {
    *scale = 0;
    for (int i = 0; i < n; ++i) q[i] = 0;
    return;
  }
  int ex;
  std::frexp(amax, &ex);             // amax = f * 2^ex, f in [0.5, 1)
  int shared_exp = (ex - 1) - 8;     // floor(log2(amax)) - emax_elem(E4M3)
  if (shared_exp < -127) shared_exp = -127;
  if (shared_exp > 127) shared_exp = 127;
  *scale = (uint8_t)(shared_exp + 127);
  const double X = std::ldexp(1.0, shared_exp);
  for (int i = 0; i < n; ++i) q[i] = oracle_e4m3_encode(v[i] / X);
}

// Quantise a [rows, cols] bf16 matrix along cols in blocks of 32.
// q: [rows, cols] E4M3 codes. scale: [rows, cols/32] E8M0 codes.
int oracle_mx_quantize_bf16(int rows, int cols, const uint16_t* in, uint8_t* q,
                            uint8_t* scale) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    double v[32];
    for (int b = 0; b < cols / 32; ++b) {
      for (int i = 0; i < 32; ++i) v[i] = bf16_to_double(in[(size_t)r * cols + b * 32 + i]);
      mx_block(v, 32, q + (size_t)r * cols + b * 32, scale + (size_t)r * (cols / 32) + b);
    }
  }
  return 0;
}

// Same rule on double input (used for the intermediate activation h).
int oracle_mx_quantize_f64(int rows, int cols, const double* in, uint8_t* q,
                           uint8_t* scale) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r)
    for (int b = 0; b < cols / 32; ++b)
      mx_block(in + (size_t)r * cols + b * 32, 32, q + (size_t)r * cols + b * 32,
               scale + (size_t)r * (cols / 32) + b);
  return 0;
}

// Dequantise: value = 2^(scale-127) * e4m3_value(q).
int oracle_mx_dequantize(int rows, int cols, const uint8_t* q, const uint8_t* scale,
                         double* out) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c) {
      const double X = std::ldexp(1.0, (int)scale[(size_t)r * (cols / 32) + c / 32] - 127);
      out[(size_t)r * cols + c] = X * oracle_e4m3_value(q[(size_t)r * cols + c]);
    }
  return 0;
}

// ---------------------------------------------------------------------------
// MXFP4 (E2M1 elements, one E8M0 scale per 32): the routed-expert weights of
// the W4A8 recipe ([Hy3] section 8.2: MXFP4 routed experts with MXFP8
// activations; the shared expert stays W8A8). Same [OCP-MX] conversion rule
// with emax_elem = 2 for E2M1:
//   shared_exp = floor(log2(amax)) - 2; X = 2^shared_exp (E8M0);
//   P_i = v_i / X rounded to nearest-even E2M1, saturating to +-6.
// Two codes per byte: element 2j in the low nibble, 2j+1 in the high nibble.
// ---------------------------------------------------------------------------

// Value of an E2M1 code (low 4 bits) from the format definition: 1 sign bit,
// 2 exponent bits (bias 1), 1 mantissa bit; no infinities or NaN.
double oracle_e2m1_value(uint8_t code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? 0.5 * m : std::ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

// Nearest E2M1 magnitude code 0..7 to a >= 0, ties to the even mantissa;
// values past 6 saturate.
static uint8_t e2m1_round_magnitude(double a) {
  if (a >= oracle_e2m1_value(7)) return 7;
  int lo = 0, hi = 7;
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (oracle_e2m1_value((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  const double dlo = a - oracle_e2m1_value((uint8_t)lo), dhi = oracle_e2m1_value((uint8_t)hi) - a;
  if (dlo < dhi) return (uint8_t)lo;
  if (dhi < dlo) return (uint8_t)hi;
  return (lo & 1) ? (uint8_t)hi : (uint8_t)lo;
}

// Sign-magnitude E2M1 code; a magnitude that rounds to zero keeps the sign.
uint8_t oracle_e2m1_encode(double v) {
  const uint8_t mag = e2m1_round_magnitude(std::fabs(v));
  return std::signbit(v) ? (uint8_t)(mag | 8) : mag;
}

// One block of n values (n <= 32, even) -> n/2 packed bytes + one scale.
static void mxfp4_block(const double* v, int n, uint8_t* q, uint8_t* scale) {
  double amax = 0.0;
  for (int i = 0; i < n; ++i) amax = std::max(amax, std::fabs(v[i]));
  for (int i = 0; i < n / 2; ++i) q[i] = 0;
  if (amax == 0.0) {
    *scale = 0;
    return;
  }
  int ex;
  std::frexp(amax, &ex);           // amax = f * 2^ex, f in [0.5, 1)
  int shared_exp = (ex - 1) - 2;   // floor(log2(amax)) - emax_elem(E2M1)
  if (shared_exp < -127) shared_exp = -127;
  if (shared_exp > 127) shared_exp = 127;
  *scale = (uint8_t)(shared_exp + 127);
  const double X = std::ldexp(1.0, shared_exp);
  for (int i = 0; i < n; ++i) q[i / 2] |= (uint8_t)(oracle_e2m1_encode(v[i] / X) << (4 * (i & 1)));
}

// Quantise a [rows, cols] bf16 matrix along cols: q [rows, cols/2] packed
// E2M1 codes, scale [rows, cols/32] E8M0 codes.
int oracle_mxfp4_quantize_bf16(int rows, int cols, const uint16_t* in, uint8_t* q,
                               uint8_t* scale) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    double v[32];
    for (int b = 0; b < cols / 32; ++b) {
      for (int i = 0; i < 32; ++i) v[i] = bf16_to_double(in[(size_t)r * cols + b * 32 + i]);
      mxfp4_block(v, 32, q + (size_t)r * (cols / 2) + b * 16, scale + (size_t)r * (cols / 32) + b);
    }
  }
  return 0;
}

// Dequantise: value = 2^(scale-127) * e2m1_value(code).
int oracle_mxfp4_dequantize(int rows, int cols, const uint8_t* q, const uint8_t* scale,
                            double* out) {
  if (rows < 0 || cols <= 0 || cols % 32) return -1;
  for (int r = 0; r < rows; ++r)
    for (int c = 0; c < cols; ++c) {
      const double X = std::ldexp(1.0, (int)scale[(size_t)r * (cols / 32) + c / 32] - 127);
      const uint8_t byte = q[(size_t)r * (cols / 2) + c / 2];
      out[(size_t)r * cols + c] = X * oracle_e2m1_value((c & 1) ? byte >> 4 : byte & 15);
    }
  return 0;
}

// One expert SwiGLU FFN row on MX operands: x is already dequantised (double);
// weights are MX codes + scales; h is MX-quantised (dynamic, per 32 along I)
// before the down projection, as the MXFP8 activation path quantises every
// Linear input ([Hy3] section 8.2: routed and shared Linears in W8A8 MXFP8).
// Weight format wfmt: 0 = E4M3 codes (one per byte), 1 = E2M1 codes (two per
// byte, [rows, cols/2]).
static double mx_weight(int wfmt, const uint8_t* q, const uint8_t* s, int cols, size_t r, int c) {
  const double X = std::ldexp(1.0, (int)s[r * (cols / 32) + c / 32] - 127);
  if (wfmt == 0) return X * oracle_e4m3_value(q[r * cols + c]);
  const uint8_t byte = q[r * (cols / 2) + c / 2];
  return X * oracle_e2m1_value((c & 1) ? byte >> 4 : byte & 15);
}

static void swiglu_row_mx(int wfmt, int H, int I, const double* x, const uint8_t* qg,
                          const uint8_t* sg, const uint8_t* qu, const uint8_t* su,
                          const uint8_t* qd, const uint8_t* sd, double* y) {
  std::vector<double> h(I), hd(I);
  std::vector<uint8_t> hq(I), hs(I / 32);
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int c = 0; c < H; ++c) {
      g += mx_weight(wfmt, qg, sg, H, i, c) * x[c];
      u += mx_weight(wfmt, qu, su, H, i, c) * x[c];
    }
    h[i] = silu(g) * u;
  }
  oracle_mx_quantize_f64(1, I, h.data(), hq.data(), hs.data());
  oracle_mx_dequantize(1, I, hq.data(), hs.data(), hd.data());
  for (int m = 0; m < H; ++m) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += mx_weight(wfmt, qd, sd, I, m, i) * hd[i];
    y[m] = acc;
  }
}

// Dense SwiGLU MLP over rows whose activations are already MX-quantised
// (xq codes [R, H], xs scales [R, H/32]) with MX weights (format wfmt, as in
// mx_weight): dequantise x, then the same row function as the MX layer (h
// re-quantised to MXFP8 per 32 along I). [Hy3] section 8.2.
int oracle_swiglu_mlp_mx(int wfmt, int R, int H, int I, const uint8_t* xq, const uint8_t* xs,
                         const uint8_t* qg, const uint8_t* sg, const uint8_t* qu,
                         const uint8_t* su, const uint8_t* qd, const uint8_t* sd, double* y) {
  if (R < 0 || H <= 0 || H % 32 || I <= 0 || I % 32 || wfmt < 0 || wfmt > 1) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < R; ++r) {
    std::vector<double> xd(H);
    oracle_mx_dequantize(1, H, xq + (size_t)r * H, xs + (size_t)r * (H / 32), xd.data());
    swiglu_row_mx(wfmt, H, I, xd.data(), qg, sg, qu, su, qd, sd, y + (size_t)r * H);
  }
  return 0;
}

// The whole layer in MX mode for a subset of tokens. x is given as bf16 and
// is MX-quantised here (dynamic activation quantisation); weights are given as
// MX codes/scales (produced by oracle_mx_quantize_bf16 from the bf16 weights,
// or for W4A8's routed experts (wfmt 1) by oracle_mxfp4_quantize_bf16; the
// shared expert is always E4M3). Routing, permutation, finalize and the shared
// add are as in oracle_layer_forward.
int oracle_layer_forward_mx(int wfmt, int T, int H, int E, int K, int I, int I_shared,
                            double scaling, int route_norm, const uint16_t* x,
                            const float* logits, const uint8_t* qg, const uint8_t* sg,
                            const uint8_t* qu, const uint8_t* su, const uint8_t* qd,
                            const uint8_t* sd, const uint8_t* qsg, const uint8_t* ssg,
                            const uint8_t* qsu, const uint8_t* ssu, const uint8_t* qsd,
                            const uint8_t* ssd, int n_sel, const int32_t* tokens,
                            double* out) {
  if (T <= 0 || H <= 0 || H % 32 || E <= 0 || K <= 0 || K > E || I <= 0 || I % 32 ||
      I_shared < 0 || I_shared % 32 || n_sel < 0 || wfmt < 0 || wfmt > 1)
    return -1;
  for (int j = 0; j < n_sel; ++j)
    if (tokens[j] < 0 || tokens[j] >= T) return -1;

  std::vector<float> sel_logits((size_t)n_sel * E);
  for (int j = 0; j < n_sel; ++j)
    std::memcpy(&sel_logits[(size_t)j * E], logits + (size_t)tokens[j] * E, sizeof(float) * E);
  std::vector<int32_t> idx((size_t)n_sel * K);
  std::vector<double> w((size_t)n_sel * K);
  oracle_route(n_sel, E, K, sel_logits.data(), scaling, route_norm, idx.data(), w.data());
  std::vector<int32_t> counts(E), offsets(E + 1), perm_src((size_t)n_sel * K),
      flat_to_perm((size_t)n_sel * K);
  oracle_permute(n_sel, K, E, idx.data(), counts.data(), offsets.data(), perm_src.data(),
                 flat_to_perm.data());

  // Dynamic MX quantisation of the selected tokens' x rows, then dequantise.
  std::vector<uint16_t> xs((size_t)n_sel * H);
  for (int j = 0; j < n_sel; ++j)
    std::memcpy(&xs[(size_t)j * H], x + (size_t)tokens[j] * H, sizeof(uint16_t) * H);
  std::vector<uint8_t> xq((size_t)n_sel * H), xsc((size_t)n_sel * (H / 32));
  std::vector<double> xd((size_t)n_sel * H);
  oracle_mx_quantize_bf16(n_sel, H, xs.data(), xq.data(), xsc.data());
  oracle_mx_dequantize(n_sel, H, xq.data(), xsc.data(), xd.data());

  const int RK = n_sel * K;
  std::vector<double> y_perm((size_t)RK * H);
  std::vector<int> row_expert(RK);
  for (int e = 0; e < E; ++e)
    for (int r = offsets[e]; r < offsets[e + 1]; ++r) row_expert[r] = e;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < RK; ++r) {
    const int e = row_expert[r];
    const int j = perm_src[r] / K;
    const size_t eIH = (size_t)e * I * H, eq = wfmt ? eIH / 2 : eIH;  // code bytes per expert
    swiglu_row_mx(wfmt, H, I, &xd[(size_t)j * H], qg + eq, sg + eIH / 32, qu + eq, su + eIH / 32,
                  qd + eq, sd + eIH / 32, &y_perm[(size_t)r * H]);
  }
  std::vector<double> s((size_t)n_sel * H, 0.0);
  if (I_shared > 0) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int j = 0; j < n_sel; ++j)
      swiglu_row_mx(0, H, I_shared, &xd[(size_t)j * H], qsg, ssg, qsu, ssu, qsd, ssd,
                    &s[(size_t)j * H]);
  }
  for (int j = 0; j < n_sel; ++j)
    for (int m = 0; m < H; ++m) {
      double acc = 0.0;
      for (int k = 0; k < K; ++k)
        acc += w[(size_t)j * K + k] * y_perm[(size_t)flat_to_perm[(size_t)j * K + k] * H + m];
      out[(size_t)j * H + m] = acc + s[(size_t)j * H + m];
    }
  return 0;
}

}  // extern "C"
