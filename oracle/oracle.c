/*
 * CPU oracle for the MoE routing / permute / MXFP8 expert-FFN path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or table with the CUDA library.
 *
 * Every function is a plain, slow, literal reading of the operator pages:
 *
 *   MoeInitRoutingV3 (gitcode.com/cann/ops-transformer, moe/moe_init_routing_v3),
 *     "计算公式" steps 1-3 and 5   -> orc_route, orc_permute
 *   moe_token_permute article (sheratonhq.com/news/115526), sections
 *     功能说明 (argSort / inverse / gather) and 返回值说明 (output shapes,
 *     MXFP8 scale layout [M, AlignUp(CeilDiv(H,32),2)])  -> orc_route, orc_permute
 *   MegaMoE README (gitcode.com/azyuli/ops-transformer, mc2/mega_moe),
 *     "A8W8-FP quantization scenario" stages 1-4 and the swiglu formula in
 *     "Activation function formulas"  -> orc_mx_block, orc_expert_row,
 *     orc_mega_moe_tokens;  "A8W4-FP quantization scenario" (FLOAT4_E2M1
 *     weights with E8M0 scales, FP8 E4M3 activations) -> the same functions
 *     with the E2M1 element format;  "A4W4-FP quantization scenario" (tokens
 *     dispatched as MXFP4 E2M1, FLOAT4_E2M1 weights, the activation
 *     re-quantised to MXFP8 E4M3 for the A8W4 second layer) -> the same
 *     functions, with the activation format of orc_act_code
 *
 * Floating point is carried in double.  Readings of what the pages leave
 * open (shared-exponent rule, rounding, saturation, sign of zero, flatten
 * order, combine precision) are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_E5M2 23
#define ORC_E4M3 24
#define ORC_E2M1 296  /* FLOAT4_E2M1: one 4-bit code per byte here (bits 0-3) */

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Number formats.
 *
 * FLOAT8_E4M3FN: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448; smallest
 * normal 2^-6; subnormals m * 2^-9.
 * FLOAT8_E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits; exponent
 * field 31 holds inf / NaN; largest finite 1.75 * 2^15 = 57344; smallest
 * normal 2^-14; subnormals m * 2^-16.
 * FLOAT4_E2M1 (OCP MX v1.0 FP4): 1 sign, 2 exponent bits (bias 1), 1
 * mantissa bit, no infinities or NaN; values 0, 0.5 (subnormal), 1, 1.5, 2,
 * 3, 4, 6; largest finite 6 = 1.5 * 2^2; smallest normal 2^0.  The sign is
 * bit 3 of the code.
 * ------------------------------------------------------------------------- */
typedef struct {
  int nbits;    /* bits of a code (8, or 4 for E2M1) */
  int mbits;    /* explicit mantissa bits */
  int bias;
  int emin;     /* exponent of the smallest normal */
  int emax;     /* exponent of the largest finite value */
  double maxv;  /* largest finite value */
} orc_fmt;

static orc_fmt fmt_of(int code) {
  orc_fmt f;
  if (code == ORC_E5M2) {
    f.nbits = 8; f.mbits = 2; f.bias = 15; f.emin = -14; f.emax = 15; f.maxv = 57344.0;
  } else if (code == ORC_E2M1) {
    f.nbits = 4; f.mbits = 1; f.bias = 1; f.emin = 0; f.emax = 2; f.maxv = 6.0;
  } else {
    f.nbits = 8; f.mbits = 3; f.bias = 7; f.emin = -6; f.emax = 8; f.maxv = 448.0;
  }
  return f;
}

/* Value of an FP8 (or FP4 E2M1) code (NaN / inf as such). */
double orc_fp8_value(uint8_t c, int code) {
  orc_fmt f = fmt_of(code);
  int sign = (c >> (f.nbits - 1)) & 1;
  int ebits = (c >> f.mbits) & ((1 << (f.nbits - 1 - f.mbits)) - 1);
  int m = c & ((1 << f.mbits) - 1);
  int etop = (1 << (f.nbits - 1 - f.mbits)) - 1;
  double v;
  if (code == ORC_E4M3 && ebits == etop && m == (1 << f.mbits) - 1) return NAN;
  if (code == ORC_E5M2 && ebits == etop) return m == 0 ? (sign ? -INFINITY : INFINITY) : NAN;
  if (ebits == 0)
    v = ldexp((double)m, f.emin - f.mbits);
  else
    v = ldexp(1.0 + (double)m / (double)(1 << f.mbits), ebits - f.bias);
  return sign ? -v : v;
}

/* Round a non-negative finite double to the binary grid with `mbits`
 * mantissa bits and smallest normal exponent `emin` (nearest, ties to even;
 * no upper bound).  The quantum at magnitude a is 2^(max(floor(log2 a), emin) - mbits). */
static double round_to_grid(double a, int mbits, int emin) {
  int e;
  if (a == 0.0) return 0.0;
  frexp(a, &e);                         /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;                        /* floor(log2 a), exact */
  if (E < emin) E = emin;
  double q = ldexp(1.0, E - mbits);
  return nearbyint(a / q) * q;          /* a / q and r * q are exact; nearbyint is ties-to-even */
}

/* FP8 (or FP4 E2M1) code of a finite double: saturate the magnitude to the
 * largest finite value, round to nearest with ties to even, keep the sign
 * (also for zero). */
uint8_t orc_fp8_round(double t, int code) {
  orc_fmt f = fmt_of(code);
  uint8_t sign = signbit(t) ? (uint8_t)(1u << (f.nbits - 1)) : 0x00;
  double a = fabs(t);
  if (a > f.maxv) a = f.maxv;
  double v = round_to_grid(a, f.mbits, f.emin);
  if (v == 0.0) return sign;
  int e;
  frexp(v, &e);
  int E = e - 1;
  if (E < f.emin) /* subnormal: v = m * 2^(emin - mbits) */
    return sign | (uint8_t)(int)(v / ldexp(1.0, f.emin - f.mbits));
  int m = (int)(v / ldexp(1.0, E - f.mbits)) - (1 << f.mbits);
  return sign | (uint8_t)((E + f.bias) << f.mbits) | (uint8_t)m;
}

/* orc_fp8_round over an array. */
void orc_fp8_round_array(const double* t, int64_t n, int code, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_round(t[i], code);
}

/* bf16 bit pattern of a finite double, one rounding (nearest, ties to even). */
uint16_t orc_bf16_round(double t) {
  uint16_t sign = signbit(t) ? 0x8000 : 0x0000;
  double v = round_to_grid(fabs(t), 7, -126);
  if (v == 0.0) return sign;
  int e;
  frexp(v, &e);
  int E = e - 1;
  if (E > 127) return sign | 0x7F80; /* overflow to infinity */
  if (E < -126) return sign | (uint16_t)(int)(v / ldexp(1.0, -133));
  int m = (int)(v / ldexp(1.0, E - 7)) - 128;
  return sign | (uint16_t)((E + 127) << 7) | (uint16_t)m;
}

double orc_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

double orc_f16_value(uint16_t b) {
  int sign = b >> 15, ebits = (b >> 10) & 31, m = b & 1023;
  double v;
  if (ebits == 31) return m ? NAN : (sign ? -INFINITY : INFINITY);
  if (ebits == 0) v = ldexp((double)m, -24);
  else v = ldexp(1.0 + m / 1024.0, ebits - 15);
  return sign ? -v : v;
}

/* ---------------------------------------------------------------------------
 * MX group quantiser Q_MX (MegaMoE README, A8W8-FP stage 1: group of 32,
 * shared exponent, FP8 elements, FLOAT8_E8M0 scale).
 *
 * Reading of the shared-exponent rule (the pages only say "extract the
 * shared exponent"): the OCP MX v1.0 rule,
 *   s = floor(log2(amax)) - emax_elem,  clamped to [-127, 127],
 *   scale code = s + 127 (E8M0), amax = 0 gives s = -127 (code 0),
 *   element = FP8(v * 2^-s) with saturation to the largest finite value.
 * A partial last group (n not a multiple of 32) uses the elements present.
 * ------------------------------------------------------------------------- */
void orc_mx_block(const double* v, int64_t n, int code, uint8_t* q, uint8_t* scale_code) {
  orc_fmt f = fmt_of(code);
  double amax = 0.0;
  for (int64_t i = 0; i < n; ++i)
    if (fabs(v[i]) > amax) amax = fabs(v[i]);
  int s;
  if (amax == 0.0) {
    s = -127;
  } else {
    int e;
    frexp(amax, &e);
    s = (e - 1) - f.emax;
    if (s < -127) s = -127;
    if (s > 127) s = 127;
  }
  *scale_code = (uint8_t)(s + 127);
  for (int64_t i = 0; i < n; ++i) q[i] = orc_fp8_round(ldexp(v[i], -s), code);
}

/* Q_MX along each row of a [rows, cols] double matrix; scales go to a
 * [rows, s_cols] byte matrix (s_cols >= ceil(cols/32); extra columns are 0). */
void orc_mx_quantize_rows(const double* x, int64_t rows, int64_t cols, int code,
                          uint8_t* q, uint8_t* scales, int64_t s_cols) {
  int64_t groups = (cols + 31) / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t g = 0; g < s_cols; ++g) scales[r * s_cols + g] = 0;
    for (int64_t g = 0; g < groups; ++g) {
      int64_t c0 = g * 32, n = cols - c0 < 32 ? cols - c0 : 32;
      orc_mx_block(x + r * cols + c0, n, code, q + r * cols + c0, scales + r * s_cols + g);
    }
  }
}

/* Element of a source row as double: dtype 0 = fp32, 1 = fp16, 27 = bf16. */
static double src_value(const void* row, int64_t i, int dtype) {
  if (dtype == 0) return (double)((const float*)row)[i];
  if (dtype == 1) return orc_f16_value(((const uint16_t*)row)[i]);
  return orc_bf16_value(((const uint16_t*)row)[i]);
}

static int64_t dtype_size(int dtype) { return dtype == 0 ? 4 : 2; }

/* Q_MX of rows of a bf16 / fp16 / fp32 matrix (weights and tests). */
void orc_mx_quantize_src(const void* x, int dtype, int64_t rows, int64_t cols, int code,
                         uint8_t* q, uint8_t* scales, int64_t s_cols) {
  int64_t es = dtype_size(dtype), groups = (cols + 31) / 32;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double buf[32];
    const char* row = (const char*)x + r * cols * es;
    for (int64_t g = 0; g < s_cols; ++g) scales[r * s_cols + g] = 0;
    for (int64_t g = 0; g < groups; ++g) {
      int64_t c0 = g * 32, n = cols - c0 < 32 ? cols - c0 : 32;
      for (int64_t i = 0; i < n; ++i) buf[i] = src_value(row, c0 + i, dtype);
      orc_mx_block(buf, n, code, q + r * cols + c0, scales + r * s_cols + g);
    }
  }
}

/* ---------------------------------------------------------------------------
 * Routing (MoeInitRoutingV3 steps 1-3; moe_token_permute 功能说明).
 *
 * Flatten order: j = i*K + k (row-major reshape(-1) of [N, K], as in the
 * permute article's golden reference); the source token of j is j / K.
 * Step 1, keyValueSort(expertIdx, rowIdx): ascending expert id, and for
 * equal ids ascending j (a stable sort).  Sorting the (id, j) pairs by the
 * pair is that order; qsort is used for it.
 * Step 2: expandedRowIdx[sortedRowIdx[d]] = d.
 * Step 3: counts[e] = number of j with id_j == e.
 * Ids outside [0, E) are left out of the sort (they have no expert): their
 * expandedRowIdx is -1 and the tail of sortedRowIdx is -1.  Returns how
 * many there were.
 * ------------------------------------------------------------------------- */
typedef struct {
  int64_t key;
  int64_t j;
} orc_kv;

static int cmp_kv(const void* a, const void* b) {
  const orc_kv* x = (const orc_kv*)a;
  const orc_kv* y = (const orc_kv*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  return x->j < y->j ? -1 : (x->j > y->j ? 1 : 0);
}

/* With an active expert range [start, end) (MoeInitRoutingV3,
 * activeExpertRangeOptional; step 6: availableIdxNum counts the ids in
 * the range): only ids in the range are sorted, counts[e - start] for the
 * experts of the range; ids in [0, num_experts) but outside the range are
 * left out like the out-of-range ones but are not errors.  Returns the
 * number of ids outside [0, num_experts). */
int64_t orc_route_range(const void* ids, int ids_is_int64, int64_t n, int64_t k, int64_t num_experts,
                        int64_t start, int64_t end, int32_t* sorted_row_idx, int32_t* expanded_row_idx,
                        int64_t* counts) {
  int64_t rows = n * k, valid = 0, bad = 0;
  orc_kv* kv = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)(rows > 0 ? rows : 1));
  for (int64_t e = start; e < end; ++e) counts[e - start] = 0;
  for (int64_t j = 0; j < rows; ++j) {
    int64_t id = ids_is_int64 ? ((const int64_t*)ids)[j] : (int64_t)((const int32_t*)ids)[j];
    expanded_row_idx[j] = -1;
    if (id < 0 || id >= num_experts) {
      ++bad;
      continue;
    }
    if (id < start || id >= end) continue;
    kv[valid].key = id;
    kv[valid].j = j;
    ++valid;
    counts[id - start] += 1;
  }
  qsort(kv, (size_t)valid, sizeof(orc_kv), cmp_kv);
  for (int64_t d = 0; d < rows; ++d) sorted_row_idx[d] = -1;
  for (int64_t d = 0; d < valid; ++d) {
    sorted_row_idx[d] = (int32_t)kv[d].j;
    expanded_row_idx[kv[d].j] = (int32_t)d;
  }
  free(kv);
  return bad;
}

int64_t orc_route(const void* ids, int ids_is_int64, int64_t n, int64_t k, int64_t num_experts,
                  int32_t* sorted_row_idx, int32_t* expanded_row_idx, int64_t* counts) {
  return orc_route_range(ids, ids_is_int64, n, k, num_experts, 0, num_experts, sorted_row_idx, expanded_row_idx,
                         counts);
}

/* ---------------------------------------------------------------------------
 * Permute (MoeInitRoutingV3 step 5 with the row-major flatten; the permute
 * article's gather form): output row d takes token sortedRowIdx[d] / K,
 * copied (code < 0: element bytes as they are) or MX-quantised (code 23/24,
 * source bf16 / fp16 / fp32, scales [m_out, s_cols]).  Rows d < m_out only.
 * ------------------------------------------------------------------------- */
void orc_permute(const void* x, int dtype, int64_t h, int64_t k, const int32_t* sorted_row_idx,
                 int64_t m_out, int code, void* out, uint8_t* scales, int64_t s_cols) {
  int64_t es = dtype_size(dtype);
#pragma omp parallel for schedule(static)
  for (int64_t d = 0; d < m_out; ++d) {
    int32_t j = sorted_row_idx[d];
    if (j < 0) continue;
    const char* src = (const char*)x + (int64_t)(j / k) * h * es;
    if (code < 0) {
      memcpy((char*)out + d * h * es, src, (size_t)(h * es));
    } else {
      orc_mx_quantize_src(src, dtype, 1, h, code, (uint8_t*)out + d * h, scales + d * s_cols, s_cols);
    }
  }
}

/* DQ_MX of one row of codes: value(q[c]) * 2^(scale[c/32] - 127). */
static void dequant_row(const uint8_t* q, const uint8_t* s, int64_t n, int code, double* out) {
  for (int64_t c = 0; c < n; ++c) out[c] = ldexp(orc_fp8_value(q[c], code), (int)s[c / 32] - 127);
}

/* ---------------------------------------------------------------------------
 * Activation (MegaMoE README, "Activation function formulas").
 * sigma(z) = 1 / (1 + e^-z), SiLU(z) = z sigma(z); clamp c (+inf when not
 * enabled), G_c = min(G, c), U_c = clip(U, -c, c):
 *   0 swiglu      A = SiLU(G_c) U_c
 *   1 swiglustep  A = min(SiLU(G), c) U_c
 *   2 swigluoai   A = G_c sigma(alpha G_c) (U_c + beta)
 *   3 situglu     A = beta tanh(G / beta) sigma(G) L(U),
 *                 L(U) = U, or beta_lin tanh(U / beta_lin) when configured
 *   4 gelu        A = Z sigma(sqrt(8/pi) (Z + 0.044715 Z^3)), element-wise
 *                 on the whole Linear1 output Z (no gate / up split)
 * p = {c, alpha, beta, beta_lin} (beta_lin 0: not configured).
 * ------------------------------------------------------------------------- */
#define ORC_SWIGLU 0
#define ORC_SWIGLUSTEP 1
#define ORC_SWIGLUOAI 2
#define ORC_SITUGLU 3
#define ORC_GELU 4

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

static double act_gated(int kind, double g, double u, const double* p) {
  double c = p[0];
  double gc = g < c ? g : c;
  double uc = u < -c ? -c : (u > c ? c : u);
  switch (kind) {
    case ORC_SWIGLUSTEP: {
      double s = g * sigmoid(g);
      return (s < c ? s : c) * uc;
    }
    case ORC_SWIGLUOAI:
      return gc * sigmoid(p[1] * gc) * (uc + p[2]);
    case ORC_SITUGLU: {
      double l = p[3] > 0.0 ? p[3] * tanh(u / p[3]) : u;
      return p[2] * tanh(g / p[2]) * sigmoid(g) * l;
    }
    default:
      return gc * sigmoid(gc) * uc;
  }
}

static double act_gelu(double z) {
  return z * sigmoid(sqrt(8.0 / acos(-1.0)) * (z + 0.044715 * z * z * z));
}

/* Activation output width for a Linear1 output width of 2I. */
static int64_t act_width(int kind, int64_t inter) { return kind == ORC_GELU ? 2 * inter : inter; }

/* ---------------------------------------------------------------------------
 * One expanded row through one expert (MegaMoE A8W8-FP / A8W4-FP stages 2-3):
 *   h[n] = sum_c DQ(x)[c] * DQ(W1)[n][c]      n in [0, 2I)   (sequential double sum)
 *   gated: G = h[0:I] (gate), U = h[I:2I] (up), A[n] = Activation(G[n], U[n]);
 *   gelu:  A[n] = GELU(h[n]) for n in [0, 2I);  A rounded to fp32
 *   Ahat, S_A = Q_MX(A) in the format a_code     (width W = I, or 2I for gelu)
 *   o[c] = sum_n DQ(Ahat)[n] * DQ(W2)[c][n]   c in [0, H), W2 [H, W]
 * Weights are in the storage layout [N_out, K_red] with E8M0 scales
 * [N_out, w_s_cols] (the pages' (., N_out, CeilDiv(K_red, 64), 2) flattened).
 * ------------------------------------------------------------------------- */
void orc_expert_row(const uint8_t* xq, const uint8_t* xs, int x_code, const uint8_t* w1,
                    const uint8_t* s1, const uint8_t* w2, const uint8_t* s2, int w_code,
                    int64_t h, int64_t inter, int a_code, int act, const double* act_p, uint8_t* aq,
                    uint8_t* as, double* o) {
  int64_t aw = act_width(act, inter);
  int64_t s1_cols = 2 * ((h + 63) / 64), s2_cols = 2 * ((aw + 63) / 64);
  double* xd = (double*)malloc(sizeof(double) * (size_t)h);
  double* wd = (double*)malloc(sizeof(double) * (size_t)(h > aw ? h : aw));
  double* hv = (double*)malloc(sizeof(double) * (size_t)(2 * inter));
  double* a = (double*)malloc(sizeof(double) * (size_t)aw);
  double* ad = (double*)malloc(sizeof(double) * (size_t)aw);
  dequant_row(xq, xs, h, x_code, xd);
  for (int64_t n = 0; n < 2 * inter; ++n) {
    dequant_row(w1 + n * h, s1 + n * s1_cols, h, w_code, wd);
    double acc = 0.0;
    for (int64_t c = 0; c < h; ++c) acc += xd[c] * wd[c];
    hv[n] = acc;
  }
  if (act == ORC_GELU) {
    for (int64_t n = 0; n < aw; ++n) a[n] = (double)(float)act_gelu(hv[n]);
  } else {
    for (int64_t n = 0; n < inter; ++n) a[n] = (double)(float)act_gated(act, hv[n], hv[inter + n], act_p);
  }
  orc_mx_quantize_rows(a, 1, aw, a_code, aq, as, (aw + 31) / 32);
  dequant_row(aq, as, aw, a_code, ad);
  for (int64_t c = 0; c < h; ++c) {
    dequant_row(w2 + c * aw, s2 + c * s2_cols, aw, w_code, wd);
    double acc = 0.0;
    for (int64_t n = 0; n < aw; ++n) acc += ad[n] * wd[n];
    o[c] = acc;
  }
  free(xd); free(wd); free(hv); free(a); free(ad);
}

/* Format of A_hat for a dispatch format: the dispatch format itself in the
 * A8W8-FP and A8W4-FP scenarios (their stage 2 re-quantises the activation
 * into the dispatch type); MXFP8 E4M3 in the A4W4-FP scenario, whose stage 2
 * re-quantises the activation into MXFP8 E4M3 so that the second layer is
 * A8W4 (MegaMoE README, "A4W4-FP quantization scenario", stages 2-3). */
int orc_act_code(int x_code) { return x_code == ORC_E2M1 ? ORC_E4M3 : x_code; }

/* ---------------------------------------------------------------------------
 * MegaMoE at ep_world_size = 1, for a list of tokens (stage 4, combine):
 *   Y[i] = sum_k W[i,k] * O[pi(i,k)] + sum_s O_s^shared[i]
 * O[pi(i,k)] is the expert row of token i for expert ids[i,k]: the row of
 * X_hat at pi(i,k) is Q_MX(x_i) whatever its position, so each output row is
 * a function of its own token only.  The sum is in double over k = 0..K-1,
 * then the shared experts; Y is reported in double and rounded once to bf16.
 * Gating weights are fp32 (gate_is_bf16 = 0) or bf16 (1), widened exactly.
 * Optionally also returns the activation codes of every (token, k) pair:
 * aq_out [n_tok, K, I], as_out [n_tok, K, I/32] (format orc_act_code(x_code)).
 * Shared experts quantise their input in shared_x_code (the parameter
 * table's shared-expert quantisation type; < 0: the dispatch type), with
 * their activation in orc_act_code(shared_x_code).
 * combine_code 23 / 24 (combineQuantMode 3 / 4, the quantisation of the
 * combine communication between ranks): each routed expert row O, rounded
 * to bf16 as it leaves GMM2, is sent as Q_MX codes in that type and enters
 * the sum as DQ_MX of them; < 0: O as computed.  Shared-expert rows are
 * local to the card and are not quantised.
 * ------------------------------------------------------------------------- */
void orc_mega_moe_tokens(const uint16_t* x, const int32_t* ids, const void* gate, int gate_is_bf16,
                         const uint8_t* w1, const uint8_t* s1, const uint8_t* w2, const uint8_t* s2,
                         const uint8_t* sw1, const uint8_t* ss1, const uint8_t* sw2,
                         const uint8_t* ss2, int64_t n_shared, int64_t h, int64_t k,
                         int64_t num_experts, int64_t inter, int x_code, int w_code,
                         int shared_w_code, const int64_t* tokens, int64_t n_tok, double* y,
                         uint16_t* y_bf16, uint8_t* aq_out, uint8_t* as_out, const uint8_t* xq_in,
                         const uint8_t* xs_in, int act, const double* act_p, int shared_x_code,
                         int combine_code) {
  int64_t aw = act_width(act, inter);
  int64_t s1_cols = 2 * ((h + 63) / 64), s2_cols = 2 * ((aw + 63) / 64);
  int64_t w1_sz = 2 * inter * h, w2_sz = h * aw;
  int64_t i_groups = (aw + 31) / 32;
  int a_code = orc_act_code(x_code);
  int sx_code = shared_x_code < 0 ? x_code : shared_x_code;
  int sa_code = orc_act_code(sx_code);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < n_tok; ++t) {
    int64_t i = tokens[t];
    uint8_t* xq = (uint8_t*)malloc((size_t)h);
    uint8_t* xs = (uint8_t*)malloc((size_t)((h + 31) / 32));
    uint8_t* sxq = (uint8_t*)malloc((size_t)h);
    uint8_t* sxs = (uint8_t*)malloc((size_t)((h + 31) / 32));
    uint8_t* cq = (uint8_t*)malloc((size_t)h);
    uint8_t* cs = (uint8_t*)malloc((size_t)((h + 31) / 32));
    uint8_t* aq = (uint8_t*)malloc((size_t)aw);
    uint8_t* as = (uint8_t*)malloc((size_t)i_groups);
    double* o = (double*)malloc(sizeof(double) * (size_t)h);
    double* acc = y + t * h;
    for (int64_t c = 0; c < h; ++c) acc[c] = 0.0;
    if (xq_in) { /* pre-quantised pass-through: X_hat and S_X as given */
      memcpy(xq, xq_in + i * h, (size_t)h);
      memcpy(xs, xs_in + i * ((h + 31) / 32), (size_t)((h + 31) / 32));
    } else {
      orc_mx_quantize_src(x + i * h, 27, 1, h, x_code, xq, xs, (h + 31) / 32);
    }
    for (int64_t kk = 0; kk < k; ++kk) {
      int32_t e = ids[i * k + kk];
      if (e < 0 || e >= num_experts) continue;
      double w = gate_is_bf16 ? orc_bf16_value(((const uint16_t*)gate)[i * k + kk])
                              : (double)((const float*)gate)[i * k + kk];
      orc_expert_row(xq, xs, x_code, w1 + e * w1_sz, s1 + e * 2 * inter * s1_cols,
                     w2 + e * w2_sz, s2 + e * h * s2_cols, w_code, h, inter, a_code, act, act_p, aq, as, o);
      if (combine_code >= 0) {  /* the row on the wire: Q_MX of its bf16 value, then DQ_MX */
        for (int64_t c = 0; c < h; ++c) o[c] = orc_bf16_value(orc_bf16_round(o[c]));
        orc_mx_quantize_rows(o, 1, h, combine_code, cq, cs, (h + 31) / 32);
        dequant_row(cq, cs, h, combine_code, o);
      }
      if (aq_out) memcpy(aq_out + (t * k + kk) * aw, aq, (size_t)aw);
      if (as_out) memcpy(as_out + (t * k + kk) * i_groups, as, (size_t)i_groups);
      for (int64_t c = 0; c < h; ++c) acc[c] += w * o[c];
    }
    if (n_shared > 0) {
      if (sx_code == x_code) {
        memcpy(sxq, xq, (size_t)h);
        memcpy(sxs, xs, (size_t)((h + 31) / 32));
      } else {
        orc_mx_quantize_src(x + i * h, 27, 1, h, sx_code, sxq, sxs, (h + 31) / 32);
      }
    }
    for (int64_t s = 0; s < n_shared; ++s) {
      orc_expert_row(sxq, sxs, sx_code, sw1 + s * w1_sz, ss1 + s * 2 * inter * s1_cols,
                     sw2 + s * w2_sz, ss2 + s * h * s2_cols, shared_w_code, h, inter, sa_code, act, act_p,
                     aq, as, o);
      for (int64_t c = 0; c < h; ++c) acc[c] += o[c];
    }
    for (int64_t c = 0; c < h; ++c) y_bf16[t * h + c] = orc_bf16_round(acc[c]);
    free(xq); free(xs); free(sxq); free(sxs); free(cq); free(cs); free(aq); free(as); free(o);
  }
}
