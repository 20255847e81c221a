/*
 * Plain, slow, single-threaded CPU oracle for the routing-and-combine path of a
 * decode-step latent-MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library. The product path (the CUDA library under
 * latent_moe_decode_gb300/) never calls, links or includes anything here, and
 * nothing here includes or calls the product path.
 *
 * Built with -O2 -ffp-contract=off: every multiply-add below is either a separate
 * FP32 multiply and add or an explicit fmaf(), exactly as written.
 *
 * The pages this follows (all from the vLLM API docs of the Kimi-K3 / GLM-5-next
 * "specialized_decode" CuTe-DSL kernels):
 *   [wide]   vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.wide
 *            - "Finalize" class and kernel; "WideRoute" class docstring and kernel;
 *              "WideScratch" buffers; module docstring (precision paragraph).
 *   [ep]     vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.moe.ep.layer
 *            - "EpMoeLayer.topk" (stock sigmoid top-16), "EpMoeLayer.stock_order"
 *              (FP32-out router GEMM), module docstring.
 *   [fin]    vllm.models.glm5next.nvidia.specialized_decode.cutedsl.finalize_publish
 *            - "_QuadFinalizePublishDeviceKernel" (metadata staging, accumulation,
 *              shared-expert add).
 *
 * Functions whose result has a plain definition are that definition written out.
 * The MXFP8 encoding and the sigmoid are encodings/approximations and follow their
 * stated steps. Every function here is pinned by the CPU tests (tests/test_oracle_*.py)
 * against closed forms, brute force or library routines; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* BF16 <-> FP32, written from the format's definition (upper 16 bits of FP32). */

static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round-to-nearest-even to BF16. NaN stays NaN (quiet bit set). */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* ------------------------------------------------------------------------- */
/* Router logits.
 * [ep] EpMoeLayer.stock_order: logits = mm(x, gate^T) with out_dtype float32; the
 * [ep] module docstring: the router logits are FP32 and the split-K partials are reduced in FP32;
 * [wide] module docstring: FP32 router logits.
 * The oracle is the tolerance reference: the exact products of BF16 values summed
 * in FP64, plus sum_j |x*w| as the forward-error denominator. */
void oracle_router_logits(const uint16_t* x, const uint16_t* w, int T, int H, int E,
                          double* logits, double* abs_sum) {
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double s = 0.0, a = 0.0;
      const uint16_t* xr = x + (size_t)t * H;
      const uint16_t* wr = w + (size_t)e * H;
      for (int j = 0; j < H; ++j) {
        double p = (double)bf16_to_f32(xr[j]) * (double)bf16_to_f32(wr[j]);
        s += p;
        a += fabs(p);
      }
      logits[(size_t)t * E + e] = s;
      if (abs_sum) abs_sum[(size_t)t * E + e] = a;
    }
  }
}

/* The same, for n sampled (token, expert) pairs only. */
void oracle_router_logits_sampled(const uint16_t* x, const uint16_t* w, int H, int n,
                                  const int32_t* tok, const int32_t* exp_,
                                  double* logits, double* abs_sum) {
  for (int i = 0; i < n; ++i) {
    double s = 0.0, a = 0.0;
    const uint16_t* xr = x + (size_t)tok[i] * H;
    const uint16_t* wr = w + (size_t)exp_[i] * H;
    for (int j = 0; j < H; ++j) {
      double p = (double)bf16_to_f32(xr[j]) * (double)bf16_to_f32(wr[j]);
      s += p;
      a += fabs(p);
    }
    logits[i] = s;
    if (abs_sum) abs_sum[i] = a;
  }
}

/* ------------------------------------------------------------------------- */
/* Latent down projection: the front GEMM's latent columns.
 * [wide] module docstring: one front GEMM over the router rows and the latent down
 * rows, the latent then rounded to BF16 a single time, as the stock GEMM's epilogue does;
 * [ep] EpMoeLayer.stock_order: front = mm(x, front^T) in BF16.
 * The exact sum is oracle_router_logits over the down-projection rows. The one
 * rounding to BF16 is done here straight from the double (nearest, ties to even):
 * going through FP32 first would round twice. BF16 keeps 8 significant bits and
 * FP32's exponent range (normal down to 2^-126, subnormal steps of 2^-133). */
uint16_t oracle_f64_to_bf16(double v) {
  if (v != v) return 0x7FC0u;
  const uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);         /* a = m * 2^e2 with m in [0.5, 1): leading bit 2^(e2-1) */
  int lead = e2 - 1;
  if (lead < -126) lead = -126; /* below the normal range the step stays 2^-133 */
  const double step = ldexp(1.0, lead - 7);
  const double r = nearbyint(a / step) * step; /* a / step is exact; default mode: ties to even */
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* overflow: infinity */
  const float f = (float)r;                                     /* exact: 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

void oracle_f64_to_bf16_array(const double* v, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(v[i]);
}

/* ------------------------------------------------------------------------- */
/* Sigmoid. The pages say only "sigmoid" ([ep] EpMoeLayer.topk, scoring func
 * "sigmoid"); they fix no numerics. Because the selected ids and weights are
 * compared bit for bit, the method's sigmoid is specified here from a published
 * method: Cody & Waite (1980) range reduction exp(y) = 2^n * exp(r), r = y - n ln2,
 * with ln2 split into a high part (12 low significand bits cleared, so n*LN2_HI is
 * exact) and a low part, then the degree-7 Taylor polynomial of exp(r) by Horner
 * with fused multiply-adds. Only IEEE basic operations are used. */

static int consts_ready = 0;
static float LOG2E_F, LN2_HI, LN2_LO, INV_FACT[8];

static void init_consts(void) {
  if (consts_ready) return;
  double ln2 = log(2.0);
  LOG2E_F = (float)(1.0 / ln2);
  float hi = (float)ln2;
  uint32_t b;
  memcpy(&b, &hi, 4);
  b &= ~0xFFFu;
  memcpy(&hi, &b, 4);
  LN2_HI = hi;
  LN2_LO = (float)(ln2 - (double)hi);
  double fact = 1.0;
  for (int i = 0; i < 8; ++i) {
    if (i > 0) fact *= (double)i;
    INV_FACT[i] = (float)(1.0 / fact);
  }
  consts_ready = 1;
}

static float pow2_f32(int k) { /* 2^k for -126 <= k <= 127 */
  return f32_from_bits((uint32_t)(k + 127) << 23);
}

/* exp(y) for -17.5 < y < 88.5 (the only range the sigmoid below uses). */
float oracle_exp_spec(float y) {
  init_consts();
  float t = y * LOG2E_F;
  float n = rintf(t); /* round half to even (default rounding mode) */
  float r = fmaf(-n, LN2_HI, y);
  r = fmaf(-n, LN2_LO, r);
  float p = INV_FACT[7];
  for (int i = 6; i >= 0; --i) p = fmaf(p, r, INV_FACT[i]);
  int ni = (int)n;
  int a = ni / 2, c = ni - a; /* two exact power-of-two scalings */
  p = p * pow2_f32(a);
  p = p * pow2_f32(c);
  return p;
}

/* sigma(x) = 1 / (1 + exp(-x)): FP32 add, correctly rounded FP32 division.
 * x >= 17.5 gives exactly 1 (exp(-x) < 2^-25, so 1 + e rounds to 1);
 * x <= -88.5 gives 0 (exp(-x) taken as +inf). NaN propagates. */
float oracle_sigmoid(float x) {
  if (isnan(x)) return x;
  if (x >= 17.5f) return 1.0f;
  if (x <= -88.5f) return 0.0f;
  float e = oracle_exp_spec(-x);
  float d = 1.0f + e;
  return 1.0f / d;
}

void oracle_sigmoid_array(const float* x, float* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = oracle_sigmoid(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Sigmoid + e_score_correction_bias top-k with renormalised weights.
 * [ep] EpMoeLayer.topk: fused_grouped_topk(x, logits, 16, renormalize, bias, 1, 1,
 *      "sigmoid", scale) -- one group, sigmoid scores, bias-corrected selection.
 * [wide] WideRoute docstring: an exact top-16 with renormalised weights.
 * [wide] WideMoE.__init__: bias = gate.e_score_correction_bias, scale =
 *      routed_scaling_factor, renorm = moe_renormalize.
 * Readings where the pages are silent: selection key c_e = s_e + bias_e (FP32 add);
 * order "c descending, then expert index ascending"; slot k holds the k-th pick;
 * weights use the unbiased scores s; the renormalising sum runs in slot order in
 * FP32; a zero sum gives zero weights; scale multiplies after renormalising and is
 * skipped when it is 1. NaN keys rank below every number; +0 and -0 tie. */

/* 1 if (a, ia) ranks before (b, ib). */
static int ranks_before(float a, int ia, float b, int ib) {
  int an = isnan(a), bn = isnan(b);
  if (an || bn) {
    if (an && bn) return ia < ib;
    return bn;
  }
  if (a > b) return 1;
  if (a < b) return 0;
  return ia < ib;
}

int oracle_topk_route(const float* logits, const float* bias, int T, int E, int K,
                      int renormalize, float scale, int32_t* ids, float* weights,
                      uint16_t* weights_bf16) {
  if (T < 0 || E < 1 || K < 1 || K > E) return -1;
  float* s = (float*)malloc(sizeof(float) * (size_t)E);
  float* c = (float*)malloc(sizeof(float) * (size_t)E);
  unsigned char* taken = (unsigned char*)malloc((size_t)E);
  if (!s || !c || !taken) {
    free(s); free(c); free(taken);
    return -2;
  }
  for (int t = 0; t < T; ++t) {
    const float* lg = logits + (size_t)t * E;
    for (int e = 0; e < E; ++e) {
      s[e] = oracle_sigmoid(lg[e]);
      c[e] = bias ? s[e] + bias[e] : s[e];
      taken[e] = 0;
    }
    int32_t* id = ids + (size_t)t * K;
    /* K passes of a linear argmax. */
    for (int k = 0; k < K; ++k) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (best < 0 || ranks_before(c[e], e, c[best], best)) best = e;
      }
      taken[best] = 1;
      id[k] = best;
    }
    float S = 0.0f;
    for (int k = 0; k < K; ++k) S = S + s[id[k]];
    for (int k = 0; k < K; ++k) {
      float wk;
      if (renormalize)
        wk = (S == 0.0f) ? 0.0f : s[id[k]] / S;
      else
        wk = s[id[k]];
      if (scale != 1.0f) wk = wk * scale;
      weights[(size_t)t * K + k] = wk;
      if (weights_bf16) weights_bf16[(size_t)t * K + k] = f32_to_bf16_rne(wk);
    }
  }
  free(s); free(c); free(taken);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Per-expert routing lists.
 * [wide] WideRoute docstring and kernel: each of a token's 16 (token, slot) pairs is
 * appended to its expert's list; the stored value is cta*16 + tid, i.e. the pair
 * code t*K + k, which is also the expanded-row index the Finalize reads.
 * Reading: the pages' append order is whatever the atomic counter gives; here each
 * list is in ascending token order (within a token the experts are distinct, so the
 * order is total), stored as CSR: offsets = exclusive prefix sum of the counts. */
int oracle_routing_lists(const int32_t* ids, int T, int K, int E, int32_t* offsets,
                         int32_t* pairs) {
  int32_t* fill = (int32_t*)calloc((size_t)E + 1, sizeof(int32_t));
  if (!fill) return -2;
  for (long i = 0; i < (long)T * K; ++i) {
    int e = ids[i];
    if (e < 0 || e >= E) {
      free(fill);
      return -1;
    }
    fill[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + fill[e];
  memset(fill, 0, sizeof(int32_t) * ((size_t)E + 1));
  for (int t = 0; t < T; ++t)
    for (int k = 0; k < K; ++k) {
      int e = ids[(size_t)t * K + k];
      pairs[offsets[e] + fill[e]] = t * K + k;
      fill[e] += 1;
    }
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Unit windows of the routing lists.
 * [wide] module docstring: the wide grouped engine takes its units from the
 * routing lists, each expert that has tokens read once per 8 of them. Read as:
 * expert e's list is cut, in list order, into consecutive windows of `window` pairs
 * (the last one shorter); the units are numbered expert by expert. */
int oracle_unit_windows(const int32_t* offsets, int E, int window, int32_t* unit_offsets,
                        int32_t* unit_expert, int32_t* unit_start, int32_t* unit_len,
                        int max_units) {
  int u = 0;
  for (int e = 0; e < E; ++e) {
    unit_offsets[e] = u;
    for (int pos = offsets[e]; pos < offsets[e + 1]; pos += window) {
      if (u >= max_units) return -1;
      int len = offsets[e + 1] - pos;
      if (len > window) len = window;
      unit_expert[u] = e;
      unit_start[u] = pos;
      unit_len[u] = len;
      ++u;
    }
  }
  unit_offsets[E] = u;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* MXFP8 quantisation of BF16 rows.
 * [wide] module docstring: MXFP8 activations; [ep] module docstring: the latent in MXFP8,
 * bit-identical to the stock mxfp8_quantize; [wide] WideRoute: the plan row of a
 * token is written from its BF16 latent. The pages define no further detail, so the
 * OCP Microscaling (MX) v1.0 reading is taken: blocks of 32 consecutive elements,
 * one E8M0 scale X = 2^se with se = floor(log2(amax)) - emax(E4M3) = floor(log2 amax) - 8,
 * clamped to the E8M0 range, elements E4M3(v / X) rounded to nearest even with
 * saturation to +-448. Scales are stored row-major [rows, cols/32].
 * A block with a NaN or an infinity gets scale 0xFF and elements 0x7F (E8M0 and
 * E4M3 NaN); an all-zero block gets scale 0 and signed zeros. */

/* floor(log2 |v|) of a nonzero finite BF16, from its exponent bits. */
static int bf16_floor_log2(uint16_t b) {
  int ex = (b >> 7) & 0xFF;
  int man = b & 0x7F;
  if (ex) return ex - 127;
  int msb = 6;
  while (!((man >> msb) & 1)) --msb;
  return msb - 133; /* subnormal: man * 2^-133 */
}

/* Round-half-even of a nonnegative double to an integer-valued double. */
static double rne_nonneg(double v) {
  double f = floor(v);
  double d = v - f;
  if (d > 0.5) return f + 1.0;
  if (d < 0.5) return f;
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* E4M3 (bias 7, 3 mantissa bits, max finite 448, no infinities) of an exactly
 * representable double y, round to nearest even, saturating. */
uint8_t oracle_e4m3_encode(double y) {
  uint8_t sign = (y < 0.0 || (y == 0.0 && signbit(y))) ? 0x80 : 0x00;
  double a = fabs(y);
  if (a == 0.0) return sign;
  if (a > 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) { /* subnormal range: step 2^-9 */
    double m = rne_nonneg(a * 512.0);
    return sign | (uint8_t)m; /* m == 8 is the smallest normal, 0x08 */
  }
  int e = (int)floor(log2(a));
  /* guard log2 rounding at exact powers of two */
  if (ldexp(1.0, e) > a) e -= 1;
  if (ldexp(1.0, e + 1) <= a) e += 1;
  double m = rne_nonneg(ldexp(a, 3 - e)); /* in [8, 16] */
  if (m == 16.0) {
    e += 1;
    m = 8.0;
  }
  int code = ((e + 7) << 3) | ((int)m - 8);
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

/* rule 0: the OCP floor rule above. rule 1: the round-up rule, X = the smallest power
 * of two with amax / X <= 448 (no element saturates): the floor exponent, plus one when
 * amax exceeds 448 times the floor scale (a block maximum whose significand is above
 * 1.75). The pages show neither; the ep page only says the stock quantiser's output is
 * matched bit for bit, so both readings are kept. */
void oracle_mxfp8_quantize_rule(const uint16_t* x, int rows, int cols, int rule, uint8_t* q,
                                uint8_t* scales) {
  int blocks = cols / 32;
  for (int r = 0; r < rows; ++r) {
    for (int b = 0; b < blocks; ++b) {
      const uint16_t* v = x + (size_t)r * cols + (size_t)b * 32;
      uint8_t* qo = q + (size_t)r * cols + (size_t)b * 32;
      int special = 0;
      float amax = 0.0f;
      uint16_t amax_bits = 0;
      for (int i = 0; i < 32; ++i) {
        float f = bf16_to_f32(v[i]);
        if (isnan(f) || isinf(f)) special = 1;
        float m = fabsf(f);
        if (m > amax) {
          amax = m;
          amax_bits = v[i] & 0x7FFF;
        }
      }
      uint8_t* so = scales + (size_t)r * blocks + b;
      if (special) {
        *so = 0xFF;
        for (int i = 0; i < 32; ++i) qo[i] = 0x7F;
        continue;
      }
      if (amax == 0.0f) {
        *so = 0;
        for (int i = 0; i < 32; ++i) qo[i] = (v[i] & 0x8000) ? 0x80 : 0x00;
        continue;
      }
      int se = bf16_floor_log2(amax_bits) - 8;
      if (rule == 1 && (double)amax > ldexp(448.0, se)) se += 1;
      if (se < -127) se = -127;
      if (se > 127) se = 127;
      *so = (uint8_t)(se + 127);
      for (int i = 0; i < 32; ++i) {
        double y = ldexp((double)bf16_to_f32(v[i]), -se); /* exact */
        qo[i] = oracle_e4m3_encode(y);
      }
    }
  }
}

void oracle_mxfp8_quantize(const uint16_t* x, int rows, int cols, uint8_t* q,
                           uint8_t* scales) {
  oracle_mxfp8_quantize_rule(x, rows, cols, 0, q, scales);
}

/* The scale bytes of oracle_mxfp8_quantize_rule in the tile layout that the
 * block-scaled tensor-core MMA of the sm_100 family (tcgen05.mma kind::mxf8f6f4 with
 * a scale vector of 32) loads through tcgen05.cp, as the PTX ISA and CUTLASS's
 * block-scaled GEMMs describe it: the [rows, nsc] scale matrix is cut into tiles of
 * 128 rows x 4 scale columns (rows padded to a multiple of 128, columns to a multiple
 * of 4); tile (i, j) occupies the 512 bytes at (i * CT + j) * 512, CT = ceil(nsc / 4),
 * and inside it the scale of row r (0..127) and column c (0..3) is byte
 * 16 * (r mod 32) + 4 * (r div 32) + c: 32 lines of 16 bytes, line l holding rows
 * l, l + 32, l + 64, l + 96. Padding bytes are 0. The wide page writes its plan rows
 * with a swizzled scale layout of its own (plan_xsf) that it does not show. */
size_t oracle_mxfp8_tcgen05_scales_bytes(int rows, int nsc) {
  const size_t rt = (size_t)(rows + 127) / 128, ct = (size_t)(nsc + 3) / 4;
  return rt * ct * 512;
}

void oracle_mxfp8_scales_tcgen05(const uint8_t* scales, int rows, int nsc, uint8_t* out) {
  const size_t ct = (size_t)(nsc + 3) / 4;
  memset(out, 0, oracle_mxfp8_tcgen05_scales_bytes(rows, nsc));
  for (int r = 0; r < rows; ++r) {
    for (int c = 0; c < nsc; ++c) {
      const size_t tile = (size_t)(r / 128) * ct + (size_t)(c / 4);
      const int rr = r % 128, cc = c % 4;
      out[tile * 512 + 16 * (rr % 32) + 4 * (rr / 32) + cc] = scales[(size_t)r * nsc + c];
    }
  }
}

/* E4M3 byte -> value (NaN for 0x7F/0xFF). */
double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* ------------------------------------------------------------------------- */
/* Finalize: out[t] = sum_k w[t,k] * rows[idx(t,k)], FP32, k in order, one BF16
 * rounding.
 * [wide] Finalize docstring and kernel: acc starts at 0, acc = fma(w, row, acc) for
 *   k = 0..15 in order, then one round-to-nearest-even pack to BF16; row 16t + k.
 * [fin] _QuadFinalizePublishDeviceKernel: metadata staging (weight read as BF16 or
 *   FP32, multiplied by routed_scaling_factor when it is not 1, zeroed when the
 *   permuted index is -1), the accumulation over k in order skipping -1 rows, and
 *   the shared-expert row added in FP32 once after all k, then one BF16 rounding.
 * row_index NULL means row t*K + k. weights_bf16 selects the weight dtype.
 * Returns -1 (and writes nothing further) on an index outside [-1, n_rows). */
int oracle_finalize(const uint16_t* rows, long n_rows, const int32_t* row_index,
                    const void* weights, int weights_bf16, const uint16_t* shared,
                    float scale, int T, int K, int H, uint16_t* out) {
  float* w = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
  long* idx = (long*)malloc(sizeof(long) * (size_t)(K > 0 ? K : 1));
  if (!w || !idx) {
    free(w); free(idx);
    return -2;
  }
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      size_t i = (size_t)t * K + k;
      long r = row_index ? (long)row_index[i] : (long)i;
      if (r < -1 || r >= n_rows) {
        free(w); free(idx);
        return -1;
      }
      float wk = weights_bf16 ? bf16_to_f32(((const uint16_t*)weights)[i])
                              : ((const float*)weights)[i];
      if (scale != 1.0f) wk = wk * scale;
      if (r == -1) wk = 0.0f;
      w[k] = wk;
      idx[k] = r;
    }
    for (int c = 0; c < H; ++c) {
      float acc = 0.0f;
      for (int k = 0; k < K; ++k) {
        if (idx[k] == -1) continue;
        acc = fmaf(w[k], bf16_to_f32(rows[(size_t)idx[k] * H + c]), acc);
      }
      if (shared) acc = acc + bf16_to_f32(shared[(size_t)t * H + c]);
      out[(size_t)t * H + c] = f32_to_bf16_rne(acc);
    }
  }
  free(w); free(idx);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* RMSNorm of the routed latent (the tolerance reference).
 * [ep] EpMoeLayer.forward / stock_order: normed = rms_norm(routed, w["norm"], eps),
 * eps defaulting to 1e-5; [wide] WideMoE.tail: the RMSNorm of the latent. The pages
 * give no formula beyond the name; the plainest reading is the usual one:
 *   y[c] = x[c] / sqrt(mean_c x[c]^2 + eps) * g[c],
 * here in FP64 from the BF16 values x (the routed latent, already rounded to BF16 by
 * Finalize) and g. The GPU's FP32 result, rounded once to BF16, is compared against
 * this value within a relative tolerance. */
void oracle_rmsnorm(const uint16_t* x, const uint16_t* g, int T, int H, double eps, double* y) {
  for (int t = 0; t < T; ++t) {
    const uint16_t* xr = x + (size_t)t * H;
    double ss = 0.0;
    for (int c = 0; c < H; ++c) {
      const double v = (double)bf16_to_f32(xr[c]);
      ss += v * v;
    }
    const double inv = 1.0 / sqrt(ss / (double)H + eps);
    for (int c = 0; c < H; ++c)
      y[(size_t)t * H + c] = (double)bf16_to_f32(xr[c]) * inv * (double)bf16_to_f32(g[c]);
  }
}

/* ------------------------------------------------------------------------- */
/* BF16 helpers exposed for the tests' own checks of the conversions. */
float oracle_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
uint16_t oracle_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
