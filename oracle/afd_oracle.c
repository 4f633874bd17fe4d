/*
 * afd_oracle.c -- plain, slow CPU oracle for the FFN-server MoE layer of
 * Attention-FFN Disaggregation (AFD).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes (one MoE layer over one aggregated decode batch):
 *   a1  tokens of M attention-instance buffers, in (buffer, row) order, form
 *       one batch X[T,H]  ("大模型推理的内存与计算解耦：AFD 架构解析与性能验证",
 *       section 2, benefit one: several attention instances feed one FFN).
 *   a2  router logits l[t,e] = sum_h x[t,h] * Wr[h,e] (+ bias[e]) in fp32, in a
 *       fixed summation order (defined below), because top-k indices must be
 *       reproducible bit for bit on any machine.
 *   a3  top-k on the logits, then softmax over the k selected logits
 *       ("MoE 大规模分布式推理工程实战", section 4.1, the router's forward:
 *       logits + dynamic bias, topk, softmax of the top-k logits).
 *   a4/a5 per-expert counts, exclusive prefix sum, expert-contiguous order
 *       (same page, section 2.2: per-destination counts, prefix-sum offsets,
 *       pack kernel; "MoE系统与AFD架构概述" section 3.3: pre-sort routing
 *       results), here per expert and stable by token index.
 *   a6..a9 per selected expert a SwiGLU FFN  y = (silu(a Wg) * (a Wu)) Wd,
 *       weighted by the routing weight and summed in slot order, plus an
 *       always-on shared expert with weight 1 when configured.
 *
 * Precision: dot products of the expert FFN accumulate in double.  The
 * intermediate h is rounded to the precision the down projection consumes
 * (fp32 / bf16 / per-128-channel e4m3).  The output is rounded once.
 * FP8 activations are quantised per row per 128 channels with
 * scale = amax/448 (fp32 division), q = e4m3(x/scale) rounded to nearest even
 * and saturated to +-448, as in the layer's FP8 configuration.
 *
 * Parity pins: see tests/test_oracle_pins.py (brute force, closed forms,
 * library routines, invariants).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_FP32 0
#define ORC_BF16 1
#define ORC_FP8 2

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32. */
static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary32 -> bf16, round to nearest, ties to even (NaN stays NaN). */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

float oracle_bf16_round(float f) { return bf16_bits_to_f32(oracle_f32_to_bf16(f)); }

/* OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign, 4 exponent bits
 * (bias 7), 3 mantissa bits; exponent field 0 is subnormal
 * (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities; the largest
 * finite magnitude is S.1111.110 = 1.75 * 2^8 = 448. */
double oracle_e4m3_decode(uint8_t q) {
  int s = (q >> 7) & 1;
  int e = (q >> 3) & 0xf;
  int m = q & 7;
  double v;
  if (e == 0xf && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* binary32 -> E4M3, round to nearest with ties to the even code, magnitudes
 * above 448 (and infinities) saturate to 448, NaN maps to the NaN code.
 * Written from the definition: the 127 non-negative finite codes are ordered
 * by value, so the result is the nearest code by a search over that order. */
uint8_t oracle_e4m3_encode(float v) {
  if (isnan(v)) return 0x7f;
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  /* largest code c in [0, 0x7e] with decode(c) <= a */
  int lo = 0, hi = 0x7e;
  while (lo < hi) {
    int mid = (lo + hi + 1) / 2;
    if (oracle_e4m3_decode((uint8_t)mid) <= a)
      lo = mid;
    else
      hi = mid - 1;
  }
  int c = lo;
  double vc = oracle_e4m3_decode((uint8_t)c);
  if (vc == a || c == 0x7e) return (uint8_t)(sign | c);
  double vn = oracle_e4m3_decode((uint8_t)(c + 1));
  double dl = a - vc, dh = vn - a;
  int pick;
  if (dl < dh)
    pick = c;
  else if (dh < dl)
    pick = c + 1;
  else
    pick = (c & 1) ? c + 1 : c; /* tie: even code (mantissa lsb 0) */
  return (uint8_t)(sign | pick);
}

/* Quantise one row of `n` fp32 values in blocks of 128 channels:
 * scale_b = amax_b / 448 (binary32 division), q = e4m3(x / scale_b);
 * an all-zero block gets scale 1 and zero codes. */
void oracle_quantize_row(const float* x, int n, uint8_t* q, float* scales) {
  for (int b0 = 0, blk = 0; b0 < n; b0 += 128, ++blk) {
    int b1 = b0 + 128 < n ? b0 + 128 : n;
    float amax = 0.0f;
    for (int i = b0; i < b1; ++i) {
      float a = fabsf(x[i]);
      if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
      scales[blk] = 1.0f;
      for (int i = b0; i < b1; ++i) q[i] = 0;
      continue;
    }
    volatile float scale = amax / 448.0f;
    scales[blk] = scale;
    for (int i = b0; i < b1; ++i) {
      volatile float r = x[i] / scale;
      q[i] = oracle_e4m3_encode(r);
    }
  }
}

/* ------------------------------------------------------------------ */
/* Inputs                                                              */
/* ------------------------------------------------------------------ */

static float load_act(const void* base, int dtype, long idx) {
  if (dtype == ORC_FP32) return ((const float*)base)[idx];
  return bf16_bits_to_f32(((const uint16_t*)base)[idx]);
}

/* ------------------------------------------------------------------ */
/* a2: router logits in the canonical order                            */
/* ------------------------------------------------------------------ */
/*
 * The canonical fp32 order of  s = sum_h x[h] * w[h]  over H channels
 * (H a multiple of 8):
 *   1. channels are grouped in chunks of 8 consecutive channels; chunk c
 *      belongs to lane (c mod 32);
 *   2. each of the 32 lanes starts from +0 and applies, for its chunks in
 *      ascending order and for the 8 channels of a chunk in ascending order,
 *      p = fma(x[h], w[h], p)  (one rounding per step);
 *   3. the 32 lane sums are folded pairwise: for o = 16, 8, 4, 2, 1,
 *      p[l] = p[l] + p[l + o] for l < o;   s = p[0];
 *   4. when a bias is present, logit = s + bias[e] (one fp32 addition).
 * Selection of the top-k set depends on every bit of the logits, so both
 * implementations of the layer evaluate exactly this expression.
 */
float oracle_canonical_dot(const float* x, const float* w, int H) {
  float p[32];
  for (int l = 0; l < 32; ++l) p[l] = 0.0f;
  int nchunk = H / 8;
  for (int c = 0; c < nchunk; ++c) {
    int l = c % 32;
    for (int j = 0; j < 8; ++j) {
      int h = 8 * c + j;
      p[l] = fmaf(x[h], w[h], p[l]);
    }
  }
  for (int o = 16; o >= 1; o /= 2)
    for (int l = 0; l < o; ++l) {
      volatile float s = p[l] + p[l + o];
      p[l] = s;
    }
  return p[0];
}

/* logits[t,e] for X[T,H] (act dtype fp32 or bf16) and Wr[H,E] (same dtype). */
void oracle_router_logits(const void* x, const void* w_r, int act_dtype, const float* bias, int T, int H,
                          int E, float* logits) {
  float* wt = (float*)malloc(sizeof(float) * (size_t)H * E); /* Wr transposed to [E,H] as fp32 */
  for (int h = 0; h < H; ++h)
    for (int e = 0; e < E; ++e) wt[(size_t)e * H + h] = load_act(w_r, act_dtype, (long)h * E + e);
#pragma omp parallel for schedule(dynamic, 4)
  for (int t = 0; t < T; ++t) {
    float* xr = (float*)malloc(sizeof(float) * H);
    for (int h = 0; h < H; ++h) xr[h] = load_act(x, act_dtype, (long)t * H + h);
    for (int e = 0; e < E; ++e) {
      float s = oracle_canonical_dot(xr, wt + (size_t)e * H, H);
      if (bias) {
        volatile float b = s + bias[e];
        s = b;
      }
      logits[(size_t)t * E + e] = s;
    }
    free(xr);
  }
  free(wt);
}

/* ------------------------------------------------------------------ */
/* a3: top-k selection and softmax over the selected logits            */
/* ------------------------------------------------------------------ */
/* Expert a ranks before expert b iff l_a > l_b, or l_a == l_b and a < b.
 * Slot j holds the j-th ranked expert.  Weights: w_j = exp(l_j - l_0) /
 * sum_i exp(l_i - l_0) over the k selected, in double, stored as fp32. */
void oracle_topk(const float* logits, int T, int E, int k, int32_t* idx, float* wts) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float* l = logits + (size_t)t * E;
    unsigned char* used = (unsigned char*)calloc((size_t)E, 1);
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (used[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict: ties keep the lower id */
      }
      used[best] = 1;
      idx[(size_t)t * k + j] = best;
    }
    double m = (double)l[idx[(size_t)t * k]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)l[idx[(size_t)t * k + j]] - m);
    for (int j = 0; j < k; ++j)
      wts[(size_t)t * k + j] = (float)(exp((double)l[idx[(size_t)t * k + j]] - m) / den);
    free(used);
  }
}

/* ------------------------------------------------------------------ */
/* a4/a5: histogram, exclusive prefix sum, stable expert-major order    */
/* ------------------------------------------------------------------ */
/* counts[e]   = #{(t,j) : idx[t,j] == e}
 * offsets[e]  = sum_{e' < e} counts[e'],  offsets[E] = T*k
 * perm[r]     = token of packed row r; rows of expert e are offsets[e] ..
 *               offsets[e+1]-1 in ascending token order
 * pos[t*k+j]  = packed row of (t, j) */
void oracle_routing_tables(const int32_t* idx, int T, int k, int E, int32_t* counts, int32_t* offsets,
                           int32_t* perm, int32_t* pos) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long i = 0; i < (long)T * k; ++i) counts[idx[i]]++;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  for (int e = 0; e < E; ++e) {
    int row = offsets[e];
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) {
          perm[row] = t;
          pos[(size_t)t * k + j] = row;
          ++row;
        }
  }
}

/* ------------------------------------------------------------------ */
/* a6..a9: expert FFN and combine                                      */
/* ------------------------------------------------------------------ */

typedef struct {
  int H, I, E, k, n_shared, dtype;
} oracle_cfg;

typedef struct {
  const void* w_router; /* [H,E], act dtype (bf16 for bf16/fp8 layers) */
  const float* router_bias; /* [E] or NULL */
  const void *w_gate, *w_up; /* [E,H,I]: fp32 / bf16 bits / e4m3 codes */
  const void* w_down;        /* [E,I,H] */
  const float *s_gate, *s_up; /* fp8: [E,H/128,I/128] */
  const float* s_down;        /* fp8: [E,I/128,H/128] */
  const void *sh_gate, *sh_up, *sh_down; /* shared expert, one expert's shapes */
  const float *sh_s_gate, *sh_s_up, *sh_s_down;
} oracle_weights;

/* element (r, c) of expert matrix [R, C] with optional 128x128 block scales */
static double weight_at(const void* w, const float* s, int dtype, long ebase, int R, int C, int r, int c,
                        const double* e4m3_table) {
  (void)R;
  long i = ebase + (long)r * C + c;
  if (dtype == ORC_FP32) return (double)((const float*)w)[i];
  if (dtype == ORC_BF16) return (double)bf16_bits_to_f32(((const uint16_t*)w)[i]);
  {
    int nbc = (C + 127) / 128;
    long sbase = (ebase / ((long)R * C)) * ((long)((R + 127) / 128) * nbc);
    double sc = (double)s[sbase + (long)(r / 128) * nbc + c / 128];
    return e4m3_table[((const uint8_t*)w)[i]] * sc;
  }
}

/* Turn an fp32 row into the values the next GEMM consumes, per layer dtype. */
static void operand_row(const float* v, int n, int dtype, double* out, const double* e4m3_table) {
  if (dtype == ORC_FP32) {
    for (int i = 0; i < n; ++i) out[i] = (double)v[i];
  } else if (dtype == ORC_BF16) {
    for (int i = 0; i < n; ++i) out[i] = (double)oracle_bf16_round(v[i]);
  } else {
    uint8_t* q = (uint8_t*)malloc((size_t)n);
    float* sc = (float*)malloc(sizeof(float) * (size_t)((n + 127) / 128));
    oracle_quantize_row(v, n, q, sc);
    for (int i = 0; i < n; ++i) out[i] = e4m3_table[q[i]] * (double)sc[i / 128];
    free(q);
    free(sc);
  }
}

/* First half of one SwiGLU expert on an operand row a[H] (double):
 * G = a Wg, U = a Wu accumulated in double, hf[i] = silu(G_i) * U_i rounded
 * once to fp32 -- the value the down projection's operand is made from. */
static void expert_hidden(const oracle_cfg* cfg, const void* wg, const void* wu, const float* sg,
                          const float* su, int e, const double* a, float* hf, const double* e4m3_table) {
  int H = cfg->H, I = cfg->I;
  double* G = (double*)calloc((size_t)I, sizeof(double));
  double* U = (double*)calloc((size_t)I, sizeof(double));
  long gbase = (long)e * H * I;
  for (int h = 0; h < H; ++h) {
    double ah = a[h];
    for (int i = 0; i < I; ++i) {
      G[i] += ah * weight_at(wg, sg, cfg->dtype, gbase, H, I, h, i, e4m3_table);
      U[i] += ah * weight_at(wu, su, cfg->dtype, gbase, H, I, h, i, e4m3_table);
    }
  }
  for (int i = 0; i < I; ++i) {
    double g = G[i];
    double silu = g / (1.0 + exp(-g));
    hf[i] = (float)(silu * U[i]);
  }
  free(G);
  free(U);
}

/* y[H] = SwiGLU expert applied to one operand row a[H] (double).  Returns the
 * number of multiply-adds performed (3*H*I). */
static long long expert_ffn(const oracle_cfg* cfg, const void* wg, const void* wu, const void* wd,
                            const float* sg, const float* su, const float* sd, int e, const double* a,
                            double* y, const double* e4m3_table) {
  int H = cfg->H, I = cfg->I;
  long long fmas = 0;
  float* hf = (float*)malloc(sizeof(float) * (size_t)I);
  double* hd = (double*)malloc(sizeof(double) * (size_t)I);
  expert_hidden(cfg, wg, wu, sg, su, e, a, hf, e4m3_table);
  fmas += 2LL * H * I;
  operand_row(hf, I, cfg->dtype, hd, e4m3_table);
  for (int c = 0; c < H; ++c) y[c] = 0.0;
  long dbase = (long)e * I * H;
  for (int i = 0; i < I; ++i) {
    double hi = hd[i];
    for (int c = 0; c < H; ++c) y[c] += hi * weight_at(wd, sd, cfg->dtype, dbase, I, H, i, c, e4m3_table);
  }
  fmas += (long long)I * H;
  free(hf);
  free(hd);
  return fmas;
}

/* The fp32 SwiGLU hidden rows (before the down projection's rounding or
 * quantisation) of n (token, expert) pairs, for tests that compare the
 * layer's intermediate operand.
 *   x      : [n, H] token rows in the activation dtype (fp32 values, or bf16
 *            bits for the bf16/fp8 layers)
 *   expert : [n] expert ids; -1 selects the shared expert
 *   hf     : [n, I] fp32 output
 * The activation operand is formed as in the full layer (bf16 values, or the
 * per-128-channel e4m3 quantisation for the fp8 layer).  Returns 0, or -1 on
 * a bad expert id. */
int oracle_expert_hidden(const oracle_cfg* cfg, const oracle_weights* w, const void* x, const int32_t* expert,
                         int n, float* hf) {
  int H = cfg->H, I = cfg->I;
  int act_dtype = cfg->dtype == ORC_FP32 ? ORC_FP32 : ORC_BF16;
  double e4m3_table[256];
  for (int c = 0; c < 256; ++c) e4m3_table[c] = oracle_e4m3_decode((uint8_t)c);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n; ++i) {
    int e = expert[i];
    if (e < -1 || e >= cfg->E || (e == -1 && !cfg->n_shared)) {
      bad = 1;
      continue;
    }
    float* xf = (float*)malloc(sizeof(float) * H);
    double* a = (double*)malloc(sizeof(double) * H);
    for (int h = 0; h < H; ++h) xf[h] = load_act(x, act_dtype, (long)i * H + h);
    operand_row(xf, H, cfg->dtype, a, e4m3_table);
    if (e < 0)
      expert_hidden(cfg, w->sh_gate, w->sh_up, w->sh_s_gate, w->sh_s_up, 0, a, hf + (size_t)i * I, e4m3_table);
    else
      expert_hidden(cfg, w->w_gate, w->w_up, w->s_gate, w->s_up, e, a, hf + (size_t)i * I, e4m3_table);
    free(xf);
    free(a);
  }
  return bad ? -1 : 0;
}

/*
 * Full layer.
 *   src[m] : [src_counts[m], H] in the activation dtype (fp32 for the fp32
 *            layer, bf16 bits otherwise); tokens are numbered in (m, row) order.
 *   tokens : the token ids whose outputs are computed (NULL = all T); routing
 *            (logits, top-k) is always evaluated for every token.
 *   out    : [n_tokens, H], fp32 for the fp32 layer, bf16 bits otherwise; row i
 *            is the output of tokens[i].
 *   idx/wts/logits (optional): [T,k], [T,k], [T,E].
 *   fma_count (optional): multiply-adds spent in expert FFNs for the computed
 *            tokens.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_moe_forward(const oracle_cfg* cfg, const oracle_weights* w, const void* const* src,
                       const int* src_counts, int M, const int32_t* tokens, int n_tokens, void* out,
                       int32_t* idx_out, float* w_out, float* logits_out, long long* fma_count) {
  int H = cfg->H, E = cfg->E, k = cfg->k;
  if (H <= 0 || cfg->I <= 0 || E <= 0 || k <= 0 || k > E || H % 8 != 0 || M < 0) return -1;
  int act_dtype = cfg->dtype == ORC_FP32 ? ORC_FP32 : ORC_BF16;
  size_t esz = act_dtype == ORC_FP32 ? 4 : 2;
  long T = 0;
  for (int m = 0; m < M; ++m) {
    if (src_counts[m] < 0) return -1;
    T += src_counts[m];
  }
  /* a1: aggregate the M buffers in (m, row) order */
  char* X = (char*)malloc(esz * (size_t)(T > 0 ? T : 1) * H);
  {
    size_t off = 0;
    for (int m = 0; m < M; ++m) {
      size_t nb = esz * (size_t)src_counts[m] * H;
      if (nb) memcpy(X + off, src[m], nb);
      off += nb;
    }
  }
  double e4m3_table[256];
  for (int c = 0; c < 256; ++c) e4m3_table[c] = oracle_e4m3_decode((uint8_t)c);

  float* logits = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1) * E);
  int32_t* idx = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1) * k);
  float* wts = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1) * k);
  oracle_router_logits(X, w->w_router, act_dtype, w->router_bias, (int)T, H, E, logits);
  oracle_topk(logits, (int)T, E, k, idx, wts);

  int n_out = tokens ? n_tokens : (int)T;
  long long total_fma = 0;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : total_fma)
  for (int i = 0; i < n_out; ++i) {
    long t = tokens ? tokens[i] : i;
    if (t < 0 || t >= T) {
      bad = 1;
      continue;
    }
    float* xf = (float*)malloc(sizeof(float) * H);
    double* a = (double*)malloc(sizeof(double) * H);
    double* y = (double*)malloc(sizeof(double) * H);
    double* acc = (double*)calloc((size_t)H, sizeof(double));
    for (int h = 0; h < H; ++h) xf[h] = load_act(X, act_dtype, t * H + h);
    operand_row(xf, H, cfg->dtype, a, e4m3_table); /* a6: activation operand */
    for (int j = 0; j < k; ++j) {
      int e = idx[t * k + j];
      double wj = (double)wts[t * k + j];
      total_fma += expert_ffn(cfg, w->w_gate, w->w_up, w->w_down, w->s_gate, w->s_up, w->s_down, e, a, y,
                              e4m3_table);
      for (int h = 0; h < H; ++h) acc[h] += wj * y[h];
    }
    if (cfg->n_shared) {
      total_fma += expert_ffn(cfg, w->sh_gate, w->sh_up, w->sh_down, w->sh_s_gate, w->sh_s_up,
                              w->sh_s_down, 0, a, y, e4m3_table);
      for (int h = 0; h < H; ++h) acc[h] += y[h];
    }
    for (int h = 0; h < H; ++h) {
      if (cfg->dtype == ORC_FP32)
        ((float*)out)[(size_t)i * H + h] = (float)acc[h];
      else
        ((uint16_t*)out)[(size_t)i * H + h] = oracle_f32_to_bf16((float)acc[h]);
    }
    free(xf);
    free(a);
    free(y);
    free(acc);
  }
  if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)T * k);
  if (w_out) memcpy(w_out, wts, sizeof(float) * (size_t)T * k);
  if (logits_out) memcpy(logits_out, logits, sizeof(float) * (size_t)T * E);
  if (fma_count) *fma_count = total_fma;
  free(X);
  free(logits);
  free(idx);
  free(wts);
  return bad ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the parallel loops that follow (n >= 1); timing only, results do not
 * depend on it (every parallel loop writes disjoint outputs or sums integers). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
