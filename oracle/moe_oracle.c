/*
 * moe_oracle.c -- plain, slow, fp64 oracle of the MoE FFN layer forward.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE LIBRARY.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load or call this code.  It
 * shares nothing with the CUDA path: no header, helper, table or constant.
 *
 * What it computes, step by step, in the order the Colibri pages give the
 * MoE pipeline ("Colibri：面向MoE架构的C语言级高效推理引擎" §2.1: router logits,
 * top-k, dispatch to the k experts, k expert matmuls, weighted sum):
 *
 *  1. router logits  l[t][e] = sum_i x[t][i] * Wr[e][i] + b[e]
 *     (the router's linear projection with bias, same page §3.2; Wr stored
 *     as [E][d] out-by-in, the channel-last rule of §3.1)
 *  2. gating: softmax over the E logits, then top-k, weights renormalised
 *     over the k ("Colibri：面向MoE模型的高性能C语言推理引擎" §1, §2.1).
 *     Experts are ordered by (logit descending, index ascending), so ties go
 *     to the lower index; slot s is the s-th expert in that order.  Because
 *     softmax is monotone and its full denominator cancels after the
 *     renormalisation, w[t][s] = exp(l_s - l_0) / sum_{j<k} exp(l_j - l_0).
 *     A NaN logit ranks below every number; among NaNs the lower index wins.
 *     Router variants (step 2 replaced; the rest of the layer unchanged):
 *     - raw-logit gate (the first page's §3.2: top-k straight on the raw
 *       logits, no softmax): the same expert order, and slot s carries the
 *       selected logit itself as its weight, w[t][s] = l_s;
 *     - hash routing ("lshu.cn/news/53496" §2): a light projection
 *       r = x W_h to hash_dims values (W_h stored [hash_dims][d]), each
 *       mapped to a 20-bit integer h_i = (int32)(r_i * 1e6) & 0xFFFFF, and
 *       the expert (h_0 ^ h_1 ^ ...) mod E, with k = 1 and weight 1.  The
 *       page's expression is C on a float routing vector, so r_i is a float
 *       sum, taken left to right, of the exact bf16 products; r_i * 1e6 is
 *       evaluated in double (the literal is a double), which is exact; the
 *       int32 conversion truncates toward zero and saturates at the int32
 *       range (NaN gives 0), which the page leaves open.
 *  3. dispatch (the dispatch kernel of the first page's §2.3): per-expert
 *     counts, exclusive prefix-sum offsets, and the canonical permutation:
 *     rows of expert e hold its tokens in ascending token order.
 *     tok[row] = token, inv[t][s] = row.
 *  4. expert FFN per routed row (SwiGLU with w1 = gate, w3 = up,
 *     w2 = down, second page §4.2): g_j = sum_i x_i Wg[e][j][i],
 *     u_j = sum_i x_i Wu[e][j][i], h_j = SiLU(g_j) u_j with
 *     SiLU(z) = z / (1 + exp(-z)), y_c = sum_j h_j Wd[e][c][j].
 *     int8 experts (symmetric per-output-channel, "lshu.cn/news/53496" §4.3):
 *     W[e][j][i] = s[e][j] * Q[e][j][i], so g_j = s_g[e][j] * sum_i x_i Q_g.
 *     int4 experts (4-bit codes with a scale and a zero point per channel,
 *     "m.nxbn.cn/news/47706" §3.2; a channel is read as an output row):
 *     W[e][j][i] = s[e][j] * (q[e][j][i] - z[e][j]) with q in 0..15 packed two
 *     to a byte along i (element 2m in the low nibble of byte m) and an
 *     integer zero point z, so g_j = s_g[e][j] * sum_i x_i (q_g - z_g).
 *     fp8 experts (the FP8 of the roadmap in "discosf.com/news/4774337" §6.3,
 *     read as the e4m3 format that Transformer Engine uses for forward-pass
 *     weights, with an fp32 scale per output channel as for int8):
 *     W[e][j][i] = s[e][j] * v(c[e][j][i]) for the byte c = sign, 4 exponent
 *     bits E (bias 7), 3 mantissa bits M: v = (-1)^sign * (1 + M/8) * 2^(E-7)
 *     for E > 0, (-1)^sign * (M/8) * 2^-6 for E = 0; E = 15 with M = 7 is NaN
 *     (there is no infinity).
 *     Mode EXACT keeps h in double; mode BF16H rounds each h_j to bf16
 *     (round to nearest even) before the down projection, which is the
 *     precision the layer's bf16 down-projection operand holds.
 *  5. combine (the combine kernel of the first page's §2.3):
 *     o[t] = sum_s w[t][s] * y(t, s).
 *
 * Every sum is a plain sequential loop in double.  Inputs are bf16 bit
 * patterns (uint16), or int8, packed int4 or e4m3 codes with float scales
 * (and uint8 zero points for int4).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
  int32_t T, d, f, E, k;
  int32_t wdtype;                 /* 0 = bf16 weights, 1 = int8 + scales,
                                     2 = int4 + scales + zero points,
                                     3 = fp8 (e4m3) + scales              */
  const uint16_t *x;              /* [T][d] bf16 bits                    */
  const uint16_t *wr;             /* [E][d] bf16 bits                    */
  const float *bias;              /* [E] or NULL                         */
  const void *wg, *wu;            /* [E][f][d] bf16 bits or int8         */
  const void *wd;                 /* [E][d][f]                           */
  const float *sg, *su;           /* [E][f] (int8 only)                  */
  const float *sd;                /* [E][d] (int8 only)                  */
  int32_t router_mode;            /* 0 softmax top-k, 1 raw logits, 2 hash */
  int32_t hash_dims;              /* hash router: rows of wh             */
  const uint16_t *wh;             /* [hash_dims][d] bf16 bits, or NULL   */
  const uint8_t *zg, *zu;         /* [E][f] zero points (int4 only)      */
  const uint8_t *zd;              /* [E][d] (int4 only)                  */
} moe_oracle_layer_t;

enum { ORACLE_EXACT = 0, ORACLE_BF16H = 1 };
enum { ROUTER_SOFTMAX = 0, ROUTER_RAW = 1, ROUTER_HASH = 2 };

/* ---------------------------------------------------------------- threads */
void moe_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int moe_oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- numbers */
static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 value (ties to even), returned as a
 * double.  Normal range: clear the low 45 of the 52 fraction bits with
 * round-half-even on the bit pattern; subnormal range: the 2^-133 grid. */
double moe_oracle_round_bf16(double v) {
  if (isnan(v) || isinf(v) || v == 0.0) return v;
  double a = fabs(v);
  if (a < 0x1p-126) return copysign(nearbyint(a * 0x1p133) * 0x1p-133, v);
  uint64_t b;
  memcpy(&b, &v, 8);
  uint64_t lsb = (b >> 45) & 1u;
  b += ((uint64_t)1 << 44) - 1u + lsb;
  b &= ~(((uint64_t)1 << 45) - 1u);
  double r;
  memcpy(&r, &b, 8);
  if (fabs(r) > 0x1.FEp127) return copysign(INFINITY, v);
  return r;
}

/* bf16 bit pattern of a value already on the bf16 grid */
uint16_t moe_oracle_bf16_bits(double v) {
  double r = moe_oracle_round_bf16(v);
  float f = (float)r;
  uint32_t u;
  memcpy(&u, &f, 4);
  if (isnan(v)) return 0x7FC0;
  return (uint16_t)(u >> 16);
}

/* Value of an e4m3 byte (sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities; exponent 15 with mantissa 7 is NaN). */
double moe_oracle_fp8_value(uint8_t c) {
  const int sign = c >> 7, ex = (c >> 3) & 0xF, man = c & 0x7;
  double mag;
  if (ex == 15 && man == 7) return NAN;
  if (ex == 0)
    mag = ldexp((double)man / 8.0, -6);  /* subnormal: (M/8) 2^(1-7) */
  else
    mag = ldexp(1.0 + (double)man / 8.0, ex - 7);
  return sign ? -mag : mag;
}

/* moe_oracle_fp8_value of every byte, filled once before the first parallel
 * loop that reads fp8 weights (the same values, looked up). */
static double fp8_table[256];
static int fp8_table_ready = 0;

static void fp8_table_fill(void) {
  if (fp8_table_ready) return;
  for (int c = 0; c < 256; ++c) fp8_table[c] = moe_oracle_fp8_value((uint8_t)c);
  fp8_table_ready = 1;
}

/* Element idx of a weight tensor before its channel scale: the bf16 value,
 * the int8 code, the int4 code minus the row's zero point `zero`, or the
 * value of the e4m3 byte. */
static double weight_elem(const moe_oracle_layer_t *L, const void *w, int64_t idx, int zero) {
  if (L->wdtype == 0) return bf16_value(((const uint16_t *)w)[idx]);
  if (L->wdtype == 1) return (double)((const int8_t *)w)[idx];
  if (L->wdtype == 3) return fp8_table[((const uint8_t *)w)[idx]];
  const uint8_t byte = ((const uint8_t *)w)[idx / 2];
  const int q = (idx % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  return (double)(q - zero);
}

/* ---------------------------------------------------------- 1. the router */
/* logits of token t into l[0..E) */
static void router_logits_row(const moe_oracle_layer_t *L, int64_t t, double *l) {
  const uint16_t *xr = L->x + t * (int64_t)L->d;
  for (int e = 0; e < L->E; ++e) {
    const uint16_t *wr = L->wr + (int64_t)e * L->d;
    double acc = 0.0;
    for (int i = 0; i < L->d; ++i) acc += bf16_value(xr[i]) * bf16_value(wr[i]);
    if (L->bias) acc += (double)L->bias[e];
    l[e] = acc;
  }
}

/* ---------------------------------------------------------- 2. top-k gate */
/* 1 if expert (a, ia) ranks before (b, ib) */
static int ranks_before(double a, int ia, double b, int ib) {
  int na = isnan(a), nb = isnan(b);
  if (na != nb) return nb;          /* the number beats the NaN */
  if (na && nb) return ia < ib;
  if (a != b) return a > b;
  return ia < ib;
}

/* Full order of the E experts by insertion sort on ranks_before. */
static void order_experts(int E, const double *l, int *order) {
  for (int e = 0; e < E; ++e) {
    int j = e;
    while (j > 0 && ranks_before(l[e], e, l[order[j - 1]], order[j - 1])) {
      order[j] = order[j - 1];
      --j;
    }
    order[j] = e;
  }
}

/* One token's gate: ids[k], w[k]; gap_k = l(k-1) - l(k) in the sorted order
 * (+inf when k == E), gap_slot = smallest adjacent gap among the k chosen
 * (+inf when k == 1).  raw != 0: the raw-logit gate (w = the logits).
 * Returns 0, or -1 on bad sizes. */
static int gate_common(int E, int k, const double *l, int32_t *ids, double *w,
                       double *gap_k, double *gap_slot, int raw) {
  if (E <= 0 || k <= 0 || k > E) return -1;
  int *order = (int *)malloc(sizeof(int) * (size_t)E);
  if (!order) return -1;
  order_experts(E, l, order);
  double l0 = l[order[0]];
  double den = 0.0;
  for (int s = 0; s < k; ++s) den += exp(l[order[s]] - l0);
  for (int s = 0; s < k; ++s) {
    ids[s] = order[s];
    w[s] = raw ? l[order[s]] : exp(l[order[s]] - l0) / den;
  }
  if (gap_k) *gap_k = (k < E) ? l[order[k - 1]] - l[order[k]] : INFINITY;
  if (gap_slot) {
    double g = INFINITY;
    for (int s = 0; s + 1 < k; ++s) {
      double dg = l[order[s]] - l[order[s + 1]];
      if (dg < g) g = dg;
    }
    *gap_slot = g;
  }
  free(order);
  return 0;
}

int moe_oracle_gate(int E, int k, const double *l, int32_t *ids, double *w,
                    double *gap_k, double *gap_slot) {
  return gate_common(E, k, l, ids, w, gap_k, gap_slot, 0);
}

int moe_oracle_gate_raw(int E, int k, const double *l, int32_t *ids, double *w,
                        double *gap_k, double *gap_slot) {
  return gate_common(E, k, l, ids, w, gap_k, gap_slot, 1);
}

/* int32 conversion of a double: truncation toward zero, saturating at the
 * int32 range, NaN -> 0 */
static int32_t trunc_sat_i32(double v) {
  if (isnan(v)) return 0;
  if (v >= 2147483647.0) return INT32_MAX;
  if (v <= -2147483648.0) return INT32_MIN;
  return (int32_t)v;
}

/* The hash router's expert of one bf16 row (d elements) under W_h
 * [hd][d]: see the header.  Returns -1 on bad sizes. */
int32_t moe_oracle_hash_expert(const uint16_t *xrow, const uint16_t *wh, int d, int hd, int E) {
  if (d <= 0 || hd <= 0 || E <= 0) return -1;
  uint32_t acc = 0;
  for (int i = 0; i < hd; ++i) {
    float r = 0.0f;
    for (int j = 0; j < d; ++j) r += (float)bf16_value(xrow[j]) * (float)bf16_value(wh[(int64_t)i * d + j]);
    acc ^= (uint32_t)trunc_sat_i32((double)r * 1e6) & 0xFFFFFu;
  }
  return (int32_t)(acc % (uint32_t)E);
}

/* The gate of token t under the layer's router; l is scratch of E doubles
 * (left holding the logits, or NaN under the hash router). */
static int gate_token(const moe_oracle_layer_t *L, int64_t t, double *l, int32_t *ids, double *w,
                      double *gap_k, double *gap_slot) {
  if (L->router_mode == ROUTER_HASH) {
    if (L->k != 1 || L->wh == NULL || L->hash_dims <= 0) return -1;
    for (int e = 0; e < L->E; ++e) l[e] = NAN;
    ids[0] = moe_oracle_hash_expert(L->x + t * (int64_t)L->d, L->wh, L->d, L->hash_dims, L->E);
    w[0] = 1.0;
    if (gap_k) *gap_k = INFINITY;
    if (gap_slot) *gap_slot = INFINITY;
    return ids[0] < 0 ? -1 : 0;
  }
  if (L->router_mode != ROUTER_SOFTMAX && L->router_mode != ROUTER_RAW) return -1;
  router_logits_row(L, t, l);
  return gate_common(L->E, L->k, l, ids, w, gap_k, gap_slot, L->router_mode == ROUTER_RAW);
}

/* Route tokens tokens[0..n) (or 0..n when tokens == NULL).  Outputs are
 * indexed by position in the list; logits may be NULL. */
int moe_oracle_route(const moe_oracle_layer_t *L, const int32_t *tokens, int64_t n,
                     double *logits, int32_t *ids, double *w, double *gap_k, double *gap_slot) {
  int bad = 0;
  #pragma omp parallel
  {
    double *l = (double *)malloc(sizeof(double) * (size_t)L->E);
    #pragma omp for schedule(dynamic, 16)
    for (int64_t p = 0; p < n; ++p) {
      int64_t t = tokens ? tokens[p] : p;
      if (!l || t < 0 || t >= L->T) { bad = 1; continue; }
      if (gate_token(L, t, l, ids + p * L->k, w + p * L->k, gap_k ? gap_k + p : NULL,
                     gap_slot ? gap_slot + p : NULL))
        bad = 1;
      if (logits) memcpy(logits + p * L->E, l, sizeof(double) * (size_t)L->E);
    }
    free(l);
  }
  return bad ? -1 : 0;
}

/* ---------------------------------------------------------- 3. dispatch */
/* Counting sort of the T*k (token, slot) pairs by expert, stable in token
 * order.  cnt[E], off[E+1], tok[T*k], inv[T*k].  Returns -1 on an id out of
 * range or a token holding one expert twice. */
int moe_oracle_dispatch(int64_t T, int E, int k, const int32_t *ids,
                        int32_t *cnt, int32_t *off, int32_t *tok, int32_t *inv) {
  if (E <= 0 || k <= 0 || T < 0) return -1;
  for (int e = 0; e < E; ++e) cnt[e] = 0;
  for (int64_t t = 0; t < T; ++t)
    for (int s = 0; s < k; ++s) {
      int32_t e = ids[t * k + s];
      if (e < 0 || e >= E) return -1;
      for (int s2 = 0; s2 < s; ++s2)
        if (ids[t * k + s2] == e) return -1;
      cnt[e] += 1;
    }
  off[0] = 0;
  for (int e = 0; e < E; ++e) off[e + 1] = off[e] + cnt[e];
  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -1;
  for (int64_t t = 0; t < T; ++t)
    for (int s = 0; s < k; ++s) {
      int32_t e = ids[t * k + s];
      int32_t r = off[e] + fill[e]++;
      tok[r] = (int32_t)t;
      inv[t * k + s] = r;
    }
  free(fill);
  return 0;
}

/* ---------------------------------------------------------- 4. one expert */
/* y[d] = FFN_e(xrow).  h is scratch of f doubles. */
static void expert_row(const moe_oracle_layer_t *L, int e, const double *xv, int mode,
                       double *h, double *y) {
  const int d = L->d, f = L->f;
  const int64_t gbase = (int64_t)e * f * d, dbase = (int64_t)e * d * f;
  const int int4 = L->wdtype == 2;
  for (int j = 0; j < f; ++j) {
    double g = 0.0, u = 0.0;
    const int zg = int4 ? L->zg[(int64_t)e * f + j] : 0, zu = int4 ? L->zu[(int64_t)e * f + j] : 0;
    for (int i = 0; i < d; ++i) {
      g += xv[i] * weight_elem(L, L->wg, gbase + (int64_t)j * d + i, zg);
      u += xv[i] * weight_elem(L, L->wu, gbase + (int64_t)j * d + i, zu);
    }
    if (L->wdtype != 0) {
      g *= (double)L->sg[(int64_t)e * f + j];
      u *= (double)L->su[(int64_t)e * f + j];
    }
    double silu = g / (1.0 + exp(-g));
    double hj = silu * u;
    h[j] = (mode == ORACLE_BF16H) ? moe_oracle_round_bf16(hj) : hj;
  }
  for (int c = 0; c < d; ++c) {
    double acc = 0.0;
    const int zd = int4 ? L->zd[(int64_t)e * d + c] : 0;
    for (int j = 0; j < f; ++j) acc += h[j] * weight_elem(L, L->wd, dbase + (int64_t)c * f + j, zd);
    if (L->wdtype != 0) acc *= (double)L->sd[(int64_t)e * d + c];
    y[c] = acc;
  }
}

/* Expert e applied to an arbitrary bf16 row (d elements). */
void moe_oracle_expert(const moe_oracle_layer_t *L, int e, const uint16_t *xrow, int mode, double *y) {
  fp8_table_fill();
  double *xv = (double *)malloc(sizeof(double) * (size_t)L->d);
  double *h = (double *)malloc(sizeof(double) * (size_t)L->f);
  for (int i = 0; i < L->d; ++i) xv[i] = bf16_value(xrow[i]);
  expert_row(L, e, xv, mode, h, y);
  free(xv);
  free(h);
}

/* ---------------------------------------------------------- 5. the layer */
/* Layer output for tokens[0..n) (all tokens when NULL): out[n][d] in double,
 * plus the gate's ids[n][k] and w[n][k] (either may be NULL). */
int moe_oracle_forward(const moe_oracle_layer_t *L, const int32_t *tokens, int64_t n, int mode,
                       double *out, int32_t *ids_out, double *w_out) {
  const int d = L->d, E = L->E, k = L->k;
  int bad = 0;
  fp8_table_fill();
  #pragma omp parallel
  {
    double *l = (double *)malloc(sizeof(double) * (size_t)E);
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)L->f);
    double *y = (double *)malloc(sizeof(double) * (size_t)d);
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    double *w = (double *)malloc(sizeof(double) * (size_t)k);
    #pragma omp for schedule(dynamic, 1)
    for (int64_t p = 0; p < n; ++p) {
      int64_t t = tokens ? tokens[p] : p;
      if (!l || !xv || !h || !y || !ids || !w || t < 0 || t >= L->T) { bad = 1; continue; }
      if (gate_token(L, t, l, ids, w, NULL, NULL)) { bad = 1; continue; }
      for (int i = 0; i < d; ++i) xv[i] = bf16_value(L->x[t * (int64_t)d + i]);
      double *o = out + p * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int s = 0; s < k; ++s) {
        expert_row(L, ids[s], xv, mode, h, y);
        for (int c = 0; c < d; ++c) o[c] += w[s] * y[c];
      }
      if (ids_out) memcpy(ids_out + p * k, ids, sizeof(int32_t) * (size_t)k);
      if (w_out) memcpy(w_out + p * k, w, sizeof(double) * (size_t)k);
    }
    free(l); free(xv); free(h); free(y); free(ids); free(w);
  }
  return bad ? -1 : 0;
}
