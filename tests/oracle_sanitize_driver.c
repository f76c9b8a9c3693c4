/*
 * Test driver that runs the fp64 oracle under AddressSanitizer and
 * UndefinedBehaviorSanitizer (built by tests/test_oracle_sanitizers.py).
 * It compiles the oracle's source into this one translation unit and calls
 * every entry point on small layers of each weight format (bf16, int8, int4,
 * fp8) and router mode (softmax, raw logits, hash), with every buffer
 * allocated at its exact size so that an access past one is reported.
 * Inputs come from a fixed linear congruential sequence: this checks memory
 * and arithmetic safety, not values (the pins do that).
 */
#include "../oracle/moe_oracle.c"

#include <stdio.h>

static uint64_t rng = 0x2545F4914F6CDD1Dull;

static uint32_t next_u32(void) {
  rng = rng * 6364136223846793005ull + 1442695040888963407ull;
  return (uint32_t)(rng >> 32);
}

/* a value in [-scale, scale) as bf16 bits (truncated) */
static uint16_t rand_bf16(float scale) {
  float f = ((float)(next_u32() >> 8) / 16777216.0f * 2.0f - 1.0f) * scale;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

static void *xmalloc(size_t n) {
  void *p = malloc(n ? n : 1);
  if (!p) {
    fprintf(stderr, "out of memory\n");
    exit(2);
  }
  return p;
}

static int run_layer(int wdtype, int router_mode) {
  const int T = 7, d = 16, f = 24, E = 5;
  const int k = router_mode == 2 ? 1 : 2, hd = router_mode == 2 ? 3 : 0;
  const size_t nw_gu = (size_t)E * f * d, nw_d = (size_t)E * d * f;
  uint16_t *x = xmalloc(sizeof(uint16_t) * (size_t)T * d);
  uint16_t *wr = xmalloc(sizeof(uint16_t) * (size_t)E * d);
  uint16_t *wh = hd ? xmalloc(sizeof(uint16_t) * (size_t)hd * d) : NULL;
  float *bias = xmalloc(sizeof(float) * (size_t)E);
  for (int i = 0; i < T * d; ++i) x[i] = rand_bf16(1.0f);
  for (int i = 0; i < E * d; ++i) wr[i] = rand_bf16(0.3f);
  for (int i = 0; i < hd * d; ++i) wh[i] = rand_bf16(0.3f);
  for (int e = 0; e < E; ++e) bias[e] = (float)e * -0.25f;

  void *wg, *wu, *wd;
  float *sg = NULL, *su = NULL, *sd = NULL;
  uint8_t *zg = NULL, *zu = NULL, *zd = NULL;
  if (wdtype == 0) {
    uint16_t *a = xmalloc(2 * nw_gu), *b = xmalloc(2 * nw_gu), *c = xmalloc(2 * nw_d);
    for (size_t i = 0; i < nw_gu; ++i) a[i] = rand_bf16(0.2f), b[i] = rand_bf16(0.2f);
    for (size_t i = 0; i < nw_d; ++i) c[i] = rand_bf16(0.2f);
    wg = a, wu = b, wd = c;
  } else {
    const size_t bg = wdtype == 2 ? nw_gu / 2 : nw_gu, bd = wdtype == 2 ? nw_d / 2 : nw_d;
    uint8_t *a = xmalloc(bg), *b = xmalloc(bg), *c = xmalloc(bd);
    for (size_t i = 0; i < bg; ++i) a[i] = (uint8_t)next_u32(), b[i] = (uint8_t)next_u32();
    for (size_t i = 0; i < bd; ++i) c[i] = (uint8_t)next_u32();
    if (wdtype == 3) /* e4m3: no NaN bytes */
      for (size_t i = 0; i < bg; ++i) {
        if ((a[i] & 0x7F) == 0x7F) a[i] ^= 1;
        if ((b[i] & 0x7F) == 0x7F) b[i] ^= 1;
        if (i < bd && (c[i] & 0x7F) == 0x7F) c[i] ^= 1;
      }
    wg = a, wu = b, wd = c;
    sg = xmalloc(sizeof(float) * (size_t)E * f);
    su = xmalloc(sizeof(float) * (size_t)E * f);
    sd = xmalloc(sizeof(float) * (size_t)E * d);
    for (int i = 0; i < E * f; ++i) sg[i] = 1e-3f, su[i] = 2e-3f;
    for (int i = 0; i < E * d; ++i) sd[i] = 1.5e-3f;
    if (wdtype == 2) {
      zg = xmalloc((size_t)E * f), zu = xmalloc((size_t)E * f), zd = xmalloc((size_t)E * d);
      for (int i = 0; i < E * f; ++i) zg[i] = (uint8_t)(next_u32() & 15), zu[i] = (uint8_t)(next_u32() & 15);
      for (int i = 0; i < E * d; ++i) zd[i] = (uint8_t)(next_u32() & 15);
    }
  }
  moe_oracle_layer_t L = {T, d, f, E, k, wdtype, x, wr, router_mode == 2 ? NULL : bias, wg, wu, wd, sg, su, sd,
                          router_mode, hd, wh, zg, zu, zd};

  int bad = 0;
  double *out = xmalloc(sizeof(double) * (size_t)T * d);
  int32_t *ids = xmalloc(sizeof(int32_t) * (size_t)T * k);
  double *w = xmalloc(sizeof(double) * (size_t)T * k);
  for (int mode = 0; mode < 2; ++mode) bad |= moe_oracle_forward(&L, NULL, T, mode, out, ids, w) != 0;
  const int32_t list[3] = {6, 0, 3};
  bad |= moe_oracle_forward(&L, list, 3, 1, out, ids, w) != 0;
  if (router_mode != 2) {
    double *lg = xmalloc(sizeof(double) * (size_t)T * E), *gk = xmalloc(sizeof(double) * T),
           *gs = xmalloc(sizeof(double) * T);
    bad |= moe_oracle_route(&L, NULL, T, lg, ids, w, gk, gs) != 0;
    free(lg), free(gk), free(gs);
  }
  int32_t *cnt = xmalloc(sizeof(int32_t) * E), *off = xmalloc(sizeof(int32_t) * (E + 1));
  int32_t *tok = xmalloc(sizeof(int32_t) * (size_t)T * k), *inv = xmalloc(sizeof(int32_t) * (size_t)T * k);
  bad |= moe_oracle_forward(&L, NULL, T, 1, out, ids, w) != 0;
  bad |= moe_oracle_dispatch(T, E, k, ids, cnt, off, tok, inv) != 0;
  double *y = xmalloc(sizeof(double) * d);
  for (int e = 0; e < E; ++e) moe_oracle_expert(&L, e, x + (size_t)(e % T) * d, e & 1, y);
  if (hd) (void)moe_oracle_hash_expert(x, wh, d, hd, E);

  free(y), free(cnt), free(off), free(tok), free(inv), free(out), free(ids), free(w);
  free(wg), free(wu), free(wd), free(sg), free(su), free(sd), free(zg), free(zu), free(zd);
  free(x), free(wr), free(wh), free(bias);
  return bad;
}

int main(void) {
  int bad = 0;
  moe_oracle_set_threads(2);
  for (int wdtype = 0; wdtype < 4; ++wdtype)
    for (int rm = 0; rm < 3; ++rm) bad |= run_layer(wdtype, rm);
  /* the gate on ties, zeros of both signs, infinities and NaN */
  const double l[6] = {1.0, 1.0, -0.0, 0.0, NAN, -INFINITY};
  int32_t ids[6];
  double w[6], gk, gs;
  bad |= moe_oracle_gate(6, 6, l, ids, w, &gk, &gs) != 0;
  bad |= moe_oracle_gate_raw(6, 3, l, ids, w, &gk, &gs) != 0;
  for (int c = 0; c < 256; ++c) (void)moe_oracle_fp8_value((uint8_t)c);
  const double specials[5] = {INFINITY, -INFINITY, NAN, 0x1p-140, -3.0e38};
  for (int i = 0; i < 5; ++i) (void)moe_oracle_bf16_bits(specials[i]);
  printf(bad ? "oracle call failed\n" : "ok\n");
  return bad;
}
