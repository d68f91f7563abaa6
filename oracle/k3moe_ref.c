/* k3moe_ref.c -- ORACLE (test infrastructure only) for the routed MoE expert FFN.
 * Plain C99, one thread, float64 arithmetic.  Sources and readings: k3moe_ref.h. */
#include "k3moe_ref.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static int shape_ok(k3ref_shape s) {
  return s.T >= 0 && s.H > 0 && s.I > 0 && s.E > 0 && s.k > 0 && s.k <= s.E && s.H % 32 == 0 &&
         s.I % 32 == 0;
}

/* E2M1 per [OCP-MX]: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * exponent 0 is subnormal: m * 2^-1; otherwise 2^(e-1) * (1 + m/2). */
double k3ref_e2m1(unsigned code) {
  const unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  const double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

/* E8M0 per [OCP-MX]: an unsigned biased exponent, 2^(byte-127); 0xFF is NaN. */
double k3ref_e8m0(unsigned byte) {
  if ((byte & 0xFFu) == 0xFFu) return NAN;
  return ldexp(1.0, (int)(byte & 0xFFu) - 127);
}

/* bf16 = the upper 16 bits of an IEEE binary32. */
double k3ref_bf16_value(uint16_t bits) {
  const uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 (8 significant bits, exponent range of
 * binary32, subnormal quantum 2^-133), ties to even; overflow gives inf. */
uint16_t k3ref_bf16_rne(double v) {
  if (isnan(v)) return (uint16_t)0x7FC0;
  const uint16_t sign = signbit(v) ? (uint16_t)0x8000 : (uint16_t)0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int ex;
  (void)frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  int q = ex - 8;      /* quantum of an 8-significant-bit value */
  if (q < -133) q = -133;
  const double r = ldexp(rint(ldexp(a, -q)), q); /* rint: round to nearest, ties even */
  const double bf16_max = ldexp(255.0, 120);      /* (2 - 2^-7) * 2^127 */
  if (r > bf16_max) return (uint16_t)(sign | 0x7F80);
  const float f = (float)r; /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFFu));
}

double k3ref_silu(double z) { return z / (1.0 + exp(-z)); }

/* Round a non-negative magnitude onto the E2M1 grid {0,.5,1,1.5,2,3,4,6},
 * nearest, ties to the even code, saturating at 6.  Returns the 3-bit code. */
static unsigned e2m1_round_mag(double q) {
  static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  if (q >= 6.0) return 7u;
  unsigned lo = 0;
  while (lo < 7 && grid[lo + 1] <= q) ++lo;
  if (grid[lo] == q) return lo;
  const double dlo = q - grid[lo], dhi = grid[lo + 1] - q;
  if (dlo < dhi) return lo;
  if (dhi < dlo) return lo + 1;
  return (lo % 2u == 0u) ? lo : lo + 1; /* tie: even code */
}

/* MXFP4 quantisation per [OCP-MX] section on conversion to MX formats:
 * X = 2^(floor(log2(amax)) - 2), clamped to the E8M0 range; element = RNE(v / X)
 * on the E2M1 grid with saturation; an all-zero block gets scale byte 0. */
void k3ref_quant_mxfp4(const uint16_t *v, int n, uint8_t *codes, uint8_t *scales) {
  for (int b = 0; b < n / 32; ++b) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) {
      const double a = fabs(k3ref_bf16_value(v[b * 32 + i]));
      if (a > amax) amax = a;
    }
    int shared = -127;
    if (amax > 0.0) {
      int ex;
      (void)frexp(amax, &ex);  /* floor(log2(amax)) = ex - 1 */
      shared = (ex - 1) - 2;
      if (shared < -127) shared = -127;
      if (shared > 127) shared = 127;
    }
    scales[b] = (uint8_t)(shared + 127);
    for (int i = 0; i < 32; ++i) {
      const double val = k3ref_bf16_value(v[b * 32 + i]);
      unsigned c = e2m1_round_mag(ldexp(fabs(val), -shared));
      if (val < 0.0) c |= 8u;
      const int e = b * 32 + i;
      if (e % 2 == 0)
        codes[e / 2] = (uint8_t)c;
      else
        codes[e / 2] = (uint8_t)(codes[e / 2] | (c << 4));
    }
  }
}

/* ---- routing: top-k of E by (logit descending, index ascending), then a
 * softmax over the selected logits ([changelog] "[0.1.0] Added": 896 routed
 * experts with top-16 selection; [article] "01": 16 of 896 woken). ---- */
typedef struct {
  float v;
  int32_t e;
} scored;

static int cmp_scored(const void *pa, const void *pb) {
  const scored *a = (const scored *)pa, *b = (const scored *)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->e < b->e) ? -1 : (a->e > b->e);
}

int k3ref_route(k3ref_shape s, const float *logits, int32_t *idx, double *w, int32_t *row_bad) {
  if (!shape_ok(s)) return -1;
  scored *buf = (scored *)malloc(sizeof(scored) * (size_t)s.E);
  if (!buf) return -1;
  int nbad = 0;
  for (int t = 0; t < s.T; ++t) {
    const float *l = logits + (size_t)t * s.E;
    int bad = 0;
    for (int e = 0; e < s.E; ++e) {
      if (isnan(l[e])) bad = 1;
      buf[e].v = l[e];
      buf[e].e = e;
    }
    int32_t *it = idx + (size_t)t * s.k;
    double *wt = w + (size_t)t * s.k;
    if (row_bad) row_bad[t] = bad;
    if (bad) {
      ++nbad;
      for (int j = 0; j < s.k; ++j) {
        it[j] = j;
        wt[j] = 1.0 / s.k;
      }
      continue;
    }
    qsort(buf, (size_t)s.E, sizeof(scored), cmp_scored);
    for (int j = 0; j < s.k; ++j) it[j] = buf[j].e;
    const double m = (double)buf[0].v; /* the row maximum */
    if (isinf(m) && m < 0) {           /* all -inf */
      for (int j = 0; j < s.k; ++j) wt[j] = 1.0 / s.k;
    } else if (isinf(m)) { /* limit of the softmax: the +inf picks share the weight */
      int ninf = 0;
      for (int j = 0; j < s.k; ++j) ninf += isinf(buf[j].v) && buf[j].v > 0;
      for (int j = 0; j < s.k; ++j) wt[j] = (isinf(buf[j].v) && buf[j].v > 0) ? 1.0 / ninf : 0.0;
    } else {
      double z = 0.0;
      for (int j = 0; j < s.k; ++j) z += exp((double)buf[j].v - m);
      for (int j = 0; j < s.k; ++j) wt[j] = exp((double)buf[j].v - m) / z;
    }
  }
  free(buf);
  return nbad;
}

/* ---- router: the score of every expert for every token, the input of the
 * top-16-of-896 selection ([changelog] "[0.1.0] Added"; [article] "01").  The
 * score is the linear form x . wr[e]; bf16 products are exact in double and
 * the sum runs in ascending h. ---- */
int k3ref_router_logits(k3ref_shape s, const uint16_t *x, const uint16_t *wr, double *logits) {
  if (!shape_ok(s)) return -1;
  double *xv = (double *)malloc(sizeof(double) * (size_t)s.H);
  if (!xv) return -1;
  for (int t = 0; t < s.T; ++t) {
    for (int h = 0; h < s.H; ++h) xv[h] = k3ref_bf16_value(x[(size_t)t * s.H + h]);
    for (int e = 0; e < s.E; ++e) {
      const uint16_t *row = wr + (size_t)e * s.H;
      double acc = 0.0;
      for (int h = 0; h < s.H; ++h) acc += xv[h] * k3ref_bf16_value(row[h]);
      logits[(size_t)t * s.E + e] = acc;
    }
  }
  free(xv);
  return 0;
}

int k3ref_router(k3ref_shape s, const uint16_t *x, const uint16_t *wr, double *logits, float *logits_f32,
                 int32_t *idx, double *w, int32_t *row_bad) {
  if (!shape_ok(s)) return -1;
  const size_t n = (size_t)s.T * s.E;
  double *l64 = (double *)malloc(sizeof(double) * (n ? n : 1));
  float *l32 = (float *)malloc(sizeof(float) * (n ? n : 1));
  int rc = -1;
  if (l64 && l32 && k3ref_router_logits(s, x, wr, l64) == 0) {
    for (size_t i = 0; i < n; ++i) l32[i] = (float)l64[i]; /* one rounding, to nearest even */
    rc = k3ref_route(s, l32, idx, w, row_bad);
    if (logits) memcpy(logits, l64, sizeof(double) * n);
    if (logits_f32) memcpy(logits_f32, l32, sizeof(float) * n);
  }
  free(l64);
  free(l32);
  return rc;
}

/* ---- bucketing: a stable counting sort of assignment ids a = t*k + j by the
 * routed expert idx[a] ([changelog] "[1.0.0] Added", chunk-union prefill: the
 * tokens of a chunk are grouped by routed expert so each unique expert is read
 * once). ---- */
int k3ref_bucket(k3ref_shape s, const int32_t *idx, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *inv) {
  if (!shape_ok(s)) return -1;
  const int A = s.T * s.k;
  for (int e = 0; e < s.E; ++e) counts[e] = 0;
  for (int a = 0; a < A; ++a) {
    if (idx[a] < 0 || idx[a] >= s.E) return -1;
    counts[idx[a]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < s.E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)s.E);
  if (!fill) return -1;
  for (int e = 0; e < s.E; ++e) fill[e] = offsets[e];
  for (int a = 0; a < A; ++a) { /* ascending a: stable */
    const int p = fill[idx[a]]++;
    perm[p] = a;
    inv[a] = p;
  }
  free(fill);
  return 0;
}

/* Row r of an MXFP4 matrix with K columns, decoded to doubles:
 * W[r][c] = E2M1(code(r,c)) * E8M0(scale[r][c/32])
 * ([overview] "layer one": half a byte per weight; [OCP-MX] block of 32).
 * The E2M1 values come from k3ref_e2m1 through a 16-entry cache. */
static void mx_row(const uint8_t *codes, const uint8_t *scales, int K, int r, double *row) {
  static double e2m1_cache[16];
  static int cached = 0;
  if (!cached) {
    for (unsigned q = 0; q < 16; ++q) e2m1_cache[q] = k3ref_e2m1(q);
    cached = 1;
  }
  double scale = 0.0;
  for (int c = 0; c < K; ++c) {
    if (c % 32 == 0) scale = k3ref_e8m0(scales[(size_t)r * (K / 32) + c / 32]);
    const uint8_t byte = codes[(size_t)r * (K / 2) + c / 2];
    const unsigned nib = (c % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
    row[c] = e2m1_cache[nib] * scale;
  }
}

/* Activation vector of n bf16 values as doubles; with a4 the values are first
 * quantised to MXFP4 and decoded back (exact). */
static void activation_values(const uint16_t *v, int n, int a4, double *out) {
  if (!a4) {
    for (int i = 0; i < n; ++i) out[i] = k3ref_bf16_value(v[i]);
    return;
  }
  uint8_t *codes = (uint8_t *)malloc((size_t)n / 2);
  uint8_t *sc = (uint8_t *)malloc((size_t)n / 32);
  k3ref_quant_mxfp4(v, n, codes, sc);
  for (int i = 0; i < n; ++i) {
    const unsigned nib = (i % 2 == 0) ? (codes[i / 2] & 0xFu) : (codes[i / 2] >> 4);
    out[i] = k3ref_e2m1(nib) * k3ref_e8m0(sc[i / 32]);
  }
  free(codes);
  free(sc);
}

static int expert_present(int e, const uint8_t *const *w13c, const uint8_t *const *w13s,
                          const uint8_t *const *w2c, const uint8_t *const *w2s) {
  return w13c[e] && w13s[e] && w2c[e] && w2s[e];
}

/* Gate/up half of one expert on one token: g = Wg x, u = Wu x, hpre = silu(g) u
 * in double, h = bf16(hpre) ([changelog] "[0.1.0] Added": GLU expert with MXFP4
 * weights).  Optional outputs (NULL to skip): hpre; g and u; gabs = sum |Wg x|
 * and uabs = sum |Wu x| (the magnitudes that bound a finite-precision sum). */
static void expert_gateup(k3ref_shape s, const double *xv, const uint8_t *w13c, const uint8_t *w13s,
                          uint16_t *h_bits, double *hpre, double *g_out, double *u_out, double *gabs,
                          double *uabs) {
  double *wg = (double *)malloc(sizeof(double) * (size_t)s.H);
  double *wu = (double *)malloc(sizeof(double) * (size_t)s.H);
  for (int r = 0; r < s.I; ++r) {
    mx_row(w13c, w13s, s.H, r, wg);        /* gate row r */
    mx_row(w13c, w13s, s.H, s.I + r, wu);  /* up row r   */
    double g = 0.0, u = 0.0, ga = 0.0, ua = 0.0;
    for (int c = 0; c < s.H; ++c) {
      g += wg[c] * xv[c];
      u += wu[c] * xv[c];
      ga += fabs(wg[c] * xv[c]);
      ua += fabs(wu[c] * xv[c]);
    }
    const double v = k3ref_silu(g) * u;
    if (hpre) hpre[r] = v;
    if (g_out) g_out[r] = g;
    if (u_out) u_out[r] = u;
    if (gabs) gabs[r] = ga;
    if (uabs) uabs[r] = ua;
    h_bits[r] = k3ref_bf16_rne(v);
  }
  free(wg);
  free(wu);
}

/* Down half: y = W2 h, with h the bf16 row (quantised to MXFP4 first with a4). */
static void expert_down(k3ref_shape s, const uint16_t *h_bits, const uint8_t *w2c, const uint8_t *w2s, int a4,
                        double *hv, double *y) {
  double *wd = (double *)malloc(sizeof(double) * (size_t)s.I);
  activation_values(h_bits, s.I, a4, hv);
  for (int r = 0; r < s.H; ++r) {
    mx_row(w2c, w2s, s.I, r, wd);
    double acc = 0.0;
    for (int c = 0; c < s.I; ++c) acc += wd[c] * hv[c];
    y[r] = acc;
  }
  free(wd);
}

/* One expert FFN on one token: the gate/up half, then the down half on its h. */
static void expert_apply(k3ref_shape s, const double *xv, const uint8_t *w13c,
                         const uint8_t *w13s, const uint8_t *w2c, const uint8_t *w2s, int a4,
                         uint16_t *h_bits, double *hv, double *y) {
  expert_gateup(s, xv, w13c, w13s, h_bits, NULL, NULL, NULL, NULL, NULL);
  expert_down(s, h_bits, w2c, w2s, a4, hv, y);
}

int k3ref_expert_gateup(k3ref_shape s, const uint16_t *x, const uint8_t *const *w13c,
                        const uint8_t *const *w13s, const uint8_t *const *w2c,
                        const uint8_t *const *w2s, const int32_t *offsets, const int32_t *perm,
                        int a4, double *hpre, uint16_t *h, double *g, double *u, double *gabs,
                        double *uabs) {
  if (!shape_ok(s)) return -1;
  double *xv = (double *)malloc(sizeof(double) * (size_t)s.H);
  if (!xv) return -1;
  for (int e = 0; e < s.E; ++e) {
    const int present = expert_present(e, w13c, w13s, w2c, w2s);
    for (int p = offsets[e]; p < offsets[e + 1]; ++p) {
      const size_t o = (size_t)p * s.I;
      if (!present) { /* [changelog] "[Unreleased] Fixed": a missing expert adds zero */
        for (int i = 0; i < s.I; ++i) {
          hpre[o + i] = 0.0;
          h[o + i] = 0;
          if (g) g[o + i] = 0.0;
          if (u) u[o + i] = 0.0;
          if (gabs) gabs[o + i] = 0.0;
          if (uabs) uabs[o + i] = 0.0;
        }
        continue;
      }
      activation_values(x + (size_t)(perm[p] / s.k) * s.H, s.H, a4, xv);
      expert_gateup(s, xv, w13c[e], w13s[e], h + o, hpre + o, g ? g + o : NULL, u ? u + o : NULL,
                    gabs ? gabs + o : NULL, uabs ? uabs + o : NULL);
    }
  }
  free(xv);
  return 0;
}

int k3ref_expert_down(k3ref_shape s, const uint16_t *h, const uint8_t *const *w13c,
                      const uint8_t *const *w13s, const uint8_t *const *w2c,
                      const uint8_t *const *w2s, const int32_t *offsets, int a4, double *Y) {
  if (!shape_ok(s)) return -1;
  double *hv = (double *)malloc(sizeof(double) * (size_t)s.I);
  if (!hv) return -1;
  for (int e = 0; e < s.E; ++e) {
    const int present = expert_present(e, w13c, w13s, w2c, w2s);
    for (int p = offsets[e]; p < offsets[e + 1]; ++p) {
      double *y = Y + (size_t)p * s.H;
      if (!present) {
        for (int r = 0; r < s.H; ++r) y[r] = 0.0;
        continue;
      }
      expert_down(s, h + (size_t)p * s.I, w2c[e], w2s[e], a4, hv, y);
    }
  }
  free(hv);
  return 0;
}

int k3ref_expert_ffn(k3ref_shape s, const uint16_t *x, const uint8_t *const *w13c,
                     const uint8_t *const *w13s, const uint8_t *const *w2c,
                     const uint8_t *const *w2s, const int32_t *offsets, const int32_t *perm,
                     int a4, double *Y, uint16_t *h_out) {
  if (!shape_ok(s)) return -1;
  double *xv = (double *)malloc(sizeof(double) * (size_t)s.H);
  double *hv = (double *)malloc(sizeof(double) * (size_t)s.I);
  uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)s.I);
  if (!xv || !hv || !hb) return -1;
  for (int e = 0; e < s.E; ++e) {
    const int present = expert_present(e, w13c, w13s, w2c, w2s);
    for (int p = offsets[e]; p < offsets[e + 1]; ++p) {
      double *y = Y + (size_t)p * s.H;
      if (!present) { /* [changelog] "[Unreleased] Fixed": a missing expert adds zero */
        for (int r = 0; r < s.H; ++r) y[r] = 0.0;
        if (h_out) memset(h_out + (size_t)p * s.I, 0, sizeof(uint16_t) * (size_t)s.I);
        continue;
      }
      const int t = perm[p] / s.k;
      activation_values(x + (size_t)t * s.H, s.H, a4, xv);
      expert_apply(s, xv, w13c[e], w13s[e], w2c[e], w2s[e], a4, hb, hv, y);
      if (h_out) memcpy(h_out + (size_t)p * s.I, hb, sizeof(uint16_t) * (size_t)s.I);
    }
  }
  free(xv);
  free(hv);
  free(hb);
  return 0;
}

/* Routing-weighted sum of the k expert outputs of each token, in j order
 * ([article] "02": one fixed accumulation order). */
int k3ref_combine(k3ref_shape s, const double *Y, const double *w, const int32_t *inv, double *out,
                  uint16_t *out_bf16) {
  if (!shape_ok(s)) return -1;
  for (int t = 0; t < s.T; ++t) {
    for (int c = 0; c < s.H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < s.k; ++j)
        acc += w[(size_t)t * s.k + j] * Y[(size_t)inv[t * s.k + j] * s.H + c];
      out[(size_t)t * s.H + c] = acc;
      if (out_bf16) out_bf16[(size_t)t * s.H + c] = k3ref_bf16_rne(acc);
    }
  }
  return 0;
}

int k3ref_moe_token(k3ref_shape s, const uint16_t *x_row, const int32_t *idx_row,
                    const double *w_row, const uint8_t *const *w13c, const uint8_t *const *w13s,
                    const uint8_t *const *w2c, const uint8_t *const *w2s, int a4, double *out_row) {
  if (!shape_ok(s)) return -1;
  double *xv = (double *)malloc(sizeof(double) * (size_t)s.H);
  double *hv = (double *)malloc(sizeof(double) * (size_t)s.I);
  double *y = (double *)malloc(sizeof(double) * (size_t)s.H);
  uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)s.I);
  if (!xv || !hv || !y || !hb) return -1;
  activation_values(x_row, s.H, a4, xv);
  for (int c = 0; c < s.H; ++c) out_row[c] = 0.0;
  for (int j = 0; j < s.k; ++j) {
    const int e = idx_row[j];
    if (e < 0 || e >= s.E) return -1;
    if (!expert_present(e, w13c, w13s, w2c, w2s)) {
      for (int c = 0; c < s.H; ++c) y[c] = 0.0;
    } else {
      expert_apply(s, xv, w13c[e], w13s[e], w2c[e], w2s[e], a4, hb, hv, y);
    }
    for (int c = 0; c < s.H; ++c) out_row[c] += w_row[j] * y[c];
  }
  free(xv);
  free(hv);
  free(y);
  free(hb);
  return 0;
}

int k3ref_moe_layer(k3ref_shape s, const float *logits, const uint16_t *x,
                    const uint8_t *const *w13c, const uint8_t *const *w13s,
                    const uint8_t *const *w2c, const uint8_t *const *w2s, int a4, double *out,
                    uint16_t *out_bf16) {
  if (!shape_ok(s)) return -1;
  const size_t A = (size_t)s.T * s.k;
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (A ? A : 1));
  double *w = (double *)malloc(sizeof(double) * (A ? A : 1));
  int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)s.E);
  int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * ((size_t)s.E + 1));
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (A ? A : 1));
  int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * (A ? A : 1));
  double *Y = (double *)malloc(sizeof(double) * (A ? A : 1) * (size_t)s.H);
  int rc = -1;
  if (idx && w && counts && offsets && perm && inv && Y && k3ref_route(s, logits, idx, w, NULL) >= 0 &&
      k3ref_bucket(s, idx, counts, offsets, perm, inv) == 0 &&
      k3ref_expert_ffn(s, x, w13c, w13s, w2c, w2s, offsets, perm, a4, Y, NULL) == 0 &&
      k3ref_combine(s, Y, w, inv, out, out_bf16) == 0)
    rc = 0;
  free(idx);
  free(w);
  free(counts);
  free(offsets);
  free(perm);
  free(inv);
  free(Y);
  return rc;
}
