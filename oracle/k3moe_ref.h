/* k3moe_ref.h -- ORACLE for the routed MoE expert FFN with MXFP4 experts.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded C99
 * implementation written from the definition of the method.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no code with the CUDA library (no headers, tables or helpers) and the CUDA
 * library never calls it.
 *
 * Sources (web pages about the kimi-k3-in-c engine; cited by title + section):
 *  [changelog]  "kimi-k3-in-c CHANGELOG walkthrough" (m.qwbw.cn/news/81998):
 *               block "[0.1.0] Added" (896 routed experts, top-16 selection,
 *               the GLU expert activation, native MXFP4 expert weights, a
 *               matmul that consumes packed nibbles directly); block
 *               "[1.0.0] Added" (chunk-union prefill: each routed unique expert
 *               fetched once per chunk, tokens bit-identical to the per-token
 *               path); block "[Unreleased] Fixed" (an expert that fails to
 *               load contributes zero, never uninitialised memory).
 *  [article]    "kimi-k3-in-c: pure C99 Kimi K3 inference engine" (chenxutan.com),
 *               section "01 four-fold compression": 896 experts per layer,
 *               16 woken per token; section "02 no dependencies": fixed
 *               accumulation order.
 *  [overview]   "kimi-k3-in-c" (pomoai.com), section "layer one: the experts
 *               are already half a byte (MXFP4)".
 *  [OCP-MX]     OCP Microscaling Formats (MX) Specification v1.0: the E2M1
 *               element encoding, the E8M0 shared scale, 32-element blocks,
 *               and the conversion rule (shared exponent = floor(log2 amax)
 *               minus the element format's largest exponent, 2 for E2M1).
 *
 * Readings taken where the pages are silent (each is a choice, listed in the
 * design notes of the repository):
 *  - routing: softmax over the router logits restricted to the top-k experts,
 *    selection on the raw logits, ties to the lower expert index, outputs in
 *    (logit descending, index ascending) order; a row with a NaN is invalid
 *    (experts 0..k-1, weights 1/k, flagged); an all -inf row gets weights 1/k;
 *    a row whose maximum is +inf splits the weight evenly over its +inf picks.
 *  - activation: silu(g) * u (SwiGLU), silu(z) = z / (1 + exp(-z)).
 *  - h = bf16 round-to-nearest-even of silu(g) * u (one fixed rounding point).
 *  - weight layout: per expert, w13 = [2I][H/2] code bytes (rows 0..I-1 gate,
 *    I..2I-1 up), w2 = [H][I/2]; low nibble = even column; scales [rows][K/32].
 *  - an expert whose four pointers are not all non-NULL is absent: its rows of
 *    Y (and h) are zero.
 *  - router: the pages name the selection (16 of 896 experts per token) but not
 *    the score; the score of expert e is read as the linear form x . wr[e]
 *    of the token's bf16 hidden state with a bf16 router row, and the route
 *    selects on those scores rounded once to fp32.
 *  - W4A4 mode ("a4"): x and h are quantised to MXFP4 by the [OCP-MX] rule
 *    (round-to-nearest-even on the E2M1 grid, saturate at 6, all-zero block ->
 *    scale byte 0, code sign bit set iff the value is < 0) before the dot
 *    products.
 */
#ifndef K3MOE_REF_H
#define K3MOE_REF_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t T, H, I, E, k;
} k3ref_shape;

/* ---- scalar definitions ---- */
double k3ref_e2m1(unsigned code);      /* 4-bit E2M1 code -> value (exact)            */
double k3ref_e8m0(unsigned byte);      /* E8M0 byte -> 2^(byte-127); 255 -> NaN       */
double k3ref_bf16_value(uint16_t bits);
uint16_t k3ref_bf16_rne(double v);     /* round-to-nearest-even, overflow -> inf      */
double k3ref_silu(double z);
/* MXFP4 quantisation of n bf16 values (n % 32 == 0): codes[n/2] (low nibble =
 * even element), scales[n/32]. */
void k3ref_quant_mxfp4(const uint16_t *v, int n, uint8_t *codes, uint8_t *scales);

/* ---- the four steps ---- */
/* idx[T][k], w[T][k] (double); row_bad[T] (may be NULL) = 1 for a NaN row.
 * Returns the number of NaN rows, or -1 on bad shape. */
int k3ref_route(k3ref_shape s, const float *logits, int32_t *idx, double *w, int32_t *row_bad);
/* counts[E], offsets[E+1], perm[A], inv[A] with A = T*k.  Returns 0 or -1. */
int k3ref_bucket(k3ref_shape s, const int32_t *idx, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *inv);
/* Y[A][H] in bucket (perm) order; h_out[A][I] (may be NULL) = the bf16 bits of h.
 * a4 = 0: W4A16 (bf16 activations), 1: W4A4.  Returns 0 or -1. */
int k3ref_expert_ffn(k3ref_shape s, const uint16_t *x, const uint8_t *const *w13c,
                     const uint8_t *const *w13s, const uint8_t *const *w2c,
                     const uint8_t *const *w2s, const int32_t *offsets, const int32_t *perm,
                     int a4, double *Y, uint16_t *h_out);
/* The two halves of k3moe_ref_expert_ffn, for checking a path that takes the
 * bf16 rounding of h as its own decision: hpre[A][I] = silu(g) u in double and
 * h[A][I] = its bf16 rounding, in bucket order (optionally g, u and the sums
 * gabs = sum_c |Wg[c] x[c]|, uabs = sum_c |Wu[c] x[c]|, [A][I] each, NULL to
 * skip); and Y[A][H] = W2 h for given bf16 h rows in bucket order (a4: each h row
 * quantised to MXFP4 first).  An absent expert gives zero rows.  expert_ffn =
 * gateup, then down on its h.  Return 0 or -1. */
int k3ref_expert_gateup(k3ref_shape s, const uint16_t *x, const uint8_t *const *w13c,
                        const uint8_t *const *w13s, const uint8_t *const *w2c,
                        const uint8_t *const *w2s, const int32_t *offsets, const int32_t *perm,
                        int a4, double *hpre, uint16_t *h, double *g, double *u, double *gabs,
                        double *uabs);
int k3ref_expert_down(k3ref_shape s, const uint16_t *h, const uint8_t *const *w13c,
                      const uint8_t *const *w13s, const uint8_t *const *w2c,
                      const uint8_t *const *w2s, const int32_t *offsets, int a4, double *Y);
/* out[T][H] = sum_j w[t][j] * Y[inv[t*k+j]] in j order; out_bf16 may be NULL. */
int k3ref_combine(k3ref_shape s, const double *Y, const double *w, const int32_t *inv, double *out,
                  uint16_t *out_bf16);

/* ---- per-token path (no bucketing): out_row[H] = sum_j w[j] * FFN_{idx[j]}(x_row) ----
 * This is the per-token formulation that the batched path must agree with. */
int k3ref_moe_token(k3ref_shape s, const uint16_t *x_row, const int32_t *idx_row,
                    const double *w_row, const uint8_t *const *w13c, const uint8_t *const *w13s,
                    const uint8_t *const *w2c, const uint8_t *const *w2s, int a4, double *out_row);

/* ---- router (the step before routing): one linear score per expert ----
 * logits[t][e] = sum_h x[t][h] * wr[e][h] over bf16 x [T][H] and the bf16
 * router matrix wr [E][H] (row e scores expert e); products and sum in double.
 * Returns 0 or -1. */
int k3ref_router_logits(k3ref_shape s, const uint16_t *x, const uint16_t *wr, double *logits);
/* Router then route: the double logits rounded once to float (round to nearest
 * even) are the fp32 logits that the route selects on; idx, w and row_bad as in
 * k3ref_route.  logits (double [T][E]) and logits_f32 may be NULL.  Returns
 * k3ref_route's value, or -1. */
int k3ref_router(k3ref_shape s, const uint16_t *x, const uint16_t *wr, double *logits, float *logits_f32,
                 int32_t *idx, double *w, int32_t *row_bad);

/* ---- whole layer: route, bucket, FFN, combine (scratch allocated with malloc) ---- */
int k3ref_moe_layer(k3ref_shape s, const float *logits, const uint16_t *x,
                    const uint8_t *const *w13c, const uint8_t *const *w13s,
                    const uint8_t *const *w2c, const uint8_t *const *w2s, int a4, double *out,
                    uint16_t *out_bf16);

#ifdef __cplusplus
}
#endif
#endif
