/* k3gen.h -- seeded, counter-based synthetic input generator.
 *
 * This module is shared by the oracle side and the GPU side of the tests and of
 * the benchmark.  It holds none of the MoE method's arithmetic: it only draws
 * random bytes, integers and normal variates from a counter-based generator,
 * so that both sides see the same input bytes.
 *
 * Generator definition (SplitMix64, Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014):
 *   gamma     = 0x9E3779B97F4A7C15
 *   mix64(z)  : z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
 *               z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
 *   base(seed, stream) = mix64(seed * gamma + mix64(stream + gamma))
 *   draw(seed, stream, n) = mix64(base + (n + 1) * gamma)      (mod 2^64)
 * Every value below is a pure function of (seed, stream, n), so any slice of
 * any tensor can be regenerated independently (per expert, per token ...).
 *
 * Derived variates:
 *   U53(d)   = (d >> 11) * 2^-53                      in [0, 1)
 *   bytes    : byte i of a stream = byte (i mod 8) of draw(i / 8), little-endian
 *   int      : lo + floor(U53(draw(n)) * (hi - lo + 1))
 *   normal   : Box-Muller with one output per pair of draws:
 *              u1 = 1 - U53(draw(2n))  (in (0,1]),  u2 = U53(draw(2n+1)),
 *              z  = sqrt(-2 ln u1) * cos(2 pi u2)                  (double)
 *   f32      : (float)(sigma * z)   (round to nearest even)
 *   bf16     : round-to-nearest-even of that f32 value to bf16
 */
#ifndef K3GEN_H
#define K3GEN_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stream ids.  Per-expert tensors use (kind << 32) | expert. */
#define K3GEN_KIND_W13_CODES 1u
#define K3GEN_KIND_W13_SCALES 2u
#define K3GEN_KIND_W2_CODES 3u
#define K3GEN_KIND_W2_SCALES 4u
#define K3GEN_KIND_X 5u
#define K3GEN_KIND_LOGITS 6u
#define K3GEN_KIND_AUX 7u

uint64_t k3gen_draw(uint64_t seed, uint64_t stream, uint64_t n);
double k3gen_u53(uint64_t seed, uint64_t stream, uint64_t n);

/* Fill out[0..n) with the uniform byte stream (seed, stream), starting at byte
 * offset `first` of that stream. */
void k3gen_bytes(uint64_t seed, uint64_t stream, uint64_t first, uint8_t *out, size_t n);
/* out[i] = lo + floor(U53(draw(first + i)) * (hi - lo + 1)), as bytes. */
void k3gen_uint8_range(uint64_t seed, uint64_t stream, uint64_t first, uint8_t *out, size_t n,
                       int lo, int hi);
/* Normal variates, element index first + i of the stream. */
void k3gen_normal_f64(uint64_t seed, uint64_t stream, uint64_t first, double *out, size_t n);
void k3gen_normal_f32(uint64_t seed, uint64_t stream, uint64_t first, float *out, size_t n,
                      double sigma);
void k3gen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t first, uint16_t *out, size_t n,
                       double sigma);
/* Uniform doubles U53. */
void k3gen_uniform_f64(uint64_t seed, uint64_t stream, uint64_t first, double *out, size_t n);

/* MXFP4 expert weights for experts [e0, e1), written back to back:
 *   w13c: (e1-e0) x [2I][H/2] code bytes (uniform bytes, stream W13_CODES|e)
 *   w13s: (e1-e0) x [2I][H/32] scale bytes (uniform in [slo, shi], stream W13_SCALES|e)
 *   w2c : (e1-e0) x [H][I/2]              (stream W2_CODES|e)
 *   w2s : (e1-e0) x [H][I/32]             (stream W2_SCALES|e)
 * Any pointer may be NULL to skip that tensor.  Work is split over nthreads
 * POSIX threads (<= 0: one thread).  Returns 0, or -1 on bad arguments. */
int k3gen_experts(uint64_t seed, int H, int I, int e0, int e1, int slo, int shi, uint8_t *w13c,
                  uint8_t *w13s, uint8_t *w2c, uint8_t *w2s, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
