/* k3moe.h -- C ABI of the GB300 (sm_103a) routed MoE expert FFN with MXFP4 experts.
 *
 * One MoE layer is four calls, each a set of hand-written CUDA kernels launched
 * on the caller's stream:
 *
 *   k3moe_route       router logits -> top-k experts and routing weights
 *   k3moe_bucket      assignments -> expert-major order (counts, offsets, perm, inv)
 *   k3moe_expert_ffn  MXFP4 SwiGLU expert FFN over the bucketed assignments
 *   k3moe_combine     routing-weighted sum of each token's k expert outputs
 *
 * The operation follows the kimi-k3-in-c engine as described by its CHANGELOG
 * walkthrough (m.qwbw.cn): "[0.1.0] Added" (896 routed experts, top-16
 * selection, a gated-linear-unit expert, native MXFP4 expert weights, a matmul
 * that reads the packed nibbles directly and never materialises a dequantised
 * expert), "[1.0.0] Added" (chunk-union prefill: the tokens of a chunk are
 * grouped by routed expert so each unique expert's weights are read once, with
 * results identical to the per-token path) and "[Unreleased] Fixed" (an expert
 * that fails to load contributes zero, never uninitialised memory); and by the
 * article "kimi-k3-in-c: pure C99 Kimi K3 inference engine" (chenxutan.com),
 * section "01" (896 experts per layer, 16 woken per token).  MXFP4 is the OCP
 * Microscaling v1.0 format: E2M1 4-bit elements, one E8M0 scale per 32.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates no device memory, never synchronises the host, and launches
 *    only on `stream` (NULL = the legacy default stream).
 *  - Row-major, densely packed layouts as documented per argument.
 *  - Host-detectable errors (NULL required pointer, bad shape, misalignment,
 *    short workspace, wrong GPU) return a negative k3moe_status and launch
 *    nothing.  A launch failure returns K3MOE_ERR_LAUNCH.
 *  - Conditions found on the device are OR-ed as K3MOE_DEV_* bits into the
 *    caller's int32 `dev_status` word (device memory; zero it beforehand and
 *    read it after synchronising).
 *  - Outputs are overwritten, never accumulated into.  T = 0 is valid (no work).
 *  - Results are deterministic: the same inputs give bitwise the same outputs.
 */
#ifndef K3MOE_H
#define K3MOE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *k3moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  K3MOE_OK = 0,
  K3MOE_ERR_ARG = -1,         /* NULL required pointer or bad enum value         */
  K3MOE_ERR_SHAPE = -2,       /* shape outside the supported range               */
  K3MOE_ERR_ALIGN = -3,       /* pointer not 16-byte aligned                     */
  K3MOE_ERR_WORKSPACE = -4,   /* workspace NULL or smaller than required         */
  K3MOE_ERR_ARCH = -5,        /* current device is not compute capability 10.3   */
  K3MOE_ERR_LAUNCH = -6,      /* a CUDA launch failed                            */
  K3MOE_ERR_UNSUPPORTED = -7, /* valid request the chosen mode cannot serve      */
  K3MOE_ERR_NOALLOC_LIMIT = -8 /* problem needs more scratch than the fixed array of
                                  k3moe_expert_ffn_noalloc holds                  */
} k3moe_status;

/* Device-side status bits (OR-ed into *dev_status). */
#define K3MOE_DEV_NONFINITE 1 /* a router logit row contained NaN                 */
#define K3MOE_DEV_BOUNDS 2    /* an index read from device memory was out of range */
#define K3MOE_DEV_TIMEOUT 4   /* a bounded device-side wait gave up               */

/* T tokens, H hidden size, I expert intermediate size, E experts, k experts per
 * token.  Supported: 0 <= T, 1 <= k <= min(E, 32), E <= 4096, H and I multiples
 * of 32 in [32, 16384], T*k < 2^31. */
typedef struct {
  int32_t T, H, I, E, k;
} k3moe_shape;

/* MXFP4 expert weights of one layer.  Each member is a DEVICE array of E device
 * pointers, one per expert.  Expert e is absent when any of its four pointers
 * is NULL: its assignments then produce zero rows (never an error).  The host
 * cannot see these pointers: an expert whose code arrays are not 16-byte aligned
 * is also treated as absent (never read through), and the call sets
 * K3MOE_DEV_BOUNDS in dev_status.
 *   w13_codes[e]  : uint8 [2I][H/2]  rows 0..I-1 are the gate projection, rows
 *                   I..2I-1 the up projection; byte c of a row holds column 2c in
 *                   its low nibble and column 2c+1 in its high nibble; each
 *                   nibble is an E2M1 code (bit 3 sign, bits 2-1 exponent, bit 0
 *                   mantissa).  16-byte aligned.
 *   w13_scales[e] : uint8 [2I][H/32] E8M0 scale of each 32-column block
 *                   (value 2^(byte-127); 255 is NaN).
 *   w2_codes[e]   : uint8 [H][I/2]   down projection, same nibble order. 16-byte aligned.
 *   w2_scales[e]  : uint8 [H][I/32]
 * Element (r, c) of a matrix = E2M1(code) * E8M0(scale[r][c/32]). */
typedef struct {
  const uint8_t *const *w13_codes;
  const uint8_t *const *w13_scales;
  const uint8_t *const *w2_codes;
  const uint8_t *const *w2_scales;
} k3moe_weights;

/* Expert FFN modes.  All compute the same function (bf16 activations, exact
 * MXFP4 weights, fp32 accumulation); they differ in how weights are streamed. */
#define K3MOE_FFN_AUTO 0   /* the library picks per call: GEMM when 5 A >= 4 E
                              (A = T*k; 0.8 assignments per expert)
                              and the shape allows it, else GEMV                      */
#define K3MOE_FFN_GEMV 1   /* CUDA-core GEMV kernels, 128-bit register loads (any shape);
                              each routed expert's weights are read once per call     */
#define K3MOE_FFN_STREAM 2 /* retired: served by the GEMV kernels (kept so that callers
                              passing it keep working); a shared-memory ring fed by
                              1-D TMA bulk copies was measured slower than the
                              register-pipelined GEMV kernels                           */
#define K3MOE_FFN_GEMM 3   /* grouped GEMMs on the tcgen05 tensor cores (weights dequantised
                              exactly to bf16, fp32 accumulators in tensor memory) for
                              token chunks; needs H and I multiples of 128
                              (else K3MOE_ERR_UNSUPPORTED).                             */
#define K3MOE_FFN_W4A4 4   /* the GEMM mode with MXFP4 activations: x and h are quantised to
                              MXFP4 per 32-block (k3moe_quantize_mxfp4's rule) before the
                              products, which are then exact; same shape rules as GEMM.
                              With H and I multiples of 256 the products run on the
                              block-scaled FP4 tensor core (tcgen05 kind::mxf4: codes
                              and E8M0 scales of both operands as stored), else on the
                              GEMM mode's kernel after exact dequantisation.
                              Never chosen by AUTO.                                     */

/* Workspace queries (bytes; 0 when the call needs none).  op is one of: */
#define K3MOE_OP_BUCKET 1
#define K3MOE_OP_EXPERT_FFN 2
#define K3MOE_OP_LAYER 3
size_t k3moe_workspace_bytes(k3moe_shape s, int op, int mode);
/* Where the expert FFN leaves h: after a k3moe_expert_ffn call with shape s and
 * mode, its workspace holds h = bf16_rne(silu(g) * u) -- the GLU expert's one
 * rounding point, before the down projection (in W4A4 mode: before its MXFP4
 * quantisation) -- as uint16 [A][I] bf16 bit patterns in bucket order, starting
 * this many bytes into the workspace (256-byte aligned).  Lets a caller check or
 * reuse the intermediate without another kernel.  (size_t)-1 for a bad shape or
 * an unsupported mode. */
size_t k3moe_workspace_h_offset(k3moe_shape s, int mode);

/* Route: for each token t, the k experts with the largest logits, ordered by
 * (logit descending, expert index ascending) -- ties go to the lower index, -0
 * equals +0 -- and weights w[t][j] = exp(l_j - m) / sum_j' exp(l_j' - m) over
 * the k picks (m = the row maximum), i.e. the softmax over all E experts
 * renormalised to the top k.  A row holding a NaN sets K3MOE_DEV_NONFINITE
 * and yields experts 0..k-1 with weights 1/k; an all -inf row yields weights
 * 1/k; a row whose maximum is +inf splits the weight evenly over its +inf picks.
 *   logits : float [T][E]      idx : int32 [T][k]      w : float [T][k]
 *   dev_status : int32 device word (may be NULL: NaN rows are then unreported). */
int k3moe_route(k3moe_shape s, const float *logits, int32_t *idx, float *w,
                int32_t *dev_status, k3moe_stream_t stream);

/* Router: the score of every expert for every token, then the route above on
 * those scores (the step that feeds the top-16-of-896 selection: kimi-k3-in-c
 * CHANGELOG walkthrough "[0.1.0] Added"; article section "01").  The pages
 * name the selection but not the score; it is the linear form
 *   logits[t][e] = sum_h x[t][h] * wr[e][h]
 * of the token's bf16 hidden state and the bf16 router row of expert e, with
 * exact products accumulated in fp32, and the route selects on these fp32
 * logits exactly as k3moe_route does (same order, ties and weights).
 *   x      : uint16 [T][H] bf16 bit patterns, 16-byte aligned
 *   wr     : uint16 [E][H] bf16 bit patterns (row e scores expert e), 16-byte aligned
 *   logits : float [T][E], written (the fp32 scores the route selected on)
 *   idx, w, dev_status : as in k3moe_route
 * Accumulation: below 64 tokens a CUDA-core kernel sums each score in a fixed
 * order whose longest chain of fp32 roundings is ceil(H/256) + 7 (so |error| <=
 * gamma(ceil(H/256) + 7) * sum_h |x[t][h] wr[e][h]|, gamma(d) = d u / (1 - d u),
 * u = 2^-24); from 64 tokens the tcgen05 tensor cores accumulate in fp32 in
 * steps of K = 16 (fixed, deterministic order), for which the stated bound is
 * gamma(ceil(H/16) + 16) with u = 2^-23.  Scores that differ by less than
 * twice the bound can therefore order differently from an exact sum.
 * Errors: as k3moe_route; x or wr misaligned -> K3MOE_ERR_ALIGN. */
int k3moe_router(k3moe_shape s, const uint16_t *x, const uint16_t *wr, float *logits, int32_t *idx, float *w,
                 int32_t *dev_status, k3moe_stream_t stream);

/* Bucket: a stable counting sort of the A = T*k assignments a = t*k + j by
 * expert idx[a] (the chunk-union grouping).
 *   counts  : int32 [E]    number of assignments per expert
 *   offsets : int32 [E+1]  exclusive prefix sum of counts (offsets[E] = A)
 *   perm    : int32 [A]    assignment ids in expert-major, then ascending, order
 *   inv     : int32 [A]    inv[perm[p]] = p
 *   ws      : workspace of k3moe_workspace_bytes(s, K3MOE_OP_BUCKET, 0) bytes
 * An idx entry outside [0, E) sets K3MOE_DEV_BOUNDS (when dev_status is given)
 * and that assignment is dropped from the counts. */
int k3moe_bucket(k3moe_shape s, const int32_t *idx, int32_t *counts, int32_t *offsets,
                 int32_t *perm, int32_t *inv, void *ws, size_t ws_bytes, int32_t *dev_status,
                 k3moe_stream_t stream);

/* Expert FFN: for each bucket position p (assignment a = perm[p], token t = a/k,
 * expert e with offsets[e] <= p < offsets[e+1]):
 *   g = W_gate,e x_t ;  u = W_up,e x_t ;  h = bf16_rne(silu(g) * u) ;
 *   Y[p] = W_down,e h          (silu(z) = z / (1 + exp(-z)))
 * Dot products accumulate in fp32 from exact products; h is rounded to bf16
 * (round to nearest even) before the down projection.
 *   x    : uint16 [T][H] bf16 bit patterns, 16-byte aligned
 *   Y    : float  [A][H] in bucket order, 16-byte aligned
 *   ws   : workspace of k3moe_workspace_bytes(s, K3MOE_OP_EXPERT_FFN, mode) bytes */
int k3moe_expert_ffn(k3moe_shape s, const uint16_t *x, const k3moe_weights *w,
                     const int32_t *offsets, const int32_t *perm, float *Y, int mode, void *ws,
                     size_t ws_bytes, int32_t *dev_status, k3moe_stream_t stream);

/* Expert FFN without a workspace argument (no counterpart on the pages: it exists
 * for callers of this library that cannot allocate device memory).  Some callers
 * cannot call cudaMalloc around the layer: cudaMalloc/cudaFree may synchronise
 * the whole device and stall other streams, a host framework may own all device
 * memory through its own pool, or the code may run where CUDA allocation calls
 * are not allowed.  This entry point takes the arguments of k3moe_expert_ffn
 * minus ws/ws_bytes; its scratch is a file-scope device array of
 * K3MOE_NOALLOC_SCRATCH_BYTES that every GPU loading the library keeps until the
 * process exits.  It calls no allocation routine.
 *  - Modes: it serves the CUDA-core GEMV kernels only.  K3MOE_FFN_AUTO (and
 *    K3MOE_FFN_STREAM) mean K3MOE_FFN_GEMV here (k3moe_expert_ffn's AUTO may pick
 *    the tensor-core GEMM for the same shape, so the two entry points can then
 *    differ within the parity tolerance, not bitwise); in GEMV mode it computes
 *    bitwise what k3moe_expert_ffn computes.  K3MOE_FFN_GEMM and K3MOE_FFN_W4A4
 *    return K3MOE_ERR_UNSUPPORTED; other values K3MOE_ERR_ARG.
 *  - Limit: a problem whose scratch, k3moe_workspace_bytes(s, K3MOE_OP_EXPERT_FFN,
 *    K3MOE_FFN_GEMV), exceeds
 *    K3MOE_NOALLOC_SCRATCH_BYTES returns K3MOE_ERR_NOALLOC_LIMIT and launches
 *    nothing (decode-sized batches fit; large prefill chunks do not).
 *  - The first call on a device looks up the array's device address with that
 *    device current (one-time set-up); make that first call before any stream
 *    capture.  Calls after a cudaDeviceReset of that device are not supported.
 *  - Every call on a device uses the same array, which keeps the previous call's
 *    contents; each call re-initialises whatever it reads.  Calls whose kernels
 *    overlap on the GPU (different streams, no ordering between them) race on the
 *    array and give wrong results: order them on one stream or with events.
 *  - A failed launch returns K3MOE_ERR_LAUNCH with its text in
 *    k3moe_last_cuda_error(), as for the other entry points. */
#define K3MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
int k3moe_expert_ffn_noalloc(k3moe_shape s, const uint16_t *x, const k3moe_weights *w,
                             const int32_t *offsets, const int32_t *perm, float *Y, int mode,
                             int32_t *dev_status, k3moe_stream_t stream);

/* MXFP4 quantisation of bf16 activations (the W4A4 mode's input step; OCP
 * Microscaling Formats v1.0, conversion to MXFP4).  Per block of 32 consecutive
 * values: shared exponent e = floor(log2 amax) - 2 clamped to [-127, 127] (an
 * all-zero block: e = -127), stored as the E8M0 byte e + 127; each element's code
 * is |v| / 2^e rounded to the nearest E2M1 value (ties to the even code),
 * saturating at 6, with the sign bit set iff v < 0 (NaN elements give code 0;
 * results for blocks holding an infinity are unspecified).
 *   n      : number of values, a multiple of 32 (rows whose length is a multiple of
 *            32 may be passed as one run)
 *   x      : bf16 [n], 16-byte aligned
 *   codes  : uint8 [n/2], 16-byte aligned; byte i holds values 2i (low nibble), 2i+1
 *   scales : uint8 [n/32]
 * Errors: n < 0 or not a multiple of 32 -> K3MOE_ERR_SHAPE; NULL -> ERR_ARG;
 * misaligned x/codes -> ERR_ALIGN; n == 0 launches nothing. */
int k3moe_quantize_mxfp4(int64_t n, const uint16_t *x, uint8_t *codes, uint8_t *scales, k3moe_stream_t stream);

/* Combine: out_f32[t] = sum_{j=0..k-1} w[t][j] * Y[inv[t*k+j]], accumulated in
 * fp32 in increasing j; out[t] = bf16_rne(out_f32[t]).
 *   Y : float [A][H]   w : float [T][k]   inv : int32 [A]
 *   out : uint16 [T][H] bf16 bit patterns (required); out_f32 : float [T][H] or NULL. */
int k3moe_combine(k3moe_shape s, const float *Y, const float *w, const int32_t *inv, uint16_t *out,
                  float *out_f32, k3moe_stream_t stream);

/* Expert cache: MXFP4 experts resident in host memory, read by the GPU, and a
 * least-recently-used arena of expert slots in device memory (no counterpart
 * API on the pages; it follows the expert-cache design of "running a 2.78T
 * model in 8 GB", section on the trunk and the expert cache: an LRU arena with
 * a batch prefetch of the step's experts, and two hit counts -- raw hits, the
 * expert is in the arena when the FFN asks for it, near 100% because of the
 * prefetch; and TRUE resident hits, the expert stayed in the arena since the
 * previous step, the measure of reads avoided).
 *   slots      : expert slots in the arena, 1 .. 2^20; a step needs at least as
 *                many as the distinct experts it routes to (else the step is
 *                refused: K3MOE_DEV_BOUNDS, nothing copied)
 *   arena      : caller-owned device memory of k3moe_cache_bytes(s, slots) bytes,
 *                256-byte aligned; it holds the bookkeeping, four device tables
 *                of E expert pointers and the slots.  Only s.H, s.I and s.E
 *                matter for its size.
 *   host_w     : the experts in host memory, in the layout of k3moe_weights: four
 *                DEVICE-readable arrays of E pointers to host arrays that the GPU
 *                can read (page-locked memory from cudaHostAlloc, or registered
 *                with cudaHostRegister), each 16-byte aligned; NULL = absent
 *   s          : the arena's shape: H, I and E = every expert it caches (up to
 *                2^20: for a stack of layers, E = layers x experts per layer, and
 *                expert l * E_layer + e is expert e of layer l); T and k unused
 *   counts     : int32 [count_n] from k3moe_bucket: the step requests expert
 *                count_base + i when counts[i] > 0 (a layer's slice of the arena's
 *                experts); count_base + count_n <= E
 *   stats      : device uint64 [4] accumulating requests, raw hits, true resident
 *                hits and bytes copied host -> arena (zero it before the first
 *                step), or NULL
 * k3moe_cache_init marks every slot empty.  k3moe_cache_fetch makes every
 * requested expert resident: hits stay; each miss, in ascending expert order,
 * takes the least recently used slot that the step does not request (ties by
 * slot index; empty slots first) and its four arrays are copied from host
 * memory by a device kernel in the same stream (no host synchronisation).
 * k3moe_cache_weights (host only, no device call) fills a k3moe_weights whose
 * four device tables inside the arena point at the resident experts' slots
 * (NULL for others): pass it to k3moe_expert_ffn after k3moe_cache_fetch (for
 * layer l of a stack, offset each table by l * E_layer).  The
 * arena's contents are the cache's state: steps on one arena must be ordered on
 * one stream. */
size_t k3moe_cache_bytes(k3moe_shape s, int slots);
int k3moe_cache_weights(k3moe_shape s, int slots, void *arena, k3moe_weights *w);
int k3moe_cache_init(k3moe_shape s, int slots, void *arena, size_t arena_bytes, k3moe_stream_t stream);
int k3moe_cache_fetch(k3moe_shape s, int slots, void *arena, size_t arena_bytes, const k3moe_weights *host_w,
                      const int32_t *counts, int32_t count_base, int32_t count_n, uint64_t *stats,
                      int32_t *dev_status, k3moe_stream_t stream);

/* The whole layer in one call: k3moe_route, k3moe_bucket, k3moe_expert_ffn and
 * k3moe_combine on `stream`, with the same arguments, outputs and results (bit
 * for bit) as the four calls; every intermediate (idx, wts, counts, offsets,
 * perm, inv, Y) is written as those calls write it.  The workspace, of
 * k3moe_workspace_bytes(s, K3MOE_OP_LAYER, mode) bytes (256-byte aligned),
 * serves the bucketing and the expert FFN in turn.  When the FFN runs the GEMV
 * kernels and the batch is small (T <= 4, E <= 1024, T*k <= 128) the route,
 * the bucketing and the FFN's preparation run as one single-block kernel: a
 * decode step is then five launches instead of seven.  Errors: the union of the
 * four calls'. */
int k3moe_layer(k3moe_shape s, const float *logits, const uint16_t *x, const k3moe_weights *w, int32_t *idx,
                float *wts, int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv, float *Y, uint16_t *out,
                float *out_f32, int mode, void *ws, size_t ws_bytes, int32_t *dev_status, k3moe_stream_t stream);

/* Combine into a residual stream (a stack of MoE layers: x_next = x + MoE(x);
 * the pages' engine adds each layer's routed experts into the residual stream):
 * out_f32[t] = residual[t] + (sum_{j} w[t][j] * Y[inv[t*k+j]], fp32 in increasing
 * j, as k3moe_combine), the residual added once after the sum; out[t] =
 * bf16_rne(out_f32[t]).  residual : uint16 [T][H] bf16 bit patterns, 16-byte
 * aligned; it may be the same buffer as out (each element is read before it is
 * written, by the same thread).  Errors as k3moe_combine; NULL residual ->
 * K3MOE_ERR_ARG. */
int k3moe_combine_residual(k3moe_shape s, const float *Y, const float *w, const int32_t *inv, const uint16_t *residual,
                           uint16_t *out, float *out_f32, k3moe_stream_t stream);

/* Self-test of the bounded waits (a test hook, not part of the path): one
 * thread waits, with the iteration bound every mbarrier wait in the tensor-core
 * kernels uses, on a phase that nothing completes, so the wait runs out: the
 * kernel ORs K3MOE_DEV_TIMEOUT into *dev_status and writes the wait's duration
 * in nanoseconds to *dev_elapsed_ns (both device pointers), then returns; the
 * context stays usable.  No copy or tensor-core operation is in flight in the
 * waiting CTA.  Errors: NULL pointer -> K3MOE_ERR_ARG; not sm_103 ->
 * K3MOE_ERR_ARCH; launch failure -> K3MOE_ERR_LAUNCH. */
int k3moe_selftest_bounded_wait(int32_t *dev_status, unsigned long long *dev_elapsed_ns, k3moe_stream_t stream);

/* Human-readable name of a k3moe_status value. */
const char *k3moe_status_string(int code);

/* The CUDA error text behind the calling thread's most recent K3MOE_ERR_LAUNCH
 * ("no error" if none).  The string is static; do not free it. */
const char *k3moe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif
#endif
