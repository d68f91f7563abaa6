// k3moe.cu -- the C ABI (include/k3moe.h): argument validation and dispatch.
// Every entry point validates on the host, launches nothing on error, and
// otherwise enqueues its kernels on the caller's stream without synchronising.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/k3moe.h"
#include "k3moe_dev.cuh"
#include "k3moe_launch.h"
#include "tc_sm103.cuh"

namespace {

using k3moe_stream = cudaStream_t;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

thread_local const char *t_last_cuda_error = "no error";

}  // namespace

namespace k3moe {

int abi_check_shape(const k3moe_shape &s) {
  if (s.T < 0 || s.E < 1 || s.E > 4096 || s.k < 1 || s.k > 32 || s.k > s.E) return K3MOE_ERR_SHAPE;
  if (s.H < 32 || s.H > 16384 || s.H % 32 || s.I < 32 || s.I > 16384 || s.I % 32) return K3MOE_ERR_SHAPE;
  if (static_cast<long long>(s.T) * s.k >= (1LL << 31)) return K3MOE_ERR_SHAPE;
  return K3MOE_OK;
}

// The kernels use sm_103a instructions: refuse any other device.
int abi_check_arch() {
  static std::mutex mu;
  static int cached[64];
  static bool init = false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();  // leave no error behind for the next call
    return K3MOE_ERR_ARCH;
  }
  std::lock_guard<std::mutex> g(mu);
  if (!init) {
    for (int i = 0; i < 64; ++i) cached[i] = 0;
    init = true;
  }
  if (cached[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cached[dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return cached[dev] == 1 ? K3MOE_OK : K3MOE_ERR_ARCH;
}

int abi_launched(int rc) {
  const cudaError_t e = cudaGetLastError();
  if (rc == 0 && e == cudaSuccess) return K3MOE_OK;
  t_last_cuda_error = cudaGetErrorString(e == cudaSuccess ? cudaErrorLaunchFailure : e);
  return K3MOE_ERR_LAUNCH;
}

}  // namespace k3moe

using k3moe::abi_check_arch;
using k3moe::abi_check_shape;
using k3moe::abi_launched;

extern "C" {

// The expert FFN path a mode resolves to for a shape (-1: unsupported).
static int resolve_ffn_mode(const k3moe_shape &s, int mode) {
  switch (mode) {
    case K3MOE_FFN_AUTO: {
      // tensor cores once the assignments reach 0.8 per expert (measured at
      // H = 7168, I = 2048, E = 896, k = 16 with independent routing: the GEMM
      // overtakes the GEMV kernels between T = 32 and T = 48); otherwise the
      // GEMV kernels, which stream each routed expert's weights once for its
      // tokens but spend CUDA-core instructions on every token
      const long long A = static_cast<long long>(s.T) * s.k;
      if (k3moe::ffn_gemm_supported(s) && 5 * A >= 4 * static_cast<long long>(s.E)) return K3MOE_FFN_GEMM;
      return K3MOE_FFN_GEMV;
    }
    case K3MOE_FFN_GEMV: return K3MOE_FFN_GEMV;
    case K3MOE_FFN_STREAM: return K3MOE_FFN_GEMV;  // retired: the GEMV kernels serve it
    case K3MOE_FFN_GEMM: return k3moe::ffn_gemm_supported(s) ? K3MOE_FFN_GEMM : -1;
    case K3MOE_FFN_W4A4: return k3moe::ffn_gemm_supported(s) ? K3MOE_FFN_W4A4 : -1;
    default: return -1;
  }
}

static size_t ffn_workspace(const k3moe_shape &s, int resolved) {
  if (resolved == K3MOE_FFN_GEMV) return k3moe::ffn_gemv_workspace(s);
  if (resolved == K3MOE_FFN_GEMM || resolved == K3MOE_FFN_W4A4) return k3moe::ffn_gemm_workspace(s);
  return 0;
}

size_t k3moe_workspace_h_offset(k3moe_shape s, int mode) {
  if (abi_check_shape(s) != K3MOE_OK) return static_cast<size_t>(-1);
  const int resolved = resolve_ffn_mode(s, mode);
  if (resolved == K3MOE_FFN_GEMV) return k3moe::ffn_gemv_h_offset(s);
  if (resolved == K3MOE_FFN_GEMM || resolved == K3MOE_FFN_W4A4) return k3moe::ffn_gemm_h_offset(s);
  return static_cast<size_t>(-1);
}

// The layer call runs bucket and expert FFN one after the other: one workspace
// serves both.
static size_t layer_workspace(const k3moe_shape &s, int resolved) {
  if (resolved < 0) return 0;
  const size_t b = k3moe::bucket_workspace(s), f = ffn_workspace(s, resolved);
  return b > f ? b : f;
}

size_t k3moe_workspace_bytes(k3moe_shape s, int op, int mode) {
  if (abi_check_shape(s) != K3MOE_OK) return 0;
  if (op == K3MOE_OP_BUCKET) return k3moe::bucket_workspace(s);
  if (op == K3MOE_OP_EXPERT_FFN) return ffn_workspace(s, resolve_ffn_mode(s, mode));
  if (op == K3MOE_OP_LAYER) return layer_workspace(s, resolve_ffn_mode(s, mode));
  return 0;
}

int k3moe_route(k3moe_shape s, const float *logits, int32_t *idx, float *w, int32_t *dev_status,
                k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (s.T == 0) return K3MOE_OK;
  if (!logits || !idx || !w) return K3MOE_ERR_ARG;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(k3moe::launch_route(s, logits, idx, w, dev_status, reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_router(k3moe_shape s, const uint16_t *x, const uint16_t *wr, float *logits, int32_t *idx, float *w,
                 int32_t *dev_status, k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (s.T == 0) return K3MOE_OK;
  if (!x || !wr || !logits || !idx || !w) return K3MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(wr)) return K3MOE_ERR_ALIGN;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(
      k3moe::launch_router(s, x, wr, logits, idx, w, dev_status, reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_bucket(k3moe_shape s, const int32_t *idx, int32_t *counts, int32_t *offsets, int32_t *perm,
                 int32_t *inv, void *ws, size_t ws_bytes, int32_t *dev_status,
                 k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (!counts || !offsets) return K3MOE_ERR_ARG;
  if (s.T > 0 && (!idx || !perm || !inv)) return K3MOE_ERR_ARG;
  const size_t need = k3moe::bucket_workspace(s);
  if (need && (!ws || ws_bytes < need || !aligned16(ws))) return K3MOE_ERR_WORKSPACE;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(k3moe::launch_bucket(s, idx, counts, offsets, perm, inv, ws, dev_status,
                                       reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_expert_ffn(k3moe_shape s, const uint16_t *x, const k3moe_weights *w, const int32_t *offsets,
                     const int32_t *perm, float *Y, int mode, void *ws, size_t ws_bytes,
                     int32_t *dev_status, k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (mode < K3MOE_FFN_AUTO || mode > K3MOE_FFN_W4A4) return K3MOE_ERR_ARG;
  const int resolved = resolve_ffn_mode(s, mode);
  if (resolved < 0) return K3MOE_ERR_UNSUPPORTED;
  if (s.T == 0) return K3MOE_OK;
  if (!x || !w || !offsets || !perm || !Y) return K3MOE_ERR_ARG;
  if (!w->w13_codes || !w->w13_scales || !w->w2_codes || !w->w2_scales) return K3MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(Y)) return K3MOE_ERR_ALIGN;
  const size_t need = ffn_workspace(s, resolved);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return K3MOE_ERR_WORKSPACE;
  if ((rc = abi_check_arch())) return rc;
  const cudaStream_t st = reinterpret_cast<k3moe_stream>(stream);
  if (resolved == K3MOE_FFN_GEMM || resolved == K3MOE_FFN_W4A4)
    return abi_launched(k3moe::launch_ffn_gemm(s, x, *w, offsets, perm, Y, ws, dev_status, st,
                                           resolved == K3MOE_FFN_W4A4));
  return abi_launched(k3moe::launch_ffn_gemv(s, x, *w, offsets, perm, Y, ws, dev_status, st));
}

// The cache's shape may cache several layers' experts: E up to 2^20 (the
// per-call shape rule E <= 4096 applies to the layer calls, not to the arena).
static int cache_check_shape(const k3moe_shape &s) {
  if (s.E < 1 || s.E > (1 << 20) || s.T < 0 || s.k < 1 || s.k > 32) return K3MOE_ERR_SHAPE;
  if (s.H < 32 || s.H > 16384 || s.H % 32 || s.I < 32 || s.I > 16384 || s.I % 32) return K3MOE_ERR_SHAPE;
  return K3MOE_OK;
}

size_t k3moe_cache_bytes(k3moe_shape s, int slots) {
  if (cache_check_shape(s) != K3MOE_OK || slots < 1 || slots > (1 << 20)) return 0;
  return k3moe::cache_arena_bytes(s, slots);
}

int k3moe_cache_weights(k3moe_shape s, int slots, void *arena, k3moe_weights *w) {
  int rc = cache_check_shape(s);
  if (rc) return rc;
  if (slots < 1 || slots > (1 << 20)) return K3MOE_ERR_SHAPE;
  if (!arena || !w) return K3MOE_ERR_ARG;
  k3moe::cache_tables(s, slots, arena, w);
  return K3MOE_OK;
}

int k3moe_cache_init(k3moe_shape s, int slots, void *arena, size_t arena_bytes, k3moe_stream_t stream) {
  int rc = cache_check_shape(s);
  if (rc) return rc;
  if (slots < 1 || slots > (1 << 20)) return K3MOE_ERR_SHAPE;
  if (!arena) return K3MOE_ERR_ARG;
  if (arena_bytes < k3moe::cache_arena_bytes(s, slots) || (reinterpret_cast<uintptr_t>(arena) & 255u))
    return K3MOE_ERR_WORKSPACE;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(k3moe::launch_cache_init(s, slots, arena, reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_cache_fetch(k3moe_shape s, int slots, void *arena, size_t arena_bytes, const k3moe_weights *host_w,
                      const int32_t *counts, int32_t count_base, int32_t count_n, uint64_t *stats,
                      int32_t *dev_status, k3moe_stream_t stream) {
  int rc = cache_check_shape(s);
  if (rc) return rc;
  if (slots < 1 || slots > (1 << 20)) return K3MOE_ERR_SHAPE;
  if (count_base < 0 || count_n < 0 || count_base > s.E - count_n) return K3MOE_ERR_SHAPE;
  if (count_n == 0) return K3MOE_OK;
  if (!arena || !host_w || !counts) return K3MOE_ERR_ARG;
  if (!host_w->w13_codes || !host_w->w13_scales || !host_w->w2_codes || !host_w->w2_scales) return K3MOE_ERR_ARG;
  if (arena_bytes < k3moe::cache_arena_bytes(s, slots) || (reinterpret_cast<uintptr_t>(arena) & 255u))
    return K3MOE_ERR_WORKSPACE;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(k3moe::launch_cache_fetch(s, slots, arena, *host_w, counts, count_base, count_n,
                                                reinterpret_cast<unsigned long long *>(stats), dev_status,
                                                reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_layer(k3moe_shape s, const float *logits, const uint16_t *x, const k3moe_weights *w, int32_t *idx,
                float *wts, int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv, float *Y, uint16_t *out,
                float *out_f32, int mode, void *ws, size_t ws_bytes, int32_t *dev_status, k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (mode < K3MOE_FFN_AUTO || mode > K3MOE_FFN_W4A4) return K3MOE_ERR_ARG;
  const int resolved = resolve_ffn_mode(s, mode);
  if (resolved < 0) return K3MOE_ERR_UNSUPPORTED;
  if (s.T == 0) return K3MOE_OK;
  if (!logits || !x || !w || !idx || !wts || !counts || !offsets || !perm || !inv || !Y || !out) return K3MOE_ERR_ARG;
  if (!w->w13_codes || !w->w13_scales || !w->w2_codes || !w->w2_scales) return K3MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(Y) || !aligned16(out) || (out_f32 && !aligned16(out_f32))) return K3MOE_ERR_ALIGN;
  const size_t need = layer_workspace(s, resolved);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255u)) return K3MOE_ERR_WORKSPACE;
  if ((rc = abi_check_arch())) return rc;
  const cudaStream_t st = reinterpret_cast<k3moe_stream>(stream);
  if (resolved == K3MOE_FFN_GEMV && k3moe::layer_front_fits(s))
    return abi_launched(k3moe::launch_layer_gemv_fast(s, logits, x, *w, idx, wts, counts, offsets, perm, inv, Y, out,
                                                      out_f32, ws, dev_status, st));
  if (k3moe::launch_route(s, logits, idx, wts, dev_status, st)) return abi_launched(-1);
  if (k3moe::launch_bucket(s, idx, counts, offsets, perm, inv, ws, dev_status, st)) return abi_launched(-1);
  int lrc;
  if (resolved == K3MOE_FFN_GEMM || resolved == K3MOE_FFN_W4A4)
    lrc = k3moe::launch_ffn_gemm(s, x, *w, offsets, perm, Y, ws, dev_status, st, resolved == K3MOE_FFN_W4A4);
  else
    lrc = k3moe::launch_ffn_gemv(s, x, *w, offsets, perm, Y, ws, dev_status, st);
  if (lrc) return abi_launched(-1);
  return abi_launched(k3moe::launch_combine(s, Y, wts, inv, nullptr, out, out_f32, st));
}

int k3moe_quantize_mxfp4(int64_t n, const uint16_t *x, uint8_t *codes, uint8_t *scales, k3moe_stream_t stream) {
  if (n < 0 || n % 32) return K3MOE_ERR_SHAPE;
  if (n == 0) return K3MOE_OK;
  if (!x || !codes || !scales) return K3MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(codes)) return K3MOE_ERR_ALIGN;
  int rc;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(k3moe::launch_quantize_mxfp4(static_cast<long long>(n), x, codes, scales,
                                               reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_combine(k3moe_shape s, const float *Y, const float *w, const int32_t *inv, uint16_t *out,
                  float *out_f32, k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (s.T == 0) return K3MOE_OK;
  if (!Y || !w || !inv || !out) return K3MOE_ERR_ARG;
  if (!aligned16(Y) || !aligned16(out) || (out_f32 && !aligned16(out_f32))) return K3MOE_ERR_ALIGN;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(
      k3moe::launch_combine(s, Y, w, inv, nullptr, out, out_f32, reinterpret_cast<k3moe_stream>(stream)));
}

int k3moe_combine_residual(k3moe_shape s, const float *Y, const float *w, const int32_t *inv, const uint16_t *residual,
                           uint16_t *out, float *out_f32, k3moe_stream_t stream) {
  int rc = abi_check_shape(s);
  if (rc) return rc;
  if (s.T == 0) return K3MOE_OK;
  if (!Y || !w || !inv || !residual || !out) return K3MOE_ERR_ARG;
  if (!aligned16(Y) || !aligned16(out) || !aligned16(residual) || (out_f32 && !aligned16(out_f32)))
    return K3MOE_ERR_ALIGN;
  if ((rc = abi_check_arch())) return rc;
  return abi_launched(
      k3moe::launch_combine(s, Y, w, inv, residual, out, out_f32, reinterpret_cast<k3moe_stream>(stream)));
}

const char *k3moe_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"

namespace {
// One thread waits, with the bound every tensor-core kernel's waits use, on an
// mbarrier phase that nothing completes (no copy or MMA is in flight into the
// CTA), then reports K3MOE_DEV_TIMEOUT and how long the wait took.
__global__ void selftest_bounded_wait_kernel(int32_t *status, unsigned long long *elapsed_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    k3moe::mb_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long t0, t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    const bool done = k3moe::mb_wait(&bar, 0);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (!done) k3moe::set_status(status, K3MOE_DEV_TIMEOUT);
    *elapsed_ns = t1 - t0;
  }
}
}  // namespace

extern "C" {

int k3moe_selftest_bounded_wait(int32_t *dev_status, unsigned long long *dev_elapsed_ns, k3moe_stream_t stream) {
  if (!dev_status || !dev_elapsed_ns) return K3MOE_ERR_ARG;
  const int rc = abi_check_arch();
  if (rc) return rc;
  selftest_bounded_wait_kernel<<<1, 32, 0, reinterpret_cast<k3moe_stream>(stream)>>>(dev_status, dev_elapsed_ns);
  return abi_launched(0);
}

const char *k3moe_status_string(int code) {
  switch (code) {
    case K3MOE_OK: return "ok";
    case K3MOE_ERR_ARG: return "invalid argument (NULL pointer or bad enum)";
    case K3MOE_ERR_SHAPE: return "unsupported shape";
    case K3MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
    case K3MOE_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case K3MOE_ERR_ARCH: return "current device is not sm_103 (GB300)";
    case K3MOE_ERR_LAUNCH: return "CUDA launch failed";
    case K3MOE_ERR_UNSUPPORTED: return "request not supported by the chosen mode";
    case K3MOE_ERR_NOALLOC_LIMIT: return "problem exceeds the fixed scratch of k3moe_expert_ffn_noalloc";
    default: return "unknown status";
  }
}

}  // extern "C"
