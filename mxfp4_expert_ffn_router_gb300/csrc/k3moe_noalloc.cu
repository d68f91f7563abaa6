// k3moe_noalloc.cu -- k3moe_expert_ffn_noalloc: the expert FFN with its scratch
// in a fixed device array, for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc when they run the layer: cudaMalloc and
// cudaFree may synchronise the device (stalling every other stream), a host
// framework may own all device memory through its own pool and forbid raw
// allocations, or the caller may run inside a host callback that may not make
// CUDA allocation calls at all.  For them this entry point takes the same
// inputs and outputs as k3moe_expert_ffn but no workspace: the scratch lives in
// g_noalloc_scratch below, a file-scope device array of
// K3MOE_NOALLOC_SCRATCH_BYTES that every GPU which loads this library holds
// until the process exits.
//
// It serves the CUDA-core GEMV kernels only (AUTO and STREAM mean GEMV): the
// decode-sized path whose scratch fits the array.  GEMM and W4A4 return
// K3MOE_ERR_UNSUPPORTED.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/k3moe.h"
#include "k3moe_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[K3MOE_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch per device ordinal.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, called once per device with that device current.  The
// cached address belongs to the device's context at that time: calls after a
// cudaDeviceReset of that device are not supported.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return K3MOE_ERR_ARCH;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return k3moe::abi_launched(-1);  // records the error text
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return K3MOE_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int k3moe_expert_ffn_noalloc(k3moe_shape s, const uint16_t *x, const k3moe_weights *w,
                                        const int32_t *offsets, const int32_t *perm, float *Y, int mode,
                                        int32_t *dev_status, k3moe_stream_t stream) {
  int rc = k3moe::abi_check_shape(s);
  if (rc) return rc;
  if (mode < K3MOE_FFN_AUTO || mode > K3MOE_FFN_W4A4) return K3MOE_ERR_ARG;
  if (mode == K3MOE_FFN_GEMM || mode == K3MOE_FFN_W4A4) return K3MOE_ERR_UNSUPPORTED;
  if (s.T == 0) return K3MOE_OK;
  if (!x || !w || !offsets || !perm || !Y) return K3MOE_ERR_ARG;
  if (!w->w13_codes || !w->w13_scales || !w->w2_codes || !w->w2_scales) return K3MOE_ERR_ARG;
  if (!aligned16(x) || !aligned16(Y)) return K3MOE_ERR_ALIGN;
  const size_t need = k3moe::ffn_gemv_workspace(s);
  if (need > K3MOE_NOALLOC_SCRATCH_BYTES) return K3MOE_ERR_NOALLOC_LIMIT;
  if ((rc = k3moe::abi_check_arch())) return rc;
  void *ws = nullptr;
  if ((rc = scratch_for_current_device(&ws))) return rc;
  // Nothing in the scratch has to start at zero: the first kernel of each call
  // (the prep kernel) writes every count and table the call reads.
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return k3moe::abi_launched(k3moe::launch_ffn_gemv(s, x, *w, offsets, perm, Y, ws, dev_status, st));
}
