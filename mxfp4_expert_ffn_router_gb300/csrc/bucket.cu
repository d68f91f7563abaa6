// bucket.cu -- deterministic stable counting sort of assignments by expert.
//
// Implements the chunk-union grouping of the kimi-k3-in-c CHANGELOG walkthrough,
// "[1.0.0] Added": the tokens of a chunk are grouped by routed expert so that each
// unique expert is fetched once per chunk.  Order inside an expert is ascending
// assignment id (a stable sort), so the grouped path visits the same pairs in
// the same order on every run.  No atomics decide an order: counts use integer
// atomics (order-free), and positions come from a warp-sequential scan.
#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

constexpr int kTile = 4096;  // assignments per tile

__device__ __forceinline__ bool valid_expert(int e, int E) { return e >= 0 && e < E; }

// Exclusive scan of cnt[0..E) (shared) into out[0..E] with 1024 threads.
__device__ void block_exclusive_scan(const int32_t *cnt, int E, int32_t *out, int32_t *warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int per = (E + 1023) / 1024;
  const int e0 = tid * per;
  int local = 0;
  for (int i = 0; i < per; ++i)
    if (e0 + i < E) local += cnt[e0 + i];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = warp_tot[lane];
    int vi = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, vi, off);
      if (lane >= off) vi += o;
    }
    warp_tot[lane] = vi - v;  // exclusive warp base
  }
  __syncthreads();
  int run = warp_tot[wid] + incl - local;
  for (int i = 0; i < per; ++i)
    if (e0 + i < E) {
      out[e0 + i] = run;
      run += cnt[e0 + i];
    }
  if (tid == 1023) out[E] = run;
  __syncthreads();
}

// One warp places the assignments [a0, a1) in order: fill[e] is the next free
// position of expert e; lanes that share an expert take consecutive slots.
__device__ void warp_place(const int32_t *__restrict__ idx, int a0, int a1, int E, int32_t *fill,
                           int32_t *__restrict__ perm, int32_t *__restrict__ inv) {
  const int lane = threadIdx.x & 31;
  for (int base = a0; base < a1; base += 32) {
    const int a = base + lane;
    const bool in = a < a1;
    const int e = in ? idx[a] : -1;
    const bool ok = in && valid_expert(e, E);
    const unsigned okmask = __ballot_sync(0xFFFFFFFFu, ok);
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, ok ? e : -1) & okmask;
    if (ok) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int pos = fill[e] + rank;
      perm[pos] = a;
      inv[a] = pos;
    } else if (in) {
      inv[a] = -1;
    }
    __syncwarp();
    if (ok && (31 - __clz(peers)) == lane) fill[e] += __popc(peers);
    __syncwarp();
  }
}

// A <= kTile: histogram, scan and placement in one block of 1024 threads.
__global__ void __launch_bounds__(1024)
    bucket_single_kernel(const int32_t *__restrict__ idx, int A, int E, int32_t *__restrict__ counts,
                         int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                         int32_t *__restrict__ inv, int32_t *status) {
  extern __shared__ int32_t sm[];
  int32_t *cnt = sm, *fill = sm + E, *wtot = sm + 2 * E + 1;
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += 1024) cnt[e] = 0;
  __syncthreads();
  bool bad = false;
  for (int a = threadIdx.x; a < A; a += 1024) {
    const int e = idx[a];
    if (valid_expert(e, E))
      atomicAdd(&cnt[e], 1);
    else
      bad = true;
  }
  if (bad) set_status(status, K3MOE_DEV_BOUNDS);
  __syncthreads();
  block_exclusive_scan(cnt, E, fill, wtot);
  for (int e = threadIdx.x; e < E; e += 1024) counts[e] = cnt[e];
  for (int e = threadIdx.x; e <= E; e += 1024) offsets[e] = fill[e];
  const int placed = fill[E];
  __syncthreads();
  if (threadIdx.x < 32) warp_place(idx, 0, A, E, fill, perm, inv);
  for (int p = placed + threadIdx.x; p < A; p += 1024) perm[p] = -1;  // only with bad ids
}

// Large A: per-tile histograms ...
__global__ void __launch_bounds__(256)
    bucket_hist_kernel(const int32_t *__restrict__ idx, int A, int E, int32_t *__restrict__ tile_hist,
                       int32_t *status) {
  extern __shared__ int32_t cnt[];
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += 256) cnt[e] = 0;
  __syncthreads();
  const int a0 = blockIdx.x * kTile, a1 = min(A, a0 + kTile);
  bool bad = false;
  for (int a = a0 + threadIdx.x; a < a1; a += 256) {
    const int e = idx[a];
    if (valid_expert(e, E))
      atomicAdd(&cnt[e], 1);
    else
      bad = true;
  }
  if (bad) set_status(status, K3MOE_DEV_BOUNDS);
  __syncthreads();
  int32_t *dst = tile_hist + static_cast<size_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += 256) dst[e] = cnt[e];
}

// ... a scan over experts and tiles (tile_hist becomes each tile's base) ...
__global__ void __launch_bounds__(1024)
    bucket_scan_kernel(int32_t *__restrict__ tile_hist, int ntiles, int E,
                       int32_t *__restrict__ counts, int32_t *__restrict__ offsets) {
  extern __shared__ int32_t sm[];
  int32_t *cnt = sm, *off = sm + E, *wtot = sm + 2 * E + 1;
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < E; e += 1024) {
    int s = 0;
    for (int t = 0; t < ntiles; ++t) s += tile_hist[static_cast<size_t>(t) * E + e];
    cnt[e] = s;
  }
  __syncthreads();
  block_exclusive_scan(cnt, E, off, wtot);
  for (int e = threadIdx.x; e < E; e += 1024) {
    counts[e] = cnt[e];
    int run = off[e];
    for (int t = 0; t < ntiles; ++t) {
      int32_t *h = tile_hist + static_cast<size_t>(t) * E + e;
      const int c = *h;
      *h = run;
      run += c;
    }
  }
  for (int e = threadIdx.x; e <= E; e += 1024) offsets[e] = off[e];
}

// ... and one warp per tile placing its assignments from the tile's bases.
__global__ void __launch_bounds__(32)
    bucket_place_kernel(const int32_t *__restrict__ idx, int A, int E,
                        const int32_t *__restrict__ tile_base, const int32_t *__restrict__ offsets,
                        int32_t *__restrict__ perm, int32_t *__restrict__ inv) {
  extern __shared__ int32_t fill[];
  pdl_wait();
  pdl_trigger();
  const int32_t *b = tile_base + static_cast<size_t>(blockIdx.x) * E;
  for (int e = threadIdx.x; e < E; e += 32) fill[e] = b[e];
  __syncwarp();
  const int a0 = blockIdx.x * kTile, a1 = min(A, a0 + kTile);
  warp_place(idx, a0, a1, E, fill, perm, inv);
  if (blockIdx.x == 0) {
    const int placed = offsets[E];
    for (int p = placed + threadIdx.x; p < A; p += 32) perm[p] = -1;  // only with bad ids
  }
}

size_t bucket_workspace(const k3moe_shape &s) {
  const long long A = static_cast<long long>(s.T) * s.k;
  const long long ntiles = (A + kTile - 1) / kTile;
  return ntiles > 1 ? static_cast<size_t>(ntiles) * s.E * sizeof(int32_t) : 0;
}

int launch_bucket(const k3moe_shape &s, const int32_t *idx, int32_t *counts, int32_t *offsets,
                  int32_t *perm, int32_t *inv, void *ws, int32_t *status, cudaStream_t st) {
  const int A = s.T * s.k;
  const int ntiles = (A + kTile - 1) / kTile;
  const size_t scan_smem = (2 * static_cast<size_t>(s.E) + 1 + 32) * sizeof(int32_t);
  if (ntiles <= 1) {
    return launch_pdl(bucket_single_kernel, dim3(1), dim3(1024), scan_smem, st, idx, A, s.E, counts,
                      offsets, perm, inv, status) == cudaSuccess
               ? 0
               : -1;
  }
  int32_t *tile = static_cast<int32_t *>(ws);
  const size_t esmem = static_cast<size_t>(s.E) * sizeof(int32_t);
  if (launch_pdl(bucket_hist_kernel, dim3(ntiles), dim3(256), esmem, st, idx, A, s.E, tile,
                 status) != cudaSuccess)
    return -1;
  if (launch_pdl(bucket_scan_kernel, dim3(1), dim3(1024), scan_smem, st, tile, ntiles, s.E, counts,
                 offsets) != cudaSuccess)
    return -1;
  if (launch_pdl(bucket_place_kernel, dim3(ntiles), dim3(32), esmem, st, idx, A, s.E,
                 static_cast<const int32_t *>(tile), static_cast<const int32_t *>(offsets), perm,
                 inv) != cudaSuccess)
    return -1;
  return 0;
}

}  // namespace k3moe
