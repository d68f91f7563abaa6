// expert_cache.cu -- host-resident MXFP4 experts with a least-recently-used
// arena of expert slots in HBM.
//
// The kimi-k3-in-c engine keeps its 1.45 TB of experts on disk and an LRU cache
// arena of experts in RAM with a batch prefetch just before use ("running a
// 2.78T model in 8 GB", the expert-cache study: raw hits -- the expert is in the
// arena when requested, near 100% because the prefetch has just read it -- and
// TRUE resident hits -- the expert stayed in the arena since the previous step,
// the only measure of avoided reads; 1,472 requests per token, 0% true resident
// hits at an 8 GB budget).  Here the experts live in host memory (Grace
// LPDDR5X, read by the GPU over NVLink-C2C) and the arena is device memory.
//
// One step (k3moe_cache_fetch, after k3moe_bucket) runs two kernels:
//  * cache_plan_kernel (one block): the requested experts are those of the
//    step's range with a nonzero count (a layer's experts inside an arena that
//    caches several layers).  Requested experts already in a slot are true
//    resident hits;
//    each miss takes, in ascending expert order, the next slot of the arena's
//    recency order among the slots not requested this step (least recently used
//    first, ties by slot index; empty slots are the oldest).  The recency order is
//    kept as an array of slots: every step it becomes [slots not used this step,
//    in their order] + [slots used this step, by slot index].  The kernel writes
//    the copy list, updates the device weight tables (pointers into the arena
//    for every resident expert, NULL otherwise: only the entries that change)
//    and adds the step's counters.
//  * cache_copy_kernel: the misses' four arrays, host -> arena, 16-byte loads
//    over the whole grid.
// Every decision is a function of the counts and the previous state, so runs are
// deterministic.
#include <cuda_runtime.h>

#include "k3moe_dev.cuh"
#include "k3moe_launch.h"

namespace k3moe {

namespace {

constexpr int kCacheThreads = 1024;

__host__ __device__ inline size_t c_align(size_t v) { return (v + 255) & ~size_t(255); }

// Byte sizes of one expert's four arrays and their offsets inside a slot.
struct SlotLayout {
  size_t sz[4], off[4], slot;
};

__host__ __device__ inline SlotLayout slot_layout(int H, int I) {
  SlotLayout L;
  L.sz[0] = static_cast<size_t>(2) * I * (H / 2);
  L.sz[1] = static_cast<size_t>(2) * I * (H / 32);
  L.sz[2] = static_cast<size_t>(H) * (I / 2);
  L.sz[3] = static_cast<size_t>(H) * (I / 32);
  size_t o = 0;
  for (int q = 0; q < 4; ++q) {
    L.off[q] = o;
    o = c_align(o + L.sz[q]);
  }
  L.slot = o;
  return L;
}

// Arena layout: bookkeeping first, then the slots.
struct ArenaLayout {
  size_t slot_of, expert_of, order, order_tmp, used, tables, copy, meta, slots, total;
};

__host__ __device__ inline ArenaLayout arena_layout(int E, int S, int H, int I) {
  ArenaLayout A;
  size_t o = 0;
  A.slot_of = o;   o = c_align(o + sizeof(int32_t) * E);       // slot of each expert, -1 = not resident
  A.expert_of = o; o = c_align(o + sizeof(int32_t) * S);       // expert in each slot, -1 = empty
  A.order = o;     o = c_align(o + sizeof(int32_t) * S);       // slots, least recently used first
  A.order_tmp = o; o = c_align(o + sizeof(int32_t) * S);
  A.used = o;      o = c_align(o + sizeof(int32_t) * S);       // per slot: requested this step
  A.tables = o;    o = c_align(o + sizeof(void *) * 4 * static_cast<size_t>(E));  // 4 device pointer arrays
  A.copy = o;      o = c_align(o + sizeof(int2) * (E < S ? E : S));  // {slot, expert} per miss
  A.meta = o;      o = c_align(o + sizeof(int32_t) * 8);       // [0] misses this step
  A.slots = o;
  A.total = o + static_cast<size_t>(S) * slot_layout(H, I).slot;
  return A;
}

// Exclusive scan of one int per thread over the block (1024 threads); returns
// the block total through *total.
__device__ __forceinline__ int block_excl_scan(int v, int *buf, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
    if (lane >= off) inc += o;
  }
  __syncthreads();
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = buf[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, wi, off);
      if (lane >= off) wi += o;
    }
    buf[lane] = wi - w;  // exclusive prefix of the warp totals
    if (lane == 31) buf[32] = wi;
  }
  __syncthreads();
  const int r = buf[warp] + inc - v;
  *total = buf[32];
  return r;
}

}  // namespace

__global__ void __launch_bounds__(kCacheThreads) cache_init_kernel(int E, int S, uint8_t *arena) {
  const ArenaLayout A = arena_layout(E, S, 1, 1);  // bookkeeping offsets do not depend on H, I
  int32_t *slot_of = reinterpret_cast<int32_t *>(arena + A.slot_of);
  int32_t *expert_of = reinterpret_cast<int32_t *>(arena + A.expert_of);
  int32_t *order = reinterpret_cast<int32_t *>(arena + A.order);
  uint8_t **tables = reinterpret_cast<uint8_t **>(arena + A.tables);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    slot_of[e] = -1;
    for (int q = 0; q < 4; ++q) tables[q * static_cast<size_t>(E) + e] = nullptr;
  }
  for (int v = threadIdx.x; v < S; v += blockDim.x) {
    expert_of[v] = -1;
    order[v] = v;
  }
}

__global__ void __launch_bounds__(kCacheThreads)
    cache_plan_kernel(int E, int S, int H, int I, uint8_t *arena, const int32_t *__restrict__ counts, int cbase,
                      int cn, unsigned long long *stats, int32_t *status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int buf[33];
  const ArenaLayout A = arena_layout(E, S, H, I);
  const SlotLayout L = slot_layout(H, I);
  int32_t *slot_of = reinterpret_cast<int32_t *>(arena + A.slot_of);
  int32_t *expert_of = reinterpret_cast<int32_t *>(arena + A.expert_of);
  int32_t *order = reinterpret_cast<int32_t *>(arena + A.order);
  int32_t *order_tmp = reinterpret_cast<int32_t *>(arena + A.order_tmp);
  int32_t *used = reinterpret_cast<int32_t *>(arena + A.used);
  uint8_t **tables = reinterpret_cast<uint8_t **>(arena + A.tables);
  int2 *copy = reinterpret_cast<int2 *>(arena + A.copy);
  int32_t *meta = reinterpret_cast<int32_t *>(arena + A.meta);
  uint8_t *slots = arena + A.slots;
  const int tid = threadIdx.x, nth = blockDim.x;

  // 1. hits: requested experts with a slot mark it used
  for (int v = tid; v < S; v += nth) used[v] = 0;
  __syncthreads();
  int nreq = 0, nhit = 0;
  for (int i = tid; i < cn; i += nth) {
    if (counts[i] > 0) {
      ++nreq;
      const int v = slot_of[cbase + i];
      if (v >= 0) {
        ++nhit;
        used[v] = 1;
      }
    }
  }
  __syncthreads();
  // 2. misses in ascending expert order (chunks of the requested range per thread)
  const int per_e = (cn + nth - 1) / nth;
  const int e0 = tid * per_e;
  int nm = 0;
  for (int i = e0; i < e0 + per_e && i < cn; ++i) nm += counts[i] > 0 && slot_of[cbase + i] < 0;
  int total_miss;
  int mbase = block_excl_scan(nm, buf, &total_miss);
  // 3. victims: the first total_miss slots of the recency order that are not used this step
  const int per_s = (S + nth - 1) / nth;
  const int p0 = tid * per_s;
  int nu = 0;
  for (int p = p0; p < p0 + per_s && p < S; ++p) nu += !used[order[p]];
  int total_unused;
  int ubase = block_excl_scan(nu, buf, &total_unused);
  if (total_miss > total_unused) {  // more distinct experts requested than slots: refuse the step
    if (tid == 0) {
      meta[0] = 0;
      set_status(status, K3MOE_DEV_BOUNDS);
    }
    return;
  }
  // victim j of the recency order -> copy[j].x
  for (int p = p0, r = ubase; p < p0 + per_s && p < S; ++p) {
    const int v = order[p];
    if (!used[v]) {
      if (r < total_miss) copy[r].x = v;
      ++r;
    }
  }
  __syncthreads();
  // miss j (ascending expert) -> copy[j].y; the victim's previous expert leaves
  for (int i = e0, r = mbase; i < e0 + per_e && i < cn; ++i) {
    if (counts[i] > 0 && slot_of[cbase + i] < 0) {
      copy[r].y = cbase + i;
      ++r;
    }
  }
  __syncthreads();
  for (int j = tid; j < total_miss; j += nth) {
    const int old = expert_of[copy[j].x];
    if (old >= 0) {
      slot_of[old] = -1;
      for (int q = 0; q < 4; ++q) tables[q * static_cast<size_t>(E) + old] = nullptr;
    }
  }
  __syncthreads();
  for (int j = tid; j < total_miss; j += nth) {
    const int v = copy[j].x, e = copy[j].y;
    expert_of[v] = e;
    slot_of[e] = v;
    used[v] = 1;
    for (int q = 0; q < 4; ++q) tables[q * static_cast<size_t>(E) + e] = slots + static_cast<size_t>(v) * L.slot + L.off[q];
  }
  __syncthreads();
  // 4. recency order: [not used, in order] + [used, by slot index]
  int nkeep = 0;
  for (int p = p0; p < p0 + per_s && p < S; ++p) nkeep += !used[order[p]];
  int kept;
  int kbase = block_excl_scan(nkeep, buf, &kept);
  for (int p = p0, r = kbase; p < p0 + per_s && p < S; ++p)
    if (!used[order[p]]) order_tmp[r++] = order[p];
  int nused = 0;
  for (int v = p0; v < p0 + per_s && v < S; ++v) nused += used[v];
  int tot_used;
  int ubase2 = block_excl_scan(nused, buf, &tot_used);
  for (int v = p0, r = kept + ubase2; v < p0 + per_s && v < S; ++v)
    if (used[v]) order_tmp[r++] = v;
  __syncthreads();
  for (int p = tid; p < S; p += nth) order[p] = order_tmp[p];
  // 5. counters: sum the per-thread request and hit counts
  int treq, thit;
  block_excl_scan(nreq, buf, &treq);
  block_excl_scan(nhit, buf, &thit);
  if (tid == 0) {
    meta[0] = total_miss;
    if (stats) {
      stats[0] += static_cast<unsigned long long>(treq);   // requests
      stats[1] += static_cast<unsigned long long>(treq);   // raw hits: every request is served from the arena
      stats[2] += static_cast<unsigned long long>(thit);   // true resident hits
      stats[3] += static_cast<unsigned long long>(total_miss) * (L.sz[0] + L.sz[1] + L.sz[2] + L.sz[3]);
    }
  }
}

// Copy the misses' arrays from host memory into their slots: the grid walks
// (miss, array, 16-byte word) with every array a multiple of 16 bytes.
__global__ void __launch_bounds__(256)
    cache_copy_kernel(int E, int S, int H, int I, uint8_t *arena, k3moe_weights host_w) {
  pdl_wait();
  pdl_trigger();
  const ArenaLayout A = arena_layout(E, S, H, I);
  const SlotLayout L = slot_layout(H, I);
  const int2 *copy = reinterpret_cast<const int2 *>(arena + A.copy);
  const int nmiss = reinterpret_cast<const int32_t *>(arena + A.meta)[0];
  uint8_t *slots = arena + A.slots;
  const size_t words[4] = {L.sz[0] / 16, L.sz[1] / 16, L.sz[2] / 16, L.sz[3] / 16};
  const size_t per = words[0] + words[1] + words[2] + words[3];
  const size_t total = per * static_cast<size_t>(nmiss);
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  constexpr int U = 4;  // loads in flight per thread
  for (size_t base = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < total; base += U * stride) {
    uint4 v[U];
    uint4 *dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const size_t w = base + u * stride;
      dst[u] = nullptr;
      if (w < total) {
        const int j = static_cast<int>(w / per);
        size_t r = w % per;
        int q = 0;
        while (q < 3 && r >= words[q]) r -= words[q++];
        const int2 c = copy[j];
        const uint8_t *const *arr = q == 0 ? host_w.w13_codes : q == 1 ? host_w.w13_scales
                                    : q == 2 ? host_w.w2_codes : host_w.w2_scales;
        const uint4 *src = reinterpret_cast<const uint4 *>(arr[c.y]);
        v[u] = src ? src[r] : make_uint4(0, 0, 0, 0);
        dst[u] = reinterpret_cast<uint4 *>(slots + static_cast<size_t>(c.x) * L.slot + L.off[q]) + r;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u]) *dst[u] = v[u];
  }
}

size_t cache_arena_bytes(const k3moe_shape &s, int slots) { return arena_layout(s.E, slots, s.H, s.I).total; }

void cache_tables(const k3moe_shape &s, int slots, void *arena, k3moe_weights *out) {
  const ArenaLayout A = arena_layout(s.E, slots, s.H, s.I);
  uint8_t **t = reinterpret_cast<uint8_t **>(static_cast<uint8_t *>(arena) + A.tables);
  out->w13_codes = t;
  out->w13_scales = t + s.E;
  out->w2_codes = t + 2 * static_cast<size_t>(s.E);
  out->w2_scales = t + 3 * static_cast<size_t>(s.E);
}

int launch_cache_init(const k3moe_shape &s, int slots, void *arena, cudaStream_t st) {
  cache_init_kernel<<<1, kCacheThreads, 0, st>>>(s.E, slots, static_cast<uint8_t *>(arena));
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_cache_fetch(const k3moe_shape &s, int slots, void *arena, const k3moe_weights &host_w,
                       const int32_t *counts, int cbase, int cn, unsigned long long *stats, int32_t *status,
                       cudaStream_t st) {
  if (launch_pdl(cache_plan_kernel, dim3(1), dim3(kCacheThreads), 0, st, s.E, slots, s.H, s.I,
                 static_cast<uint8_t *>(arena), counts, cbase, cn, stats, status) != cudaSuccess)
    return -1;
  return launch_pdl(cache_copy_kernel, dim3(4 * sm_count()), dim3(256), 0, st, s.E, slots, s.H, s.I,
                    static_cast<uint8_t *>(arena), host_w) == cudaSuccess
             ? 0
             : -1;
}

}  // namespace k3moe
