// Thread-block-cluster helpers shared by the kernels that split a row over a
// cluster and meet in distributed shared memory (sampling, rejection
// acceptance): cluster rank and barrier, remote shared-memory loads, a total
// order on float32 values with (key, index) packing for first-maximum
// argmaxes, and a launch with a cluster shape and programmatic serialisation.
#pragma once

#include "tv_common.cuh"

namespace tv {

// --------------------------------------------------------------- cluster helpers

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ uint64_t ld_cluster_u64(const void* local, uint32_t rank) {
  uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(r) : "memory");
  return v;
}

// ------------------------------------------------------------ argmax machinery

// Total order of float32 values as unsigned keys: NaN above +inf, -0 == +0.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0xFFFFFFFFu;
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (key, index) packed so that the unsigned maximum is the largest key with
// the smallest index. 0 is below every real candidate.
__device__ __forceinline__ uint64_t pack_best(uint32_t key, int idx) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~idx);
}
__device__ __forceinline__ int best_index(uint64_t p) {
  return static_cast<int>(~static_cast<uint32_t>(p));
}

struct ThreadBest {
  uint32_t key = 0;
  int idx = -1;
  // indices reach a thread in increasing order, so strict > keeps the first
  __device__ __forceinline__ void offer(float x, int i) {
    const uint32_t k = order_key(x);
    if (k > key) { key = k; idx = i; }
  }
  __device__ __forceinline__ uint64_t packed() const { return idx < 0 ? 0ull : pack_best(key, idx); }
};

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Slice [v0, v1) of a vocab of `vocab` entries for CTA `rank` of `csize`.
__device__ __forceinline__ void slice_of(int vocab, int rank, int csize, int& v0, int& v1) {
  const int per = ((vocab + csize - 1) / csize + 3) & ~3;
  v0 = min(vocab, rank * per);
  v1 = min(vocab, v0 + per);
}

// Checks shared by both kernels; the result is the same in every CTA of a
// cluster (it depends only on the request's inputs).
__device__ __forceinline__ int temperature_flags(float t, bool have_noise) {
  if (t != t || t < 0.0f) return TV_ST_BAD_TEMPERATURE;
  if (t > 0.0f && !have_noise) return TV_ST_BAD_TEMPERATURE;
  return 0;
}

// Partials of one row: each warp publishes its maximum in s_red[warp]; after
// the barrier (cluster-wide when the row is split over a cluster) a warp
// combines the csize x nw partials, reading the other CTAs' slots through
// distributed shared memory.
__device__ __forceinline__ void publish_warp_best(uint64_t v, uint64_t* s_red) {
  v = warp_max_u64(v);
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = v;
}

__device__ __forceinline__ uint64_t combine_partials(const uint64_t* s_red, int csize, int nw) {
  const int lane = threadIdx.x & 31;
  uint64_t v = 0ull;
  for (int j = lane; j < csize * nw; j += 32) {
    const int r = j / nw, w = j - r * nw;
    const uint64_t x = csize > 1 ? ld_cluster_u64(&s_red[w], r) : s_red[w];
    v = x > v ? x : v;
  }
  return warp_max_u64(v);
}

__device__ __forceinline__ void row_barrier(int csize) {
  if (csize > 1) cluster_sync_all();    // also a barrier of this CTA's threads
  else __syncthreads();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, int csize,
                                      cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = csize;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace tv
