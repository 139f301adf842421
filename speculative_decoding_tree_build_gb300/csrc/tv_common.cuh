// Shared device/host helpers of libtreeverify (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/treeverify.h"

#define TV_TREE_FLAGS (TV_ST_BAD_SIZE | TV_ST_BAD_ROOT | TV_ST_BAD_PARENT)

namespace tv {

// ---------------------------------------------------------------- host side

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Per-device facts queried once (benign race: every writer stores the same value).
constexpr int kMaxDevices = 64;

inline int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

inline int device_sm_count(int dev) {
  static int cache[kMaxDevices] = {0};
  if (cache[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cache[dev] = sms;
  }
  return cache[dev];
}

// 1 when the device is sm_103 (GB300), 0 otherwise, -1 on error
inline int device_is_sm103(int dev) {
  static int cache[kMaxDevices] = {0};   // 0 unknown, 1 yes, 2 no
  if (cache[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return -1;
    cache[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return cache[dev] == 1 ? 1 : 0;
}

// Raise a kernel's dynamic shared-memory limit once per device (and again
// only if a larger size is needed).
template <typename Kernel>
inline bool ensure_smem(Kernel k, size_t bytes, size_t* done_per_device, int dev) {
  if (done_per_device[dev] >= bytes) return true;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return false;
  done_per_device[dev] = bytes;
  return true;
}

inline int check_geom(const tv_geom* g) {
  if (g == nullptr) return TV_ERR_NULL_POINTER;
  if (g->head_dim != 64 && g->head_dim != 128) return TV_ERR_BAD_GEOMETRY;
  if (g->num_kv_heads < 1 || g->num_q_heads < 1) return TV_ERR_BAD_GEOMETRY;
  if (g->num_q_heads % g->num_kv_heads != 0) return TV_ERR_BAD_GEOMETRY;
  if (g->num_q_heads / g->num_kv_heads > 16) return TV_ERR_BAD_GEOMETRY;
  if (g->block_size != TV_BLOCK_SIZE) return TV_ERR_BAD_GEOMETRY;
  if (!(g->rope_base > 0.0f)) return TV_ERR_BAD_GEOMETRY;
  if (g->rope_style != 0 && g->rope_style != 1) return TV_ERR_BAD_GEOMETRY;
  return TV_OK;
}

// The commit kernels move accepted rows through a shared-memory staging
// buffer of stage_bytes, whole K+V rows (all KV heads) at a time; a geometry
// whose one row does not fit cannot be committed.
inline int check_commit_geom(const tv_geom* g, int stage_bytes) {
  const long long row_bytes = 2ll * g->num_kv_heads * g->head_dim * 2;
  return row_bytes <= stage_bytes ? TV_OK : TV_ERR_BAD_GEOMETRY;
}

// --------------------------------------------------------------- device side

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Pack two floats into a bf16x2 word (lo in bits 0..15), round-to-nearest-even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: a grid launched with programmatic stream
// serialisation may start while the previous grid on the stream runs; it
// must wait here before touching anything that grid reads or writes.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the next grid on the stream (if launched programmatically) to start
// being scheduled; its CTAs still wait in grid_dependency_wait.
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- host launch

// Launch with programmatic stream serialisation. Every kernel launched this
// way calls grid_dependency_wait() before its first global memory access, so
// stream order is kept; what is gained is the launch latency, which overlaps
// the previous grid's tail.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace tv
