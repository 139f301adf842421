// Dense tree-mask export for callers whose attention takes a dense mask.
//
// Definitions: "Beam Search、约束解码与 Tree/Self Speculation", section
// "Packed tree attention" (the tree mask is [N, P+N]: every node sees the
// whole committed prefix and, among the tree nodes, exactly its ancestor
// chain and itself; as bool or as an additive -inf mask) and "02 · Token Tree
// 与 Tree Attention" §3 (the builder's mask modes FULL_MASK and QLEN_ONLY next
// to the bit-packed one this library keeps).
//
// Input: the bit-packed rows of tv_tree_build. Output, request after request
// (row-major, no padding): FULL_MASK [N_b][P_b + N_b], QLEN_ONLY [N_b][N_b];
// elements uint8 (1 visible, 0 masked) or float32 (0 visible, -inf masked).
// One CTA writes kMaskRows rows of one request, one warp per row; each lane
// writes whole 16-byte groups of its row (the row edges, which need not be
// 16-byte aligned, are written with narrower stores). Write-bandwidth-bound
// for long rows, latency-bound at the sizes of one verification step.
#include "tv_common.cuh"

namespace tv {

constexpr int kMaskThreads = 256;
constexpr int kMaskRows = kMaskThreads / 32;     // one warp per row

// Elements before request b's block: sum over earlier requests of N (P + N)
// (or N * N), reduced by the whole CTA.
__device__ long long mask_block_offset(const int32_t* cu_nodes, const int32_t* prompt_len, int b,
                                       bool full, long long* red) {
  long long part = 0;
  for (int i = threadIdx.x; i < b; i += blockDim.x) {
    const long long n = cu_nodes[i + 1] - cu_nodes[i];
    part += n * ((full ? max(prompt_len[i], 0) : 0) + n);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
  __syncthreads();
  long long total = 0;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) total += red[w];
  return total;
}

template <typename T>
__device__ __forceinline__ T mask_value(bool visible);
template <>
__device__ __forceinline__ uint8_t mask_value<uint8_t>(bool visible) { return visible ? 1 : 0; }
template <>
__device__ __forceinline__ float mask_value<float>(bool visible) { return visible ? 0.0f : -INFINITY; }

template <typename T>
__global__ void __launch_bounds__(kMaskThreads)
tree_mask_dense_kernel(const uint32_t* __restrict__ mask_bits, const int32_t* __restrict__ cu_nodes,
                       const int32_t* __restrict__ prompt_len, const int32_t* __restrict__ status,
                       int words, bool full, T* __restrict__ out) {
  __shared__ long long red[kMaskThreads / 32];
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const long long base = mask_block_offset(cu_nodes, prompt_len, b, full, red);
  const int t0 = cu_nodes[b];
  const int n = cu_nodes[b + 1] - t0;
  const int p = full ? max(prompt_len[b], 0) : 0;
  if (status[b] != 0 || n <= 0) return;
  const long long width = static_cast<long long>(p) + n;
  constexpr int kVec = 16 / sizeof(T);                     // elements per 16-byte group
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kMaskRows + static_cast<int>(threadIdx.x >> 5);
  if (r < n) {
    const uint32_t* bits = mask_bits + static_cast<size_t>(t0 + r) * words;
    T* row = out + base + static_cast<long long>(r) * width;
    // element e of the row is visible iff e < p, or bit (e - p) of the row
    auto value = [&](long long e) -> T {
      if (e < p) return mask_value<T>(true);
      const int j = static_cast<int>(e - p);
      return mask_value<T>((bits[j >> 5] >> (j & 31)) & 1u);
    };
    // head up to the first 16-byte boundary, aligned body, tail
    const uintptr_t addr = reinterpret_cast<uintptr_t>(row);
    const long long head = min(width, static_cast<long long>(((16 - (addr & 15)) & 15) / sizeof(T)));
    for (long long e = lane; e < head; e += 32) row[e] = value(e);
    const long long body = (width - head) / kVec;
    for (long long g = lane; g < body; g += 32) {
      const long long e0 = head + g * kVec;
      union { uint4 v; T x[kVec]; } u;
      if (e0 + kVec <= p) {
#pragma unroll
        for (int i = 0; i < kVec; ++i) u.x[i] = mask_value<T>(true);
      } else {
#pragma unroll
        for (int i = 0; i < kVec; ++i) u.x[i] = value(e0 + i);
      }
      *reinterpret_cast<uint4*>(row + e0) = u.v;
    }
    for (long long e = head + body * kVec + lane; e < width; e += 32) row[e] = value(e);
  }
}

}  // namespace tv

extern "C" int tv_tree_mask_dense(const uint32_t* mask_bits, const int32_t* cu_nodes,
                                  const int32_t* prompt_len, const int32_t* status, int32_t batch,
                                  int32_t max_nodes, int32_t mode, int32_t dtype, void* out,
                                  void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || batch > 65535) return TV_ERR_BAD_SIZE;
  if (mode != TV_MASK_FULL && mode != TV_MASK_QLEN_ONLY) return TV_ERR_BAD_SIZE;
  if (dtype != TV_MASK_BOOL && dtype != TV_MASK_ADDITIVE_F32) return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!mask_bits || !cu_nodes || !prompt_len || !status || !out) return TV_ERR_NULL_POINTER;
  if (dtype == TV_MASK_ADDITIVE_F32 && !tv::aligned(out, 4)) return TV_ERR_MISALIGNED;
  const int words = (max_nodes + 31) / 32;
  const dim3 grid((max_nodes + tv::kMaskRows - 1) / tv::kMaskRows, batch);
  const bool full = mode == TV_MASK_FULL;
  cudaError_t err;
  if (dtype == TV_MASK_BOOL)
    err = tv::launch_pdl(tv::tree_mask_dense_kernel<uint8_t>, grid, dim3(tv::kMaskThreads), 0,
                         tv::as_stream(stream), mask_bits, cu_nodes, prompt_len,
                         static_cast<const int32_t*>(status), words, full,
                         static_cast<uint8_t*>(out));
  else
    err = tv::launch_pdl(tv::tree_mask_dense_kernel<float>, grid, dim3(tv::kMaskThreads), 0,
                         tv::as_stream(stream), mask_bits, cu_nodes, prompt_len,
                         static_cast<const int32_t*>(status), words, full,
                         static_cast<float*>(out));
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
