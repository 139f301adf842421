// tv_tree_build: parent list -> ancestor bit mask, depth positions,
// retrieve_index / next_token / next_sibling.
//
// Definitions: "02 · Token Tree 与 Tree Attention" §3 (mask rule; positions =
// prompt length + depth, siblings share a position; the builder's outputs) and
// "Beam Search、约束解码与 Tree/Self Speculation" section "Packed tree
// attention" (topologically packed nodes, ancestor-only visibility).
//
// One CTA per request. Integer work only: every output is bit-exact.
#include "tv_common.cuh"

#include <climits>

namespace tv {

constexpr int kBuildThreads = 256;

__global__ void __launch_bounds__(kBuildThreads)
tree_build_kernel(const int32_t* __restrict__ parents, const int32_t* __restrict__ cu_nodes,
                  const int32_t* __restrict__ prompt_len, int max_nodes, int words,
                  uint32_t* __restrict__ mask, int32_t* __restrict__ depth_out,
                  int32_t* __restrict__ positions, int32_t* __restrict__ retrieve_index,
                  int32_t* __restrict__ next_token, int32_t* __restrict__ next_sibling,
                  int32_t* __restrict__ status) {
  __shared__ int s_par[TV_MAX_NODES];
  __shared__ int s_child[TV_MAX_NODES];
  __shared__ int s_bad;
  grid_dependency_wait();                 // inputs written by the previous kernel are visible
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int t0 = cu_nodes[b];
  const int n = cu_nodes[b + 1] - t0;
  const int plen = prompt_len[b];
  if (n < 1 || n > max_nodes || plen < 0) {
    if (threadIdx.x == 0) status[b] = TV_ST_BAD_SIZE;
    return;
  }
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int bad = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int p = parents[t0 + i];
    s_par[i] = p;
    s_child[i] = INT_MAX;
    if (i == 0) {
      if (p != -1) bad |= TV_ST_BAD_ROOT;
    } else if (p < 0 || p >= i) {
      bad |= TV_ST_BAD_PARENT;
    }
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) status[b] = s_bad;
    return;
  }
  for (int i = threadIdx.x + 1; i < n; i += blockDim.x) atomicMin(&s_child[s_par[i]], i);
  __syncthreads();

  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int t = t0 + i;
    // Walk the chain i -> root. Indices strictly decrease along it, so the
    // mask words are produced from the highest word down and each word is
    // written exactly once.
    uint32_t* row = mask + static_cast<size_t>(t) * words;
    int w = words - 1;
    uint32_t acc = 0;
    int d = -1;
    for (int a = i; a != -1; a = s_par[a]) {
      const int aw = a >> 5;
      while (w > aw) {
        row[w] = acc;
        acc = 0;
        --w;
      }
      acc |= 1u << (a & 31);
      ++d;
    }
    for (; w >= 0; --w) {
      row[w] = acc;
      acc = 0;
    }
    depth_out[t] = d;
    positions[t] = plen + d;
    retrieve_index[t] = t;
    const int c = s_child[i];
    next_token[t] = (c == INT_MAX) ? -1 : c;
    int sib = -1;
    if (i != 0) {
      const int p = s_par[i];
      for (int j = i + 1; j < n; ++j) {
        if (s_par[j] == p) {
          sib = j;
          break;
        }
      }
    }
    next_sibling[t] = sib;
  }
  if (threadIdx.x == 0) status[b] = 0;
}

}  // namespace tv

extern "C" int tv_tree_build(const int32_t* parents, const int32_t* cu_nodes,
                             const int32_t* prompt_len, int32_t batch, int32_t max_nodes,
                             uint32_t* mask_bits, int32_t* depth, int32_t* positions,
                             int32_t* retrieve_index, int32_t* next_token,
                             int32_t* next_sibling, int32_t* status, void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES) return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!parents || !cu_nodes || !prompt_len || !mask_bits || !depth || !positions ||
      !retrieve_index || !next_token || !next_sibling || !status)
    return TV_ERR_NULL_POINTER;
  const int words = (max_nodes + 31) / 32;
  const cudaError_t err = tv::launch_pdl(tv::tree_build_kernel, dim3(batch), dim3(tv::kBuildThreads), 0,
                                         tv::as_stream(stream), parents, cu_nodes, prompt_len,
                                         static_cast<int>(max_nodes), words, mask_bits, depth, positions,
                                         retrieve_index, next_token, next_sibling, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
