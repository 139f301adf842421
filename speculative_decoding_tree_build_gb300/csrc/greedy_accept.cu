// tv_greedy_accept: greedy walk of the candidate tree against the target's
// per-node greedy tokens.
//
// Definition: "02 · Token Tree 与 Tree Attention" §4 (from the root accept the
// child whose token equals the target's choice and continue from it; when no
// child matches the target's token is the correction), "Beam Search、约束解码与
// Tree/Self Speculation" three-part experiment (verify_tree keeps the branches
// matching the target at each depth and stops at the first miss) and
// "Accelerating Speculative Decoding with Block Diffusion Draft Trees" §7.2
// (the first mismatching target token becomes the next bonus token).
//
// One CTA per request: the request's arrays are staged into shared memory
// with coalesced loads, then one thread walks first-child / next-sibling links
// there (shared-memory latency instead of a chain of dependent global loads).
#include "tv_step.cuh"

namespace tv {

constexpr int kAcceptThreads = 128;

__global__ void __launch_bounds__(kAcceptThreads)
greedy_accept_kernel(const int32_t* __restrict__ target_ids,
                     const int32_t* __restrict__ draft_tokens,
                     const int32_t* __restrict__ cu_nodes, const int32_t* __restrict__ next_token,
                     const int32_t* __restrict__ next_sibling, int max_nodes, int max_depth,
                     int32_t* __restrict__ accept_path, int32_t* __restrict__ accept_len,
                     int32_t* __restrict__ bonus, int32_t* __restrict__ status) {
  __shared__ WalkSmem w;
  grid_dependency_wait();                 // inputs written by the previous kernel are visible
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int st = status[b];               // loaded together with the node range
  const int t0 = cu_nodes[b];
  const int n = cu_nodes[b + 1] - t0;
  if (st != 0) return;
  if (n < 1 || n > max_nodes) {
    if (threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  greedy_walk(target_ids, draft_tokens, next_token, next_sibling, t0, n, max_depth, w);
  if (w.bad) {
    if (threadIdx.x == 0) atomicOr(&status[b], w.bad);
    return;
  }
  const int len = w.len;
  int32_t* row = accept_path + static_cast<size_t>(b) * (max_depth + 1);
  for (int k = threadIdx.x; k <= max_depth; k += blockDim.x) row[k] = k <= len ? w.path[k] : -1;
  if (threadIdx.x == 0) {
    accept_len[b] = len;
    bonus[b] = w.bonus;
  }
}

}  // namespace tv

extern "C" int tv_greedy_accept(const int32_t* target_ids, const int32_t* draft_tokens,
                                const int32_t* cu_nodes, const int32_t* next_token,
                                const int32_t* next_sibling, int32_t batch, int32_t max_nodes,
                                int32_t max_depth, int32_t* accept_path, int32_t* accept_len,
                                int32_t* bonus, int32_t* status, void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || max_depth < 0)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!target_ids || !draft_tokens || !cu_nodes || !next_token || !next_sibling ||
      !accept_path || !accept_len || !bonus || !status)
    return TV_ERR_NULL_POINTER;
  const cudaError_t err = tv::launch_pdl(tv::greedy_accept_kernel, dim3(batch), dim3(tv::kAcceptThreads), 0,
                                         tv::as_stream(stream), target_ids, draft_tokens, cu_nodes,
                                         next_token, next_sibling, static_cast<int>(max_nodes),
                                         static_cast<int>(max_depth), accept_path, accept_len, bonus, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
