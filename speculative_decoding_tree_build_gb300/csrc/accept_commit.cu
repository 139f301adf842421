// tv_accept_commit: tv_greedy_accept followed by tv_kv_commit in one kernel.
// The accepted path stays in shared memory between the walk and the row
// moves, and the step has one launch (and one grid-to-grid dependency) less.
// Definitions and behaviour are those of the two calls (see tv_step.cuh).
#include "tv_step.cuh"

namespace tv {

constexpr int kFusedThreads = 256;
constexpr int kFusedStage = 64 * 1024;

__global__ void __launch_bounds__(kFusedThreads)
accept_commit_kernel(const int32_t* __restrict__ target_ids,
                     const int32_t* __restrict__ draft_tokens,
                     const int32_t* __restrict__ cu_nodes, const int32_t* __restrict__ next_token,
                     const int32_t* __restrict__ next_sibling, int max_nodes, int max_depth,
                     int32_t* __restrict__ accept_path, int32_t* __restrict__ accept_len,
                     int32_t* __restrict__ bonus, const int32_t* __restrict__ prompt_len,
                     int32_t* __restrict__ block_table, int32_t* __restrict__ n_blocks,
                     int max_blocks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                     int num_blocks, int hkv, int head_vecs, int32_t* __restrict__ new_len,
                     int32_t* __restrict__ released, int32_t* __restrict__ released_count,
                     int32_t* __restrict__ status) {
  extern __shared__ uint4 stage[];
  __shared__ WalkSmem w;
  __shared__ int s_blk[2 * TV_MAX_NODES];
  __shared__ int s_flag;
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int st = status[b];               // scalars of both stages in one round trip
  const int t0 = cu_nodes[b];
  const int n = cu_nodes[b + 1] - t0;
  const int plen = prompt_len[b];
  const int held = n_blocks[b];
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
  const int a = w.len;
  int32_t* row = accept_path + static_cast<size_t>(b) * (max_depth + 1);
  for (int k = threadIdx.x; k <= max_depth; k += blockDim.x) row[k] = k <= a ? w.path[k] : -1;
  if (threadIdx.x == 0) {
    accept_len[b] = a;
    bonus[b] = w.bonus;
  }
  if (plen < 0 || held < 0 || held > max_blocks) {
    if (threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int flag = commit_rows(w.path, a, plen, held, block_table + static_cast<size_t>(b) * max_blocks,
                               max_blocks, k_cache, v_cache, num_blocks, hkv, head_vecs, stage,
                               kFusedStage, s_blk, &s_flag, &new_len[b],
                               released + static_cast<size_t>(b) * max_blocks, &released_count[b],
                               &n_blocks[b]);
  if (flag && threadIdx.x == 0) atomicOr(&status[b], flag);
}

}  // namespace tv

extern "C" int tv_accept_commit(const tv_geom* geom, const int32_t* target_ids,
                                const int32_t* draft_tokens, const int32_t* cu_nodes,
                                const int32_t* next_token, const int32_t* next_sibling,
                                int32_t batch, int32_t max_nodes, int32_t max_depth,
                                int32_t* accept_path, int32_t* accept_len, int32_t* bonus,
                                const int32_t* prompt_len, int32_t* block_table,
                                int32_t* n_blocks, int32_t max_blocks_per_req, void* k_cache,
                                void* v_cache, int32_t num_blocks, int32_t* new_len,
                                int32_t* released, int32_t* released_count, int32_t* status,
                                void* stream) {
  int rc = tv::check_geom(geom);
  if (rc != TV_OK) return rc;
  rc = tv::check_commit_geom(geom, tv::kFusedStage);
  if (rc != TV_OK) return rc;
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || max_depth < 0 ||
      max_blocks_per_req < 1 || num_blocks < 1)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!target_ids || !draft_tokens || !cu_nodes || !next_token || !next_sibling || !accept_path ||
      !accept_len || !bonus || !prompt_len || !block_table || !n_blocks || !k_cache || !v_cache ||
      !new_len || !released || !released_count || !status)
    return TV_ERR_NULL_POINTER;
  if (!tv::aligned(k_cache, 16) || !tv::aligned(v_cache, 16)) return TV_ERR_MISALIGNED;
  static size_t smem_set[tv::kMaxDevices] = {0};
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  if (!tv::ensure_smem(tv::accept_commit_kernel, tv::kFusedStage, smem_set, dev)) return TV_ERR_CUDA;
  const cudaError_t err = tv::launch_pdl(
      tv::accept_commit_kernel, dim3(batch), dim3(tv::kFusedThreads), tv::kFusedStage,
      tv::as_stream(stream), target_ids, draft_tokens, cu_nodes, next_token, next_sibling,
      static_cast<int>(max_nodes), static_cast<int>(max_depth), accept_path, accept_len, bonus,
      prompt_len, block_table, n_blocks, static_cast<int>(max_blocks_per_req),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), static_cast<int>(num_blocks),
      geom->num_kv_heads, geom->head_dim / 8, new_len, released, released_count, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
