// tv_kv_commit: move the accepted path's tentative K/V rows to the committed
// slots and release the blocks past the new end.
//
// Definition: "Beam Search、约束解码与 Tree/Self Speculation" section
// "Tree/Self Speculation" ([10,11] -> [10,11,4,7]; every other tentative node
// is rolled back), "02 · Token Tree 与 Tree Attention" §4 (the chosen path's KV
// becomes the next round's prompt, the rest is discarded, pages are
// reclaimed) and "投机解码的树状注意力验证…" section "实现中的 KV Cache 与批处理约束"
// (a contiguous tree region in node order; a paged cache frees or reuses
// pages).
//
// Slot P+path[k] moves to slot P+k for k = 1..a. path[k] >= k, so a
// destination slot can be the source of an EARLIER k only. The rows are
// therefore moved in ascending chunks, each chunk staged in shared memory
// (all of its reads before any of its writes); later chunks only read slots
// that no earlier chunk wrote. One CTA per request; byte moves are exact.
#include "tv_step.cuh"

namespace tv {

constexpr int kCommitThreads = 256;
constexpr int kCommitSmem = 64 * 1024;

__global__ void __launch_bounds__(kCommitThreads)
kv_commit_kernel(const int32_t* __restrict__ accept_path, const int32_t* __restrict__ accept_len,
                 int max_depth, const int32_t* __restrict__ prompt_len,
                 int32_t* __restrict__ block_table, int32_t* __restrict__ n_blocks,
                 int max_blocks, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                 int num_blocks, int hkv, int head_vecs, int32_t* __restrict__ new_len,
                 int32_t* __restrict__ released, int32_t* __restrict__ released_count,
                 int32_t* __restrict__ status) {
  extern __shared__ uint4 stage[];
  __shared__ int s_path[TV_MAX_NODES];
  __shared__ int s_blk[2 * TV_MAX_NODES];
  __shared__ int s_flag;
  grid_dependency_wait();                 // inputs written by the previous kernel are visible
  grid_launch_dependents();
  const int b = blockIdx.x;
  // one memory round trip: the request's scalars and its whole path row
  // (max_depth + 1 entries, valid memory whatever the accepted length)
  const int st = status[b];
  const int a = accept_len[b];
  const int plen = prompt_len[b];
  const int held = n_blocks[b];
  const int32_t* path = accept_path + static_cast<size_t>(b) * (max_depth + 1);
  for (int k = threadIdx.x; k <= max_depth && k < TV_MAX_NODES; k += blockDim.x) s_path[k] = path[k];
  __syncthreads();
  if (st != 0) return;
  if (a < 0 || a > max_depth || a >= TV_MAX_NODES || plen < 0 || held < 0 || held > max_blocks) {
    if (threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int flag = commit_rows(s_path, a, plen, held, block_table + static_cast<size_t>(b) * max_blocks,
                               max_blocks, k_cache, v_cache, num_blocks, hkv, head_vecs, stage,
                               kCommitSmem, s_blk, &s_flag, &new_len[b],
                               released + static_cast<size_t>(b) * max_blocks, &released_count[b],
                               &n_blocks[b]);
  if (flag && threadIdx.x == 0) atomicOr(&status[b], flag);
}

}  // namespace tv

extern "C" int tv_kv_commit(const tv_geom* geom, int32_t batch, const int32_t* accept_path,
                            const int32_t* accept_len, int32_t max_depth,
                            const int32_t* prompt_len, int32_t* block_table, int32_t* n_blocks,
                            int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                            int32_t num_blocks, int32_t* new_len, int32_t* released,
                            int32_t* released_count, int32_t* status, void* stream) {
  int rc = tv::check_geom(geom);
  if (rc != TV_OK) return rc;
  rc = tv::check_commit_geom(geom, tv::kCommitSmem);
  if (rc != TV_OK) return rc;
  if (batch < 0 || max_depth < 0 || max_blocks_per_req < 1 || num_blocks < 1)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!accept_path || !accept_len || !prompt_len || !block_table || !n_blocks || !k_cache ||
      !v_cache || !new_len || !released || !released_count || !status)
    return TV_ERR_NULL_POINTER;
  if (!tv::aligned(k_cache, 16) || !tv::aligned(v_cache, 16)) return TV_ERR_MISALIGNED;
  static size_t smem_set[tv::kMaxDevices] = {0};
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  if (!tv::ensure_smem(tv::kv_commit_kernel, tv::kCommitSmem, smem_set, dev)) return TV_ERR_CUDA;
  const int head_vecs = geom->head_dim / 8;
  const cudaError_t err = tv::launch_pdl(
      tv::kv_commit_kernel, dim3(batch), dim3(tv::kCommitThreads), tv::kCommitSmem, tv::as_stream(stream),
      accept_path, accept_len, static_cast<int>(max_depth), prompt_len, block_table, n_blocks,
      static_cast<int>(max_blocks_per_req), static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
      static_cast<int>(num_blocks), geom->num_kv_heads, head_vecs, new_len, released, released_count, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
