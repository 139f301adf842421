// EAGLE-2 dynamic-tree selection on the device.
//
// Definitions ("02 · Token Tree 与 Tree Attention"): §3 - EAGLE grows the
// tree layer by layer, each step expanding the top-k nodes of the current
// layer; §5 - EAGLE-2 scores every node by its prefix survival probability
// (the product of the drafter's probabilities along its path) and keeps the
// N_tree most promising nodes globally.
//
// A request's candidates come in generation order (a parent before its
// children): the drafter's log-probability of the candidate's token under its
// parent, the parent candidate (-1 for the root's children) and the token.
// One CTA per request stages them in shared memory and
//  - derives every candidate's score (parent's score + own log-probability,
//    float32, in that order) and depth, one tree level per round;
//  - tv_eagle_expand_select: ranks the candidates of one layer (score
//    descending, generation order on ties) and returns the top k;
//  - tv_eagle_rerank: ranks all candidates (score descending, then
//    shallower, then earlier generated), keeps the first n_keep, checks they
//    are prefix-closed and packs them breadth first (depth, parent's packed
//    index, generation order) into a parent list for tv_tree_build.
// Ranks are counts of larger keys in shared memory: exact, order-independent
// and free of sorting networks at these sizes (a few hundred to a few
// thousand candidates). Every thread takes part: a candidate's comparisons
// are split over several threads whose partial counts meet in shared
// memory. The breadth-first packing works on the kept nodes only, gathered
// by their (unique) global rank.
#include "tv_common.cuh"

namespace tv {

constexpr int kEagleThreads = 1024;
constexpr int kEagleMaxCands = 4096;

__device__ __forceinline__ uint32_t eagle_float_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0u;                     // NaN scores rank last
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct EagleSmem {
  float score[kEagleMaxCands];
  int parent[kEagleMaxCands];
  int depth[kEagleMaxCands];
};

// Stage a request's candidates and derive score and depth. Returns the
// request's status flags (the same value in every thread).
__device__ int eagle_stage(const float* logp, const int32_t* parent, int m, EagleSmem& s,
                           float* lp) {
  int bad = 0;
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    const int p = parent[c];
    lp[c] = logp[c];
    s.parent[c] = p;
    s.depth[c] = 0;                          // 0: not derived yet
    if (p < -1 || p >= c) bad = 1;
  }
  if (__syncthreads_or(bad)) return TV_ST_BAD_PARENT;
  // one level per round: a candidate whose parent is derived derives itself
  for (int round = 0; round < m; ++round) {
    int pending = 0;
    for (int c = threadIdx.x; c < m; c += blockDim.x) {
      if (s.depth[c] != 0) continue;
      const int p = s.parent[c];
      if (p < 0) {
        s.score[c] = lp[c];
        s.depth[c] = 1;
      } else if (round > 0 && s.depth[p] == round) {   // parent derived last round
        s.score[c] = __fadd_rn(s.score[p], lp[c]);
        s.depth[c] = round + 1;
      } else {
        pending = 1;
      }
    }
    // candidates derived this round have depth round + 1; they are read as
    // parents only in the next round, after the barrier
    if (!__syncthreads_or(pending)) break;
  }
  return 0;
}


// rank[i] = number of keys larger than key[i], i < n (keys are distinct).
// All threads call it. With fewer keys than threads, each key's comparisons
// are split over up to 32 threads.
__device__ void eagle_rank(const uint64_t* key, int n, int* rank) {
  const int nt = blockDim.x;
  const int slices = n >= nt ? 1 : min(32, nt / max(n, 1));
  for (int i = threadIdx.x; i < n; i += nt) rank[i] = 0;
  __syncthreads();
  const int work = n * slices;
  for (int w = threadIdx.x; w < work; w += nt) {
    const int i = w % n, sl = w / n;
    const int j0 = static_cast<int>(static_cast<long long>(n) * sl / slices);
    const int j1 = static_cast<int>(static_cast<long long>(n) * (sl + 1) / slices);
    const uint64_t ki = key[i];
    int cnt = 0;
    for (int j = j0; j < j1; ++j) cnt += key[j] > ki ? 1 : 0;
    if (slices == 1) rank[i] = cnt;
    else if (cnt) atomicAdd(&rank[i], cnt);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kEagleThreads)
eagle_expand_select_kernel(const float* __restrict__ logp, const int32_t* __restrict__ parent,
                           const int32_t* __restrict__ cand_count, int max_cands, int layer,
                           int k, int32_t* __restrict__ selected, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem[];
  EagleSmem& s = *reinterpret_cast<EagleSmem*>(smem);
  float* lp = reinterpret_cast<float*>(smem + sizeof(EagleSmem));
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int st = status[b];
  const int m = cand_count[b];
  if (st != 0) return;
  if (m < 0 || m > max_cands) {
    if (threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const size_t base = static_cast<size_t>(b) * max_cands;
  const int flags = eagle_stage(logp + base, parent + base, m, s, lp);
  if (flags) {
    if (threadIdx.x == 0) atomicOr(&status[b], flags);
    return;
  }
  uint64_t* key = reinterpret_cast<uint64_t*>(lp + kEagleMaxCands);    // [max_cands]
  int* lc = reinterpret_cast<int*>(key + kEagleMaxCands);               // the layer's candidates
  int* rank = reinterpret_cast<int*>(lp);                               // log-probs no longer needed
  __shared__ int s_nl;
  int32_t* out = selected + static_cast<size_t>(b) * k;
  for (int r = threadIdx.x; r < k; r += blockDim.x) out[r] = -1;
  if (threadIdx.x == 0) s_nl = 0;
  __syncthreads();
  // the layer's candidates (in any order: the key carries the generation index)
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    if (s.depth[c] != layer) continue;
    const int i = atomicAdd(&s_nl, 1);
    lc[i] = c;
    key[i] = (static_cast<uint64_t>(eagle_float_key(s.score[c])) << 32) | static_cast<uint32_t>(~c);
  }
  __syncthreads();
  const int nl = s_nl;
  eagle_rank(key, nl, rank);
  for (int i = threadIdx.x; i < nl; i += blockDim.x)
    if (rank[i] < k) out[rank[i]] = lc[i];
}

__global__ void __launch_bounds__(kEagleThreads)
eagle_rerank_kernel(const float* __restrict__ logp, const int32_t* __restrict__ parent,
                    const int32_t* __restrict__ token, const int32_t* __restrict__ cand_count,
                    int max_cands, int n_keep, const int32_t* __restrict__ root_tokens,
                    int32_t* __restrict__ parents_out, int32_t* __restrict__ tokens_out,
                    int32_t* __restrict__ cu_nodes, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) unsigned char smem[];
  EagleSmem& s = *reinterpret_cast<EagleSmem*>(smem);
  float* lp = reinterpret_cast<float*>(smem + sizeof(EagleSmem));      // [max_cands]
  int* packed = reinterpret_cast<int*>(lp + kEagleMaxCands);           // [max_cands]
  int* start = packed + kEagleMaxCands;                                // [kEagleMaxCands + 2]
  uint64_t* key = reinterpret_cast<uint64_t*>(start + kEagleMaxCands + 2);  // [max_cands]
  int* kn = reinterpret_cast<int*>(key + kEagleMaxCands);              // kept nodes by rank
  int* ppk = kn + TV_MAX_NODES;                                        // parent's packed index
  int* rank = reinterpret_cast<int*>(lp);                              // log-probs no longer needed
  __shared__ int s_maxd;
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int n_out = n_keep + 1;
  if (threadIdx.x == 0) {
    cu_nodes[b] = b * n_out;
    if (b == gridDim.x - 1) cu_nodes[b + 1] = (b + 1) * n_out;
  }
  const int st = status[b];
  const int m = cand_count[b];
  if (st != 0) return;
  if (m < n_keep || m > max_cands) {
    if (threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const size_t base = static_cast<size_t>(b) * max_cands;
  const int flags = eagle_stage(logp + base, parent + base, m, s, lp);
  if (flags) {
    if (threadIdx.x == 0) atomicOr(&status[b], flags);
    return;
  }
  for (int i = threadIdx.x; i < kEagleMaxCands + 2; i += blockDim.x) start[i] = 0;
  if (threadIdx.x == 0) s_maxd = 0;
  // global rank: score descending, then shallower, then earlier generated
  for (int c = threadIdx.x; c < m; c += blockDim.x)
    key[c] = (static_cast<uint64_t>(eagle_float_key(s.score[c])) << 32) |
             static_cast<uint32_t>(~((static_cast<uint32_t>(s.depth[c]) << 12) | c));
  __syncthreads();
  eagle_rank(key, m, rank);
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    const bool kept = rank[c] < n_keep;
    packed[c] = kept ? -2 : -1;
    if (kept) {
      kn[rank[c]] = c;
      atomicAdd(&start[s.depth[c] + 1], 1);
      atomicMax(&s_maxd, s.depth[c]);
    }
  }
  __syncthreads();
  // the kept set must be prefix-closed (a child never outscores its parent
  // unless a log-probability is positive)
  int open = 0;
  for (int c = threadIdx.x; c < m; c += blockDim.x)
    if (packed[c] == -2 && s.parent[c] >= 0 && packed[s.parent[c]] == -1) open = 1;
  if (__syncthreads_or(open)) {
    if (threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int maxd = s_maxd;
  if (threadIdx.x == 0) {
    start[1] = 1;                                          // after the root
    for (int d = 2; d <= maxd; ++d) start[d] += start[d - 1];
  }
  __syncthreads();
  // breadth first over the kept nodes, level by level, by (parent's packed
  // index, generation order): first every kept node of the level notes its
  // parent's packed index (the parents' level is final), then each ranks
  // itself among them
  for (int d = 1; d <= maxd; ++d) {
    for (int i = threadIdx.x; i < n_keep; i += blockDim.x) {
      const int c = kn[i];
      ppk[i] = s.depth[c] != d ? -1 : s.parent[c] < 0 ? 0 : packed[s.parent[c]];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_keep; i += blockDim.x) {
      const int pc = ppk[i];
      if (pc < 0) continue;
      const int c = kn[i];
      int r = 0;
      for (int j = 0; j < n_keep; ++j) {
        const int pj = ppk[j];
        r += (pj >= 0 && (pj < pc || (pj == pc && kn[j] < c))) ? 1 : 0;
      }
      packed[c] = start[d] + r;
    }
    __syncthreads();
  }
  const size_t out0 = static_cast<size_t>(b) * n_out;
  const int32_t* tok = token + base;
  if (threadIdx.x == 0) {
    parents_out[out0] = -1;
    tokens_out[out0] = root_tokens ? root_tokens[b] : -1;
  }
  for (int c = threadIdx.x; c < m; c += blockDim.x) {
    const int pk = packed[c];
    if (pk < 1) continue;
    parents_out[out0 + pk] = s.parent[c] < 0 ? 0 : packed[s.parent[c]];
    tokens_out[out0 + pk] = tok[c];
  }
}

static size_t expand_smem_bytes() {
  return sizeof(EagleSmem) + kEagleMaxCands * (sizeof(float) + sizeof(uint64_t) + sizeof(int));
}
static size_t rerank_smem_bytes() {
  return sizeof(EagleSmem) + kEagleMaxCands * (sizeof(float) + sizeof(int)) +
         (kEagleMaxCands + 2) * sizeof(int) + kEagleMaxCands * sizeof(uint64_t) +
         2 * TV_MAX_NODES * sizeof(int);
}

}  // namespace tv

extern "C" int tv_eagle_expand_select(const float* logp, const int32_t* parent,
                                      const int32_t* cand_count, int32_t batch,
                                      int32_t max_cands, int32_t layer, int32_t k,
                                      int32_t* selected, int32_t* status, void* stream) {
  if (batch < 0 || max_cands < 1 || max_cands > tv::kEagleMaxCands || layer < 1 || k < 1 ||
      k > max_cands)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!logp || !parent || !cand_count || !selected || !status) return TV_ERR_NULL_POINTER;
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  static size_t done[tv::kMaxDevices] = {0};
  const size_t smem = tv::expand_smem_bytes();
  if (!tv::ensure_smem(tv::eagle_expand_select_kernel, smem, done, dev)) return TV_ERR_CUDA;
  const cudaError_t err = tv::launch_pdl(tv::eagle_expand_select_kernel, dim3(batch),
                                         dim3(tv::kEagleThreads), smem, tv::as_stream(stream),
                                         logp, parent, cand_count, static_cast<int>(max_cands),
                                         static_cast<int>(layer), static_cast<int>(k), selected,
                                         status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

extern "C" int tv_eagle_rerank(const float* logp, const int32_t* parent, const int32_t* token,
                               const int32_t* cand_count, int32_t batch, int32_t max_cands,
                               int32_t n_keep, const int32_t* root_tokens, int32_t* parents,
                               int32_t* tokens, int32_t* cu_nodes, int32_t* status,
                               void* stream) {
  if (batch < 0 || max_cands < 1 || max_cands > tv::kEagleMaxCands || n_keep < 1 ||
      n_keep > TV_MAX_NODES - 1 || n_keep > max_cands)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!logp || !parent || !token || !cand_count || !parents || !tokens || !cu_nodes || !status)
    return TV_ERR_NULL_POINTER;
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  static size_t done[tv::kMaxDevices] = {0};
  const size_t smem = tv::rerank_smem_bytes();
  if (!tv::ensure_smem(tv::eagle_rerank_kernel, smem, done, dev)) return TV_ERR_CUDA;
  const cudaError_t err = tv::launch_pdl(tv::eagle_rerank_kernel, dim3(batch),
                                         dim3(tv::kEagleThreads), smem, tv::as_stream(stream),
                                         logp, parent, token, cand_count,
                                         static_cast<int>(max_cands), static_cast<int>(n_keep),
                                         root_tokens, parents, tokens, cu_nodes, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
