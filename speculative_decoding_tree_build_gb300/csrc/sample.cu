// Sampling acceptance: the verifier samples its own token at each node.
//
// Definitions:
//  - "解码：采样、束搜索和推测性解码", "高效离散采样" / "Gumbel Max技巧": a draw
//    from Categorical(softmax(h)) is argmax_v (h_v + g_v) with Gumbel noise g;
//    the noise is prepared ahead, so a draw is an add and an argmax.
//  - "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
//    §7.2-§7.3: the verifier walks from the root, picks a token at the current
//    node with its own decoding rule (greedy or temperature sampling), moves to
//    the child carrying that token, and otherwise stops with the token as the
//    next bonus. The walk is lossless whatever the drafter proposed.
//
// Decision rule per node, in float32 exactly as written (no contraction):
//    x_v = fl(fl(h_v * fl(1 / T)) + g_v),  token = first argmax_v x_v;
// T == 0 takes the argmax of h itself. A NaN counts as the largest value and
// +0 equals -0, so the first NaN wins and zeros of either sign tie.
//
// GB300 layout: the node's logits row (and noise row) is split across a
// thread-block cluster; every CTA streams its slice with 128-bit loads and the
// partial argmaxes meet in distributed shared memory. Both kernels are
// HBM-bound streams (8 bytes per vocabulary entry when sampling, 4 greedy).
//
//  sample_tokens_kernel    one cluster per node: the target's choice at every
//                          node of every request.
//  sampled_accept_kernel   one cluster per request: the walk itself. Only the
//                          nodes on the walk are sampled (the others' choices
//                          are never used), one row per step; the cluster
//                          agrees on the next node from the shared partials.
#include "tv_cluster.cuh"

namespace tv {

constexpr int kSampleThreads = 256;
constexpr int kWalkThreads = 1024;
constexpr int kSampleUnroll = 4;      // float4 loads in flight per array per thread

__device__ __forceinline__ float sample_value(float h, float g, float inv_t) {
  return __fadd_rn(__fmul_rn(h, inv_t), g);
}

// Scan logits[v0, v1) (and the noise) of one row; the row start is 16-byte
// aligned and v0 % 4 == 0. Threads tid, tid + nthr, ... of the CTA take
// consecutive float4 groups.
template <bool kSample>
__device__ __forceinline__ uint64_t scan_slice(const float* __restrict__ h_row,
                                               const float* __restrict__ g_row, int v0, int v1,
                                               float inv_t, int tid, int nthr) {
  ThreadBest tb;
  const int nvec = (v1 - v0) >> 2;
  const float4* h4 = reinterpret_cast<const float4*>(h_row + v0);
  const float4* g4 = reinterpret_cast<const float4*>(kSample ? g_row + v0 : h_row + v0);
  int j = tid;
  for (; j + (kSampleUnroll - 1) * nthr < nvec; j += kSampleUnroll * nthr) {
    float4 hv[kSampleUnroll], gv[kSampleUnroll];
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) hv[u] = __ldcs(h4 + j + u * nthr);
    if (kSample) {
#pragma unroll
      for (int u = 0; u < kSampleUnroll; ++u) gv[u] = __ldcs(g4 + j + u * nthr);
    }
#pragma unroll
    for (int u = 0; u < kSampleUnroll; ++u) {
      const int i = v0 + 4 * (j + u * nthr);
      if (kSample) {
        tb.offer(sample_value(hv[u].x, gv[u].x, inv_t), i);
        tb.offer(sample_value(hv[u].y, gv[u].y, inv_t), i + 1);
        tb.offer(sample_value(hv[u].z, gv[u].z, inv_t), i + 2);
        tb.offer(sample_value(hv[u].w, gv[u].w, inv_t), i + 3);
      } else {
        tb.offer(hv[u].x, i);
        tb.offer(hv[u].y, i + 1);
        tb.offer(hv[u].z, i + 2);
        tb.offer(hv[u].w, i + 3);
      }
    }
  }
  for (; j < nvec; j += nthr) {
    const float4 hv = __ldcs(h4 + j);
    const int i = v0 + 4 * j;
    if (kSample) {
      const float4 gv = __ldcs(g4 + j);
      tb.offer(sample_value(hv.x, gv.x, inv_t), i);
      tb.offer(sample_value(hv.y, gv.y, inv_t), i + 1);
      tb.offer(sample_value(hv.z, gv.z, inv_t), i + 2);
      tb.offer(sample_value(hv.w, gv.w, inv_t), i + 3);
    } else {
      tb.offer(hv.x, i);
      tb.offer(hv.y, i + 1);
      tb.offer(hv.z, i + 2);
      tb.offer(hv.w, i + 3);
    }
  }
  // ragged tail (fewer than 4 entries) goes to the threads after the last
  // vector group, which keeps each thread's indices increasing
  const int tail0 = v0 + 4 * nvec;
  if (tail0 + tid < v1 && tid < 4) {
    const int i = tail0 + tid;
    const float x = kSample ? sample_value(__ldcs(h_row + i), __ldcs(g_row + i), inv_t)
                            : __ldcs(h_row + i);
    tb.offer(x, i);
  }
  return tb.packed();
}

// ------------------------------------------------------------ per-node sampling

__global__ void __launch_bounds__(kSampleThreads, 4)
sample_tokens_kernel(const float* __restrict__ logits, long long logits_ld,
                     const float* __restrict__ gumbel, long long gumbel_ld,
                     const int32_t* __restrict__ cu_nodes, const float* __restrict__ temperature,
                     int max_nodes, int vocab, int csize, int32_t* __restrict__ tokens,
                     int32_t* __restrict__ status) {
  __shared__ uint64_t s_red[32];
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int node = blockIdx.x / csize;
  const int rank = csize > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int st = status[b];
  const int t0 = cu_nodes[b];
  const int n = cu_nodes[b + 1] - t0;
  const float temp = temperature[b];
  // every CTA of a cluster takes the same branch below (same b and node)
  if (st != 0 || node >= n) return;
  if (n > max_nodes) {
    if (node == 0 && rank == 0 && threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int tflag = temperature_flags(temp, gumbel != nullptr);
  if (tflag) {
    if (node == 0 && rank == 0 && threadIdx.x == 0) atomicOr(&status[b], tflag);
    return;
  }
  const size_t t = static_cast<size_t>(t0 + node);
  int v0, v1;
  slice_of(vocab, rank, csize, v0, v1);
  const uint64_t best = temp > 0.0f
      ? scan_slice<true>(logits + t * logits_ld, gumbel + t * gumbel_ld, v0, v1,
                         __frcp_rn(temp), threadIdx.x, blockDim.x)
      : scan_slice<false>(logits + t * logits_ld, nullptr, v0, v1, 1.0f, threadIdx.x,
                          blockDim.x);
  publish_warp_best(best, s_red);
  row_barrier(csize);
  if (rank == 0 && threadIdx.x < 32) {
    const uint64_t v = combine_partials(s_red, csize, blockDim.x >> 5);
    if (threadIdx.x == 0) tokens[t] = best_index(v);
  }
  if (csize > 1) cluster_sync_all();    // keep every slot alive until rank 0 has read it
}

// ------------------------------------------------------------------- fused walk

__global__ void __launch_bounds__(kWalkThreads, 1)
sampled_accept_kernel(const float* __restrict__ logits, long long logits_ld,
                      const float* __restrict__ gumbel, long long gumbel_ld,
                      const int32_t* __restrict__ cu_nodes, const float* __restrict__ temperature,
                      const int32_t* __restrict__ parents, const int32_t* __restrict__ draft_tokens,
                      int max_nodes, int max_depth, int vocab, int csize,
                      int32_t* __restrict__ accept_path, int32_t* __restrict__ accept_len,
                      int32_t* __restrict__ bonus, int32_t* __restrict__ status) {
  __shared__ int s_par[TV_MAX_NODES];
  __shared__ int s_tok[TV_MAX_NODES];
  __shared__ int s_path[TV_MAX_NODES];
  __shared__ uint64_t s_red[32];
  __shared__ uint64_t s_cta[2];           // this CTA's maximum, by step parity
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int rank = csize > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int st = status[b];
  const int t0 = cu_nodes[b];
  const int n = cu_nodes[b + 1] - t0;
  const float temp = temperature[b];
  if (st != 0) return;                  // uniform across the cluster
  if (n < 1 || n > max_nodes) {
    if (rank == 0 && threadIdx.x == 0) atomicOr(&status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int tflag = temperature_flags(temp, gumbel != nullptr);
  if (tflag) {
    if (rank == 0 && threadIdx.x == 0) atomicOr(&status[b], tflag);
    return;
  }
  // the tree is staged through registers (n <= 1024 = one node per thread)
  // so that its loads overlap the root row's
  int my_par = -1, my_tok = 0;
  if (threadIdx.x < n) {
    my_par = parents[t0 + threadIdx.x];
    my_tok = draft_tokens[t0 + threadIdx.x];
  }
  int v0, v1;
  slice_of(vocab, rank, csize, v0, v1);
  const bool sample = temp > 0.0f;
  const float inv_t = sample ? __frcp_rn(temp) : 1.0f;
  int cur = 0, len = 0, tok = 0, bad = 0;
  // every warp of every CTA derives the same (cur, len, tok, bad) from the
  // same partials, so all run the loop equally often and meet every barrier
  for (int step = 0;; ++step) {
    const int ph = step & 1;
    const size_t t = static_cast<size_t>(t0 + cur);
    const uint64_t best = sample
        ? scan_slice<true>(logits + t * logits_ld, gumbel + t * gumbel_ld, v0, v1, inv_t,
                           threadIdx.x, blockDim.x)
        : scan_slice<false>(logits + t * logits_ld, nullptr, v0, v1, 1.0f, threadIdx.x,
                            blockDim.x);
    if (step == 0 && threadIdx.x < n) {
      s_par[threadIdx.x] = my_par;
      s_tok[threadIdx.x] = my_tok;
    }
    // CTA maximum first (one barrier), then one value per CTA crosses the
    // cluster: every warp reads the csize values it needs by itself
    publish_warp_best(best, s_red);
    __syncthreads();
    if (warp == 0) {
      uint64_t v = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0ull;
      v = warp_max_u64(v);
      if (lane == 0) s_cta[ph] = v;
    }
    row_barrier(csize);
    tok = best_index(combine_partials(&s_cta[ph], csize, 1));
    // children of cur are later nodes whose parent is cur; the smallest index
    // carrying the token wins. Each warp searches on its own (no barrier).
    int c = -1;
    for (int base = cur + 1; base < n; base += 32) {
      const int i = base + lane;
      const uint32_t m = __ballot_sync(0xffffffffu, i < n && s_par[i] == cur && s_tok[i] == tok);
      if (m) { c = base + __ffs(m) - 1; break; }
    }
    if (c < 0) break;
    if (len + 1 >= n) { bad = 1; break; }             // parents were validated: unreachable
    ++len;
    if (threadIdx.x == 0) s_path[len] = c;
    cur = c;
  }
  if (csize > 1) cluster_sync_all();    // partials stay readable until every CTA is done
  if (rank != 0) return;
  if (threadIdx.x == 0) s_path[0] = 0;
  __syncthreads();
  if (bad || len > max_depth) {
    if (threadIdx.x == 0) atomicOr(&status[b], bad ? TV_ST_BAD_SIZE : TV_ST_PATH_OVERFLOW);
    return;
  }
  int32_t* row = accept_path + static_cast<size_t>(b) * (max_depth + 1);
  for (int k = threadIdx.x; k <= max_depth; k += blockDim.x) row[k] = k <= len ? s_path[k] : -1;
  if (threadIdx.x == 0) {
    accept_len[b] = len;
    bonus[b] = tok;
  }
}

// ------------------------------------------------------------------ host side

static int check_rows(const float* logits, long long logits_ld, const float* gumbel,
                      long long gumbel_ld, int vocab) {
  if (vocab < 1 || vocab > (1 << 30) || logits_ld < vocab || (gumbel && gumbel_ld < vocab))
    return TV_ERR_BAD_SIZE;
  if (!aligned(logits, 16) || (logits_ld & 3)) return TV_ERR_MISALIGNED;
  if (gumbel && (!aligned(gumbel, 16) || (gumbel_ld & 3))) return TV_ERR_MISALIGNED;
  return TV_OK;
}

// Cluster size for the fused walk: the requests' clusters together cover at
// most half the SMs, at most 8 CTAs each (measured on GB300: 16-CTA clusters
// and a fuller machine both lengthened the per-step latency chain).
static int walk_cluster_size(int batch, int dev) {
  const int sms = device_sm_count(dev);
  if (sms <= 0) return -1;
  int c = 1;
  while (c < 8 && batch * c * 2 * 2 <= sms) c *= 2;
  return c;
}

}  // namespace tv

extern "C" int tv_sample_tokens(const float* logits, int64_t logits_ld, const float* gumbel,
                                int64_t gumbel_ld, const int32_t* cu_nodes,
                                const float* temperature, int32_t batch, int32_t max_nodes,
                                int32_t vocab, int32_t* tokens, int32_t* status, void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || batch > 65535)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!logits || !cu_nodes || !temperature || !tokens || !status) return TV_ERR_NULL_POINTER;
  int rc = tv::check_rows(logits, logits_ld, gumbel, gumbel_ld, vocab);
  if (rc != TV_OK) return rc;
  const int dev = tv::current_device();
  const int sms = dev < 0 ? -1 : tv::device_sm_count(dev);
  if (sms <= 0) return TV_ERR_CUDA;
  // One CTA per node streams its row; only when the nodes cannot cover the
  // SMs is a row split over a cluster (measured on GB300: clusters cost more
  // than the last partial wave they would even out once rows >= SMs).
  const long long rows = static_cast<long long>(batch) * max_nodes;
  int csize = 1;
  while (csize < 8 && rows * csize * 2 <= sms && vocab >= csize * 2 * 4096) csize *= 2;
  const cudaError_t err = tv::launch_cluster_pdl(
      tv::sample_tokens_kernel, dim3(max_nodes * csize, batch), dim3(tv::kSampleThreads), csize,
      tv::as_stream(stream), logits, static_cast<long long>(logits_ld), gumbel,
      static_cast<long long>(gumbel_ld), cu_nodes, temperature, static_cast<int>(max_nodes),
      static_cast<int>(vocab), csize, tokens, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

extern "C" int tv_sampled_accept(const float* logits, int64_t logits_ld, const float* gumbel,
                                 int64_t gumbel_ld, const int32_t* cu_nodes,
                                 const float* temperature, const int32_t* parents,
                                 const int32_t* draft_tokens, int32_t batch, int32_t max_nodes,
                                 int32_t max_depth, int32_t vocab, int32_t* accept_path,
                                 int32_t* accept_len, int32_t* bonus, int32_t* status,
                                 void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || max_depth < 0 || batch > 65535)
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!logits || !cu_nodes || !temperature || !parents || !draft_tokens || !accept_path ||
      !accept_len || !bonus || !status)
    return TV_ERR_NULL_POINTER;
  int rc = tv::check_rows(logits, logits_ld, gumbel, gumbel_ld, vocab);
  if (rc != TV_OK) return rc;
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  const int csize = tv::walk_cluster_size(batch, dev);
  if (csize <= 0) return TV_ERR_CUDA;
  const cudaError_t err = tv::launch_cluster_pdl(
      tv::sampled_accept_kernel, dim3(csize, batch), dim3(tv::kWalkThreads), csize,
      tv::as_stream(stream), logits, static_cast<long long>(logits_ld), gumbel,
      static_cast<long long>(gumbel_ld), cu_nodes, temperature, parents, draft_tokens,
      static_cast<int>(max_nodes), static_cast<int>(max_depth), static_cast<int>(vocab), csize,
      accept_path, accept_len, bonus, status);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
