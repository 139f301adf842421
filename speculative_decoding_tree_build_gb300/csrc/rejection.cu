// Rejection-sampling verification along one chosen path.
//
// Definitions: "02 · Token Tree 与 Tree Attention" §4 - the target's one
// forward gives logits at every node; one best path (by path log-probability)
// is chosen and accepted left to right with the min(1, p/q) rule; on a
// rejection a correction token is sampled at the current node, after a fully
// accepted path the bonus token is sampled at the last node. "解码：采样、束
// 搜索和推测性解码" ("Gumbel Max技巧"): argmax_v (log w_v + g_v) draws from
// w / sum(w). The correction is drawn from the residual max(0, p - q) (from p
// when that is zero everywhere), the lossless form of the rule.
//
// One cluster per request (a CTA per vocabulary slice):
//  1. every CTA stages the tree, sums each node's draft log-probabilities
//     from the root (float64, one tree level per round) and walks up from the
//     best leaf to get the path;
//  2. for every path node each CTA reduces its slice of the target row (max,
//     sum of exp(h / T), first argmax) and of the draft row (max, sum of
//     exp(d)); one cluster barrier, then every CTA combines all slices'
//     partials through distributed shared memory into the log-sum-exps;
//  3. the per-edge decisions r < p(x) / q(x) are scalar work (the needed
//     logits are gathered in parallel first), identical in every CTA;
//  4. the stop node's rows are scanned once more for the Gumbel-max draw
//     (residual first, p as the fallback), combined like step 2.
#include "tv_cluster.cuh"

namespace tv {

constexpr int kRejThreads = 1024;
constexpr int kRejMaxPath = 64;          // path nodes reduced per pass (longer paths: several)

struct RejParams {
  const float* target;                   // [T][target_ld]
  const float* draft;                    // [T][draft_ld]
  const float* gumbel;                   // [T][gumbel_ld] or null (greedy requests only)
  const float* uniforms;                 // [T]
  const float* temperature;              // [batch]
  const float* draft_logp;               // [T]
  const int32_t* cu_nodes;
  const int32_t* parents;
  const int32_t* draft_tokens;
  int32_t* accept_path;
  int32_t* accept_len;
  int32_t* bonus;
  int32_t* status;
  long long target_ld, draft_ld, gumbel_ld;
  int max_nodes, max_depth, vocab, csize;
};

// Per path node and CTA slice: target (max, sum of exp(h*inv - max), argmax
// key) and draft (max, sum of exp(d - max)).
struct RejPart {
  float tm, ts, dm, ds;
  uint64_t amax;
};

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float nm = fmaxf(m, m2);
  if (nm == -INFINITY) return;
  s = (m == -INFINITY ? 0.0f : s * fast_exp2((m - nm) * 1.4426950408889634f)) +
      (m2 == -INFINITY ? 0.0f : s2 * fast_exp2((m2 - nm) * 1.4426950408889634f));
  m = nm;
}

__global__ void __launch_bounds__(kRejThreads, 1) rejection_accept_kernel(const __grid_constant__ RejParams p) {
  __shared__ int s_par[TV_MAX_NODES];
  __shared__ int s_path[TV_MAX_NODES];
  __shared__ double s_score[TV_MAX_NODES];
  __shared__ unsigned char s_leaf[TV_MAX_NODES];
  __shared__ RejPart s_part[kRejMaxPath];          // this CTA's partials (read by the cluster)
  __shared__ double s_lse_t[kRejMaxPath], s_lse_d[kRejMaxPath];
  __shared__ int s_amax[kRejMaxPath];
  __shared__ float s_wm[32], s_ws[32], s_wdm[32], s_wds[32];
  __shared__ uint64_t s_wk[32], s_wk2[32];
  __shared__ uint64_t s_draw[2];
  __shared__ double s_hx[kRejMaxPath], s_dx[kRejMaxPath];
  __shared__ int s_plen, s_best, s_stop, s_acc, s_rej;
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int csize = p.csize;
  const int rank = csize > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int st = p.status[b];
  const int t0 = p.cu_nodes[b];
  const int n = p.cu_nodes[b + 1] - t0;
  const float temp = p.temperature[b];
  if (st != 0) return;                                   // uniform across the cluster
  if (n < 1 || n > p.max_nodes) {
    if (rank == 0 && threadIdx.x == 0) atomicOr(&p.status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int tflag = temperature_flags(temp, p.gumbel != nullptr);
  if (tflag) {
    if (rank == 0 && threadIdx.x == 0) atomicOr(&p.status[b], tflag);
    return;
  }
  // ---- 1. path: best cumulative draft log-probability, root to leaf
  int bad_root = 0, bad_par = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int par = p.parents[t0 + i];
    s_par[i] = par;
    s_leaf[i] = 1;
    s_score[i] = i == 0 ? 0.0 : static_cast<double>(p.draft_logp[t0 + i]);
    if (i == 0 && par != -1) bad_root = 1;
    if (i > 0 && (par < 0 || par >= i)) bad_par = 1;
  }
  bad_root = __syncthreads_or(bad_root);
  bad_par = __syncthreads_or(bad_par);
  if (bad_root || bad_par) {
    if (rank == 0 && threadIdx.x == 0)
      atomicOr(&p.status[b], (bad_root ? TV_ST_BAD_ROOT : 0) | (bad_par ? TV_ST_BAD_PARENT : 0));
    return;
  }
  for (int i = threadIdx.x + 1; i < n; i += blockDim.x) s_leaf[s_par[i]] = 0;
  // scores: one tree level per round (a node adds its parent's finished score)
  {
    __shared__ int s_depth[TV_MAX_NODES];
    for (int i = threadIdx.x; i < n; i += blockDim.x) s_depth[i] = i == 0 ? 1 : 0;
    __syncthreads();
    for (int round = 1; round < n; ++round) {
      int pending = 0;
      for (int i = threadIdx.x + 1; i < n; i += blockDim.x) {
        if (s_depth[i] != 0) continue;
        if (s_depth[s_par[i]] == round) {
          s_score[i] = s_score[s_par[i]] + s_score[i];
          s_depth[i] = round + 1;
        } else {
          pending = 1;
        }
      }
      if (!__syncthreads_or(pending)) break;
    }
  }
  {
    // best leaf: largest score, smallest index on ties
    double bs = -INFINITY;
    int bi = INT_MAX;
    for (int i = threadIdx.x; i < n; i += blockDim.x)
      if (s_leaf[i] && (s_score[i] > bs || (s_score[i] == bs && i < bi))) { bs = s_score[i]; bi = i; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (os > bs || (os == bs && oi < bi)) { bs = os; bi = oi; }
    }
    __shared__ double s_bs[32];
    __shared__ int s_bi[32];
    if (lane == 0) { s_bs[warp] = bs; s_bi[warp] = bi; }
    __syncthreads();
    if (threadIdx.x == 0) {
      double cs = s_bs[0];
      int ci = s_bi[0];
      for (int w = 1; w < nw; ++w)
        if (s_bs[w] > cs || (s_bs[w] == cs && s_bi[w] < ci)) { cs = s_bs[w]; ci = s_bi[w]; }
      // walk up, then reverse into root-first order
      int len = 0, u = ci;
      while (u >= 0 && len < TV_MAX_NODES) { s_path[len++] = u; u = s_par[u]; }
      for (int a = 0, z = len - 1; a < z; ++a, --z) { const int t = s_path[a]; s_path[a] = s_path[z]; s_path[z] = t; }
      s_plen = len;
    }
    __syncthreads();
  }
  const int plen = s_plen;
  int v0, v1;
  slice_of(p.vocab, rank, csize, v0, v1);
  const bool sample = temp > 0.0f;
  const float inv_t = sample ? __frcp_rn(temp) : 1.0f;
  const float kL2e = 1.4426950408889634f;
  // ---- 2./3. log-sum-exps of the path rows, then the decisions, in passes
  // of kRejMaxPath path nodes (a pass ends where a rejection happened)
  int acc = 0;                     // accepted edges so far
  int stop = -1;                   // path index of the node the draw happens at
  bool rejected = false;
  for (int base = 0; base < plen && stop < 0; base += kRejMaxPath) {
    const int cnt = min(kRejMaxPath, plen - base);
    for (int k = 0; k < cnt; ++k) {
      const size_t u = static_cast<size_t>(t0 + s_path[base + k]);
      const float* hr = p.target + u * p.target_ld;
      const float* dr = p.draft + u * p.draft_ld;
      float tm = -INFINITY, ts = 0.0f, dm = -INFINITY, ds = 0.0f;
      ThreadBest tb;
      for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
        const float h = __ldcs(hr + v);
        tb.offer(h, v);
        const float x = sample ? __fmul_rn(h, inv_t) : h;
        lse_merge(tm, ts, x, 1.0f);
        lse_merge(dm, ds, __ldcs(dr + v), 1.0f);
      }
      uint64_t key = tb.packed();
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lse_merge(tm, ts, __shfl_xor_sync(0xffffffffu, tm, o), __shfl_xor_sync(0xffffffffu, ts, o));
        lse_merge(dm, ds, __shfl_xor_sync(0xffffffffu, dm, o), __shfl_xor_sync(0xffffffffu, ds, o));
        const uint64_t ok = __shfl_xor_sync(0xffffffffu, key, o);
        key = ok > key ? ok : key;
      }
      if (lane == 0) { s_wm[warp] = tm; s_ws[warp] = ts; s_wdm[warp] = dm; s_wds[warp] = ds; s_wk[warp] = key; }
      __syncthreads();
      if (threadIdx.x == 0) {
        RejPart r = {s_wm[0], s_ws[0], s_wdm[0], s_wds[0], s_wk[0]};
        for (int w = 1; w < nw; ++w) {
          lse_merge(r.tm, r.ts, s_wm[w], s_ws[w]);
          lse_merge(r.dm, r.ds, s_wdm[w], s_wds[w]);
          r.amax = s_wk[w] > r.amax ? s_wk[w] : r.amax;
        }
        s_part[k] = r;
      }
      __syncthreads();
    }
    row_barrier(csize);
    // combine the cluster's partials (each CTA for itself)
    if (threadIdx.x < cnt) {
      const int k = threadIdx.x;
      float tm = -INFINITY, ts = 0.0f, dm = -INFINITY, ds = 0.0f;
      uint64_t am = 0ull;
      for (int r = 0; r < csize; ++r) {
        RejPart q;
        if (csize > 1) {
          const uint64_t* src = reinterpret_cast<const uint64_t*>(&s_part[k]);
          uint64_t w0 = ld_cluster_u64(src, r), w1 = ld_cluster_u64(src + 1, r), w2 = ld_cluster_u64(src + 2, r);
          q.tm = __uint_as_float(static_cast<uint32_t>(w0));
          q.ts = __uint_as_float(static_cast<uint32_t>(w0 >> 32));
          q.dm = __uint_as_float(static_cast<uint32_t>(w1));
          q.ds = __uint_as_float(static_cast<uint32_t>(w1 >> 32));
          q.amax = w2;
        } else {
          q = s_part[k];
        }
        lse_merge(tm, ts, q.tm, q.ts);
        lse_merge(dm, ds, q.dm, q.ds);
        am = q.amax > am ? q.amax : am;
      }
      s_lse_t[k] = static_cast<double>(tm) + log(static_cast<double>(ts));
      s_lse_d[k] = static_cast<double>(dm) + log(static_cast<double>(ds));
      s_amax[k] = best_index(am);
    }
    // the logits of each edge's token, gathered in parallel
    if (threadIdx.x < cnt && base + threadIdx.x + 1 < plen) {
      const int k = threadIdx.x;
      const size_t u = static_cast<size_t>(t0 + s_path[base + k]);
      const int x = p.draft_tokens[t0 + s_path[base + k + 1]];
      const bool inside = x >= 0 && x < p.vocab;
      s_hx[k] = inside ? static_cast<double>(p.target[u * p.target_ld + x]) : -INFINITY;
      s_dx[k] = inside ? static_cast<double>(p.draft[u * p.draft_ld + x]) : -INFINITY;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int a = acc, s_at = -1;
      bool rej = false;
      for (int k = 0; k < cnt; ++k) {
        const int pi = base + k;
        if (pi + 1 >= plen) { s_at = pi; break; }         // the last node: bonus draw
        const int x = p.draft_tokens[t0 + s_path[pi + 1]];
        double pt;
        if (sample) pt = exp(static_cast<double>(__fmul_rn(static_cast<float>(s_hx[k]), inv_t)) - s_lse_t[k]);
        else pt = (x == s_amax[k]) ? 1.0 : 0.0;
        const double qd = exp(s_dx[k] - s_lse_d[k]);
        // a token outside the vocabulary is rejected
        const double ratio = (x < 0 || x >= p.vocab) ? 0.0 : (qd > 0.0 ? pt / qd : INFINITY);
        const double r = static_cast<double>(p.uniforms[t0 + s_path[pi + 1]]);
        if (r < ratio) { ++a; continue; }
        s_at = pi;
        rej = true;
        break;
      }
      s_acc = a;
      s_stop = s_at;
      s_rej = rej;
    }
    __syncthreads();
    acc = s_acc;
    stop = s_stop;
    rejected = s_rej;
    if (stop >= 0) {
      // keep the stop node's log-sum-exps for the draw
      if (threadIdx.x == 0) {
        const int k = stop - base;
        s_lse_t[0] = s_lse_t[k];
        s_lse_d[0] = s_lse_d[k];
        s_amax[0] = s_amax[k];
      }
      __syncthreads();
    }
    row_barrier(csize);                        // partials read before the next pass rewrites them
  }
  // ---- 4. the draw at the stop node
  const size_t su = static_cast<size_t>(t0 + s_path[stop]);
  int tok;
  if (!sample) {
    // all of p on the first argmax: the residual's mass, and p's, sits there
    tok = s_amax[0];
  } else {
    const float* hr = p.target + su * p.target_ld;
    const float* dr = p.draft + su * p.draft_ld;
    const float* gr = p.gumbel + su * p.gumbel_ld;
    const float lt = static_cast<float>(s_lse_t[0]), ld = static_cast<float>(s_lse_d[0]);
    ThreadBest res, pb;
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
      const float x = __fmul_rn(__ldcs(hr + v), inv_t);
      const float g = __ldcs(gr + v);
      pb.offer(__fadd_rn(x, g), v);                      // log p_v + g_v up to a constant
      if (rejected) {
        const float pv = expf(x - lt), qv = expf(__ldcs(dr + v) - ld);
        const float w = pv - qv;
        if (w > 0.0f) res.offer(__fadd_rn(logf(w), g), v);
      }
    }
    uint64_t k1 = res.packed(), k2 = pb.packed();
    k1 = warp_max_u64(k1);
    k2 = warp_max_u64(k2);
    if (lane == 0) { s_wk[warp] = k1; s_wk2[warp] = k2; }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t a1 = 0ull, a2 = 0ull;
      for (int w = 0; w < nw; ++w) { a1 = s_wk[w] > a1 ? s_wk[w] : a1; a2 = s_wk2[w] > a2 ? s_wk2[w] : a2; }
      s_draw[0] = a1;
      s_draw[1] = a2;
    }
    row_barrier(csize);
    uint64_t a1 = 0ull, a2 = 0ull;
    for (int r = 0; r < csize; ++r) {
      const uint64_t x1 = csize > 1 ? ld_cluster_u64(&s_draw[0], r) : s_draw[0];
      const uint64_t x2 = csize > 1 ? ld_cluster_u64(&s_draw[1], r) : s_draw[1];
      a1 = x1 > a1 ? x1 : a1;
      a2 = x2 > a2 ? x2 : a2;
    }
    tok = (rejected && a1 != 0ull) ? best_index(a1) : best_index(a2);
  }
  if (csize > 1) cluster_sync_all();             // remote reads done before any CTA exits
  if (rank != 0) return;
  if (acc > p.max_depth) {
    if (threadIdx.x == 0) atomicOr(&p.status[b], TV_ST_PATH_OVERFLOW);
    return;
  }
  int32_t* row = p.accept_path + static_cast<size_t>(b) * (p.max_depth + 1);
  for (int k = threadIdx.x; k <= p.max_depth; k += blockDim.x) row[k] = k <= acc ? s_path[k] : -1;
  if (threadIdx.x == 0) {
    p.accept_len[b] = acc;
    p.bonus[b] = tok;
  }
}

}  // namespace tv

extern "C" int tv_rejection_accept(const float* target_logits, int64_t target_ld,
                                   const float* draft_logits, int64_t draft_ld,
                                   const float* gumbel, int64_t gumbel_ld, const float* uniforms,
                                   const int32_t* cu_nodes, const float* temperature,
                                   const int32_t* parents, const int32_t* draft_tokens,
                                   const float* draft_logp, int32_t batch, int32_t max_nodes,
                                   int32_t max_depth, int32_t vocab, int32_t* accept_path,
                                   int32_t* accept_len, int32_t* bonus, int32_t* status,
                                   void* stream) {
  if (batch < 0 || max_nodes < 1 || max_nodes > TV_MAX_NODES || max_depth < 0 || batch > 65535 ||
      vocab < 1 || vocab > (1 << 30) || target_ld < vocab || draft_ld < vocab ||
      (gumbel && gumbel_ld < vocab))
    return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!target_logits || !draft_logits || !uniforms || !cu_nodes || !temperature || !parents ||
      !draft_tokens || !draft_logp || !accept_path || !accept_len || !bonus || !status)
    return TV_ERR_NULL_POINTER;
  const int dev = tv::current_device();
  const int sms = dev < 0 ? -1 : tv::device_sm_count(dev);
  if (sms <= 0) return TV_ERR_CUDA;
  int csize = 1;
  while (csize < 8 && batch * csize * 2 * 2 <= sms) csize *= 2;
  tv::RejParams p;
  p.target = target_logits;
  p.draft = draft_logits;
  p.gumbel = gumbel;
  p.uniforms = uniforms;
  p.temperature = temperature;
  p.draft_logp = draft_logp;
  p.cu_nodes = cu_nodes;
  p.parents = parents;
  p.draft_tokens = draft_tokens;
  p.accept_path = accept_path;
  p.accept_len = accept_len;
  p.bonus = bonus;
  p.status = status;
  p.target_ld = target_ld;
  p.draft_ld = draft_ld;
  p.gumbel_ld = gumbel ? gumbel_ld : 0;
  p.max_nodes = max_nodes;
  p.max_depth = max_depth;
  p.vocab = vocab;
  p.csize = csize;
  const cudaError_t err = tv::launch_cluster_pdl(tv::rejection_accept_kernel, dim3(csize, batch),
                                                 dim3(tv::kRejThreads), csize,
                                                 tv::as_stream(stream), p);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
