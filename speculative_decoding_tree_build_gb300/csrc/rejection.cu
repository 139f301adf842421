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
//     from the root (float64, one tree level per round), picks the best leaf
//     by integer keys of those sums and walks up from it to get the path;
//  2. the CTA's warps split the path rows of a pass (a row per warp at most) between
//     them and reduce their segment of each row with 128-bit loads: sampling
//     requests keep the online maximum and sum of exp(h / T) and of exp(d)
//     (the log-sum-exps of p and q), greedy ones only the first argmax of h
//     (p is one-hot, so q never matters and the drafter's rows are not read);
//  3. one cluster barrier, then one warp per path row combines the cluster's
//     partials (a lane per CTA, through distributed shared memory) and
//     decides its edge, r < p(x) / q(x); a ballot finds the first rejection;
//  4. sampling requests scan the stop node's rows once more for the
//     Gumbel-max draw (residual first, p as the fallback).
#include "tv_cluster.cuh"

namespace tv {

constexpr int kRejThreads = 512;
constexpr int kRejWarps = kRejThreads / 32;
constexpr int kRejMaxPath = kRejWarps;   // path rows per pass: at least one warp per row
constexpr int kRejUnroll = 4;            // float4 loads in flight per lane and row array
constexpr float kRejLog2e = 1.4426950408889634f;
static_assert(kRejWarps <= 32, "one lane per warp in the block-level maxima");

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
  int vec;                               // bit 0/1/2: target/draft/noise rows 16-byte aligned
};

// One (row, slice) partial: target (max, sum of exp(h/T - max)), drafter
// (max, sum of exp(d - max)), packed first-argmax key of h. 24 bytes, read
// remotely as three 64-bit words.
struct RejPart {
  float tm, ts, dm, ds;
  uint64_t amax;
};

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float nm = fmaxf(m, m2);
  if (nm == -INFINITY) return;
  s = (m == -INFINITY ? 0.0f : s * fast_exp2((m - nm) * kRejLog2e)) +
      (m2 == -INFINITY ? 0.0f : s2 * fast_exp2((m2 - nm) * kRejLog2e));
  m = nm;
}

// Running maximum m and sum s of exp(x - m); -inf entries add nothing.
__device__ __forceinline__ void online_add(float& m, float& s, float x) {
  if (x > m) {
    s = s * fast_exp2((m - x) * kRejLog2e) + 1.0f;
    m = x;
  } else if (x != -INFINITY) {
    s += fast_exp2((x - m) * kRejLog2e);
  }
}

// Four entries at once: one rescale at most. exp2 of -inf is 0, so -inf
// entries (and the empty start, m = -inf, s = 0) need no test.
__device__ __forceinline__ void online_add4(float& m, float& s, float a, float b, float c,
                                            float d) {
  const float mx = fmaxf(fmaxf(a, b), fmaxf(c, d));
  if (mx == -INFINITY) return;
  if (mx > m) {
    s *= fast_exp2((m - mx) * kRejLog2e);
    m = mx;
  }
  s += (fast_exp2((a - m) * kRejLog2e) + fast_exp2((b - m) * kRejLog2e)) +
       (fast_exp2((c - m) * kRejLog2e) + fast_exp2((d - m) * kRejLog2e));
}

// Total order on float64 path sums as unsigned keys (NaN as -inf, -0 as +0),
// so the best leaf is found with integer reductions (float64 is slow here);
// every key is above 0, the key of "no leaf".
__device__ __forceinline__ uint64_t score_key(double x) {
  uint64_t u = static_cast<uint64_t>(__double_as_longlong(x));
  const uint64_t mag = u & 0x7FFFFFFFFFFFFFFFull;
  if (mag > 0x7FF0000000000000ull) u = 0xFFF0000000000000ull;   // NaN -> -inf
  if (mag == 0) u = 0;                                           // -0 -> +0
  return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// Warp-wide (largest key, smallest index among it); lanes without a
// candidate hold (0, INT_MAX).
__device__ __forceinline__ void warp_best_leaf(uint64_t& key, int& idx) {
  const uint32_t hi = static_cast<uint32_t>(key >> 32), lo = static_cast<uint32_t>(key);
  const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? lo : 0u);
  idx = __reduce_min_sync(0xffffffffu, (hi == mhi && lo == mlo) ? idx : INT_MAX);
  key = (static_cast<uint64_t>(mhi) << 32) | mlo;
}

__device__ __forceinline__ void part_identity(RejPart& r) {
  r.tm = -INFINITY; r.ts = 0.0f; r.dm = -INFINITY; r.ds = 0.0f; r.amax = 0ull;
}

__device__ __forceinline__ void part_merge(RejPart& a, const RejPart& b) {
  lse_merge(a.tm, a.ts, b.tm, b.ts);
  lse_merge(a.dm, a.ds, b.dm, b.ds);
  a.amax = b.amax > a.amax ? b.amax : a.amax;
}

__device__ __forceinline__ RejPart part_shfl_xor(const RejPart& a, int o) {
  RejPart r;
  r.tm = __shfl_xor_sync(0xffffffffu, a.tm, o);
  r.ts = __shfl_xor_sync(0xffffffffu, a.ts, o);
  r.dm = __shfl_xor_sync(0xffffffffu, a.dm, o);
  r.ds = __shfl_xor_sync(0xffffffffu, a.ds, o);
  r.amax = __shfl_xor_sync(0xffffffffu, a.amax, o);
  return r;
}

__device__ __forceinline__ RejPart part_warp_merge(RejPart a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) part_merge(a, part_shfl_xor(a, o));
  return a;
}

// One element of a path row: greedy keeps the first argmax of h, sampling
// the two running log-sum-exps.
template <bool kSample>
__device__ __forceinline__ void row_element(RejPart& r, ThreadBest& tb, float h, float d, int v,
                                            float inv_t) {
  if (kSample) {
    online_add(r.tm, r.ts, __fmul_rn(h, inv_t));
    online_add(r.dm, r.ds, d);
  } else {
    tb.offer(h, v);
  }
}

// A warp's reduction of columns [a, b) of one target row (and drafter row
// when sampling). a is a multiple of 4; with `vec` the rows are read as
// float4, kRejUnroll loads in flight per lane and array.
template <bool kSample>
__device__ __forceinline__ RejPart reduce_segment(const float* hr, const float* dr, int a, int b,
                                                  bool vec, float inv_t, int lane) {
  RejPart r;
  part_identity(r);
  ThreadBest tb;
  if (vec) {
    const int b4 = a + ((b - a) & ~3);
    for (int v = a + lane * 4; v < b4; v += kRejUnroll * 128) {
      float4 h4[kRejUnroll], d4[kRejUnroll];
#pragma unroll
      for (int j = 0; j < kRejUnroll; ++j) {
        const int vj = v + j * 128;
        if (vj < b4) {
          h4[j] = __ldcs(reinterpret_cast<const float4*>(hr + vj));
          if (kSample) d4[j] = __ldcs(reinterpret_cast<const float4*>(dr + vj));
        }
      }
#pragma unroll
      for (int j = 0; j < kRejUnroll; ++j) {
        const int vj = v + j * 128;
        if (vj < b4) {
          if (kSample) {
            online_add4(r.tm, r.ts, __fmul_rn(h4[j].x, inv_t), __fmul_rn(h4[j].y, inv_t),
                        __fmul_rn(h4[j].z, inv_t), __fmul_rn(h4[j].w, inv_t));
            online_add4(r.dm, r.ds, d4[j].x, d4[j].y, d4[j].z, d4[j].w);
          } else {
            tb.offer(h4[j].x, vj);
            tb.offer(h4[j].y, vj + 1);
            tb.offer(h4[j].z, vj + 2);
            tb.offer(h4[j].w, vj + 3);
          }
        }
      }
    }
    for (int v = b4 + lane; v < b; v += 32)
      row_element<kSample>(r, tb, __ldcs(hr + v), kSample ? __ldcs(dr + v) : 0.0f, v, inv_t);
  } else {
#pragma unroll 4
    for (int v = a + lane; v < b; v += 32)
      row_element<kSample>(r, tb, __ldcs(hr + v), kSample ? __ldcs(dr + v) : 0.0f, v, inv_t);
  }
  r.amax = tb.packed();
  return part_warp_merge(r);
}

}  // namespace tv

namespace tv {

// Draw keys of one element of the stop row: the residual's log(p - q) + g
// (after a rejection) and p's fl(h / T) + g.
__device__ __forceinline__ void draw_element(ThreadBest& res, ThreadBest& pb, float h, float d,
                                             float g, int v, float inv_t, float lt, float ld,
                                             bool rejected) {
  const float x = __fmul_rn(h, inv_t);
  pb.offer(__fadd_rn(x, g), v);
  if (rejected) {
    const float w = expf(x - lt) - expf(d - ld);
    if (w > 0.0f) res.offer(__fadd_rn(logf(w), g), v);
  }
}

__global__ void __launch_bounds__(kRejThreads, 1)
    rejection_accept_kernel(const __grid_constant__ RejParams p) {
  __shared__ int s_par[TV_MAX_NODES];
  __shared__ int s_tok[TV_MAX_NODES];
  __shared__ int s_path[TV_MAX_NODES];
  __shared__ int s_depth[TV_MAX_NODES];
  __shared__ float s_unif[TV_MAX_NODES];
  __shared__ double s_score[TV_MAX_NODES];
  __shared__ unsigned char s_leaf[TV_MAX_NODES];
  __shared__ RejPart s_pw[kRejWarps];              // per-warp partials of this CTA
  __shared__ RejPart s_part[kRejMaxPath];          // per-row partials of this CTA (read remotely)
  __shared__ float s_hx[kRejMaxPath], s_dx[kRejMaxPath];
  __shared__ float s_lt[kRejMaxPath], s_ld[kRejMaxPath];
  __shared__ int s_am[kRejMaxPath], s_dec[kRejMaxPath];
  __shared__ uint64_t s_bk[kRejWarps];
  __shared__ int s_bi[kRejWarps];
  __shared__ uint64_t s_wk[kRejWarps], s_wk2[kRejWarps], s_draw[2];
  __shared__ int s_plen;
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int csize = p.csize;
  const int rank = csize > 1 ? static_cast<int>(cluster_rank()) : 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int st = p.status[b];
  const int t0 = p.cu_nodes[b];
  const int n = p.cu_nodes[b + 1] - t0;
  const float temp = p.temperature[b];
  // every early exit below depends only on the request's inputs, so it is
  // taken by all CTAs of the cluster alike
  if (st != 0) return;
  if (n < 1 || n > p.max_nodes) {
    if (rank == 0 && threadIdx.x == 0) atomicOr(&p.status[b], TV_ST_BAD_SIZE);
    return;
  }
  const int tflag = temperature_flags(temp, p.gumbel != nullptr);
  if (tflag) {
    if (rank == 0 && threadIdx.x == 0) atomicOr(&p.status[b], tflag);
    return;
  }
  // ---- 1. the chosen path: largest cumulative draft log-probability
  int bad_root = 0, bad_par = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int par = p.parents[t0 + i];
    s_par[i] = par;
    s_tok[i] = p.draft_tokens[t0 + i];
    s_unif[i] = p.uniforms[t0 + i];
    s_leaf[i] = 1;
    s_depth[i] = i == 0 ? 1 : 0;
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
  // one tree level per round: a node adds its parent's finished score (the
  // parent's level was set in an earlier round, so its score is final)
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
  {
    // the best leaf by integer keys (a NaN score counts as -inf)
    uint64_t bk = 0ull;
    int bi = INT_MAX;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      if (!s_leaf[i]) continue;
      const uint64_t k = score_key(s_score[i]);
      if (k > bk) { bk = k; bi = i; }        // a thread's indices increase: ties keep the first
    }
    warp_best_leaf(bk, bi);
    if (lane == 0) { s_bk[warp] = bk; s_bi[warp] = bi; }
    __syncthreads();
    if (warp == 0) {
      bk = lane < kRejWarps ? s_bk[lane] : 0ull;
      bi = lane < kRejWarps ? s_bi[lane] : INT_MAX;
      warp_best_leaf(bk, bi);
      if (lane == 0) {
        // the leaf's level is its path length; fill root-first
        int u = bi;
        const int len = s_depth[bi];
        s_plen = len;
        for (int k = len - 1; k >= 0 && u >= 0; --k) { s_path[k] = u; u = s_par[u]; }
      }
    }
    __syncthreads();
  }
  const int plen = s_plen;
  int v0, v1;
  slice_of(p.vocab, rank, csize, v0, v1);
  const bool sample = temp > 0.0f;
  const float inv_t = sample ? __frcp_rn(temp) : 1.0f;
  const bool vec_t = p.vec & 1, vec_d = (p.vec & 2) != 0, vec_g = (p.vec & 4) != 0;
  // ---- 2./3. passes of up to kRejMaxPath path rows
  int acc = 0;                 // accepted edges
  int stop = -1;               // path index of the node the draw happens at
  bool rejected = false;
  for (int base = 0; stop < 0; base += kRejMaxPath) {
    const int cnt = min(kRejMaxPath, plen - base);
    // the logits of each edge's token (sampling), fetched while the rows stream
    if (sample && threadIdx.x < cnt && base + threadIdx.x + 1 < plen) {
      const int k = threadIdx.x;
      const size_t u = static_cast<size_t>(t0 + s_path[base + k]);
      const int x = s_tok[s_path[base + k + 1]];
      const bool inside = x >= 0 && x < p.vocab;
      s_hx[k] = inside ? p.target[u * p.target_ld + x] : -INFINITY;
      s_dx[k] = inside ? p.draft[u * p.draft_ld + x] : -INFINITY;
    }
    // warps split over the rows: wpr warps per row, each a segment of the slice
    const int wpr = kRejWarps / cnt;
    const int k = warp / wpr, seg = warp % wpr;
    if (k < cnt) {
      const size_t u = static_cast<size_t>(t0 + s_path[base + k]);
      const int seglen = (((v1 - v0) + wpr - 1) / wpr + 3) & ~3;
      const int a = min(v1, v0 + seg * seglen), e = min(v1, a + seglen);
      const float* hr = p.target + u * p.target_ld;
      const float* dr = p.draft + u * p.draft_ld;
      const RejPart r = sample ? reduce_segment<true>(hr, dr, a, e, vec_t && vec_d, inv_t, lane)
                               : reduce_segment<false>(hr, dr, a, e, vec_t, inv_t, lane);
      if (lane == 0) s_pw[warp] = r;
    }
    __syncthreads();
    if (warp < cnt) {
      RejPart r;
      part_identity(r);
      if (lane < wpr) r = s_pw[warp * wpr + lane];
      r = part_warp_merge(r);
      if (lane == 0) s_part[warp] = r;
    }
    row_barrier(csize);
    // one warp per row: combine the cluster's partials, decide the edge
    if (warp < cnt) {
      RejPart r;
      part_identity(r);
      if (lane < csize) {
        if (csize > 1) {
          const uint64_t* src = reinterpret_cast<const uint64_t*>(&s_part[warp]);
          const uint64_t w0 = ld_cluster_u64(src, lane), w1 = ld_cluster_u64(src + 1, lane);
          const uint64_t w2 = ld_cluster_u64(src + 2, lane);
          r.tm = __uint_as_float(static_cast<uint32_t>(w0));
          r.ts = __uint_as_float(static_cast<uint32_t>(w0 >> 32));
          r.dm = __uint_as_float(static_cast<uint32_t>(w1));
          r.ds = __uint_as_float(static_cast<uint32_t>(w1 >> 32));
          r.amax = w2;
        } else {
          r = s_part[warp];
        }
      }
      r = part_warp_merge(r);
      if (lane == 0) {
        const int pi = base + warp;
        const float lt = r.tm + logf(r.ts), ld = r.dm + logf(r.ds);
        const int am = best_index(r.amax);
        int dec = 0;                                 // 0: the walk stops at this node
        if (pi + 1 < plen) {
          const int c = s_path[pi + 1];
          const int x = s_tok[c];
          if (x < 0 || x >= p.vocab) {
            dec = 0;                                 // outside the vocabulary: rejected
          } else if (!sample) {
            dec = x == am;                           // p is one-hot on the first argmax
          } else {
            const float hx = s_hx[warp], dx = s_dx[warp];
            if (hx == -INFINITY) {
              dec = 0;                               // p(x) = 0
            } else if (dx == -INFINITY) {
              dec = 1;                               // q(x) = 0 < p(x)
            } else {
              const float ratio = expf((__fmul_rn(hx, inv_t) - lt) - (dx - ld));
              dec = s_unif[c] < ratio;
            }
          }
        }
        s_dec[warp] = dec;
        s_lt[warp] = lt;
        s_ld[warp] = ld;
        s_am[warp] = am;
      }
    }
    __syncthreads();
    // the first row whose edge is not accepted (every warp finds it itself)
    const unsigned stops = __ballot_sync(0xffffffffu, lane < cnt && s_dec[lane] == 0);
    if (stops != 0u) {
      const int ks = __ffs(stops) - 1;
      acc += ks;
      stop = base + ks;
      rejected = stop + 1 < plen;
    } else {
      acc += cnt;
      row_barrier(csize);                  // partials read everywhere before they are rewritten
    }
  }
  // ---- 4. the draw at the stop node
  const int ks = stop % kRejMaxPath;
  int tok = s_am[ks];                      // greedy: all of p, and of the residual, is there
  if (sample) {
    const size_t su = static_cast<size_t>(t0 + s_path[stop]);
    const float* hr = p.target + su * p.target_ld;
    const float* dr = p.draft + su * p.draft_ld;
    const float* gr = p.gumbel + su * p.gumbel_ld;
    const float lt = s_lt[ks], ld = s_ld[ks];
    ThreadBest res, pb;
    if (vec_t && vec_g && (vec_d || !rejected)) {
      const int b4 = v0 + ((v1 - v0) & ~3);
      for (int v = v0 + threadIdx.x * 4; v < b4; v += 4 * kRejThreads) {
        const float4 h4 = __ldcs(reinterpret_cast<const float4*>(hr + v));
        const float4 g4 = __ldcs(reinterpret_cast<const float4*>(gr + v));
        const float4 d4 = rejected ? __ldcs(reinterpret_cast<const float4*>(dr + v))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
        draw_element(res, pb, h4.x, d4.x, g4.x, v, inv_t, lt, ld, rejected);
        draw_element(res, pb, h4.y, d4.y, g4.y, v + 1, inv_t, lt, ld, rejected);
        draw_element(res, pb, h4.z, d4.z, g4.z, v + 2, inv_t, lt, ld, rejected);
        draw_element(res, pb, h4.w, d4.w, g4.w, v + 3, inv_t, lt, ld, rejected);
      }
      for (int v = b4 + threadIdx.x; v < v1; v += kRejThreads)
        draw_element(res, pb, __ldcs(hr + v), rejected ? __ldcs(dr + v) : 0.0f, __ldcs(gr + v), v,
                     inv_t, lt, ld, rejected);
    } else {
      for (int v = v0 + threadIdx.x; v < v1; v += kRejThreads)
        draw_element(res, pb, __ldcs(hr + v), rejected ? __ldcs(dr + v) : 0.0f, __ldcs(gr + v), v,
                     inv_t, lt, ld, rejected);
    }
    const uint64_t k1 = warp_max_u64(res.packed()), k2 = warp_max_u64(pb.packed());
    if (lane == 0) { s_wk[warp] = k1; s_wk2[warp] = k2; }
    __syncthreads();
    if (warp == 0) {
      const uint64_t a1 = warp_max_u64(lane < kRejWarps ? s_wk[lane] : 0ull);
      const uint64_t a2 = warp_max_u64(lane < kRejWarps ? s_wk2[lane] : 0ull);
      if (lane == 0) { s_draw[0] = a1; s_draw[1] = a2; }
    }
    row_barrier(csize);
    if (rank == 0 && warp == 0) {
      uint64_t x1 = 0ull, x2 = 0ull;
      if (lane < csize) {
        x1 = csize > 1 ? ld_cluster_u64(&s_draw[0], lane) : s_draw[0];
        x2 = csize > 1 ? ld_cluster_u64(&s_draw[1], lane) : s_draw[1];
      }
      x1 = warp_max_u64(x1);
      x2 = warp_max_u64(x2);
      tok = (rejected && x1 != 0ull) ? best_index(x1) : best_index(x2);
    }
  }
  if (csize > 1) cluster_sync_all();        // remote reads done before any CTA exits
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
  // one CTA per vocabulary slice; clusters while a CTA per SM stays for every slice
  // one CTA (one SM) per vocabulary slice: the widest portable power-of-two
  // cluster that keeps the whole batch within half the SMs
  int csize = 1;
  while (csize < 8 && batch * csize * 2 <= sms) csize *= 2;
  auto rows16 = [](const void* ptr, int64_t ld) {
    return ptr != nullptr && (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0 && ld % 4 == 0;
  };
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
  p.vec = (rows16(target_logits, target_ld) ? 1 : 0) | (rows16(draft_logits, draft_ld) ? 2 : 0) |
          (rows16(gumbel, gumbel_ld) ? 4 : 0);
  const cudaError_t err = tv::launch_cluster_pdl(tv::rejection_accept_kernel, dim3(csize, batch),
                                                 dim3(tv::kRejThreads), csize,
                                                 tv::as_stream(stream), p);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
