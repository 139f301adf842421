// DDTree draft-tree construction on the device.
//
// Definitions ("Accelerating Speculative Decoding with Block Diffusion Draft
// Trees"):
//  - §3-§4.1: the drafter gives one factorised distribution per position,
//    q_i = softmax(h_i); a prefix's log-score is the sum of its positions'
//    log-probabilities.
//  - §4.2 (Proposition 2): the B most probable prefixes are prefix-closed and
//    form the optimal tree; §4.3 (Lemma 1): only each depth's top-K tokens,
//    K = min(B, |V|), can appear in it.
//  - §5 (Algorithm 1): best-first enumeration over rank tuples - pop the best
//    tuple, offer its next sibling (last rank + 1) and its first child
//    (append rank 1); B pops give the tree. §6-§7.1: the tree is flattened
//    depth by depth after the root.
//
// Two grids:
//  ddtree_topk_kernel   one CTA per (request, position) row: streams the row's
//                       V logits once (128-bit loads, two 4096-logit chunks in
//                       flight while one is processed), admits the logits that
//                       could still be in the top K into a shared-memory
//                       candidate buffer behind a histogram threshold, and
//                       accumulates the row's log-sum-exp on the way; the
//                       survivors are ranked by a bucket sort at the end.
//                       HBM-bound: 4 bytes per vocabulary entry.
//  ddtree_heap_kernel   one CTA per request: the top-K log-probabilities go to
//                       shared memory, then one warp runs Algorithm 1. The
//                       frontier holds one offer per tree node (its next
//                       unselected child, which is what the page's sibling
//                       and first-child pushes amount to), kept in the
//                       owning lane's registers; each pop is a two-step warp
//                       max (redux.sync) over the lanes' best offers.
//                       Latency-bound: B dependent pops.
//
// Ordering and precision (readings of the pages): ranks order tokens by logit
// descending, equal logits by token id ascending; log q = h - logsumexp(h);
// a prefix's score is its parent's score plus its own log-probability, added
// in float32; equal scores pop the shallower prefix, then the one whose parent
// popped first. Output: root, then depth by depth, pop order within a depth.
#include "tv_common.cuh"

namespace tv {

constexpr int kTopkThreads = 512;
constexpr int kTopkVec = 2;                                  // float4 per thread per chunk
constexpr int kTopkChunk = kTopkThreads * kTopkVec * 4;      // 4096 logits
constexpr int kTopkCap = kTopkChunk + kTopkChunk / 2;       // candidate buffer entries
constexpr int kTopkMaxK = 1024;
constexpr int kHeapThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;

// float -> unsigned key in the same order (NaN above +inf, -0 == +0)
__device__ __forceinline__ uint32_t float_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (x != x) return 0xFFFFFFFFu;
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// (logit, token) -> 64-bit key: larger logit first, then smaller token
__device__ __forceinline__ uint64_t cand_key(float x, int tok) {
  return (static_cast<uint64_t>(float_key(x)) << 32) | static_cast<uint32_t>(~tok);
}

// ---------------------------------------------------------------- top-K rows
//
// Admission: a logit enters the candidate buffer when it is >= the lower edge
// of histogram bin b_cur (bins = top 12 bits of the order key, an eighth of
// an octave). After each chunk one thread raises b_cur while the admitted
// keys in bins above it still number >= K, so every key that can be in the
// final top K is kept and the admission rate falls as the row streams. When
// the buffer nears capacity, keys below the threshold are filtered out (and
// only if that is not enough - a row of near-equal logits - is it sorted and
// cut to K). At the end the candidates are bucketed by bin in descending
// order and ranked inside their bucket, which gives the sorted top K.

constexpr int kTopkBins = 4096;
constexpr int kTopkBucketCap = 2048;     // candidates the final bucket sort handles

struct TopkShared {
  int count;                  // entries in the buffer
  int last_count;
  int above;                  // buffer keys in bins >= b_cur
  int b_cur;
  float tau;                  // admit x >= tau
  int n_cand;
  double lse;
  float wm[32];
  float ws[32];
  uint32_t wt[32];
};

__device__ __forceinline__ int key_bin(uint64_t key) { return static_cast<int>(key >> 52); }

// lower edge of bin b as a float threshold (bins below -inf's admit all)
__device__ __forceinline__ float bin_floor(int b) {
  const uint32_t k = static_cast<uint32_t>(b) << 20;
  return k <= 0x007FFFFFu ? -INFINITY : key_float(k);
}

// Sort buf[0, n) descending (bitonic network over the next power of two,
// zero keys padding). All threads call it.
__device__ void bitonic_desc(uint64_t* buf, int n) {
  int p2 = 1;
  while (p2 < n) p2 <<= 1;
  for (int i = n + threadIdx.x; i < p2; i += blockDim.x) buf[i] = 0ull;
  __syncthreads();
  for (int size = 2; size <= p2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < p2 / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const uint64_t x = buf[lo], y = buf[hi];
        if ((x < y) == desc) { buf[lo] = y; buf[hi] = x; }
      }
      __syncthreads();
    }
  }
}

// Keep the buffer keys in bins >= b_cur, moved to the front (via `tmp`).
__device__ void filter_buffer(uint64_t* buf, uint64_t* tmp, TopkShared& sh) {
  const int n = sh.count;
  const int b_cur = sh.b_cur;
  __syncthreads();
  if (threadIdx.x == 0) sh.n_cand = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += blockDim.x) {
    const int i = i0 + threadIdx.x;
    const bool keep = i < n && key_bin(buf[i]) >= b_cur;
    const uint32_t m = __ballot_sync(0xffffffffu, keep);
    int base = 0;
    if ((threadIdx.x & 31) == 0 && m) base = atomicAdd(&sh.n_cand, __popc(m));
    base = __shfl_sync(0xffffffffu, base, 0);
    if (keep) tmp[base + __popc(m & ((1u << (threadIdx.x & 31)) - 1u))] = buf[i];
  }
  __syncthreads();
  const int kept = sh.n_cand;
  for (int i = threadIdx.x; i < kept; i += blockDim.x) buf[i] = tmp[i];
  if (threadIdx.x == 0) { sh.count = kept; sh.last_count = kept; }
  __syncthreads();
}

// Threshold from the histogram, in parallel: b_cur = the highest bin whose
// suffix count (keys in bins >= it) is still >= k; above = that count.
__device__ void threshold_from_hist(const uint32_t* hist, int k, TopkShared& sh) {
  constexpr int per = kTopkBins / kTopkThreads;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b_hi = kTopkBins - threadIdx.x * per;           // bins [b_hi - per, b_hi)
  uint32_t loc = 0;
#pragma unroll
  for (int j = 1; j <= per; ++j) loc += hist[b_hi - j];
  uint32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.wt[warp] = incl;
  __syncthreads();
  uint32_t run = incl - loc;
  for (int w = 0; w < warp; ++w) run += sh.wt[w];
  // the crossing bin is this thread's if the count reaches k inside its range
  const uint32_t need = static_cast<uint32_t>(k);
  if (run < need && run + loc >= need) {
    for (int j = 1; j <= per; ++j) {
      run += hist[b_hi - j];
      if (run >= need) {
        sh.b_cur = b_hi - j;
        sh.above = static_cast<int>(run);
        sh.tau = bin_floor(b_hi - j);
        break;
      }
    }
  }
  __syncthreads();
}

// Sort the buffer, keep k keys, rebuild the histogram and threshold from them.
__device__ void sort_cut(uint64_t* buf, uint32_t* hist, int k, TopkShared& sh) {
  bitonic_desc(buf, sh.count);
  for (int i = threadIdx.x; i < kTopkBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += blockDim.x) atomicAdd(&hist[key_bin(buf[i])], 1u);
  if (threadIdx.x == 0) { sh.count = k; sh.last_count = k; }
  __syncthreads();
  threshold_from_hist(hist, k, sh);
}

__device__ __forceinline__ void load_chunk(const float* h, int base, int vocab, int tid,
                                           float (&x)[kTopkVec * 4]) {
#pragma unroll
  for (int u = 0; u < kTopkVec; ++u) {
    const int i = base + (tid + u * kTopkThreads) * 4;
    if (i + 3 < vocab) {
      const float4 v = __ldcs(reinterpret_cast<const float4*>(h + i));
      x[u * 4 + 0] = v.x; x[u * 4 + 1] = v.y; x[u * 4 + 2] = v.z; x[u * 4 + 3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[u * 4 + e] = i + e < vocab ? __ldcs(h + i + e) : -INFINITY;
    }
  }
}

__global__ void __launch_bounds__(kTopkThreads, 2)
ddtree_topk_kernel(const float* __restrict__ logits, long long ld, int vocab, int k,
                   int32_t* __restrict__ top_tokens, float* __restrict__ top_logq) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t* buf = reinterpret_cast<uint64_t*>(smem_raw);                   // kTopkCap
  uint64_t* tmp = buf + kTopkCap;                                           // kTopkBucketCap
  uint32_t* hist = reinterpret_cast<uint32_t*>(tmp + kTopkBucketCap);       // kTopkBins
  uint32_t* pos = hist + kTopkBins;                                         // kTopkBins
  __shared__ TopkShared sh;
  grid_dependency_wait();
  grid_launch_dependents();
  const int row = blockIdx.x;
  const float* h = logits + static_cast<size_t>(row) * ld;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kTopkBins; i += blockDim.x) hist[i] = 0;
  if (tid == 0) {
    sh.count = 0; sh.last_count = 0; sh.above = 0; sh.b_cur = 0; sh.tau = -INFINITY;
  }
  __syncthreads();
  float m = -INFINITY, s = 0.0f;                            // running log-sum-exp state
  float tau = -INFINITY;
  float x[kTopkVec * 4], nx[kTopkVec * 4], nnx[kTopkVec * 4];
  load_chunk(h, 0, vocab, tid, x);
  if (kTopkChunk < vocab) load_chunk(h, kTopkChunk, vocab, tid, nx);
  for (int base = 0; base < vocab; base += kTopkChunk) {
    // two chunks' loads are in flight while this one is processed
    if (base + 2 * kTopkChunk < vocab) load_chunk(h, base + 2 * kTopkChunk, vocab, tid, nnx);
    float cm = x[0];
#pragma unroll
    for (int e = 1; e < kTopkVec * 4; ++e) cm = fmaxf(cm, x[e]);
    const float nm = fmaxf(m, cm);
    if (nm != -INFINITY) {
      const float nml = nm * kLog2e;
      float acc = s * fast_exp2(m * kLog2e - nml);
#pragma unroll
      for (int e = 0; e < kTopkVec * 4; ++e) acc += fast_exp2(fmaf(x[e], kLog2e, -nml));
      s = acc;
      m = nm;
    }
    // admission: one warp scan of the admitted counts, one atomic per warp;
    // most warps skip it once tau has risen
    if (__any_sync(0xffffffffu, cm >= tau)) {
      uint32_t amask = 0;
#pragma unroll
      for (int e = 0; e < kTopkVec * 4; ++e) {
        const int i = base + (tid + (e >> 2) * kTopkThreads) * 4 + (e & 3);
        if (i < vocab && x[e] >= tau) amask |= 1u << e;
      }
      const int cnt = __popc(amask);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int slot = 0;
      if (lane == 31 && incl > 0) slot = atomicAdd(&sh.count, incl);
      slot = __shfl_sync(0xffffffffu, slot, 31) + incl - cnt;
#pragma unroll
      for (int e = 0; e < kTopkVec * 4; ++e) {
        if (amask & (1u << e)) {
          const int i = base + (tid + (e >> 2) * kTopkThreads) * 4 + (e & 3);
          const uint64_t key = cand_key(x[e], i);
          buf[slot++] = key;
          atomicAdd(&hist[key_bin(key)], 1u);
        }
      }
    }
    __syncthreads();
    if (base == 0) {
      // first chunk: the threshold jumps from nothing to the k-th key's bin
      if (tid == 0) sh.last_count = sh.count;
      threshold_from_hist(hist, k, sh);
    } else {
      if (tid == 0) {
        // raise the threshold while the keys above it still number >= k
        int above = sh.above + (sh.count - sh.last_count);
        int b = sh.b_cur;
        while (b + 1 < kTopkBins && above - static_cast<int>(hist[b]) >= k) {
          above -= static_cast<int>(hist[b]);
          ++b;
        }
        sh.above = above;
        sh.b_cur = b;
        sh.last_count = sh.count;
        sh.tau = bin_floor(b);
      }
      __syncthreads();
    }
    if (sh.count > kTopkCap - kTopkChunk) {
      // the filtered keys must fit the bucket area; otherwise sort and cut
      if (sh.above <= kTopkBucketCap) filter_buffer(buf, tmp, sh);
      else sort_cut(buf, hist, k, sh);
    }
    tau = sh.tau;
#pragma unroll
    for (int e = 0; e < kTopkVec * 4; ++e) { x[e] = nx[e]; nx[e] = nnx[e]; }
  }
  __syncthreads();
  // log-sum-exp of the row: combine (m, s) over warps, one float64 log
  {
    float wm_ = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm_ = fmaxf(wm_, __shfl_xor_sync(0xffffffffu, wm_, o));
    float ws_ = (m == -INFINITY) ? 0.0f : s * fast_exp2((m - wm_) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ws_ += __shfl_xor_sync(0xffffffffu, ws_, o);
    if (lane == 0) { sh.wm[warp] = wm_; sh.ws[warp] = ws_; }
  }
  // final candidates: keys in bins >= b_cur (sorted and cut first when they
  // would not fit the bucket area)
  if (sh.above > kTopkBucketCap) sort_cut(buf, hist, k, sh);
  filter_buffer(buf, tmp, sh);
  if (warp == 0) {
    const int nw = kTopkThreads / 32;
    const float wmv = lane < nw ? sh.wm[lane] : -INFINITY;
    float rm = wmv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rm = fmaxf(rm, __shfl_xor_sync(0xffffffffu, rm, o));
    double t = (lane < nw && wmv != -INFINITY)
                   ? static_cast<double>(sh.ws[lane]) * static_cast<double>(fast_exp2((wmv - rm) * kLog2e))
                   : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) sh.lse = rm == -INFINITY ? -INFINITY : static_cast<double>(rm) + log(t);
  }
  const int n = sh.count;
  // bucket the candidates by bin (descending), then rank inside each bucket
  for (int i = tid; i < kTopkBins; i += blockDim.x) hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) atomicAdd(&hist[key_bin(buf[i])], 1u);
  __syncthreads();
  {
    // exclusive prefix from the top bin down: pos[b] = keys in bins > b
    constexpr int per = kTopkBins / kTopkThreads;
    const int b_hi = kTopkBins - tid * per;                 // this thread: bins [b_hi - per, b_hi)
    uint32_t loc = 0;
#pragma unroll
    for (int j = 1; j <= per; ++j) loc += hist[b_hi - j];
    uint32_t incl = loc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.wt[warp] = incl;
    __syncthreads();
    uint32_t run = incl - loc;
    for (int w = 0; w < warp; ++w) run += sh.wt[w];
#pragma unroll
    for (int j = 1; j <= per; ++j) {
      pos[b_hi - j] = run;
      run += hist[b_hi - j];
    }
  }
  __syncthreads();
  // scatter into buckets (pos advances to each bucket's end), then each key's
  // rank = keys in higher bins + larger keys in its own bin
  for (int i = tid; i < n; i += blockDim.x) {
    const uint64_t key = buf[i];
    tmp[atomicAdd(&pos[key_bin(key)], 1u)] = key;
  }
  __syncthreads();
  for (int i = tid; i < n; i += blockDim.x) {
    const uint64_t key = tmp[i];
    const int b = key_bin(key);
    const int end = static_cast<int>(pos[b]);
    const int beg = end - static_cast<int>(hist[b]);
    int r = beg;
    for (int j = beg; j < end; ++j) r += tmp[j] > key;
    if (r < k) buf[r] = key;                                // final rank
  }
  __syncthreads();
  const double lse = sh.lse;
  for (int r = tid; r < k; r += blockDim.x) {
    const uint64_t key = buf[r];
    const float xv = key_float(static_cast<uint32_t>(key >> 32));
    top_tokens[static_cast<size_t>(row) * k + r] = static_cast<int32_t>(~static_cast<uint32_t>(key));
    top_logq[static_cast<size_t>(row) * k + r] =
        lse == -INFINITY ? -INFINITY : static_cast<float>(static_cast<double>(xv) - lse);
  }
}

// ---------------------------------------------------------------- the heap

// Offer of a node (its next unselected child): score, then shallower, then
// earlier parent; the offered rank rides in the low bits (one offer per
// parent, so it never decides).
__device__ __forceinline__ uint64_t offer_key(float score, int child_depth, int parent, int r) {
  const uint32_t tie = (static_cast<uint32_t>(child_depth) << 20) |
                       (static_cast<uint32_t>(parent) << 10) | static_cast<uint32_t>(r);
  return (static_cast<uint64_t>(float_key(score)) << 32) | static_cast<uint32_t>(~tie);
}

// Algorithm 1 in one warp. Non-root node j (pop order 1..n-1) keeps its
// current offer (the key of its next unselected child) in lane (j-1) % 32,
// register slot (j-1) / 32; lane 0 also holds the root's. A pop is two
// warp-wide maxima (redux.sync) over the lanes' best offers; the key names
// the parent, the child's depth and rank, so every lane computes the two new
// offers (the parent's next rank, the new node's first child) from shared
// memory without divergence, and only the owners store them.
template <int S>
__device__ void heap_warp(const float* lq, int L, int k, int n_nodes, int* depth, int* parent,
                          int* rank, float* score) {
  const int lane = threadIdx.x & 31;
  uint64_t off[S];
#pragma unroll
  for (int i = 0; i < S; ++i) off[i] = 0ull;
  uint64_t root_off = lane == 0 ? offer_key(lq[0], 1, 0, 0) : 0ull;
  if (lane == 0) { depth[0] = 0; parent[0] = -1; rank[0] = 0; score[0] = 0.0f; }
  __syncwarp();
  uint64_t best = root_off;
  for (int v = 1; v < n_nodes; ++v) {
    const uint32_t hi = static_cast<uint32_t>(best >> 32);
    const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t lo = hi == mh ? static_cast<uint32_t>(best) : 0u;
    const uint32_t ml = __reduce_max_sync(0xffffffffu, lo);
    if (mh == 0u) break;        // no offer left: cannot happen while v < n_nodes
    const uint32_t tie = ~ml;
    const int r = static_cast<int>(tie & 1023u);          // rank of the child taken
    const int u = static_cast<int>((tie >> 10) & 1023u);  // its parent
    const int du = static_cast<int>(tie >> 20) - 1;       // depth of the parent
    const float sv = key_float(mh);
    // both new offers, computed by every lane
    const float su = score[u];
    const float l_next = r + 1 < k ? lq[du * k + r + 1] : 0.0f;
    const bool deeper = du + 1 < L;
    const float l_first = deeper ? lq[(du + 1) * k] : 0.0f;
    const uint64_t nu = r + 1 < k ? offer_key(__fadd_rn(su, l_next), du + 1, u, r + 1) : 0ull;
    const uint64_t nv = deeper ? offer_key(__fadd_rn(sv, l_first), du + 2, v, 0) : 0ull;
    const int lv = (v - 1) & 31, sl_v = (v - 1) >> 5;
    const int lu = u == 0 ? 0 : (u - 1) & 31, sl_u = u == 0 ? -1 : (u - 1) >> 5;
#pragma unroll
    for (int i = 0; i < S; ++i) {
      if (lane == lv && i == sl_v) off[i] = nv;
      if (lane == lu && i == sl_u) off[i] = nu;
    }
    if (lane == 0 && u == 0) root_off = nu;
    if (lane == 0) { score[v] = sv; depth[v] = du + 1; parent[v] = u; rank[v] = r; }
    __syncwarp();
    // lane maximum: pairwise, then a tree
    uint64_t t[(S + 1) / 2];
#pragma unroll
    for (int i = 0; i < (S + 1) / 2; ++i)
      t[i] = 2 * i + 1 < S ? (off[2 * i + 1] > off[2 * i] ? off[2 * i + 1] : off[2 * i]) : off[2 * i];
#pragma unroll
    for (int w = 1; w < (S + 1) / 2; w <<= 1)
#pragma unroll
      for (int i = 0; i + w < (S + 1) / 2; i += 2 * w) t[i] = t[i + w] > t[i] ? t[i + w] : t[i];
    best = t[0] > root_off ? t[0] : root_off;
  }
}

__global__ void __launch_bounds__(kHeapThreads)
ddtree_heap_kernel(const float* __restrict__ top_logq, const int32_t* __restrict__ top_tokens,
                   int L, int k, int n_nodes, const int32_t* __restrict__ root_tokens,
                   int32_t* __restrict__ parents, int32_t* __restrict__ tokens,
                   int32_t* __restrict__ cu_nodes) {
  extern __shared__ __align__(16) unsigned char smem[];
  float* lq = reinterpret_cast<float*>(smem);                               // [L][k]
  int* depth = reinterpret_cast<int*>(lq + L * k);                          // [n]
  int* parent = depth + n_nodes;                                            // [n]
  int* rank = parent + n_nodes;                                             // [n]
  int* slot = rank + n_nodes;                                               // [n]
  float* score = reinterpret_cast<float*>(slot + n_nodes);                  // [n]
  int* start = reinterpret_cast<int*>(score + n_nodes);                     // [L + 2]
  grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const float* src = top_logq + static_cast<size_t>(b) * L * k;
  for (int i = threadIdx.x; i < L * k; i += blockDim.x) lq[i] = src[i];
  for (int i = threadIdx.x; i < L + 2; i += blockDim.x) start[i] = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const int non_root = n_nodes - 1;
    if (non_root <= 32 * 1) heap_warp<1>(lq, L, k, n_nodes, depth, parent, rank, score);
    else if (non_root <= 32 * 2) heap_warp<2>(lq, L, k, n_nodes, depth, parent, rank, score);
    else if (non_root <= 32 * 4) heap_warp<4>(lq, L, k, n_nodes, depth, parent, rank, score);
    else if (non_root <= 32 * 8) heap_warp<8>(lq, L, k, n_nodes, depth, parent, rank, score);
    else if (non_root <= 32 * 16) heap_warp<16>(lq, L, k, n_nodes, depth, parent, rank, score);
    else heap_warp<32>(lq, L, k, n_nodes, depth, parent, rank, score);
    __syncwarp();
    // depth-major order, pop order within a depth
    for (int j = lane; j < n_nodes; j += 32) atomicAdd(&start[depth[j] + 1], 1);
    __syncwarp();
    if (lane == 0)
      for (int d = 1; d <= L + 1; ++d) start[d] += start[d - 1];
    __syncwarp();
    for (int j0 = 0; j0 < n_nodes; j0 += 32) {
      const int j = j0 + lane;
      const bool act = j < n_nodes;
      const unsigned am = __ballot_sync(0xffffffffu, act);
      if (act) {
        const int d = depth[j];
        const unsigned peers = __match_any_sync(am, d);
        const int pos = start[d] + __popc(peers & ((1u << lane) - 1u));
        slot[j] = pos;
        __syncwarp(am);
        if (lane == __ffs(peers) - 1) start[d] += __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  const size_t out0 = static_cast<size_t>(b) * n_nodes;
  for (int j = threadIdx.x; j < n_nodes; j += blockDim.x) {
    const int s = slot[j];
    parents[out0 + s] = j == 0 ? -1 : slot[parent[j]];
    tokens[out0 + s] = j == 0 ? (root_tokens ? root_tokens[b] : -1)
                              : top_tokens[(static_cast<size_t>(b) * L + depth[j] - 1) * k + rank[j]];
  }
  if (threadIdx.x == 0) {
    cu_nodes[b] = b * n_nodes;
    if (b == gridDim.x - 1) cu_nodes[b + 1] = (b + 1) * n_nodes;
  }
}

static size_t heap_smem_bytes(int L, int k, int n) {
  return static_cast<size_t>(L) * k * 4 + static_cast<size_t>(n) * 4 * 5 +
         static_cast<size_t>(L + 2) * 4;
}

}  // namespace tv

extern "C" int tv_ddtree_nodes(int32_t depth_L, int32_t k, int32_t budget) {
  if (depth_L < 1 || k < 1 || budget < 1 || budget > TV_MAX_NODES - 1) return TV_ERR_BAD_SIZE;
  long long total = 0, level = 1;
  for (int d = 1; d <= depth_L && total < budget; ++d) {
    level = level * k;
    if (level > budget) level = budget;        // enough to know the minimum
    total += level;
  }
  return static_cast<int>((total < budget ? total : budget) + 1);
}

extern "C" int tv_ddtree_topk(const float* logits, int64_t logits_ld, int32_t rows, int32_t vocab,
                              int32_t k, int32_t* top_tokens, float* top_logq, void* stream) {
  if (rows < 0 || vocab < 1 || vocab > (1 << 30) || k < 1 || k > tv::kTopkMaxK || k > vocab ||
      logits_ld < vocab)
    return TV_ERR_BAD_SIZE;
  if (rows == 0) return TV_OK;
  if (!logits || !top_tokens || !top_logq) return TV_ERR_NULL_POINTER;
  if (!tv::aligned(logits, 16) || (logits_ld & 3)) return TV_ERR_MISALIGNED;
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  static size_t done[tv::kMaxDevices] = {0};
  const size_t smem = static_cast<size_t>(tv::kTopkCap + tv::kTopkBucketCap) * sizeof(uint64_t) +
                      2 * tv::kTopkBins * sizeof(uint32_t);
  if (!tv::ensure_smem(tv::ddtree_topk_kernel, smem, done, dev)) return TV_ERR_CUDA;
  const cudaError_t err = tv::launch_pdl(tv::ddtree_topk_kernel, dim3(rows), dim3(tv::kTopkThreads),
                                         smem, tv::as_stream(stream), logits,
                                         static_cast<long long>(logits_ld), static_cast<int>(vocab),
                                         static_cast<int>(k), top_tokens, top_logq);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

extern "C" int tv_ddtree_build(const float* top_logq, const int32_t* top_tokens, int32_t batch,
                               int32_t depth_L, int32_t k, int32_t budget,
                               const int32_t* root_tokens, int32_t* parents, int32_t* tokens,
                               int32_t* cu_nodes, void* stream) {
  const int n = tv_ddtree_nodes(depth_L, k, budget);
  if (n < 0 || batch < 0 || k > tv::kTopkMaxK) return TV_ERR_BAD_SIZE;
  const size_t smem = tv::heap_smem_bytes(depth_L, k, n);
  if (smem > 200 * 1024) return TV_ERR_BAD_SIZE;
  if (batch == 0) return TV_OK;
  if (!top_logq || !top_tokens || !parents || !tokens || !cu_nodes) return TV_ERR_NULL_POINTER;
  const int dev = tv::current_device();
  if (dev < 0) return TV_ERR_CUDA;
  static size_t done[tv::kMaxDevices] = {0};
  if (!tv::ensure_smem(tv::ddtree_heap_kernel, smem, done, dev)) return TV_ERR_CUDA;
  const cudaError_t err = tv::launch_pdl(tv::ddtree_heap_kernel, dim3(batch), dim3(tv::kHeapThreads),
                                         smem, tv::as_stream(stream), top_logq, top_tokens,
                                         static_cast<int>(depth_L), static_cast<int>(k), n,
                                         root_tokens, parents, tokens, cu_nodes);
  return err == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
