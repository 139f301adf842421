// Packed tree attention on the 5th-generation tensor cores (tcgen05 + TMEM,
// TMA-fed), plus the depth-RoPE / tentative-KV pre-pass.
//
// What is computed (identical to the definition the oracle restates): for
// every tree node i and query head h of a request with P committed tokens,
//   o = softmax(q_i k^T * scale) v  over the P prompt keys and the keys of
//   i's ancestor chain (i included),
// with q and the tree keys rotated at position P + depth(i) -
// "Beam Search、约束解码与 Tree/Self Speculation", section "Packed tree
// attention" and its packed-vs-branch experiment; "02 · Token Tree 与 Tree
// Attention" §3 (visible = prompt ∪ ancestors, RoPE at tree depth).
//
// Two launches on the caller's stream:
//  1. rope_append_kernel: rotates q (into the workspace) and k (into the
//     tentative cache slots P + i, with the raw v) - "投机解码的树状注意力验证…",
//     section "实现中的 KV Cache 与批处理约束": the tree's tentative KV is a
//     contiguous region in node order. It also zero-fills the rest of the last
//     page so every row a tile reads is finite.
//  2. attn_tc_kernel: keys are cache slots [0, P + N); slots >= P are tested
//     against the node's ancestor bit row. One CTA per SM, warp-specialised:
//       warp 0      TMA producer: Q tiles and 16-row K pages (4-D tensor
//                   maps over the paged pools, 128-byte swizzle)
//       warp 1      MMA issuer: S = Q K^T (A, B in shared memory) and
//                   O += P V (P read from Tensor Memory), fp32 accumulators
//       warp 2      TMA producer for V (K and V are released separately)
//       warps 3-10  two 128-thread softmax groups, one Tensor Memory lane
//                   (= one query row) per thread, ping-ponging two 128-row
//                   M tiles so the tensor core always has work.
//     Query rows of a unit are (node, query head in the GQA group), node
//     major, so one K/V tile feeds up to 256 rows. Work plan: a unit is
//     (request, KV head, group of up to 256 rows); all units' key tiles are
//     laid end to end and every CTA takes an equal contiguous share, computed
//     on the device from cu_nodes/prompt_len (no host round trip), so each
//     CTA moves the same amount of KV whatever the prompt-length mix.
//  3. attn_merge_kernel: a unit cut between CTAs left one partial per CTA;
//     this grid merges them (log-sum-exp), many CTAs and loads in flight.
//  Launches 2 and 3 use programmatic dependent launch so their prologues
//  overlap the previous grid's tail. No CTA ever waits for another CTA.
#include <cudaTypedefs.h>

#include "tv_sm100.cuh"

namespace tv {

constexpr int kTcBN = 128;          // keys per tile
constexpr int kTcStages = 2;        // K/V pipeline depth
constexpr int kTcThreads = 352;     // 11 warps
constexpr int kTcMaxBatch = 4096;
constexpr int kRopeNodes = 4;       // nodes per pre-pass CTA
constexpr int kRopeBatch = 4;       // loads in flight per pre-pass thread
constexpr int kRopeThreads = 256;
constexpr int kTaskInts = 16;       // merge-task record per attention CTA

// floats of one partial-result slot: O [D/4 column blocks][256 rows] float4,
// then the per-row reference max and sum
__host__ __device__ constexpr size_t kSlotFloats(int d) { return static_cast<size_t>(256) * (d + 2); }

struct TcParams {
  CUtensorMap qmap;      // rotated q in the workspace, dims (D, G, Hkv, T_cap)
  CUtensorMap kmap;      // K pool, dims (D, 16, Hkv, num_blocks)
  CUtensorMap vmap;      // V pool
  const int32_t* cu_nodes;
  const int32_t* prompt_len;
  const uint32_t* mask;
  const int32_t* block_table;
  const int32_t* status;
  __nv_bfloat16* out;
  int32_t* tasks;        // kTaskInts per CTA: the split unit this CTA starts (merge work)
  float* partials;       // two slots per CTA
  int32_t* status_rw;
  int batch, max_nodes, t_cap, hq, hkv, group, npm, words, max_blocks, grid;
  float scale_log2;
};

struct RopeParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int32_t* cu_nodes;
  const int32_t* positions;
  const int32_t* prompt_len;
  const int32_t* block_table;
  const int32_t* n_blocks;
  __nv_bfloat16* q_rot;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  int32_t* status;
  int batch, max_nodes, t_cap, hq, hkv, max_blocks, num_blocks, rope_style;
  float inv_freq[64];
};

// ------------------------------------------------------------ pre-pass

template <int D>
__global__ void __launch_bounds__(kRopeThreads) rope_append_kernel(const __grid_constant__ RopeParams p) {
  constexpr int D2 = D / 2;
  __shared__ float2 s_cs[kRopeNodes][D2];
  __shared__ int s_blk[kRopeNodes];      // cache block of each node's tentative slot
  grid_launch_dependents();              // the attention grid may start its prologue
  const int b = blockIdx.y;
  const int t0 = p.cu_nodes[b];
  const int n = p.cu_nodes[b + 1] - t0;
  const int plen = p.prompt_len[b];
  if (n < 1 || n > p.max_nodes || plen < 0) return;             // tree_build flagged it
  if (static_cast<long long>(t0) + n > p.t_cap || t0 < 0) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status + b, TV_ST_BAD_SIZE);
    return;
  }
  if (p.status[b] & TV_TREE_FLAGS) return;
  const int i0 = blockIdx.x * kRopeNodes;
  if (i0 >= n) return;
  const int i1 = min(n, i0 + kRopeNodes);
  // every block holding slots [0, P + n) must be held and in range
  const long long slots = static_cast<long long>(plen) + n;
  const int nlb = static_cast<int>((slots + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE);
  const int32_t* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  int bad = (nlb > p.n_blocks[b] || nlb > p.max_blocks) ? 1 : 0;
  for (int lb = threadIdx.x; !bad && lb < nlb; lb += blockDim.x) {
    const int blk = trow[lb];
    if (blk < 0 || blk >= p.num_blocks) bad = 1;
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status + b, TV_ST_BAD_BLOCK);
    return;
  }
  if (threadIdx.x < i1 - i0) s_blk[threadIdx.x] = trow[(plen + i0 + threadIdx.x) / TV_BLOCK_SIZE];
  for (int idx = threadIdx.x; idx < (i1 - i0) * D2; idx += blockDim.x) {
    const int nd = idx / D2, pr = idx % D2;
    float sn, cs;
    sincosf(static_cast<float>(p.positions[t0 + i0 + nd]) * p.inv_freq[pr], &sn, &cs);
    s_cs[nd][pr] = make_float2(cs, sn);
  }
  __syncthreads();
  const bool style0 = p.rope_style == 0;
  // Work item = one 16-byte vector (8 bf16) of one head of one node; style 0
  // rotates the pairs inside the vector, style 1 pairs vector v with vector
  // v + D/16. Each thread loads kRopeBatch items before storing any, so the
  // loads overlap instead of waiting one by one.
  constexpr int VPH = D / 8;
  const int vpn = style0 ? VPH : VPH / 2;
  const int heads = p.hq + 2 * p.hkv;
  const int per_node = heads * vpn;
  const int total = (i1 - i0) * per_node;
  auto src_of = [&](int idx, int& nd, int& h, int& v) -> const uint4* {
    nd = idx / per_node;
    const int rem = idx % per_node;
    h = rem / vpn;
    v = rem % vpn;
    const int t = t0 + i0 + nd;
    if (h < p.hq) return reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(t) * p.hq + h) * D);
    if (h < p.hq + p.hkv)
      return reinterpret_cast<const uint4*>(p.k_new + (static_cast<size_t>(t) * p.hkv + h - p.hq) * D);
    return reinterpret_cast<const uint4*>(p.v_new + (static_cast<size_t>(t) * p.hkv + h - p.hq - p.hkv) * D);
  };
  for (int base = threadIdx.x; base < total; base += kRopeBatch * blockDim.x) {
    uint4 xa[kRopeBatch], xb[kRopeBatch];
#pragma unroll
    for (int u = 0; u < kRopeBatch; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx < total) {
        int nd, h, v;
        const uint4* src = src_of(idx, nd, h, v);
        xa[u] = src[v];
        xb[u] = style0 ? xa[u] : src[v + VPH / 2];
      }
    }
#pragma unroll
    for (int u = 0; u < kRopeBatch; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx >= total) break;
      int nd, h, v;
      src_of(idx, nd, h, v);
      const int i = i0 + nd;
      const float2* cs = s_cs[nd];
      uint4* dst;
      if (h < p.hq) {
        dst = reinterpret_cast<uint4*>(p.q_rot + (static_cast<size_t>(t0 + i) * p.hq + h) * D);
      } else {
        const bool isv = h >= p.hq + p.hkv;
        const int hh = isv ? h - p.hq - p.hkv : h - p.hq;
        const int slot = plen + i;
        dst = reinterpret_cast<uint4*>(
            (isv ? p.v_cache : p.k_cache) +
            ((static_cast<size_t>(s_blk[nd]) * p.hkv + hh) * TV_BLOCK_SIZE + slot % TV_BLOCK_SIZE) * D);
        if (isv) {                                              // value: plain copy
          dst[v] = xa[u];
          if (!style0) dst[v + VPH / 2] = xb[u];
          continue;
        }
      }
      if (style0) {
        const uint32_t w[4] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 c = cs[v * 4 + e];
          const float a = bf16_lo(w[e]), bb = bf16_hi(w[e]);
          o[e] = pack_bf16x2(a * c.x - bb * c.y, bb * c.x + a * c.y);
        }
        dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
      } else {
        const uint32_t wa[4] = {xa[u].x, xa[u].y, xa[u].z, xa[u].w};
        const uint32_t wb[4] = {xb[u].x, xb[u].y, xb[u].z, xb[u].w};
        uint32_t oa[4], ob[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int pr0 = v * 8 + 2 * e;                        // element index in the first half
          const float2 c0 = cs[pr0], c1 = cs[pr0 + 1];
          const float a0 = bf16_lo(wa[e]), a1 = bf16_hi(wa[e]);
          const float b0 = bf16_lo(wb[e]), b1 = bf16_hi(wb[e]);
          oa[e] = pack_bf16x2(a0 * c0.x - b0 * c0.y, a1 * c1.x - b1 * c1.y);
          ob[e] = pack_bf16x2(b0 * c0.x + a0 * c0.y, b1 * c1.x + a1 * c1.y);
        }
        dst[v] = make_uint4(oa[0], oa[1], oa[2], oa[3]);
        dst[v + VPH / 2] = make_uint4(ob[0], ob[1], ob[2], ob[3]);
      }
    }
  }
  // zero the rest of the last page so every row of a loaded page is finite
  if (i1 == n) {
    const int end = plen + n;
    const int pad = (TV_BLOCK_SIZE - end % TV_BLOCK_SIZE) % TV_BLOCK_SIZE;
    const int blk = trow[(end - 1) / TV_BLOCK_SIZE];
    for (int idx = threadIdx.x; idx < pad * p.hkv * VPH * 2; idx += blockDim.x) {
      const int kv = idx / (pad * p.hkv * VPH);
      int rem = idx % (pad * p.hkv * VPH);
      const int r = rem / (p.hkv * VPH);
      rem %= p.hkv * VPH;
      const int h = rem / VPH, v = rem % VPH;
      const int row = end % TV_BLOCK_SIZE + r;
      __nv_bfloat16* base = kv ? p.v_cache : p.k_cache;
      reinterpret_cast<uint4*>(base + ((static_cast<size_t>(blk) * p.hkv + h) * TV_BLOCK_SIZE + row) * D)[v] =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// ------------------------------------------------------------ attention

struct TcSeg {
  int b, t0, n, plen, kvh, rg, node0, mt, tile0, tile1, ntiles;
  bool whole, skip, valid;
  long long t_next, unit_t0;
  int my_slot;
};

struct TcShape {
  int t0, n, plen, nrg, tiles;
};

__device__ __forceinline__ TcShape tc_shape(const TcParams& p, int b) {
  TcShape r;
  r.t0 = p.cu_nodes[b];
  r.n = p.cu_nodes[b + 1] - r.t0;
  r.plen = p.prompt_len[b];
  if (r.n < 1 || r.n > p.max_nodes || r.plen < 0 || r.t0 < 0 ||
      static_cast<long long>(r.t0) + r.n > p.t_cap) {
    r.nrg = r.tiles = 0;
    return r;
  }
  r.nrg = (r.n + 2 * p.npm - 1) / (2 * p.npm);
  r.tiles = static_cast<int>((static_cast<long long>(r.plen) + r.n + kTcBN - 1) / kTcBN);
  return r;
}

// exclusive prefix of per-request tile counts (all threads call)
__device__ void tc_plan_prefix(const TcParams& p, int* s_pre, int* s_tmp) {
  const int nt = blockDim.x, tid = threadIdx.x;
  const int per = (p.batch + nt - 1) / nt;
  const int lo = min(p.batch, tid * per), hi = min(p.batch, lo + per);
  int sum = 0;
  for (int b = lo; b < hi; ++b) {
    const TcShape r = tc_shape(p, b);
    sum += p.hkv * r.nrg * r.tiles;
  }
  // block-wide exclusive scan of the per-thread sums (warp shuffles, then
  // one warp scans the per-warp totals)
  const int lane = tid & 31, wid = tid >> 5, nw = (nt + 31) >> 5;
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_tmp[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = lane < nw ? s_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) s_tmp[32 + lane] = w;            // inclusive per-warp totals
    if (lane == nw - 1) s_pre[p.batch] = w;
  }
  __syncthreads();
  int run = x - sum + (wid > 0 ? s_tmp[32 + wid - 1] : 0);
  for (int b = lo; b < hi; ++b) {
    s_pre[b] = run;
    const TcShape r = tc_shape(p, b);
    run += p.hkv * r.nrg * r.tiles;
  }
  __syncthreads();
}

__device__ __forceinline__ long long tc_cta_start(long long total, int grid, int c) {
  const long long q = total / grid, rem = total % grid;
  return c * q + min(static_cast<long long>(c), rem);
}

__device__ __forceinline__ int tc_cta_of(long long total, int grid, long long t) {
  const long long q = total / grid, rem = total % grid;
  const long long big = rem * (q + 1);
  if (t < big) return static_cast<int>(t / (q + 1));
  return static_cast<int>(rem + (t - big) / q);
}

// Segment of this CTA's tile range that starts at global tile t.
__device__ TcSeg tc_segment(const TcParams& p, const int* s_pre, long long t, long long s,
                            long long e) {
  TcSeg g;
  g.valid = t < e;
  if (!g.valid) return g;
  int lo = 0, hi = p.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const TcShape r = tc_shape(p, b);
  const long long local = t - s_pre[b];
  const int unit = static_cast<int>(local / r.tiles);
  g.b = b;
  g.t0 = r.t0;
  g.n = r.n;
  g.plen = r.plen;
  g.kvh = unit / r.nrg;
  g.rg = unit % r.nrg;
  g.node0 = g.rg * 2 * p.npm;
  const int nodes_u = min(2 * p.npm, r.n - g.node0);
  g.mt = (nodes_u + p.npm - 1) / p.npm;
  g.ntiles = r.tiles;
  g.tile0 = static_cast<int>(local % r.tiles);
  g.tile1 = static_cast<int>(min(static_cast<long long>(r.tiles), g.tile0 + (e - t)));
  g.t_next = t + (g.tile1 - g.tile0);
  g.whole = g.tile0 == 0 && g.tile1 == r.tiles;
  g.unit_t0 = s_pre[b] + static_cast<long long>(unit) * r.tiles;
  g.my_slot = 2 * blockIdx.x + (t == s ? 0 : 1);
  g.skip = (p.status[b] & (TV_TREE_FLAGS | TV_ST_BAD_BLOCK)) != 0;
  return g;
}

// 32 bits of visibility for key slots [k0, k0 + 32) of a row whose node has
// ancestor bit row mrow (tree key j = slot - plen).
__device__ __forceinline__ uint32_t visible_bits(const uint32_t* mrow, int words, int plen, int n,
                                                 int k0) {
  uint32_t bits;
  if (k0 + 32 <= plen) return 0xFFFFFFFFu;
  bits = k0 >= plen ? 0u : ((1u << (plen - k0)) - 1u);
  const int j0 = k0 - plen;                          // may be negative
  if (j0 + 32 > 0 && j0 < n) {
    const int wi = j0 >= 0 ? (j0 >> 5) : -1;
    const int sh = j0 - 32 * wi;
    const uint32_t lo = (wi >= 0 && wi < words) ? __ldg(mrow + wi) : 0u;
    const uint32_t hi = (wi + 1 >= 0 && wi + 1 < words) ? __ldg(mrow + wi + 1) : 0u;
    uint32_t tb = __funnelshift_r(lo, hi, sh);
    if (j0 + 32 > n) tb &= (n - j0 >= 32) ? 0xFFFFFFFFu : ((1u << (n - j0)) - 1u);
    if (j0 < 0) tb &= ~((1u << (-j0)) - 1u);
    bits |= tb;
  }
  return bits;
}

template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;
  static constexpr uint32_t kHalfBytes = 128 * 128;                 // 128 rows x 128 B
  static constexpr uint32_t kQBytes = 2 * kHalves * kHalfBytes;     // two M tiles
  static constexpr uint32_t kTileBytes = kHalves * kHalfBytes;      // one K or V tile
  static constexpr uint32_t kSmem = kQBytes + 2 * kTcStages * kTileBytes;
};

struct TcBars {
  uint64_t q_full, q_empty, drain;
  uint64_t k_full[kTcStages], v_full[kTcStages], k_empty[kTcStages], v_empty[kTcStages];
  uint64_t s_ready[2], p_ready[2], o_done[2], o_free[2];
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kQBytes;
  uint8_t* sV = sK + kTcStages * C::kTileBytes;
  int* s_pre = reinterpret_cast<int*>(sV + kTcStages * C::kTileBytes);
  __shared__ TcBars bars;
  __shared__ int s_tmp[kTcThreads];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    mbar_init(&bars.drain, 1);
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    for (int m = 0; m < 2; ++m) {
      mbar_init(&bars.s_ready[m], 1);
      mbar_init(&bars.p_ready[m], 4);
      mbar_init(&bars.o_done[m], 1);
      mbar_init(&bars.o_free[m], 4);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.qmap);
    tma_prefetch_desc(&p.kmap);
    tma_prefetch_desc(&p.vmap);
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  tc_plan_prefix(p, s_pre, s_tmp);        // contains __syncthreads; reads only call inputs
  tc_fence_after();
  grid_launch_dependents();               // the merge grid may start its prologue
  grid_dependency_wait();                 // rotated q, tentative KV and status are written
  const uint32_t tbase = s_tmem;
  volatile int* abort = &s_abort;
  const long long total = s_pre[p.batch];
  const long long cs = tc_cta_start(total, p.grid, blockIdx.x);
  const long long ce = tc_cta_start(total, p.grid, blockIdx.x + 1);
  const int G = p.group, npm = p.npm;
  const int32_t* table_base = p.block_table;

  if (warp == 0 || warp == 2) {
    // ================================================= TMA producers
    // warp 0 streams Q and K, warp 2 streams V. K of a stage is free once the
    // S MMAs that read it finished, V once the PV MMAs did, so the two
    // streams run ahead independently. The whole warp runs the loop: lane j
    // fetches page j's block-table entry (one coalesced load per tile) and
    // issues that page's copies.
    const bool is_k = warp == 0;
    uint64_t* full = is_k ? bars.k_full : bars.v_full;
    uint64_t* empty = is_k ? bars.k_empty : bars.v_empty;
    uint8_t* dst_base = is_k ? sK : sV;
    const CUtensorMap* map = is_k ? &p.kmap : &p.vmap;
    uint32_t it = 0, qs = 0;
    bool ok = true;
    for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); ok && g.valid;
         g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
      if (g.skip) continue;
      if (is_k) {
        ok = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(&bars.q_empty, (qs & 1) ^ 1, abort) : false, 0);
        if (!ok) break;
        ++qs;
        if (lane == 0) {
          const uint32_t qbox = 64u * 2u * G * npm;
          mbar_arrive_expect_tx(&bars.q_full, qbox * C::kHalves * g.mt);
          for (int m = 0; m < g.mt; ++m)
            for (int h = 0; h < C::kHalves; ++h)
              tma_load_4d(sQ + (m * C::kHalves + h) * C::kHalfBytes, &p.qmap, h * 64, 0, g.kvh,
                          g.t0 + g.node0 + m * npm, &bars.q_full);
        }
      }
      const int32_t* trow = table_base + static_cast<size_t>(g.b) * p.max_blocks;
      const long long end = static_cast<long long>(g.plen) + g.n;
      for (int t = g.tile0; t < g.tile1; ++t, ++it) {
        const int s = it % kTcStages;
        const int p0 = t * (kTcBN / TV_BLOCK_SIZE);
        const long long hi = min(end, static_cast<long long>(t + 1) * kTcBN);
        const int np = static_cast<int>((hi + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE) - p0;
        const int blk = lane < np ? __ldg(trow + p0 + lane) : 0;
        ok = __shfl_sync(0xffffffffu,
                         lane == 0 ? mbar_wait(&empty[s], ((it / kTcStages) & 1) ^ 1, abort) : false, 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], np * C::kHalves * 2048u);
        __syncwarp();
        if (lane < np) {
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h)
            tma_load_4d(dst_base + s * C::kTileBytes + lane * 2048 + h * C::kHalfBytes, map, h * 64, 0,
                        g.kvh, blk, &full[s]);
        }
      }
    }
    // never leave copies in flight: wait for the stages this warp filled
    for (uint32_t k = (it > kTcStages ? it - kTcStages : 0); lane == 0 && k < it; ++k) {
      volatile int no_abort = 0;
      mbar_wait(&full[k % kTcStages], (k / kTcStages) & 1, &no_abort);
    }
  } else if (warp == 1) {
    // ================================================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kTcBN, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
      // A single thread issues every MMA, so the issue path must be short:
      // the shared-memory descriptors are built once here and each K step
      // only adds a compile-time offset (the start-address field is the low
      // 14 bits, in 16-byte units; stage bases are far below 256 KB, so the
      // addition never carries out of the field).
      const uint64_t dQ0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dQ1 = smem_desc_sw128(smem_u32(sQ) + C::kHalves * C::kHalfBytes, 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dK1 = smem_desc_sw128(smem_u32(sK) + C::kTileBytes, 16, 1024);
      const uint64_t dV0 = smem_desc_sw128(smem_u32(sV), C::kHalfBytes, 1024);
      const uint64_t dV1 = smem_desc_sw128(smem_u32(sV) + C::kTileBytes, C::kHalfBytes, 1024);
      static_assert(kTcStages == 2, "descriptor bases are precomputed for two stages");
      uint32_t it = 0, qs = 0, pc[2] = {0, 0}, of[2] = {0, 0};
      bool used[2] = {false, false};
      bool ok = true;
      auto issue_s = [&](int m, int s) {
        const uint32_t d = tbase + m * 256;
        const uint64_t a0 = m ? dQ1 : dQ0;
        const uint64_t b0 = s ? dK1 : dK0;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          constexpr uint32_t kStep = 32 / 16;                       // 32 bytes per K step
          const uint64_t off = (k / 4) * (C::kHalfBytes / 16) + (k % 4) * kStep;
          mma_ss(d, a0 + off, b0 + off, idS, k > 0 ? 1u : 0u);
        }
        mma_commit(&bars.s_ready[m]);
      };
      auto issue_pv = [&](int m, int s, int kchunks, bool accumulate) {
        const uint32_t d = tbase + m * 256 + 128;
        const uint32_t a = tbase + m * 256;
        const uint64_t b0 = s ? dV1 : dV0;
#pragma unroll
        for (int k = 0; k < kTcBN / 16; ++k) {
          if (k < kchunks) mma_ts(d, a + k * 8, b0 + k * (2048 / 16), idO, (accumulate || k > 0) ? 1u : 0u);
        }
      };
      for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); ok && g.valid;
           g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
        if (g.skip) continue;
        if (!(ok = mbar_wait(&bars.q_full, qs & 1, abort))) break;
        ++qs;
        tc_fence_after();
        const int nt = g.tile1 - g.tile0;
        const long long end = static_cast<long long>(g.plen) + g.n;
        bool pv_started[2] = {false, false};
        // Ping-pong order per step i: PV_0(i-1), S_0(i), PV_1(i-1), S_1(i).
        // S_m(i) reuses the Tensor Memory columns P_m(i-1) occupies, so it is
        // issued after PV_m(i-1); tcgen05 MMAs from one thread run in order.
        // A PV never waits for the next K tile.
        for (int i = 0; i <= nt && ok; ++i) {
          const uint32_t iti = it + i;
          const int s = iti % kTcStages;
          const int sp = (iti - 1) % kTcStages;
          int kch = 0;
          if (i > 0) {
            const long long hi = min(end, static_cast<long long>(g.tile0 + i) * kTcBN);
            kch = static_cast<int>((hi - static_cast<long long>(g.tile0 + i - 1) * kTcBN + 15) / 16);
          }
          for (int m = 0; m < g.mt && ok; ++m) {
            if (i > 0) {
              if (!(ok = mbar_wait(&bars.p_ready[m], pc[m] & 1, abort))) break;
              ++pc[m];
              if (!pv_started[m] && used[m]) {
                if (!(ok = mbar_wait(&bars.o_free[m], of[m] & 1, abort))) break;
                ++of[m];
              }
              if (m == 0 && !(ok = mbar_wait(&bars.v_full[sp], ((iti - 1) / kTcStages) & 1, abort))) break;
              tc_fence_after();
              issue_pv(m, sp, kch, pv_started[m]);
              pv_started[m] = true;
              if (i == nt) mma_commit(&bars.o_done[m]);
            }
            if (i < nt) {
              if (m == 0) {
                if (!(ok = mbar_wait(&bars.k_full[s], (iti / kTcStages) & 1, abort))) break;
                tc_fence_after();
              }
              issue_s(m, s);
            }
          }
          if (!ok) break;
          if (i > 0) mma_commit(&bars.v_empty[sp]);
          if (i < nt) mma_commit(&bars.k_empty[s]);
          if (i == nt - 1) mma_commit(&bars.q_empty);    // the last S of the segment
        }
        for (int m = 0; m < g.mt; ++m) used[m] = true;
        it += nt;
      }
      // drain: every MMA issued so far completes before Tensor Memory is freed
      mma_commit(&bars.drain);
      volatile int no_abort = 0;
      mbar_wait(&bars.drain, 0, &no_abort);
    }
  } else {
    // ================================================= softmax groups
    const int m = (warp - 3) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + m * 256 + lane_addr;
    const uint32_t tO = tS + 128;
    uint32_t sc = 0, oc = 0;
    bool ok = true;
    for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); ok && g.valid;
         g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
      if (g.skip) continue;
      const int nt = g.tile1 - g.tile0;
      const int nd = g.node0 + m * npm + row / G;    // node of this row
      const bool row_valid = m < g.mt && row < G * npm && nd < g.n;
      const bool warp_live = __any_sync(0xffffffffu, row_valid);
      float m_ref = -INFINITY, l_sum = 0.f;
      if (m < g.mt) {
        const uint32_t* mrow = p.mask + static_cast<size_t>(g.t0 + (row_valid ? nd : 0)) * p.words;
        for (int i = 0; i < nt && ok; ++i) {
          if (!(ok = mbar_wait(&bars.s_ready[m], sc & 1, abort))) break;
          ++sc;
          tc_fence_after();
          if (warp_live) {
            const int k0 = (g.tile0 + i) * kTcBN;
            float s[kTcBN];
            uint32_t* su = reinterpret_cast<uint32_t*>(s);
#pragma unroll
            for (int c = 0; c < kTcBN / 32; ++c) tmem_ld32(tS + c * 32, su + c * 32);
            tmem_ld_wait();
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kTcBN / 32; ++c) {
              const uint32_t vis = row_valid ? visible_bits(mrow, p.words, g.plen, g.n, k0 + c * 32) : 0u;
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const float v = ((vis >> e) & 1u) ? s[c * 32 + e] : -INFINITY;
                s[c * 32 + e] = v;
                mx = fmaxf(mx, v);
              }
            }
            // Lazy rescale: keep the reference max until a score exceeds it by
            // 2^8; p stays <= 2^8 and O, l share the same reference.
            const float mxs = mx * p.scale_log2;
            float alpha = 1.f;
            if (mxs > m_ref + 8.f) {
              alpha = (i > 0 && m_ref != -INFINITY) ? fast_exp2(m_ref - mxs) : 1.f;
              l_sum *= alpha;
              m_ref = mxs;
            }
            const float base = m_ref == -INFINITY ? 0.f : m_ref;
#pragma unroll
            for (int c = 0; c < kTcBN / 32; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float p0 = fast_exp2(fmaf(s[c * 32 + 2 * e], p.scale_log2, -base));
                const float p1 = fast_exp2(fmaf(s[c * 32 + 2 * e + 1], p.scale_log2, -base));
                l_sum += p0 + p1;
                pk[e] = pack_bf16x2(p0, p1);
              }
              tmem_st16(tS + c * 16, pk);
            }
            if (alpha != 1.f) {                         // O holds earlier tiles: rescale it
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tmem_st32(tO + c * 32, o);
              }
            }
            tmem_st_wait();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.p_ready[m]);
        }
        if (ok && (ok = mbar_wait(&bars.o_done[m], oc & 1, abort))) {
          ++oc;
          tc_fence_after();
          if (warp_live) {
            const int h = g.kvh * G + row % G;
            if (g.whole) {
              __nv_bfloat16* dst = p.out + (static_cast<size_t>(g.t0 + nd) * p.hq + h) * D;
              const float inv = 1.f / l_sum;
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                if (row_valid) {
                  uint4* d4 = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
                  for (int q = 0; q < 4; ++q)
                    d4[q] = make_uint4(
                        pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                        pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                        pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                        pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
                }
              }
            } else {
              // partial of a split unit, stored column-block major so the
              // 128 rows of a group write (and the merge reads) contiguously
              float4* part = reinterpret_cast<float4*>(p.partials + static_cast<size_t>(g.my_slot) * kSlotFloats(D));
              const int r = m * 128 + row;
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tO + c * 32, o);
                tmem_ld_wait();
                if (row_valid) {
#pragma unroll
                  for (int q = 0; q < 8; ++q)
                    part[(c * 8 + q) * 256 + r] =
                        make_float4(__uint_as_float(o[4 * q]), __uint_as_float(o[4 * q + 1]),
                                    __uint_as_float(o[4 * q + 2]), __uint_as_float(o[4 * q + 3]));
                }
              }
              if (row_valid) {
                float* ml = reinterpret_cast<float*>(part + (D / 4) * 256);
                ml[r] = m_ref;
                ml[256 + r] = l_sum;
              }
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.o_free[m]);
        }
      }
      if (!ok) break;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  if (threadIdx.x == 0) {
    // Merge task for the unit this CTA's range starts (a unit cut at this
    // CTA's end, whose first tile is in this range); the merge kernel reads it.
    int32_t* rec = p.tasks + blockIdx.x * kTaskInts;
    int valid = 0;
    TcSeg last;
    last.valid = false;
    for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); g.valid; g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
      if (s_abort) atomicOr(p.status_rw + g.b, TV_ST_TIMEOUT);   // flag what this CTA touched
      last = g;
    }
    if (!s_abort && last.valid && !last.skip && last.tile0 == 0 && last.tile1 < last.ntiles) {
      valid = 1;
      rec[1] = last.b;
      rec[2] = last.kvh;
      rec[3] = last.node0;
      rec[4] = last.mt;
      rec[5] = last.t0;
      rec[6] = last.n;
      rec[7] = blockIdx.x;                                              // first contributor
      rec[8] = tc_cta_of(total, p.grid, last.unit_t0 + last.ntiles - 1); // last contributor
      rec[9] = last.my_slot;                                            // its slot
    }
    rec[0] = valid;
  }
}

// ------------------------------------------------------------ merge of split units
//
// A unit whose key tiles were cut between CTAs c_first..c_last left one
// partial (unnormalised O, reference max m, sum l, all per row) per
// contributor. Merging is the usual log-sum-exp combination:
//   out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c.
// kMergeSplit CTAs per split unit (32 rows each, 8 threads per row); each
// thread loads kMergeChunk contributors' partials at once.

struct MergeParams {
  const int32_t* tasks;
  const float* partials;
  __nv_bfloat16* out;
  int hq, group, npm;
};

constexpr int kMergeThreads = 256;
constexpr int kMergeSplit = 8;      // CTAs per unit (32 rows each)
constexpr int kMergeChunk = 4;      // contributors whose loads are in flight together

template <int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const __grid_constant__ MergeParams p) {
  grid_dependency_wait();            // the attention grid's partials and tasks are visible
  const int c = blockIdx.x / kMergeSplit, part_cta = blockIdx.x % kMergeSplit;
  const int32_t* rec = p.tasks + c * kTaskInts;
  if (rec[0] == 0) return;
  const int kvh = rec[2], node0 = rec[3], mt = rec[4], t0 = rec[5], n = rec[6];
  const int c_first = rec[7], c_last = rec[8], first_slot = rec[9];
  constexpr int kRowsCta = 256 / kMergeSplit;         // 32 rows per CTA
  constexpr int kParts = kMergeThreads / kRowsCta;    // 8 threads per row
  constexpr int kVecs = D / 4 / kParts;               // float4 per thread
  const int r = part_cta * kRowsCta + threadIdx.x % kRowsCta;
  const int part = threadIdx.x / kRowsCta;
  const int mm = r >> 7, rr = r & 127;
  const int G = p.group;
  const int nd = node0 + mm * p.npm + rr / G;
  if (mm >= mt || rr >= G * p.npm || nd >= n) return;
  const int nc = c_last - c_first + 1;
  // single pass, online log-sum-exp over chunks of contributors
  float m_run = -INFINITY, l_run = 0.f;
  float4 acc[kVecs];
#pragma unroll
  for (int v = 0; v < kVecs; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nc; k0 += kMergeChunk) {
    float mc[kMergeChunk], lc[kMergeChunk];
    float4 x[kMergeChunk][kVecs];
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      const int k = k0 + u;
      mc[u] = -INFINITY;
      lc[u] = 0.f;
      if (k < nc) {
        const int sl = k == 0 ? first_slot : 2 * (c_first + k);
        const float* base = p.partials + static_cast<size_t>(sl) * kSlotFloats(D);
        mc[u] = __ldcg(base + D * 256 + r);
        lc[u] = __ldcg(base + D * 256 + 256 + r);
        const float4* o4 = reinterpret_cast<const float4*>(base);
#pragma unroll
        for (int v = 0; v < kVecs; ++v) x[u][v] = __ldcg(o4 + (part * kVecs + v) * 256 + r);
      }
    }
    float m_new = m_run;
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) m_new = fmaxf(m_new, mc[u]);
    if (m_new == -INFINITY) continue;
    const float sc = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new);
    l_run *= sc;
#pragma unroll
    for (int v = 0; v < kVecs; ++v) {
      acc[v].x *= sc;
      acc[v].y *= sc;
      acc[v].z *= sc;
      acc[v].w *= sc;
    }
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      if (mc[u] == -INFINITY) continue;
      const float w = fast_exp2(mc[u] - m_new);
      l_run += w * lc[u];
#pragma unroll
      for (int v = 0; v < kVecs; ++v) {
        acc[v].x += w * x[u][v].x;
        acc[v].y += w * x[u][v].y;
        acc[v].z += w * x[u][v].z;
        acc[v].w += w * x[u][v].w;
      }
    }
    m_run = m_new;
  }
  const float inv = 1.f / l_run;
  const int h = kvh * G + rr % G;
  uint2* dst = reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(t0 + nd) * p.hq + h) * D +
                                        part * kVecs * 4);
#pragma unroll
  for (int v = 0; v < kVecs; ++v)
    dst[v] = make_uint2(pack_bf16x2(acc[v].x * inv, acc[v].y * inv),
                        pack_bf16x2(acc[v].z * inv, acc[v].w * inv));
}

// ------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

static bool encode_4d(CUtensorMap* map, void* base, const cuuint64_t dims[4],
                      const cuuint64_t strides[3], const cuuint32_t box[4]) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct TcLayout {
  size_t task_bytes, partial_bytes, qrot_bytes, total;
  int npm;
};

static TcLayout tc_layout(int batch, int hq, int hkv, int max_nodes, int head_dim, int grid) {
  TcLayout L;
  const int group = hq / hkv;
  L.npm = 128 / group;
  L.task_bytes = (static_cast<size_t>(grid) * kTaskInts * sizeof(int32_t) + 255) / 256 * 256;
  L.partial_bytes = static_cast<size_t>(2) * grid * kSlotFloats(head_dim) * sizeof(float);
  L.partial_bytes = (L.partial_bytes + 255) / 256 * 256;
  L.qrot_bytes = static_cast<size_t>(batch) * max_nodes * hq * head_dim * 2;
  L.total = L.task_bytes + L.partial_bytes + L.qrot_bytes;
  return L;
}

int tc_grid() {
  const int dev = current_device();
  return dev < 0 ? -1 : device_sm_count(dev);
}

size_t tc_workspace_bytes(int batch, int hq, int hkv, int max_nodes, int head_dim, int grid) {
  return tc_layout(batch, hq, hkv, max_nodes, head_dim, grid).total;
}

int launch_attention_tc(const tv_geom* geom, int batch, int max_nodes, const void* q,
                        const void* k_new, const void* v_new, const int32_t* cu_nodes,
                        const int32_t* positions, const uint32_t* mask, const int32_t* prompt_len,
                        const int32_t* block_table, const int32_t* n_blocks, int max_blocks,
                        void* k_cache, void* v_cache, int num_blocks, void* out, void* workspace,
                        size_t ws_bytes, int32_t* status, cudaStream_t stream) {
  const int grid = tc_grid();
  if (grid <= 0) return TV_ERR_CUDA;
  if (batch > kTcMaxBatch) return TV_ERR_BAD_SIZE;
  const int D = geom->head_dim, hq = geom->num_q_heads, hkv = geom->num_kv_heads;
  const int group = hq / hkv;
  const TcLayout L = tc_layout(batch, hq, hkv, max_nodes, D, grid);
  if (ws_bytes < L.total) return TV_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  __nv_bfloat16* q_rot = reinterpret_cast<__nv_bfloat16*>(ws + L.task_bytes + L.partial_bytes);
  const int t_cap = batch * max_nodes;

  RopeParams rp;
  rp.q = static_cast<const __nv_bfloat16*>(q);
  rp.k_new = static_cast<const __nv_bfloat16*>(k_new);
  rp.v_new = static_cast<const __nv_bfloat16*>(v_new);
  rp.cu_nodes = cu_nodes;
  rp.positions = positions;
  rp.prompt_len = prompt_len;
  rp.block_table = block_table;
  rp.n_blocks = n_blocks;
  rp.q_rot = q_rot;
  rp.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  rp.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  rp.status = status;
  rp.batch = batch;
  rp.max_nodes = max_nodes;
  rp.t_cap = t_cap;
  rp.hq = hq;
  rp.hkv = hkv;
  rp.max_blocks = max_blocks;
  rp.num_blocks = num_blocks;
  rp.rope_style = geom->rope_style;
  for (int i = 0; i < 64; ++i)
    rp.inv_freq[i] = i < D / 2 ? static_cast<float>(pow(double(geom->rope_base), -2.0 * i / D)) : 0.f;

  TcParams tp;
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(group),
                                static_cast<cuuint64_t>(hkv), static_cast<cuuint64_t>(t_cap)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(group) * D * 2,
                                   static_cast<cuuint64_t>(hq) * D * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(group), 1, static_cast<cuuint32_t>(L.npm)};
    if (!encode_4d(&tp.qmap, q_rot, dims, strides, box)) return TV_ERR_CUDA;
  }
  {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), TV_BLOCK_SIZE, static_cast<cuuint64_t>(hkv),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(TV_BLOCK_SIZE) * D * 2,
                                   static_cast<cuuint64_t>(hkv) * TV_BLOCK_SIZE * D * 2};
    const cuuint32_t box[4] = {64, TV_BLOCK_SIZE, 1, 1};
    if (!encode_4d(&tp.kmap, k_cache, dims, strides, box)) return TV_ERR_CUDA;
    if (!encode_4d(&tp.vmap, v_cache, dims, strides, box)) return TV_ERR_CUDA;
  }
  tp.cu_nodes = cu_nodes;
  tp.prompt_len = prompt_len;
  tp.mask = mask;
  tp.block_table = block_table;
  tp.status = status;
  tp.out = static_cast<__nv_bfloat16*>(out);
  tp.tasks = reinterpret_cast<int32_t*>(ws);
  tp.partials = reinterpret_cast<float*>(ws + L.task_bytes);
  tp.status_rw = status;
  tp.batch = batch;
  tp.max_nodes = max_nodes;
  tp.t_cap = t_cap;
  tp.hq = hq;
  tp.hkv = hkv;
  tp.group = group;
  tp.npm = L.npm;
  tp.words = (max_nodes + 31) / 32;
  tp.max_blocks = max_blocks;
  tp.grid = grid;
  const double scale = geom->softmax_scale > 0.f ? geom->softmax_scale : 1.0 / sqrt(double(D));
  tp.scale_log2 = static_cast<float>(scale * 1.4426950408889634);

  MergeParams mp;
  mp.tasks = tp.tasks;
  mp.partials = tp.partials;
  mp.out = tp.out;
  mp.hq = hq;
  mp.group = group;
  mp.npm = L.npm;

  const dim3 rgrid((max_nodes + kRopeNodes - 1) / kRopeNodes, batch);
  static size_t smem_set128[kMaxDevices] = {0}, smem_set64[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0) return TV_ERR_CUDA;
  const size_t smem_fixed = (D == 128 ? TcCfg<128>::kSmem : TcCfg<64>::kSmem) + 1024;
  const size_t smem = smem_fixed + static_cast<size_t>(batch + 1) * sizeof(int);
  if (smem > 227 * 1024) return TV_ERR_BAD_SIZE;

  // The attention and merge grids are launched with programmatic stream
  // serialisation: each may start (prologue, Tensor Memory allocation, work
  // plan) while the grid before it finishes, and waits in griddepcontrol.wait
  // before reading what that grid writes.
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t acfg = {};
  acfg.gridDim = dim3(grid);
  acfg.blockDim = dim3(kTcThreads);
  acfg.dynamicSmemBytes = smem;
  acfg.stream = stream;
  acfg.attrs = pdl;
  acfg.numAttrs = 1;
  cudaLaunchConfig_t mcfg = acfg;
  mcfg.gridDim = dim3(grid * kMergeSplit);
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.dynamicSmemBytes = 0;
  cudaError_t err;
  if (D == 128) {
    rope_append_kernel<128><<<rgrid, kRopeThreads, 0, stream>>>(rp);
    if (!ensure_smem(attn_tc_kernel<128>, smem, smem_set128, dev)) return TV_ERR_CUDA;
    err = cudaLaunchKernelEx(&acfg, attn_tc_kernel<128>, tp);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&mcfg, attn_merge_kernel<128>, mp);
  } else {
    rope_append_kernel<64><<<rgrid, kRopeThreads, 0, stream>>>(rp);
    if (!ensure_smem(attn_tc_kernel<64>, smem, smem_set64, dev)) return TV_ERR_CUDA;
    err = cudaLaunchKernelEx(&acfg, attn_tc_kernel<64>, tp);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&mcfg, attn_merge_kernel<64>, mp);
  }
  if (err != cudaSuccess) return TV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
