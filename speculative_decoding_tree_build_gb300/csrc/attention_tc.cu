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
// Three launches on the caller's stream:
//  1. rope_append_kernel: rotates q (into the workspace) and k (into the
//     tentative cache slots P + i, with the raw v) - "投机解码的树状注意力验证…",
//     section "实现中的 KV Cache 与批处理约束": the tree's tentative KV is a
//     contiguous region in node order. It also zero-fills the rest of the last
//     page so every row a tile reads is finite.
//  2. attn_tc_kernel: keys are cache slots [0, P + N); slots >= P are tested
//     against the node's ancestor bit row. One CTA per SM, warp-specialised:
//       warps 0, 3  TMA producers: warp 0 the Q tiles and per 128-key step
//                   the K pages, warp 3 the V pages (4-D tensor maps over the
//                   paged pools, 128-byte swizzle), each with its own barrier
//       warp 1      MMA issuer for both 128-row M tiles: S = Q K^T (A, B in
//                   shared memory, N = 128 keys) and O += P V (P read from
//                   Tensor Memory), fp32 accumulators. The issue order
//                   S0(j), PV1(j-1), S1(j), PV0(j) makes the tensor core
//                   alternate between the tiles, so each tile's softmax runs
//                   while the tensor core works on the other tile; a
//                   one-tile unit alternates between both score buffers.
//       warp 2      prefetches the first prompt K/V pages into L2 while the
//                   pre-pass finishes, then idles (it keeps the softmax
//                   warps on their lane quarters)
//       warps 4-11  two 128-thread softmax groups (one per M tile), one
//                   Tensor Memory lane (= one query row) per thread.
//     Query rows of a unit are (node, query head in the GQA group), node
//     major, spread evenly over the eight 32-row quarters of the two M tiles,
//     so one K/V tile feeds up to 256 rows. Work plan: a unit is (request,
//     KV head, group of up to 256 rows); all units' key tiles are laid end to
//     end and every CTA takes a contiguous share of equal estimated cost
//     (two-tile steps, one-tile steps and a fixed cost per unit weighted as
//     measured), computed on the device from cu_nodes/prompt_len (no host
//     round trip), so the CTAs finish together whatever the mix.
//  3. attn_merge_kernel: a unit cut between CTAs left one partial per CTA;
//     this grid merges them (log-sum-exp), many CTAs and loads in flight.
//  Launches 2 and 3 use programmatic dependent launch so their prologues
//  overlap the previous grid's tail. No CTA ever waits for another CTA.
#include <algorithm>

#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "tv_sm100.cuh"

namespace tv {

constexpr int kTcBN = 128;          // keys per work-plan tile = per pipeline step (S width)
constexpr int kTcThreads = 384;     // 12 warps
constexpr int kTcMaxBatch = 4096;
constexpr int kRopeNodes = 1;       // nodes per pre-pass CTA
constexpr int kRopeBatch = 3;       // loads in flight per pre-pass thread
constexpr int kRopeThreads = 256;
constexpr int kRopeMinBlocks = 8;   // 32 registers a thread: the whole SM's threads may run the pre-pass
constexpr int kTaskInts = 16;       // merge-task record per attention CTA

// bytes of one partial-result slot: O / l as fp16 [D/8 column blocks][256
// rows] x 16 B, then the per-row reference max and sum (fp32)
__host__ __device__ constexpr size_t kSlotBytes(int d) { return static_cast<size_t>(256) * (2 * d + 8); }

struct TcParams {
  CUtensorMap qmap;      // rotated q in the workspace, dims (D, G, Hkv, T_cap), box (64, G, 1, npq)
  CUtensorMap kmap;      // K pool, dims (D, 16, Hkv, num_blocks)
  CUtensorMap vmap;      // V pool
  const int32_t* cu_nodes;
  const int32_t* prompt_len;
  const uint32_t* mask;
  const int32_t* block_table;
  const int32_t* status;
  __nv_bfloat16* out;
  int32_t* tasks;        // kTaskInts per CTA: the split unit this CTA starts (merge work)
  uint8_t* partials;     // two slots of kSlotBytes(D) per CTA
  int32_t* status_rw;
  int batch, max_nodes, t_cap, hq, hkv, group, npq, words, max_blocks, num_blocks, grid;   // npq = 32 / G nodes per quarter
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

template <int D, bool kStyle0>
__global__ void __launch_bounds__(kRopeThreads, kRopeMinBlocks) rope_append_kernel(const __grid_constant__ RopeParams p) {
  constexpr int D2 = D / 2;
  __shared__ float2 s_cs[kRopeNodes][D2];
  __shared__ int s_blk[kRopeNodes];      // cache block of each node's tentative slot
  grid_dependency_wait();                // inputs written by the previous kernel are visible
  grid_launch_dependents();              // the attention grid may start its prologue
  // blockIdx.x = request, blockIdx.y = node chunk: the CTAs are dispatched
  // chunk by chunk, so those past a short tree's last node (which return at
  // once) come after every request's first nodes
  const int b = blockIdx.x;
  // the request's scalars, loaded together (one memory round trip)
  const int t0 = p.cu_nodes[b];
  const int t1 = p.cu_nodes[b + 1];
  const int plen = p.prompt_len[b];
  const int st = p.status[b];
  const int held = p.n_blocks[b];
  const int n = t1 - t0;
  if (n < 1 || n > p.max_nodes || plen < 0) return;             // tree_build flagged it
  if (static_cast<long long>(t0) + n > p.t_cap || t0 < 0) {
    if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(p.status + b, TV_ST_BAD_SIZE);
    return;
  }
  if (st & TV_TREE_FLAGS) return;
  const int i0 = blockIdx.y * kRopeNodes;
  if (i0 >= n) return;
  const int i1 = min(n, i0 + kRopeNodes);
  constexpr bool style0 = kStyle0;
  // Work item = one 16-byte vector (8 bf16) of one head of one node; style 0
  // rotates the pairs inside the vector, style 1 pairs vector v with vector
  // v + D/16. A thread loads kBatch items before storing any, and the
  // first batch (every item, for the 8B geometry) is loaded before the
  // block-table check, so the CTA waits on memory about twice, not five times.
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
  // style 1 holds two vectors per item, so it keeps fewer items in flight
  // within the 32-register budget
  constexpr int kBatch = kStyle0 ? kRopeBatch : 1;
  uint4 xa[kBatch], xb[kBatch];
  auto load_batch = [&](int base) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx < total) {
        int nd, h, v;
        const uint4* src = src_of(idx, nd, h, v);
        xa[u] = src[v];
        xb[u] = style0 ? xa[u] : src[v + VPH / 2];
      }
    }
  };
  load_batch(threadIdx.x);
  // every block holding slots [0, P + n) must be held and in range (the
  // loads of a thread are independent, so they are all in flight at once)
  const long long slots = static_cast<long long>(plen) + n;
  const int nlb = static_cast<int>((slots + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE);
  const int32_t* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  int bad = (nlb > held || nlb > p.max_blocks) ? 1 : 0;
  if (!bad) {
#pragma unroll 8
    for (int lb = threadIdx.x; lb < nlb; lb += blockDim.x) {
      const int blk = trow[lb];
      bad |= (blk < 0 || blk >= p.num_blocks) ? 1 : 0;
    }
  }
  if (threadIdx.x < i1 - i0) s_blk[threadIdx.x] = bad ? 0 : trow[(plen + i0 + threadIdx.x) / TV_BLOCK_SIZE];
  for (int idx = threadIdx.x; idx < (i1 - i0) * D2; idx += blockDim.x) {
    const int nd = idx / D2, pr = idx % D2;
    float sn, cs;
    sincosf(static_cast<float>(p.positions[t0 + i0 + nd]) * p.inv_freq[pr], &sn, &cs);
    s_cs[nd][pr] = make_float2(cs, sn);
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(p.status + b, TV_ST_BAD_BLOCK);
    return;
  }
  for (int base = threadIdx.x; base < total; base += kBatch * blockDim.x) {
    if (base != static_cast<int>(threadIdx.x)) load_batch(base);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
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
  int b, t0, n, plen, kvh, node0, nodes, mt, tile0, tile1, ntiles;
  bool whole, skip, valid;
  long long t_next, unit_t0;
  int my_slot;
};

struct TcShape {
  int t0, n, plen, nrg, tiles;
};

// Nodes per unit: two M tiles of four 32-lane quarters, 32 / G nodes each.
__host__ __device__ __forceinline__ int tc_unit_nodes(int npq) { return 8 * npq; }

__device__ __forceinline__ TcShape tc_shape(const TcParams& p, int b) {
  TcShape r;
  r.t0 = p.cu_nodes[b];
  const int t1 = p.cu_nodes[b + 1];
  r.plen = p.prompt_len[b];
  r.n = t1 - r.t0;
  if (r.n < 1 || r.n > p.max_nodes || r.plen < 0 || r.t0 < 0 ||
      static_cast<long long>(r.t0) + r.n > p.t_cap) {
    r.nrg = r.tiles = 0;
    return r;
  }
  r.nrg = (r.n + tc_unit_nodes(p.npq) - 1) / tc_unit_nodes(p.npq);
  r.tiles = static_cast<int>((static_cast<long long>(r.plen) + r.n + kTcBN - 1) / kTcBN);
  return r;
}

// Work plan. The tiles of all units form one global sequence (request,
// KV head, row group, key tile), and each CTA takes a contiguous range of it.
// The ranges are cut by estimated cost rather than by tile count: a 128-key
// step of a two-tile unit costs more than one of a one-tile unit, and every
// unit has a fixed cost (Q load, pipeline fill, epilogue). In cost units a
// unit is laid out as [kCostUnit + w | w | w ...] (w per tile); tile k starts
// at 0 for k = 0, else at kCostUnit + k * w; CTA c owns the tiles whose start
// lies in [floor(c W / grid), floor((c + 1) W / grid)), W the total cost.
constexpr int kCostTwo = 10;        // one step of a two-tile unit
constexpr int kCostOne = 7;         // one step of a one-tile unit
constexpr int kCostUnit = 21;       // fixed cost of a unit

__device__ __forceinline__ int tc_mt(int nodes, int npq) { return (nodes + 4 * npq - 1) / (4 * npq); }

__device__ __forceinline__ int tc_step_cost(int mt) { return mt == 2 ? kCostTwo : kCostOne; }

// row group rg of a request: its M tiles
__device__ __forceinline__ int tc_rg_mt(const TcShape& r, int rg, int npq) {
  return tc_mt(min(tc_unit_nodes(npq), r.n - rg * tc_unit_nodes(npq)), npq);
}

__device__ __forceinline__ int tc_unit_cost(const TcShape& r, int rg, int npq) {
  return kCostUnit + r.tiles * tc_step_cost(tc_rg_mt(r, rg, npq));
}

// cost of one KV head's units of a request (all row groups)
__device__ __forceinline__ int tc_head_cost(const TcShape& r, int npq) {
  if (r.nrg == 0) return 0;
  return (r.nrg - 1) * tc_unit_cost(r, 0, npq) + tc_unit_cost(r, r.nrg - 1, npq);
}

// Exclusive prefixes of per-request tile counts (s_pre) and costs (sw_pre),
// entry `batch` holding the totals (all threads call).
__device__ void tc_plan_prefix(const TcParams& p, int* s_pre, int* sw_pre, int* s_tmp) {
  const int nt = blockDim.x, tid = threadIdx.x;
  const int per = (p.batch + nt - 1) / nt;
  const int lo = min(p.batch, tid * per), hi = min(p.batch, lo + per);
  int sum = 0, wsum = 0;
  for (int b = lo; b < hi; ++b) {
    const TcShape r = tc_shape(p, b);
    sum += p.hkv * r.nrg * r.tiles;
    wsum += p.hkv * tc_head_cost(r, p.npq);
  }
  // block-wide exclusive scans of the per-thread sums (warp shuffles, then
  // one warp scans the per-warp totals)
  const int lane = tid & 31, wid = tid >> 5, nw = (nt + 31) >> 5;
  int x = sum, xw = wsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    const int yw = __shfl_up_sync(0xffffffffu, xw, o);
    if (lane >= o) {
      x += y;
      xw += yw;
    }
  }
  if (lane == 31) {
    s_tmp[wid] = x;
    s_tmp[16 + wid] = xw;
  }
  __syncthreads();
  if (wid == 0) {
    int v = lane < nw ? s_tmp[lane] : 0;
    int vw = lane < nw ? s_tmp[16 + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      const int yw = __shfl_up_sync(0xffffffffu, vw, o);
      if (lane >= o) {
        v += y;
        vw += yw;
      }
    }
    if (lane < nw) {                                  // inclusive per-warp totals
      s_tmp[32 + lane] = v;
      s_tmp[48 + lane] = vw;
    }
    if (lane == nw - 1) {
      s_pre[p.batch] = v;
      sw_pre[p.batch] = vw;
    }
  }
  __syncthreads();
  int run = x - sum + (wid > 0 ? s_tmp[32 + wid - 1] : 0);
  int wrun = xw - wsum + (wid > 0 ? s_tmp[48 + wid - 1] : 0);
  for (int b = lo; b < hi; ++b) {
    s_pre[b] = run;
    sw_pre[b] = wrun;
    const TcShape r = tc_shape(p, b);
    run += p.hkv * r.nrg * r.tiles;
    wrun += p.hkv * tc_head_cost(r, p.npq);
  }
  __syncthreads();
}

// last request whose prefix entry is <= x (requests without work share their
// successor's entry, so they are passed over)
__device__ __forceinline__ int tc_find_request(const int* pre, int batch, long long x) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// First global tile of CTA c: the first tile whose cost position is at least
// floor(c W / grid) (the total tile count for c = grid).
__device__ long long tc_cta_start(const TcParams& p, const int* s_pre, const int* sw_pre, int c) {
  const long long W = sw_pre[p.batch];
  if (c >= p.grid || W == 0) return s_pre[p.batch];
  const long long x = W * c / p.grid;
  const int b = tc_find_request(sw_pre, p.batch, x);
  const TcShape r = tc_shape(p, b);
  const int wk = tc_head_cost(r, p.npq);
  const long long local = x - sw_pre[b];
  const int kvh = static_cast<int>(local / wk);
  int rem = static_cast<int>(local % wk), rg = 0;
  for (; rg < r.nrg - 1; ++rg) {
    const int wu = tc_unit_cost(r, rg, p.npq);
    if (rem < wu) break;
    rem -= wu;
  }
  const int w = tc_step_cost(tc_rg_mt(r, rg, p.npq));
  const int k = rem <= 0 ? 0 : max(1, (rem - kCostUnit + w - 1) / w);   // may be r.tiles: the next unit's first
  return s_pre[b] + static_cast<long long>(kvh * r.nrg + rg) * r.tiles + k;
}

// The CTA whose range holds global tile t.
__device__ int tc_cta_of(const TcParams& p, const int* s_pre, const int* sw_pre, long long t) {
  const long long W = sw_pre[p.batch];
  const int b = tc_find_request(s_pre, p.batch, t);
  const TcShape r = tc_shape(p, b);
  const long long local = t - s_pre[b];
  const int unit = static_cast<int>(local / r.tiles), k = static_cast<int>(local % r.tiles);
  const int kvh = unit / r.nrg, rg = unit % r.nrg;
  const long long pos = sw_pre[b] + static_cast<long long>(kvh) * tc_head_cost(r, p.npq) +
                        static_cast<long long>(rg) * tc_unit_cost(r, 0, p.npq) +
                        (k == 0 ? 0 : kCostUnit + static_cast<long long>(k) * tc_step_cost(tc_rg_mt(r, rg, p.npq)));
  return static_cast<int>(min(static_cast<long long>(p.grid - 1), ((pos + 1) * p.grid - 1) / W));
}

// Segment of this CTA's tile range that starts at global tile t. Without
// `use_status` only the geometry is known (skip stays false): the form that
// may run before the dependency wait, since the pre-pass writes status.
__device__ TcSeg tc_segment(const TcParams& p, const int* s_pre, long long t, long long s,
                            long long e, bool use_status = true) {
  TcSeg g;
  g.valid = t < e;
  if (!g.valid) return g;
  int lo = 0, hi = p.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int st = use_status ? p.status[b] : 0;   // loaded together with the request's shape
  const TcShape r = tc_shape(p, b);
  const long long local = t - s_pre[b];
  const int unit = static_cast<int>(local / r.tiles);
  const int rg = unit % r.nrg;
  g.b = b;
  g.t0 = r.t0;
  g.n = r.n;
  g.plen = r.plen;
  g.kvh = unit / r.nrg;
  g.node0 = rg * tc_unit_nodes(p.npq);
  g.nodes = min(tc_unit_nodes(p.npq), r.n - g.node0);
  g.mt = (g.nodes + 4 * p.npq - 1) / (4 * p.npq);
  g.ntiles = r.tiles;
  g.tile0 = static_cast<int>(local % r.tiles);
  g.tile1 = static_cast<int>(min(static_cast<long long>(r.tiles), g.tile0 + (e - t)));
  g.t_next = t + (g.tile1 - g.tile0);
  g.whole = g.tile0 == 0 && g.tile1 == r.tiles;
  g.unit_t0 = s_pre[b] + static_cast<long long>(unit) * r.tiles;
  g.my_slot = 2 * blockIdx.x + (t == s ? 0 : 1);
  g.skip = (st & (TV_TREE_FLAGS | TV_ST_BAD_BLOCK)) != 0;
  return g;
}

// Query rows of a unit. An M tile is four 32-lane quarters (a warp may only
// reach the Tensor Memory lanes of its own quarter, warp % 4). The unit's
// nodes are spread in node order over the 4 * mt quarters as evenly as
// possible, G rows per node (node major, query head minor), so the softmax
// warps of all four SM sub-partitions get near-equal row counts.
struct RowSplit {
  int base, extra;   // quarter j holds base + (j < extra ? 1 : 0) nodes
};

__device__ __forceinline__ RowSplit row_split(int nodes, int mt) {
  RowSplit r;
  r.base = nodes / (4 * mt);
  r.extra = nodes % (4 * mt);
  return r;
}

__device__ __forceinline__ int quarter_first(const RowSplit& r, int j) {
  return j * r.base + min(j, r.extra);
}

__device__ __forceinline__ int quarter_count(const RowSplit& r, int j) {
  return r.base + (j < r.extra ? 1 : 0);
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

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Shared memory and Tensor Memory plan of the attention CTA.
//  smem: Q of the two M tiles ([tile][64-column half][128 rows x 128 B]),
//        then kStages K stages and kStages V stages ([half][128 keys x 128 B]
//        each), all in the 128-byte-swizzled layout TMA writes and the
//        tensor core reads.
//  TMEM: S0 = columns [0, 128), S1 = [128, 256) (fp32 scores of one 128-key
//        step; the softmax writes P as bf16 pairs into the first 64 columns
//        of the same buffer), O0 and O1 from column 256 (D columns each).
template <int D>
struct TcCfg {
  static constexpr int kHalves = D / 64;                            // 64-column halves of a row
  static constexpr uint32_t kQHalfBytes = 128 * 128;                // Q: 128 rows x 128 B
  static constexpr uint32_t kQBytes = 2 * kHalves * kQHalfBytes;    // two M tiles
  static constexpr uint32_t kHalfBytes = kTcBN * 128;               // K or V: 128 keys x 128 B
  static constexpr uint32_t kStageBytes = kHalves * kHalfBytes;     // one K or one V stage
  static constexpr int kStages = D == 128 ? 2 : 4;                  // 128 KB of K/V either way
  static constexpr uint32_t kSmem = kQBytes + 2 * kStages * kStageBytes;
  static constexpr uint32_t kOCol = 256;
};

constexpr int kTcMaxStages = 4;

// Arrival counts: K and V stages are filled by the producer (one
// arrive.expect_tx plus the copies' bytes) and released by one tcgen05
// commit of the MMA issuer (k_empty once the step's S MMAs are done, v_empty
// once its PV MMAs are done); q_empty, s_full, o_done and pv_done are
// commits as well; p_full and o_free take one arrival per softmax warp of
// the group.
struct TcBars {
  uint64_t q_full, q_empty;
  uint64_t k_full[kTcMaxStages], k_empty[kTcMaxStages];
  uint64_t v_full[kTcMaxStages], v_empty[kTcMaxStages];
  uint64_t s_full[3], p_full[3], o_done[2], o_free[2];
  uint64_t pv_done, drain;
};

// Score / P barrier of (role t, score buffer b). Each has one producer and
// one consumer that sees every phase in order: a parity wait cannot tell a
// phase that is one ahead from one behind, so no role may skip phases of a
// barrier another role drives. Index 0: buffer 0 (tile 0, or the even steps
// of a one-tile segment); 1: buffer 1 in a one-tile segment (softmax group
// 0); 2: buffer 1 as tile 1's scores (softmax group 1).
__device__ __forceinline__ int sp_bar(int t, int b) { return t == 1 ? 2 : b; }

// 128-key steps of a segment (the last one may be partial)
__device__ __forceinline__ int tc_steps(const TcSeg& g) {
  const long long end = static_cast<long long>(g.plen) + g.n;
  const long long hi = min(end, static_cast<long long>(g.tile1) * kTcBN);
  return static_cast<int>((hi - static_cast<long long>(g.tile0) * kTcBN + kTcBN - 1) / kTcBN);
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams p) {
  using C = TcCfg<D>;
  constexpr int kStages = C::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kQBytes;
  uint8_t* sV = sK + kStages * C::kStageBytes;
  int* s_pre = reinterpret_cast<int*>(sV + kStages * C::kStageBytes);
  int* sw_pre = s_pre + p.batch + 1;
  __shared__ TcBars bars;
  __shared__ int s_tmp[64];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ TcSeg s_last;                // the last segment of this CTA's range (merge task)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    s_last.valid = false;
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.k_full[s], 1);
      mbar_init(&bars.k_empty[s], 1);
      mbar_init(&bars.v_full[s], 1);
      mbar_init(&bars.v_empty[s], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 4);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.o_done[t], 1);
      mbar_init(&bars.o_free[t], 4);
    }
    mbar_init(&bars.pv_done, 1);
    mbar_init(&bars.drain, 1);
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
  tc_plan_prefix(p, s_pre, sw_pre, s_tmp);   // contains __syncthreads; reads only call inputs
  tc_fence_after();
  const long long cs = tc_cta_start(p, s_pre, sw_pre, blockIdx.x);
  const long long ce = tc_cta_start(p, s_pre, sw_pre, blockIdx.x + 1);
  if (cs == ce && threadIdx.x < 256) {
    // A CTA without tiles may still lie between the contributors of a unit
    // split across CTAs; its first partial slot, which the merge reads, then
    // holds no keys (m = -inf, l = 0).
    float* ml = reinterpret_cast<float*>(p.partials + static_cast<size_t>(2 * blockIdx.x) * kSlotBytes(D) +
                                         static_cast<size_t>(256) * 2 * D);
    ml[threadIdx.x] = -INFINITY;
    ml[256 + threadIdx.x] = 0.f;
  }
  const int G = p.group, npq = p.npq;
  const int32_t* table_base = p.block_table;
  if (warp == 2) {
    // While the pre-pass finishes, the otherwise idle warp pulls the prompt
    // K/V pages of this CTA's first steps into L2 (the producer warp goes
    // straight on to its Q and K/V copies). The pre-pass writes only the
    // tree's slots (from P on), rotated q and status; the block table and the
    // prompt pages were complete before it started, so they may be read
    // before the wait. The same table entries then sit in L1 for the producer.
    const TcSeg g = tc_segment(p, s_pre, cs, cs, ce, false);
    if (g.valid) {
      const int32_t* trow = table_base + static_cast<size_t>(g.b) * p.max_blocks;
      const int nh = min(tc_steps(g), kStages);
      for (int j = 0; j < nh; ++j) {
        const long long k0 = static_cast<long long>(g.tile0 + j) * kTcBN;
        // stop at the tree's slots, and within the request's table row (an
        // oversized prompt is flagged only by the pre-pass)
        if (k0 + kTcBN > g.plen || (k0 + kTcBN) / TV_BLOCK_SIZE > p.max_blocks) break;
        if (lane < kTcBN / TV_BLOCK_SIZE) {
          const int blk = __ldg(trow + k0 / TV_BLOCK_SIZE + lane);
          if (blk >= 0 && blk < p.num_blocks) {
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
              tma_prefetch_4d(&p.kmap, h * 64, 0, g.kvh, blk);
              tma_prefetch_4d(&p.vmap, h * 64, 0, g.kvh, blk);
            }
          }
        }
      }
    }
  }
  grid_launch_dependents();               // the merge grid may start its prologue
  grid_dependency_wait();                 // rotated q, tentative KV and status are written
  const uint32_t tbase = s_tmem;
  volatile int* abort = &s_abort;

  if (warp == 0 || warp == 3) {
    // ================================================= TMA producers
    // Warp 0 streams Q per segment and the K pages of every 128-key step
    // (eight 16-row pages, two 64-column boxes each) into K stages; warp 3
    // streams the V pages into V stages. K and V have their own barriers, so
    // the S MMAs of a step start as soon as its keys have landed, and a K
    // stage is refilled as soon as the step's S MMAs read it, while its V is
    // still in use. In each warp lane l issues box l (page l / halves,
    // 64-column half l % halves) after fetching that page's block-table entry.
    const bool kw = warp == 0;
    uint64_t* full = kw ? bars.k_full : bars.v_full;
    uint64_t* empty = kw ? bars.k_empty : bars.v_empty;
    const CUtensorMap* map = kw ? &p.kmap : &p.vmap;
    uint8_t* stage0 = kw ? sK : sV;
    uint32_t hc = 0, qs = 0;           // steps whose copies were issued; segments
    bool ok = true;
    for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); ok && g.valid;
         g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
      if (kw && lane == 0) s_last = g;
      if (g.skip) continue;
      if (kw) {
        ok = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(&bars.q_empty, (qs & 1) ^ 1, abort) : false, 0);
        if (!ok) break;
        ++qs;
        // one box of npq nodes x G heads (<= 32 rows) per quarter and half,
        // lane l issuing box l (quarter l / halves, half l % halves);
        // quarters without nodes are not loaded
        const RowSplit rs = row_split(g.nodes, g.mt);
        const uint32_t qbox = 64u * 2u * G * npq;
        const int nq = min(4 * g.mt, g.nodes);
        if (lane == 0) mbar_arrive_expect_tx(&bars.q_full, qbox * C::kHalves * nq);
        __syncwarp();
        if (lane < nq * C::kHalves) {
          const int j = lane / C::kHalves, h = lane % C::kHalves;
          tma_load_4d(sQ + ((j >> 2) * C::kHalves + h) * C::kQHalfBytes + (j & 3) * 4096, &p.qmap,
                      h * 64, 0, g.kvh, g.t0 + g.node0 + quarter_first(rs, j), &bars.q_full);
        }
      }
      const int32_t* trow = table_base + static_cast<size_t>(g.b) * p.max_blocks;
      const long long end = static_cast<long long>(g.plen) + g.n;
      const int nh = tc_steps(g);
      for (int j = 0; j < nh; ++j) {
        const int s = hc % kStages;
        const uint32_t ph = ((hc / kStages) & 1) ^ 1;
        const long long k0 = static_cast<long long>(g.tile0 + j) * kTcBN;
        const int np = static_cast<int>((min(end, k0 + kTcBN) - k0 + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE);
        const int pg = lane / C::kHalves, h = lane % C::kHalves;
        const bool mine = pg < np;
        const int blk = mine ? __ldg(trow + k0 / TV_BLOCK_SIZE + pg) : 0;
        ok = __shfl_sync(0xffffffffu, lane == 0 ? mbar_wait(&empty[s], ph, abort) : false, 0);
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], np * C::kHalves * 2048u);
        __syncwarp();
        if (mine)
          tma_load_4d(stage0 + s * C::kStageBytes + h * C::kHalfBytes + pg * 2048, map, h * 64, 0, g.kvh,
                      blk, &full[s]);
        ++hc;
      }
    }
    // never leave copies in flight: wait for the last kStages stages this
    // warp filled (and the last Q)
    for (uint32_t k = (hc > kStages ? hc - kStages : 0); lane == 0 && k < hc; ++k) {
      volatile int no_abort = 0;
      mbar_wait(&full[k % kStages], (k / kStages) & 1, &no_abort);
    }
    if (kw && lane == 0 && qs > 0) {
      volatile int no_abort = 0;
      mbar_wait(&bars.q_full, (qs - 1) & 1, &no_abort);
    }
  } else if (warp == 1) {
    // ================================================= MMA issuer
    // One thread issues every MMA, so the tensor core alternates between the
    // two M tiles: per 128-key step j of a two-tile segment
    //   S0(j) = Q0 K(j)^T,  O1 += P1(j-1) V(j-1),  S1(j) = Q1 K(j)^T,  O0 += P0(j) V(j)
    // and while the tensor core runs PV1 and S1, the softmax of tile 0 turns
    // S0 into P0, and vice versa. MMAs of one thread execute in order, so
    // S_t(j+1) may overwrite the columns P_t(j) occupies once PV_t(j) is
    // issued, and the commit that signals S_t(j) also covers PV_t(j-1): the
    // softmax may then rescale O_t in place. A one-tile segment alternates
    // between both score buffers instead,
    //   S(0), S(1), PV(0), S(2), PV(1), S(3), ...
    // so S(j+1) is computed while the softmax works on S(j); there the PV
    // completions are signalled separately for the softmax's rare O rescale.
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, kTcBN, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
      // descriptors built once; each K step only adds a compile-time offset
      // (the start-address field is the low 14 bits, in 16-byte units, and
      // shared-memory addresses stay below 256 KB, so it never carries out)
      const uint64_t dQ0 = smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dQ1 = smem_desc_sw128(smem_u32(sQ) + C::kHalves * C::kQHalfBytes, 16, 1024);
      const uint64_t dK = smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dV = smem_desc_sw128(smem_u32(sV), C::kHalfBytes, 1024);
      uint32_t hc = 0, qs = 0, pc[3] = {0, 0, 0}, of[2] = {0, 0};   // pc: P phases seen per barrier
      bool used[2] = {false, false}, ok = true;
      // S = Q_t K(stage s)^T into score buffer b (its barrier: role t)
      auto issue_s = [&](int t, int s, int b) {
        const uint64_t dq = t == 0 ? dQ0 : dQ1;
        const uint64_t bk = dK + s * (C::kStageBytes / 16);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)                        // 32 bytes per K step
          mma_ss(tbase + b * 128, dq + (k / 4) * (C::kQHalfBytes / 16) + (k % 4) * 2,
                 bk + (k / 4) * (C::kHalfBytes / 16) + (k % 4) * 2, idS, k > 0 ? 1u : 0u);
        mma_commit(&bars.s_full[sp_bar(t, b)]);
      };
      // waits for P_t in buffer b and, before the tile's first PV of a
      // segment, for the epilogue to have read O_t out; then O_t += P V(stage
      // s) for step j (16-key chunks past the request's last key are not
      // issued: their V rows were never loaded)
      auto issue_pv = [&](int t, int s, int b, int j, const TcSeg& g) -> bool {
        const int bi = sp_bar(t, b);
        if (!mbar_wait(&bars.p_full[bi], pc[bi] & 1, abort)) return false;
        ++pc[bi];
        if (j == 0 && used[t]) {
          if (!mbar_wait(&bars.o_free[t], of[t] & 1, abort)) return false;
          ++of[t];
        }
        tc_fence_after();
        const long long end = static_cast<long long>(g.plen) + g.n;
        const long long k0 = static_cast<long long>(g.tile0 + j) * kTcBN;
        const int kch = static_cast<int>((min(end, k0 + kTcBN) - k0 + 15) / 16);
        const uint32_t tO = tbase + C::kOCol + t * D;
        const uint64_t bv = dV + s * (C::kStageBytes / 16);
        if (kch == kTcBN / 16) {
#pragma unroll
          for (int k = 0; k < kTcBN / 16; ++k)
            mma_ts(tO, tbase + b * 128 + k * 8, bv + k * (2048 / 16), idO, (j > 0 || k > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int k = 0; k < kTcBN / 16; ++k)
            if (k < kch)
              mma_ts(tO, tbase + b * 128 + k * 8, bv + k * (2048 / 16), idO, (j > 0 || k > 0) ? 1u : 0u);
        }
        return true;
      };
      for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); ok && g.valid;
           g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
        if (g.skip) continue;
        if (!(ok = mbar_wait(&bars.q_full, qs & 1, abort))) break;
        ++qs;
        tc_fence_after();
        const int nh = tc_steps(g);
        if (g.mt == 2) {
          for (int j = 0; j < nh && ok; ++j) {
            const uint32_t h = hc + j;
            const int s = h % kStages;
            const uint32_t ph = (h / kStages) & 1;
            if (!(ok = mbar_wait(&bars.k_full[s], ph, abort))) break;
            tc_fence_after();
            issue_s(0, s, 0);
            if (j > 0) {
              const int sp = (h - 1) % kStages;
              if (!(ok = issue_pv(1, sp, 1, j - 1, g))) break;
              mma_commit(&bars.v_empty[sp]);                  // both tiles' PV of step j-1 issued
            }
            issue_s(1, s, 1);
            mma_commit(&bars.k_empty[s]);
            if (j == nh - 1) mma_commit(&bars.q_empty);       // the segment's last S MMAs
            if (!(ok = mbar_wait(&bars.v_full[s], ph, abort))) break;
            if (!(ok = issue_pv(0, s, 0, j, g))) break;
            if (j == nh - 1) mma_commit(&bars.o_done[0]);
          }
          if (ok) {
            const int sl = (hc + nh - 1) % kStages;
            if ((ok = issue_pv(1, sl, 1, nh - 1, g))) {
              mma_commit(&bars.v_empty[sl]);
              mma_commit(&bars.o_done[1]);
            }
          }
          used[1] = true;
        } else {
          auto s_step = [&](int j) -> bool {
            const uint32_t h = hc + j;
            const int s = h % kStages;
            if (!mbar_wait(&bars.k_full[s], (h / kStages) & 1, abort)) return false;
            tc_fence_after();
            issue_s(0, s, j & 1);
            mma_commit(&bars.k_empty[s]);
            if (j == nh - 1) mma_commit(&bars.q_empty);
            return true;
          };
          ok = s_step(0);
          if (ok && nh > 1) ok = s_step(1);
          for (int j = 0; j < nh && ok; ++j) {
            const uint32_t h = hc + j;
            const int s = h % kStages;
            if (!(ok = mbar_wait(&bars.v_full[s], (h / kStages) & 1, abort))) break;
            if (!(ok = issue_pv(0, s, j & 1, j, g))) break;
            mma_commit(&bars.v_empty[s]);
            mma_commit(&bars.pv_done);
            if (j == nh - 1) mma_commit(&bars.o_done[0]);
            if (j + 2 < nh) ok = s_step(j + 2);
          }
        }
        hc += nh;
        used[0] = true;
      }
      // drain: every MMA this thread issued completes before Tensor Memory is freed
      mma_commit(&bars.drain);
      volatile int no_abort = 0;
      mbar_wait(&bars.drain, 0, &no_abort);
    }
  } else if (warp >= 4) {
    // ================================================= softmax groups
    // warps 4-7 serve M tile 0, warps 8-11 M tile 1; warp w owns Tensor
    // Memory lanes 32 * (w % 4) .. +31, one query row per thread. A step's
    // 128 scores are taken in two halves of 64; P of each half goes as bf16
    // pairs into the buffer's columns already read. In a one-tile segment
    // group 0 takes every step, from both score buffers in turn.
    const int t = (warp - 4) >> 2;
    const int qd = warp & 3;
    const int j4 = 4 * t + qd;                         // quarter of the unit's rows
    const uint32_t lane_addr = static_cast<uint32_t>(qd * 32) << 16;
    const uint32_t tO = tbase + C::kOCol + t * D + lane_addr;
    const uint64_t scale2 = f32x2_pack(p.scale_log2, p.scale_log2);
    uint32_t sc[2] = {0, 0}, oc = 0, pvc = 0;        // sc: score phases seen per buffer
    bool ok = true;
    for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); ok && g.valid;
         g = tc_segment(p, s_pre, g.t_next, cs, ce)) {
      if (g.skip) continue;
      const int nh = tc_steps(g);
      const bool one = g.mt == 1;
      if (one && t == 1) continue;           // group 0 takes both buffers here
      const RowSplit rs = row_split(g.nodes, g.mt);
      const int cnt = quarter_count(rs, j4);
      const bool warp_live = cnt > 0;                  // uniform over the warp
      const bool row_valid = lane < G * cnt;
      const int nd = g.node0 + quarter_first(rs, j4) + (row_valid ? lane / G : 0);   // node of this row
      float m_ref = -INFINITY;
      uint64_t l2 = f32x2_pack(0.f, 0.f);              // running row sum, two partial sums
      const uint32_t* mrow = p.mask + static_cast<size_t>(g.t0 + nd) * p.words;
      for (int j = 0; j < nh && ok; ++j) {
        const int b = one ? (j & 1) : t;
        if (!(ok = mbar_wait(&bars.s_full[sp_bar(t, b)], sc[b] & 1, abort))) break;
        ++sc[b];
        tc_fence_after();
        if (warp_live) {
          const uint32_t tS = tbase + b * 128 + lane_addr;
          const int k0 = (g.tile0 + j) * kTcBN;
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            const int kh = k0 + hf * 64;
            uint32_t a[64];
            tmem_ld32(tS + hf * 64, a);
            tmem_ld32(tS + hf * 64 + 32, a + 32);
            tmem_ld_wait();
            if (kh + 64 > g.plen) {                    // the half reaches past the prompt: mask it
#pragma unroll
              for (int c = 0; c < 2; ++c) {
                const uint32_t vis = row_valid ? visible_bits(mrow, p.words, g.plen, g.n, kh + c * 32) : 0u;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (!((vis >> e) & 1u)) a[c * 32 + e] = 0xFF800000u;   // -inf
              }
            }
            float x0 = -INFINITY, x1 = -INFINITY, x2 = -INFINITY, x3 = -INFINITY;
#pragma unroll
            for (int e = 0; e < 64; e += 8) {
              x0 = fmax3(x0, __uint_as_float(a[e]), __uint_as_float(a[e + 1]));
              x1 = fmax3(x1, __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3]));
              x2 = fmax3(x2, __uint_as_float(a[e + 4]), __uint_as_float(a[e + 5]));
              x3 = fmax3(x3, __uint_as_float(a[e + 6]), __uint_as_float(a[e + 7]));
            }
            const float mxs = fmax3(x0, x1, fmaxf(x2, x3)) * p.scale_log2;
            // Lazy rescale: the reference max moves only when a score exceeds
            // it by 2^8, so p stays <= 2^8 and O, l share one reference. A
            // move rescales O (once its previous step's PV is complete) and,
            // in the second half, the P already written for the first half.
            // The Tensor Memory accesses are warp-wide, so a warp rescales
            // when any of its rows moved (alpha = 1 for the others).
            float alpha = 1.f;
            if (mxs > m_ref + 8.f) {
              if (m_ref != -INFINITY) alpha = fast_exp2(m_ref - mxs);
              m_ref = mxs;
            }
            if (__any_sync(0xffffffffu, alpha != 1.f)) {
              l2 = f32x2_mul(l2, f32x2_pack(alpha, alpha));
              if (j > 0) {
                if (one) {                             // PV(j - 1) may still be running
                  volatile int* ab = abort;
                  ok = mbar_wait(&bars.pv_done, (pvc + j - 1) & 1, ab);
                  tc_fence_after();
                }
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
              if (hf == 1) {
                uint32_t o[32];
                tmem_st_wait();                        // the first half's P is in place
                tmem_ld32(tS, o);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = pack_bf16x2(bf16_lo(o[e]) * alpha, bf16_hi(o[e]) * alpha);
                tmem_st32(tS, o);
              }
            }
            const float base = m_ref == -INFINITY ? 0.f : m_ref;
            const uint64_t nb2 = f32x2_pack(-base, -base);
            // p = 2^(s * scale * log2(e) - base), two at a time, as bf16 pairs
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                float y0, y1;
                f32x2_unpack(f32x2_fma(f32x2_pack(__uint_as_float(a[c * 32 + 2 * e]),
                                                  __uint_as_float(a[c * 32 + 2 * e + 1])),
                                       scale2, nb2), y0, y1);
                const float p0 = fast_exp2(y0), p1 = fast_exp2(y1);
                const uint64_t pp = f32x2_pack(p0, p1);
                l2 = f32x2_add(l2, pp);
                pk[e] = pack_bf16x2(p0, p1);
              }
              tmem_st16(tS + hf * 32 + c * 16, pk);
            }
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[sp_bar(t, b)]);
      }
      if (one) pvc += nh;
      if (ok && (ok = mbar_wait(&bars.o_done[t], oc & 1, abort))) {
        ++oc;
        tc_fence_after();
        if (warp_live) {
          float la, lb;
          f32x2_unpack(l2, la, lb);
          const float l_sum = la + lb;
          const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
          if (g.whole) {
            const int h = g.kvh * G + lane % G;
            __nv_bfloat16* dst = p.out + (static_cast<size_t>(g.t0 + nd) * p.hq + h) * D;
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
            // partial of a split unit: O / l as fp16 (a convex combination of
            // value rows, so well inside fp16 range) in [D/8 column blocks]
            // [256 rows] 16-byte vectors, so a quarter's 32 rows write (and the
            // merge reads) 512 contiguous bytes; then the row's m and l
            uint8_t* slot = p.partials + static_cast<size_t>(g.my_slot) * kSlotBytes(D);
            uint4* o16 = reinterpret_cast<uint4*>(slot);
            const int r = j4 * 32 + lane;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_ld_wait();
              if (row_valid) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  o16[(c * 4 + q) * 256 + r] = make_uint4(
                      pack_half2(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv),
                      pack_half2(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv),
                      pack_half2(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv),
                      pack_half2(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv));
              }
            }
            if (row_valid) {
              float* ml = reinterpret_cast<float*>(slot + static_cast<size_t>(256) * 2 * D);
              ml[r] = m_ref;
              ml[256 + r] = l_sum;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.o_free[t]);
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
    const TcSeg last = s_last;            // recorded by the producer as it walked the range
    if (s_abort) {
      for (TcSeg g = tc_segment(p, s_pre, cs, cs, ce); g.valid; g = tc_segment(p, s_pre, g.t_next, cs, ce))
        atomicOr(p.status_rw + g.b, TV_ST_TIMEOUT);               // flag what this CTA touched
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
      rec[8] = tc_cta_of(p, s_pre, sw_pre, last.unit_t0 + last.ntiles - 1);   // last contributor
      rec[9] = last.my_slot;                                            // its slot
      rec[10] = last.nodes;
    }
    rec[0] = valid;
  }
}

// ------------------------------------------------------------ merge of split units
//
// A unit whose key tiles were cut between CTAs c_first..c_last left one
// partial (normalised o_c = O_c / l_c, reference max m_c, sum l_c, per row)
// per contributor. The merge is the usual log-sum-exp combination:
//   out = sum_c w_c o_c / sum_c w_c,  w_c = 2^(m_c - M) l_c,  M = max_c m_c.
// A work item is one quarter of a split unit's rows (32 rows, 8 threads per
// row); each thread loads kMergeChunk contributors at once. The grid is one
// resident wave: every CTA reads all task flags at once, lists the valid
// records in shared memory, and takes items blockIdx.x, + gridDim.x, ...
// of that list, so the work spreads evenly whatever records are empty.

struct MergeParams {
  const int32_t* tasks;
  const uint8_t* partials;
  __nv_bfloat16* out;
  int hq, group;
  int ntask;            // task records: one per attention CTA
};

constexpr int kMergeThreads = 256;
constexpr int kMergeSplit = 8;      // CTAs per unit: one per row quarter
constexpr int kMergeChunk = 2;      // contributors whose loads are in flight together
constexpr int kMergeMinBlocks = 4;  // resident merge CTAs per SM the register budget allows
constexpr int kMergeMaxTasks = 1024;

__device__ __forceinline__ float2 half2_to_float2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// Row quarter j of the split unit described by task record rec.
template <int D>
__device__ __forceinline__ void merge_one(const MergeParams& p, const int32_t* rec, int j) {
  const int kvh = rec[2], node0 = rec[3], mt = rec[4], t0 = rec[5];
  const int c_first = rec[7], c_last = rec[8], first_slot = rec[9], nodes = rec[10];
  if ((j >> 2) >= mt) return;
  const int G = p.group;
  const RowSplit rs = row_split(nodes, mt);
  const int cnt = quarter_count(rs, j);
  constexpr int kParts = kMergeThreads / 32;          // 8 threads per row
  constexpr int kVecs = D / 8 / kParts;               // 16-byte vectors (8 fp16) per thread
  const int lane = threadIdx.x & 31, part = threadIdx.x >> 5;
  if (lane >= G * cnt) return;
  const int nd = node0 + quarter_first(rs, j) + lane / G;
  const int r = j * 32 + lane;
  const int nc = c_last - c_first + 1;
  float m_run = -INFINITY, l_run = 0.f;
  float acc[kVecs][8];
#pragma unroll
  for (int v = 0; v < kVecs; ++v)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[v][e] = 0.f;
  for (int k0 = 0; k0 < nc; k0 += kMergeChunk) {
    float mc[kMergeChunk], lc[kMergeChunk];
    uint4 x[kMergeChunk][kVecs];
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      const int k = k0 + u;
      mc[u] = -INFINITY;
      lc[u] = 0.f;
      if (k < nc) {
        const int sl = k == 0 ? first_slot : 2 * (c_first + k);
        const uint8_t* base = p.partials + static_cast<size_t>(sl) * kSlotBytes(D);
        const float* ml = reinterpret_cast<const float*>(base + static_cast<size_t>(256) * 2 * D);
        mc[u] = __ldcg(ml + r);
        lc[u] = __ldcg(ml + 256 + r);
        const uint4* o16 = reinterpret_cast<const uint4*>(base);
#pragma unroll
        for (int v = 0; v < kVecs; ++v) x[u][v] = __ldcg(o16 + (part * kVecs + v) * 256 + r);
      }
    }
    float m_new = m_run;
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) m_new = fmaxf(m_new, mc[u]);
    if (m_new == -INFINITY) continue;
    const float sc = m_run == -INFINITY ? 0.f : fast_exp2(m_run - m_new);
    l_run *= sc;
#pragma unroll
    for (int v = 0; v < kVecs; ++v)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[v][e] *= sc;
#pragma unroll
    for (int u = 0; u < kMergeChunk; ++u) {
      if (mc[u] == -INFINITY) continue;
      const float w = fast_exp2(mc[u] - m_new) * lc[u];
      l_run += w;
#pragma unroll
      for (int v = 0; v < kVecs; ++v) {
        const uint32_t xs[4] = {x[u][v].x, x[u][v].y, x[u][v].z, x[u][v].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = half2_to_float2(xs[e]);
          acc[v][2 * e] = fmaf(w, f.x, acc[v][2 * e]);
          acc[v][2 * e + 1] = fmaf(w, f.y, acc[v][2 * e + 1]);
        }
      }
    }
    m_run = m_new;
  }
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
  const int h = kvh * G + lane % G;
  uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<size_t>(t0 + nd) * p.hq + h) * D) + part * kVecs;
#pragma unroll
  for (int v = 0; v < kVecs; ++v)
    dst[v] = make_uint4(pack_bf16x2(acc[v][0] * inv, acc[v][1] * inv), pack_bf16x2(acc[v][2] * inv, acc[v][3] * inv),
                        pack_bf16x2(acc[v][4] * inv, acc[v][5] * inv), pack_bf16x2(acc[v][6] * inv, acc[v][7] * inv));
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads, kMergeMinBlocks)
    attn_merge_kernel(const __grid_constant__ MergeParams p) {
  __shared__ int s_list[kMergeMaxTasks];
  __shared__ int s_wsum[kMergeThreads / 32];
  grid_dependency_wait();            // the attention grid's partials and tasks are visible
  grid_launch_dependents();
  // compact the valid task records (in record order), one flag per thread
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int nvalid = 0;
  for (int base = 0; base < p.ntask; base += kMergeThreads) {
    const int c = base + threadIdx.x;
    const bool v = c < p.ntask && __ldcg(p.tasks + static_cast<size_t>(c) * kTaskInts) != 0;
    const unsigned bal = __ballot_sync(0xffffffffu, v);
    if (lane == 0) s_wsum[warp] = __popc(bal);
    __syncthreads();
    int before = nvalid;
    for (int w = 0; w < warp; ++w) before += s_wsum[w];
    if (v) s_list[before + __popc(bal & ((1u << lane) - 1u))] = c;
    for (int w = 0; w < kMergeThreads / 32; ++w) nvalid += s_wsum[w];
    __syncthreads();
  }
  for (int k = blockIdx.x; k < nvalid * kMergeSplit; k += gridDim.x)
    merge_one<D>(p, p.tasks + static_cast<size_t>(s_list[k / kMergeSplit]) * kTaskInts, k % kMergeSplit);
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
  int npq;
};

static TcLayout tc_layout(int batch, int hq, int hkv, int max_nodes, int head_dim, int grid) {
  TcLayout L;
  const int group = hq / hkv;
  L.npq = 32 / group;
  L.task_bytes = (static_cast<size_t>(grid) * kTaskInts * sizeof(int32_t) + 255) / 256 * 256;
  L.partial_bytes = static_cast<size_t>(2) * grid * kSlotBytes(head_dim);
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
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(group), 1, static_cast<cuuint32_t>(L.npq)};
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
  tp.partials = reinterpret_cast<uint8_t*>(ws + L.task_bytes);
  tp.status_rw = status;
  tp.batch = batch;
  tp.max_nodes = max_nodes;
  tp.t_cap = t_cap;
  tp.hq = hq;
  tp.hkv = hkv;
  tp.group = group;
  tp.npq = L.npq;
  tp.words = (max_nodes + 31) / 32;
  tp.max_blocks = max_blocks;
  tp.num_blocks = num_blocks;
  tp.grid = grid;
  const double scale = geom->softmax_scale > 0.f ? geom->softmax_scale : 1.0 / sqrt(double(D));
  tp.scale_log2 = static_cast<float>(scale * 1.4426950408889634);

  MergeParams mp;
  mp.tasks = tp.tasks;
  mp.partials = tp.partials;
  mp.out = tp.out;
  mp.hq = hq;
  mp.group = group;
  mp.ntask = grid;

  const dim3 rgrid(batch, (max_nodes + kRopeNodes - 1) / kRopeNodes);
  static size_t smem_set128[kMaxDevices] = {0}, smem_set64[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0) return TV_ERR_CUDA;
  const size_t smem_fixed = (D == 128 ? TcCfg<128>::kSmem : TcCfg<64>::kSmem) + 1024;
  const size_t smem = smem_fixed + static_cast<size_t>(batch + 1) * 2 * sizeof(int);
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
  // the merge grid: one resident wave (never more CTAs than there can be
  // work items)
  static int merge_per_sm[2][kMaxDevices] = {{0}};
  int& mps = merge_per_sm[D == 128 ? 0 : 1][dev];
  if (mps == 0) {
    int n = 0;
    const cudaError_t oe = D == 128
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_merge_kernel<128>, kMergeThreads, 0)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_merge_kernel<64>, kMergeThreads, 0);
    mps = (oe == cudaSuccess && n > 0) ? n : 1;
  }
  const int sms = device_sm_count(dev);
  if (grid > kMergeMaxTasks) return TV_ERR_BAD_SIZE;            // one task record per CTA
  const int mgrid = std::max(1, std::min(grid * kMergeSplit, std::max(sms, 1) * mps));
  cudaLaunchConfig_t mcfg = acfg;
  mcfg.gridDim = dim3(mgrid);
  mcfg.blockDim = dim3(kMergeThreads);
  mcfg.dynamicSmemBytes = 0;
  cudaError_t err;
  if (D == 128) {
    if (!ensure_smem(attn_tc_kernel<128>, smem, smem_set128, dev)) return TV_ERR_CUDA;
    err = rp.rope_style == 0 ? launch_pdl(rope_append_kernel<128, true>, rgrid, dim3(kRopeThreads), 0, stream, rp)
                             : launch_pdl(rope_append_kernel<128, false>, rgrid, dim3(kRopeThreads), 0, stream, rp);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&acfg, attn_tc_kernel<128>, tp);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&mcfg, attn_merge_kernel<128>, mp);
  } else {
    if (!ensure_smem(attn_tc_kernel<64>, smem, smem_set64, dev)) return TV_ERR_CUDA;
    err = rp.rope_style == 0 ? launch_pdl(rope_append_kernel<64, true>, rgrid, dim3(kRopeThreads), 0, stream, rp)
                             : launch_pdl(rope_append_kernel<64, false>, rgrid, dim3(kRopeThreads), 0, stream, rp);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&acfg, attn_tc_kernel<64>, tp);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&mcfg, attn_merge_kernel<64>, mp);
  }
  if (err != cudaSuccess) return TV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
