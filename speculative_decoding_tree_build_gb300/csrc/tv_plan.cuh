// Device-side split-KV work plan shared by the attention kernels.
//
// Work unit = (request b, KV head, row group). A row group is up to kRows
// query rows; row r of a request is (node r / G, query head kvh*G + r % G),
// G = Hq / Hkv. A unit's key sequence is ceil(P_b / BN) prompt tiles followed
// by ceil(N_b / BN) tree tiles. All units' tiles are laid end to end and the
// grid's CTAs take equal contiguous ranges of that sequence, so every CTA gets
// the same amount of KV traffic whatever the prompt-length mix. A unit cut
// between CTAs is merged by its last-arriving contributor (no CTA ever waits
// for another). The plan is computed by every CTA from cu_nodes/prompt_len,
// so no host round trip and no extra launch is needed.
#pragma once

#include "tv_common.cuh"

namespace tv {

struct PlanParams {
  int batch, max_nodes, group, hkv, rows_per_unit, keys_per_tile, nrg_max, grid;
};

struct ReqShape {
  int t0, n, plen, nrg, tiles;
};

__device__ __forceinline__ ReqShape req_shape(const int32_t* cu_nodes, const int32_t* prompt_len,
                                              const PlanParams& pp, int b) {
  ReqShape r;
  r.t0 = cu_nodes[b];
  r.n = cu_nodes[b + 1] - r.t0;
  r.plen = prompt_len[b];
  if (r.n < 1 || r.n > pp.max_nodes || r.plen < 0) {
    r.nrg = 0;
    r.tiles = 0;
    return r;
  }
  const int rows = pp.group * r.n;
  r.nrg = (rows + pp.rows_per_unit - 1) / pp.rows_per_unit;
  r.tiles = (r.plen + pp.keys_per_tile - 1) / pp.keys_per_tile +
            (r.n + pp.keys_per_tile - 1) / pp.keys_per_tile;
  return r;
}

// Exclusive prefix of per-request tile counts into s_pre[0..batch]
// (s_pre[batch] = total). Called by all threads of the block.
__device__ inline void plan_prefix(const int32_t* cu_nodes, const int32_t* prompt_len,
                                   const PlanParams& pp, long long* s_pre, long long* s_tmp) {
  const int nt = blockDim.x;
  const int tid = threadIdx.x;
  const int per = (pp.batch + nt - 1) / nt;
  const int lo = min(pp.batch, tid * per), hi = min(pp.batch, lo + per);
  long long sum = 0;
  for (int b = lo; b < hi; ++b) {
    const ReqShape r = req_shape(cu_nodes, prompt_len, pp, b);
    sum += static_cast<long long>(pp.hkv) * r.nrg * r.tiles;
  }
  s_tmp[tid] = sum;
  __syncthreads();
  if (tid == 0) {
    long long run = 0;
    for (int i = 0; i < nt; ++i) {
      const long long v = s_tmp[i];
      s_tmp[i] = run;
      run += v;
    }
    s_pre[pp.batch] = run;
  }
  __syncthreads();
  long long run = s_tmp[tid];
  for (int b = lo; b < hi; ++b) {
    s_pre[b] = run;
    const ReqShape r = req_shape(cu_nodes, prompt_len, pp, b);
    run += static_cast<long long>(pp.hkv) * r.nrg * r.tiles;
  }
  __syncthreads();
}

// CTA c owns tiles [cta_start(c), cta_start(c+1)).
__device__ __forceinline__ long long cta_start(long long total, int grid, int c) {
  const long long q = total / grid, rem = total % grid;
  return c * q + min(static_cast<long long>(c), rem);
}

__device__ __forceinline__ int cta_of_tile(long long total, int grid, long long t) {
  const long long q = total / grid, rem = total % grid;
  const long long big = rem * (q + 1);
  if (t < big) return static_cast<int>(t / (q + 1));
  return static_cast<int>(rem + (t - big) / q);
}

// request owning global tile t: largest b with s_pre[b] <= t and a non-empty range
__device__ __forceinline__ int request_of_tile(const long long* s_pre, int batch, long long t) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pre[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Workspace layout: [counters: int32 per unit][partial slots]
// partial slot s: O fp32 [rows][D], then m fp32 [rows], then l fp32 [rows].
__host__ __device__ inline size_t ws_counter_bytes(int batch, int hkv, int nrg_max) {
  const size_t c = static_cast<size_t>(batch) * hkv * nrg_max * sizeof(int32_t);
  return (c + 255) / 256 * 256;
}

__host__ __device__ inline size_t ws_slot_floats(int rows, int head_dim) {
  return static_cast<size_t>(rows) * (head_dim + 2);
}

}  // namespace tv
