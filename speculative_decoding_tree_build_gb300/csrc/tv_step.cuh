// Device bodies of the step's last two stages, shared by their own kernels
// (tv_greedy_accept, tv_kv_commit) and the fused tv_accept_commit kernel.
// Each runs in one CTA per request.
#pragma once

#include "tv_common.cuh"

namespace tv {

// Shared-memory state of one request's greedy walk.
struct WalkSmem {
  int tgt[TV_MAX_NODES];
  int tok[TV_MAX_NODES];
  int first[TV_MAX_NODES];
  int next[TV_MAX_NODES];
  int path[TV_MAX_NODES];
  int len, bonus, bad;
};

// Greedy acceptance walk ("02 · Token Tree 与 Tree Attention" §4: from the
// root take the child whose token equals the target's choice, stop at the
// first miss whose target token is the bonus; "Beam Search、约束解码与
// Tree/Self Speculation" verify_tree; "Accelerating Speculative Decoding with
// Block Diffusion Draft Trees" §7.2). The request's arrays are staged with
// coalesced loads, then one thread follows first-child / next-sibling links in
// shared memory. Leaves w.path[0..len], w.len, w.bonus and w.bad (a status
// flag or 0) for every thread.
__device__ __forceinline__ void greedy_walk(const int32_t* target_ids, const int32_t* draft_tokens,
                                            const int32_t* next_token, const int32_t* next_sibling,
                                            int t0, int n, int max_depth, WalkSmem& w) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    w.tgt[i] = target_ids[t0 + i];
    w.tok[i] = draft_tokens[t0 + i];
    w.first[i] = next_token[t0 + i];
    w.next[i] = next_sibling[t0 + i];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int len = 0, cur = 0, bad = 0;
    w.path[0] = 0;
    while (true) {
      const int want = w.tgt[cur];
      int c = w.first[cur];
      int guard = 0;
      while (c != -1 && w.tok[c] != want) {
        c = w.next[c];
        // links come from tv_tree_build; a corrupted list must not loop or
        // index outside the request
        if (c >= n || c < -1 || ++guard > n) { bad = 1; break; }
      }
      if (bad || c == -1) {
        w.bonus = want;
        break;
      }
      if (c <= cur || c >= n || len + 1 >= n) { bad = 1; break; }
      w.path[++len] = c;
      cur = c;
    }
    w.len = len;
    w.bad = bad ? TV_ST_BAD_SIZE : (len > max_depth ? TV_ST_PATH_OVERFLOW : 0);
  }
  __syncthreads();
}

// Commit / rollback of one request's tentative KV ("Beam Search、约束解码与
// Tree/Self Speculation", section "Tree/Self Speculation": [10,11] ->
// [10,11,4,7], every other tentative node rolled back; "02 · Token Tree 与
// Tree Attention" §4: the chosen path's KV becomes the next prompt, pages are
// reclaimed; "投机解码的树状注意力验证…", "实现中的 KV Cache 与批处理约束").
//
// Slot P+path[k] moves to slot P+k for k = 1..a. path[k] >= k, so a
// destination slot can be the source of an EARLIER k only: rows move in
// ascending chunks staged in shared memory (all of a chunk's reads before any
// of its writes); later chunks only read slots no earlier chunk wrote. Then
// the held blocks past the new end are released. `path` is in shared memory.
// Returns a status flag (0 when committed); outputs are untouched otherwise.
__device__ __forceinline__ int commit_rows(const int* path, int a, int plen, int held,
                                           int32_t* table, int max_blocks, uint4* k_cache,
                                           uint4* v_cache, int num_blocks, int hkv, int head_vecs,
                                           uint4* stage, int stage_bytes, int* blk,
                                           int* flag, int32_t* new_len, int32_t* released_row,
                                           int32_t* released_count, int32_t* n_blocks) {
  if (threadIdx.x == 0) *flag = 0;
  __syncthreads();
  int bad = 0;
  for (int k = threadIdx.x; k <= a; k += blockDim.x) {
    const int pk = path[k];
    if (k == 0) {
      if (pk != 0) bad |= TV_ST_BAD_SIZE;
      continue;
    }
    if (pk <= path[k - 1]) { bad |= TV_ST_BAD_SIZE; continue; }
    // source and destination blocks of row k
    const long long src = static_cast<long long>(plen) + pk, dst = plen + k;
    const long long lbs = src / TV_BLOCK_SIZE, lbd = dst / TV_BLOCK_SIZE;
    int bs = -1, bd = -1;
    if (lbs < held && lbs < max_blocks) bs = table[lbs];
    if (lbd < held && lbd < max_blocks) bd = table[lbd];
    if (bs < 0 || bs >= num_blocks || bd < 0 || bd >= num_blocks) bad |= TV_ST_BAD_BLOCK;
    blk[2 * k] = bs;
    blk[2 * k + 1] = bd;
  }
  if (bad) atomicOr(flag, bad);
  __syncthreads();
  if (*flag) return *flag;

  // rows to move (k with path[k] == k is already in place)
  const int row_vecs = 2 * hkv * head_vecs;   // K and V, all heads
  const int chunk_rows = stage_bytes / (row_vecs * 16);
  if (chunk_rows < 1) return TV_ST_BAD_SIZE;   // a row larger than the stage (the host rejects it)
  for (int k0 = 1; k0 <= a; k0 += chunk_rows) {
    const int k1 = min(a + 1, k0 + chunk_rows);
    const int total = (k1 - k0) * row_vecs;
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
      const int r = e / row_vecs, rem = e % row_vecs;
      const int k = k0 + r;
      if (path[k] == k) continue;
      const int kv = rem / (hkv * head_vecs), h = (rem / head_vecs) % hkv, v = rem % head_vecs;
      const int slot = (plen + path[k]) % TV_BLOCK_SIZE;
      const size_t idx = ((static_cast<size_t>(blk[2 * k]) * hkv + h) * TV_BLOCK_SIZE + slot) *
                             head_vecs + v;
      stage[e] = kv ? v_cache[idx] : k_cache[idx];
    }
    __syncthreads();
    for (int e = threadIdx.x; e < total; e += blockDim.x) {
      const int r = e / row_vecs, rem = e % row_vecs;
      const int k = k0 + r;
      if (path[k] == k) continue;
      const int kv = rem / (hkv * head_vecs), h = (rem / head_vecs) % hkv, v = rem % head_vecs;
      const int slot = (plen + k) % TV_BLOCK_SIZE;
      const size_t idx = ((static_cast<size_t>(blk[2 * k + 1]) * hkv + h) * TV_BLOCK_SIZE + slot) *
                             head_vecs + v;
      if (kv) v_cache[idx] = stage[e]; else k_cache[idx] = stage[e];
    }
    __syncthreads();
  }

  // release the blocks past the new end
  const long long nl = static_cast<long long>(plen) + 1 + a;
  const int keep = static_cast<int>((nl + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE);
  const int count = held > keep ? held - keep : 0;
  for (int j = threadIdx.x; j < max_blocks; j += blockDim.x) {
    if (j < count && keep + j < max_blocks) {
      released_row[j] = table[keep + j];
      table[keep + j] = -1;
    } else {
      released_row[j] = -1;
    }
  }
  if (threadIdx.x == 0) {
    *new_len = static_cast<int>(nl);
    *released_count = count;
    *n_blocks = held < keep ? held : keep;
  }
  return 0;
}

}  // namespace tv
