// Packed tree attention, warp-level tensor-core (mma.sync) kernel.
//
// Computes, for every tree node i and query head h of a request, softmax of
// q_i k^T * scale over the committed prompt keys plus the keys of i's ancestor
// chain (itself included), times V - "Beam Search、约束解码与 Tree/Self
// Speculation", section "Packed tree attention" and its packed-vs-branch
// experiment; "02 · Token Tree 与 Tree Attention" §3 (visible = prompt ∪
// ancestors; RoPE at depth position). The fresh Q/K are rotated here at their
// depth positions and the rotated K plus raw V are written to the request's
// tentative cache slots P + i ("投机解码的树状注意力验证…", section "实现中的 KV Cache
// 与批处理约束": a contiguous tree region in node order).
//
// Work split (see tv_plan.cuh): 128 query rows (8 warps x m16) per unit, 64
// keys per tile, prompt tiles streamed through shared memory with cp.async
// double buffering, tree tiles built in shared memory from the rotated fresh
// K/V; the ancestor mask is applied as a bit test. Online softmax in fp32
// (log2 domain), bf16 operands, fp32 accumulation.
#include "tv_plan.cuh"

namespace tv {

struct AttnParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int32_t* cu_nodes;
  const int32_t* positions;
  const uint32_t* mask;
  const int32_t* prompt_len;
  const int32_t* block_table;
  const int32_t* n_blocks;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  __nv_bfloat16* out;
  int32_t* counters;
  float* partials;
  int32_t* status;
  int hq, hkv, group, words, max_blocks, num_blocks, rope_style;
  float scale_log2;
  float inv_freq[64];
  PlanParams plan;
};

constexpr int kMmaRows = 128;
constexpr int kMmaBN = 64;
constexpr int kMmaThreads = 256;

template <int D>
struct MmaCfg {
  static constexpr int LD = D + 8;                       // padded row (elements)
  static constexpr size_t kQBytes = size_t(kMmaRows) * LD * 2;
  static constexpr size_t kTileBytes = size_t(kMmaBN) * LD * 2;
  static constexpr size_t kFixed = kQBytes + 4 * kTileBytes;
};

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                        const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                          const void* p) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}

__device__ __forceinline__ void mma16816(float* c, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const int sz = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// RoPE of one element pair (fp32 rotation of bf16 inputs).
__device__ __forceinline__ void rope_pair(float a, float b, int pos, float inv, float& o0,
                                          float& o1) {
  float sn, cs;
  sincosf(static_cast<float>(pos) * inv, &sn, &cs);
  o0 = a * cs - b * sn;
  o1 = b * cs + a * sn;
}

// Validate every block covering slots [0, P + n) of request b. All threads call.
__device__ bool request_blocks_ok(const AttnParams& p, int b, int plen, int n) {
  const long long slots = static_cast<long long>(plen) + n;
  const int nlb = static_cast<int>((slots + TV_BLOCK_SIZE - 1) / TV_BLOCK_SIZE);
  const int held = p.n_blocks[b];
  int bad = (nlb > held || nlb > p.max_blocks) ? 1 : 0;
  const int32_t* row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  for (int lb = threadIdx.x; !bad && lb < nlb && lb < p.max_blocks; lb += blockDim.x) {
    const int blk = row[lb];
    if (blk < 0 || blk >= p.num_blocks) bad = 1;
  }
  return __syncthreads_or(bad) == 0;
}

template <int D>
__device__ void mma_segment(const AttnParams& p, const ReqShape& r, int b, int kvh, int rg,
                            int tile0, int tile1, bool whole, int my_slot, int unit_id,
                            long long unit_t0, long long total, uint8_t* smem, int* s_flag) {
  using C = MmaCfg<D>;
  constexpr int LD = C::LD;
  constexpr int D2 = D / 2;
  constexpr int NT = D / 8;        // n8 tiles of the output
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem);
  __nv_bfloat16* sK0 = reinterpret_cast<__nv_bfloat16*>(smem + C::kQBytes);
  __nv_bfloat16* sV0 = sK0 + 2 * kMmaBN * LD;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int G = p.group;
  const int row_lo = rg * kMmaRows;
  const int row_hi = min(row_lo + kMmaRows, G * r.n);
  const int nrows = row_hi - row_lo;
  const int npt = (r.plen + kMmaBN - 1) / kMmaBN;
  const bool style0 = p.rope_style == 0;
  const int32_t* trow = p.block_table + static_cast<size_t>(b) * p.max_blocks;

  // ---- queries: rotate at depth position, round to bf16, stage in smem
  for (int idx = tid; idx < kMmaRows * D2; idx += kMmaThreads) {
    const int lr = idx / D2, pr = idx % D2;
    const int i0 = style0 ? 2 * pr : pr, i1 = style0 ? 2 * pr + 1 : pr + D2;
    float x0 = 0.f, x1 = 0.f;
    if (lr < nrows) {
      const int row = row_lo + lr;
      const int node = row / G, h = kvh * G + row % G;
      const __nv_bfloat16* gq = p.q + (static_cast<size_t>(r.t0 + node) * p.hq + h) * D;
      rope_pair(__bfloat162float(gq[i0]), __bfloat162float(gq[i1]), p.positions[r.t0 + node],
                p.inv_freq[pr], x0, x1);
    }
    sQ[lr * LD + i0] = __float2bfloat16_rn(x0);
    sQ[lr * LD + i1] = __float2bfloat16_rn(x1);
  }

  auto issue_prompt = [&](int tile, int buf) {
    __nv_bfloat16* sK = sK0 + buf * kMmaBN * LD;
    __nv_bfloat16* sV = sV0 + buf * kMmaBN * LD;
    constexpr int VPR = D / 8;   // 16-byte vectors per row
    for (int idx = tid; idx < kMmaBN * VPR; idx += kMmaThreads) {
      const int kk = idx / VPR, v = idx % VPR;
      const int key = tile * kMmaBN + kk;
      const bool valid = key < r.plen;
      const __nv_bfloat16* srck = p.k_cache;
      const __nv_bfloat16* srcv = p.v_cache;
      if (valid) {
        const size_t off = ((static_cast<size_t>(trow[key / TV_BLOCK_SIZE]) * p.hkv + kvh) *
                                TV_BLOCK_SIZE + key % TV_BLOCK_SIZE) * D + v * 8;
        srck += off;
        srcv += off;
      }
      cp_async16(sK + kk * LD + v * 8, srck, valid);
      cp_async16(sV + kk * LD + v * 8, srcv, valid);
    }
    cp_async_commit();
  };

  auto fill_tree = [&](int tile, int buf) {
    __nv_bfloat16* sK = sK0 + buf * kMmaBN * LD;
    __nv_bfloat16* sV = sV0 + buf * kMmaBN * LD;
    const int tb = (tile - npt) * kMmaBN;
    for (int idx = tid; idx < kMmaBN * D2; idx += kMmaThreads) {
      const int kk = idx / D2, pr = idx % D2;
      const int i0 = style0 ? 2 * pr : pr, i1 = style0 ? 2 * pr + 1 : pr + D2;
      const int jn = tb + kk;
      __nv_bfloat16 k0 = __float2bfloat16_rn(0.f), k1 = k0, v0 = k0, v1 = k0;
      if (jn < r.n) {
        const size_t base = (static_cast<size_t>(r.t0 + jn) * p.hkv + kvh) * D;
        float x0, x1;
        rope_pair(__bfloat162float(p.k_new[base + i0]), __bfloat162float(p.k_new[base + i1]),
                  p.positions[r.t0 + jn], p.inv_freq[pr], x0, x1);
        k0 = __float2bfloat16_rn(x0);
        k1 = __float2bfloat16_rn(x1);
        v0 = p.v_new[base + i0];
        v1 = p.v_new[base + i1];
        if (rg == 0) {   // exactly one unit per (request, KV head) writes the tentative slots
          const int slot = r.plen + jn;
          const size_t off = ((static_cast<size_t>(trow[slot / TV_BLOCK_SIZE]) * p.hkv + kvh) *
                                  TV_BLOCK_SIZE + slot % TV_BLOCK_SIZE) * D;
          p.k_cache[off + i0] = k0;
          p.k_cache[off + i1] = k1;
          p.v_cache[off + i0] = v0;
          p.v_cache[off + i1] = v1;
        }
      }
      sK[kk * LD + i0] = k0;
      sK[kk * LD + i1] = k1;
      sV[kk * LD + i0] = v0;
      sV[kk * LD + i1] = v1;
    }
  };

  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const bool warp_live = warp * 16 < nrows;
  // nodes of this thread's two rows (for the tree mask)
  int node_r[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int lr = warp * 16 + g + hh * 8;
    node_r[hh] = lr < nrows ? (row_lo + lr) / G : -1;
  }

  int buf = 0;
  if (tile0 < npt) issue_prompt(tile0, 0);
  for (int tile = tile0; tile < tile1; ++tile) {
    const bool prompt = tile < npt;
    if (prompt) {
      if (tile + 1 < tile1 && tile + 1 < npt) {
        issue_prompt(tile + 1, buf ^ 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
    } else {
      fill_tree(tile, buf);
    }
    __syncthreads();
    if (warp_live) {
      const __nv_bfloat16* sK = sK0 + buf * kMmaBN * LD;
      const __nv_bfloat16* sV = sV0 + buf * kMmaBN * LD;
      float s[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, sQ + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3,
                  sK + (j * 8 + (lane & 7) + (lane >> 4) * 8) * LD + kk * 16 + ((lane >> 3) & 1) * 8);
          mma16816(s[j], a0, a1, a2, a3, b0, b1);
          mma16816(s[j + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      // scale into the log2 domain and mask
      uint32_t mw[2][2] = {{0u, 0u}, {0u, 0u}};
      const int tb = (tile - npt) * kMmaBN;
      if (!prompt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (node_r[hh] >= 0) {
            const uint32_t* mrow = p.mask + static_cast<size_t>(r.t0 + node_r[hh]) * p.words;
            const int w0 = tb >> 5;
            mw[hh][0] = w0 < p.words ? mrow[w0] : 0u;
            mw[hh][1] = w0 + 1 < p.words ? mrow[w0 + 1] : 0u;
          }
        }
      }
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int hh = e >> 1;
          const int kl = j * 8 + 2 * tq + (e & 1);
          bool valid;
          if (prompt) {
            valid = tile * kMmaBN + kl < r.plen;
          } else {
            const int jn = tb + kl;
            valid = jn < r.n && ((mw[hh][kl >> 5] >> (jn & 31)) & 1u);
          }
          const float v = valid ? s[j][e] * p.scale_log2 : -INFINITY;
          s[j][e] = v;
          mx[hh] = fmaxf(mx[hh], v);
        }
      }
      float alpha[2], base[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
        mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
        const float m_new = fmaxf(m_run[hh], mx[hh]);
        base[hh] = m_new == -INFINITY ? 0.f : m_new;
        alpha[hh] = fast_exp2(m_run[hh] - base[hh]);
        m_run[hh] = m_new;
        l_run[hh] *= alpha[hh];
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[j][0] *= alpha[0];
        o[j][1] *= alpha[0];
        o[j][2] *= alpha[1];
        o[j][3] *= alpha[1];
      }
      uint32_t pa[8][2];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = fast_exp2(s[j][0] - base[0]), p1 = fast_exp2(s[j][1] - base[0]);
        const float p2 = fast_exp2(s[j][2] - base[1]), p3 = fast_exp2(s[j][3] - base[1]);
        l_run[0] += p0 + p1;
        l_run[1] += p2 + p3;
        pa[j][0] = pack_bf16x2(p0, p1);
        pa[j][1] = pack_bf16x2(p2, p3);
      }
#pragma unroll
      for (int kk = 0; kk < kMmaBN / 16; ++kk) {
        const uint32_t a0 = pa[2 * kk][0], a1 = pa[2 * kk][1];
        const uint32_t a2 = pa[2 * kk + 1][0], a3 = pa[2 * kk + 1][1];
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3,
                    sV + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + j * 8 + (lane >> 4) * 8);
          mma16816(o[j], a0, a1, a2, a3, b0, b1);
          mma16816(o[j + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
    __syncthreads();
    buf ^= 1;
  }

  // ---- epilogue
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 1);
    l_run[hh] += __shfl_xor_sync(0xffffffffu, l_run[hh], 2);
  }
  if (whole) {
    if (warp_live) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int lr = warp * 16 + g + hh * 8;
        if (lr >= nrows) continue;
        const int row = row_lo + lr;
        const int node = row / G, h = kvh * G + row % G;
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(r.t0 + node) * p.hq + h) * D;
        const float inv = 1.f / l_run[hh];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          *reinterpret_cast<uint32_t*>(dst + j * 8 + 2 * tq) =
              pack_bf16x2(o[j][2 * hh] * inv, o[j][2 * hh + 1] * inv);
        }
      }
    }
    return;
  }
  // split unit: publish the partial (unnormalised O, running max, sum)
  const size_t slot_floats = ws_slot_floats(kMmaRows, D);
  float* part = p.partials + static_cast<size_t>(my_slot) * slot_floats;
  if (warp_live) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int lr = warp * 16 + g + hh * 8;
      if (lr >= nrows) continue;
#pragma unroll
      for (int j = 0; j < NT; ++j)
        *reinterpret_cast<float2*>(part + static_cast<size_t>(lr) * D + j * 8 + 2 * tq) =
            make_float2(o[j][2 * hh], o[j][2 * hh + 1]);
      if (tq == 0) {
        part[kMmaRows * D + lr] = m_run[hh];
        part[kMmaRows * D + kMmaRows + lr] = l_run[hh];
      }
    }
  }
  __threadfence();
  __syncthreads();
  const int c_first = cta_of_tile(total, p.plan.grid, unit_t0);
  const int c_last = cta_of_tile(total, p.plan.grid, unit_t0 + r.tiles - 1);
  if (tid == 0) {
    const int prev = atomicAdd(p.counters + unit_id, 1);
    *s_flag = prev == c_last - c_first;
  }
  __syncthreads();
  if (!*s_flag) return;
  __threadfence();
  // last contributor: merge every contributor's partial
  for (int idx = tid; idx < nrows * (D / 4); idx += kMmaThreads) {
    const int lr = idx / (D / 4), d4 = idx % (D / 4);
    float mmax = -INFINITY;
    for (int c = c_first; c <= c_last; ++c) {
      const int sl = (c == c_first && cta_start(total, p.plan.grid, c) != unit_t0) ? 2 * c + 1 : 2 * c;
      const float* ps = p.partials + static_cast<size_t>(sl) * slot_floats;
      mmax = fmaxf(mmax, __ldcg(ps + kMmaRows * D + lr));
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
    for (int c = c_first; c <= c_last; ++c) {
      const int sl = (c == c_first && cta_start(total, p.plan.grid, c) != unit_t0) ? 2 * c + 1 : 2 * c;
      const float* ps = p.partials + static_cast<size_t>(sl) * slot_floats;
      const float mc = __ldcg(ps + kMmaRows * D + lr);
      if (mc == -INFINITY) continue;
      const float wgt = fast_exp2(mc - mmax);
      lsum += wgt * __ldcg(ps + kMmaRows * D + kMmaRows + lr);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(ps + static_cast<size_t>(lr) * D) + d4);
      acc.x += wgt * v.x;
      acc.y += wgt * v.y;
      acc.z += wgt * v.z;
      acc.w += wgt * v.w;
    }
    const float inv = 1.f / lsum;
    const int row = row_lo + lr;
    const int node = row / G, h = kvh * G + row % G;
    __nv_bfloat16* dst = p.out + (static_cast<size_t>(r.t0 + node) * p.hq + h) * D + d4 * 4;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  }
  if (tid == 0) p.counters[unit_id] = 0;   // leave the workspace zeroed for the next call
}

template <int D>
__global__ void __launch_bounds__(kMmaThreads, 1) attn_mma_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ long long s_tmp[kMmaThreads];
  __shared__ int s_flag;
  long long* s_pre = reinterpret_cast<long long*>(smem + MmaCfg<D>::kFixed);
  plan_prefix(p.cu_nodes, p.prompt_len, p.plan, s_pre, s_tmp);
  const long long total = s_pre[p.plan.batch];
  const int c = blockIdx.x;
  const long long s = cta_start(total, p.plan.grid, c), e = cta_start(total, p.plan.grid, c + 1);
  int checked_b = -1;
  bool checked_ok = false;
  for (long long t = s; t < e;) {
    const int b = request_of_tile(s_pre, p.plan.batch, t);
    const ReqShape r = req_shape(p.cu_nodes, p.prompt_len, p.plan, b);
    const long long local = t - s_pre[b];
    const int unit = static_cast<int>(local / r.tiles);
    const int tile0 = static_cast<int>(local % r.tiles);
    const int tile1 = static_cast<int>(min(static_cast<long long>(r.tiles), tile0 + (e - t)));
    const long long unit_t0 = s_pre[b] + static_cast<long long>(unit) * r.tiles;
    const bool first_seg = t == s;
    t += tile1 - tile0;
    if (p.status[b] & TV_TREE_FLAGS) continue;
    if (b != checked_b) {
      checked_ok = request_blocks_ok(p, b, r.plen, r.n);
      checked_b = b;
      if (!checked_ok && threadIdx.x == 0) atomicOr(p.status + b, TV_ST_BAD_BLOCK);
    }
    if (!checked_ok) continue;
    const int kvh = unit / r.nrg, rg = unit % r.nrg;
    const bool whole = tile0 == 0 && tile1 == r.tiles;
    const int my_slot = first_seg ? 2 * c : 2 * c + 1;
    const int unit_id = (b * p.hkv + kvh) * p.plan.nrg_max + rg;
    mma_segment<D>(p, r, b, kvh, rg, tile0, tile1, whole, my_slot, unit_id, unit_t0, total, smem,
                   &s_flag);
    __syncthreads();
  }
}

}  // namespace tv

// ---------------------------------------------------------------------------
// host side

namespace tv {

int mma_grid() {
  const int dev = current_device();
  return dev < 0 ? -1 : device_sm_count(dev);
}

// Bytes at the start of the workspace that must be zero before a call (the
// per-unit arrival counters).
size_t mma_counter_bytes(int batch, int hkv, int group, int max_nodes) {
  return ws_counter_bytes(batch, hkv, (group * max_nodes + kMmaRows - 1) / kMmaRows);
}

size_t mma_workspace_bytes(int batch, int hkv, int group, int max_nodes, int head_dim, int grid) {
  const int nrg_max = (group * max_nodes + kMmaRows - 1) / kMmaRows;
  return ws_counter_bytes(batch, hkv, nrg_max) +
         static_cast<size_t>(2) * grid * ws_slot_floats(kMmaRows, head_dim) * sizeof(float);
}

int launch_attention_mma(const tv_geom* geom, int batch, int max_nodes, const void* q,
                         const void* k_new, const void* v_new, const int32_t* cu_nodes,
                         const int32_t* positions, const uint32_t* mask, const int32_t* prompt_len,
                         const int32_t* block_table, const int32_t* n_blocks, int max_blocks,
                         void* k_cache, void* v_cache, int num_blocks, void* out, void* workspace,
                         size_t ws_bytes, int32_t* status, cudaStream_t stream) {
  const int grid = mma_grid();
  if (grid <= 0) return TV_ERR_CUDA;
  const int D = geom->head_dim;
  const int group = geom->num_q_heads / geom->num_kv_heads;
  if (ws_bytes < mma_workspace_bytes(batch, geom->num_kv_heads, group, max_nodes, D, grid))
    return TV_ERR_WORKSPACE;
  AttnParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k_new = static_cast<const __nv_bfloat16*>(k_new);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new);
  p.cu_nodes = cu_nodes;
  p.positions = positions;
  p.mask = mask;
  p.prompt_len = prompt_len;
  p.block_table = block_table;
  p.n_blocks = n_blocks;
  p.k_cache = static_cast<__nv_bfloat16*>(k_cache);
  p.v_cache = static_cast<__nv_bfloat16*>(v_cache);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.status = status;
  p.hq = geom->num_q_heads;
  p.hkv = geom->num_kv_heads;
  p.group = group;
  p.words = (max_nodes + 31) / 32;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.rope_style = geom->rope_style;
  const double scale = geom->softmax_scale > 0.f ? geom->softmax_scale : 1.0 / sqrt(double(D));
  p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
  for (int i = 0; i < 64; ++i)
    p.inv_freq[i] = i < D / 2 ? static_cast<float>(pow(double(geom->rope_base), -2.0 * i / D)) : 0.f;
  p.plan.batch = batch;
  p.plan.max_nodes = max_nodes;
  p.plan.group = group;
  p.plan.hkv = geom->num_kv_heads;
  p.plan.rows_per_unit = kMmaRows;
  p.plan.keys_per_tile = kMmaBN;
  p.plan.nrg_max = (group * max_nodes + kMmaRows - 1) / kMmaRows;
  p.plan.grid = grid;
  p.counters = static_cast<int32_t*>(workspace);
  p.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        ws_counter_bytes(batch, p.hkv, p.plan.nrg_max));
  const size_t smem_fixed = D == 128 ? MmaCfg<128>::kFixed : MmaCfg<64>::kFixed;
  const size_t smem = smem_fixed + static_cast<size_t>(batch + 1) * sizeof(long long);
  if (smem > 227 * 1024) return TV_ERR_BAD_SIZE;
  static size_t smem_set128[kMaxDevices] = {0}, smem_set64[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0) return TV_ERR_CUDA;
  if (D == 128) {
    if (!ensure_smem(attn_mma_kernel<128>, smem, smem_set128, dev)) return TV_ERR_CUDA;
    attn_mma_kernel<128><<<grid, kMmaThreads, smem, stream>>>(p);
  } else {
    if (!ensure_smem(attn_mma_kernel<64>, smem, smem_set64, dev)) return TV_ERR_CUDA;
    attn_mma_kernel<64><<<grid, kMmaThreads, smem, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}

}  // namespace tv
