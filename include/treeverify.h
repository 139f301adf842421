/*
 * treeverify.h - C interface of the GB300 (sm_103a) token-tree verification
 * library, libtreeverify.so.
 *
 * One verification step of tree speculative decoding runs four calls on the
 * caller's CUDA stream:
 *
 *   tv_tree_build             parent list -> bit-packed ancestor mask, depth
 *                             positions, retrieve_index / next_token /
 *                             next_sibling (tv_tree_mask_dense exports the
 *                             mask densely for other attention code)
 *   tv_tree_attention_verify  depth-RoPE of the tree's fresh Q/K, tentative KV
 *                             write, GQA attention over the paged prompt cache
 *                             plus each node's ancestors
 *   tv_greedy_accept          longest accepted path + bonus token
 *   tv_kv_commit              move the accepted K/V rows to the committed
 *                             slots and release the blocks past the new end
 *
 * Sources of the definitions (web pages, cited by title and section):
 *   [GLOSSARY] "Beam Search、约束解码与 Tree/Self Speculation"
 *   [ATLAS]    "02 · Token Tree 与 Tree Attention"
 *   [WIBLOG]   "投机解码的树状注意力验证：一次前向如何并行校验多条候选路径"
 *   [DDTREE]   "Accelerating Speculative Decoding with Block Diffusion Draft Trees"
 *   [DECODE]   "解码：采样、束搜索和推测性解码"
 *
 * Sampling acceptance (the verifier samples itself, [DDTREE] §7.2-§7.3) adds
 * two calls that take the target's per-node logits instead of its argmax ids:
 *
 *   tv_sample_tokens          the target's sampled (or greedy) token at every node
 *   tv_sampled_accept         the verifier walk, sampling only the nodes it visits
 *
 * Rejection-sampling acceptance ([ATLAS] §4: one chosen path accepted edge by
 * edge with the min(1, p/q) rule) takes the drafter's logits as well:
 *
 *   tv_rejection_accept       chosen path, per-edge acceptance, correction draw
 *
 * Draft-tree construction ([DDTREE] §4-§5) builds the tree that tv_tree_build
 * consumes from a block drafter's per-position logits:
 *
 *   tv_ddtree_topk            per position: top-K tokens and log-probabilities
 *   tv_ddtree_build           best-first heap (Algorithm 1) -> parent lists
 *
 * EAGLE-2 dynamic trees ([ATLAS] §3, §5) are selected from a drafter's
 * layer-by-layer candidates:
 *
 *   tv_eagle_expand_select    per layer: the top-k candidates to expand next
 *   tv_eagle_rerank           global top-N by survival probability -> parent lists
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All array arguments are DEVICE pointers owned by the caller. The library
 *    allocates no device memory, keeps no state between calls and never
 *    synchronises the stream. Scratch space comes from the caller's workspace.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *  - A batch holds `batch` requests whose nodes are concatenated:
 *    request b owns flattened nodes [cu_nodes[b], cu_nodes[b+1]) (cu_nodes is
 *    int32 [batch+1], cu_nodes[0] = 0, non-decreasing). Within a request node
 *    0 is the root - the bonus token confirmed by the previous step, depth 0 -
 *    and parent indices are local: parent[0] = -1, 0 <= parent[i] < i.
 *    This topological packing is the packed layout of [GLOSSARY] section
 *    "Packed tree attention" with the root of [ATLAS] §2 added as node 0.
 *  - Paged KV pools k_cache / v_cache are bf16 [num_blocks][Hkv][16][D]
 *    (block size 16). block_table is int32 [batch][max_blocks_per_req]:
 *    slot s of request b lives in block block_table[b][s / 16], row s % 16.
 *    n_blocks[b] is how many leading table entries request b holds.
 *  - Return value: TV_OK or a negative TV_ERR_* code from host-side argument
 *    checks (nothing is launched then). Errors in the DATA are reported per
 *    request in `status` (int32 [batch], TV_ST_* flags); a request with a
 *    non-zero status keeps its outputs untouched. No call traps or aborts.
 *  - batch == 0 is a valid no-op.
 */
#ifndef TREEVERIFY_H_
#define TREEVERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host-side return codes */
#define TV_OK 0
#define TV_ERR_NULL_POINTER (-1)   /* a required pointer is NULL */
#define TV_ERR_BAD_GEOMETRY (-2)   /* head_dim not 64/128, Hq % Hkv != 0, block_size != 16, bad rope */
#define TV_ERR_BAD_SIZE (-3)       /* batch < 0, max_nodes outside [1, 1024], max_depth < 0, ... */
#define TV_ERR_WORKSPACE (-4)      /* workspace smaller than tv_workspace_bytes() */
#define TV_ERR_MISALIGNED (-5)     /* a bf16 array is not 16-byte aligned (workspace: 256) */
#define TV_ERR_CUDA (-6)           /* a CUDA runtime/driver call failed */
#define TV_ERR_DEVICE (-7)         /* the current device is not sm_103 */

/* per-request status flags (OR-ed; 0 = fine) */
#define TV_ST_BAD_SIZE 1           /* node count outside [1, max_nodes], prompt_len < 0, bad path */
#define TV_ST_BAD_ROOT 2           /* parent[0] != -1 */
#define TV_ST_BAD_PARENT 4         /* parent[i] outside [0, i-1] for some i >= 1 */
#define TV_ST_BAD_BLOCK 8          /* a needed block-table entry is missing or out of range */
#define TV_ST_PATH_OVERFLOW 16     /* accepted path longer than max_depth */
#define TV_ST_TIMEOUT 32           /* a bounded device wait gave up; that request's outputs are invalid */
#define TV_ST_BAD_TEMPERATURE 64   /* temperature negative or NaN, or > 0 with no noise array */

#define TV_MAX_NODES 1024          /* largest tree (root included) per request */
#define TV_BLOCK_SIZE 16

typedef struct tv_geom {
  int32_t num_q_heads;     /* Hq */
  int32_t num_kv_heads;    /* Hkv; query head h reads KV head h / (Hq / Hkv) */
  int32_t head_dim;        /* D: 64 or 128 */
  int32_t block_size;      /* must be 16 */
  float rope_base;         /* RoPE base (10000 in [GLOSSARY]'s experiment); > 0 */
  float softmax_scale;     /* <= 0 means 1 / sqrt(D) ([GLOSSARY] packed_attention) */
  int32_t rope_style;      /* 0: pairs (2i, 2i+1) as in [GLOSSARY]; 1: pairs (i, i + D/2) */
} tv_geom;

/*
 * Workspace size for tv_tree_attention_verify on the CURRENT device.
 * The workspace holds the rotated queries, split-KV partial results and
 * merge records of one call. Its contents need no initialisation (every call
 * writes what it reads); calls that overlap on the GPU must use different
 * workspaces.
 * Returns TV_OK and writes *bytes, or a TV_ERR_* code.
 */
int tv_workspace_bytes(const tv_geom* geom, int32_t batch, int32_t max_nodes, size_t* bytes);

/*
 * Tree metadata ([ATLAS] §3 "Tree attention 的 mask 规则": the builder turns
 * the parent list into a tree mask, RoPE positions and retrieve_* arrays;
 * positions = prompt length + depth, e.g. depths [0,1,1,2] with prompt 7 give
 * [7,8,8,9]; [GLOSSARY] "Packed tree attention": each node sees its ancestor
 * chain, never siblings or cousins).
 *
 *  parents        int32 [T]            local parent index per node (see above)
 *  cu_nodes       int32 [batch+1]
 *  prompt_len     int32 [batch]        committed tokens P_b already in the cache
 *  max_nodes      largest node count allowed per request (1..1024); W = ceil(max_nodes/32)
 *  mask_bits      uint32 [T][W] out    bit (j%32) of word j/32 of row t set iff
 *                                      local node j is an ancestor of t or t itself
 *  depth          int32 [T] out        root depth 0
 *  positions      int32 [T] out        P_b + depth
 *  retrieve_index int32 [T] out        flattened index of the node (cu_nodes[b] + i)
 *  next_token     int32 [T] out        smallest-index child, -1 if none
 *  next_sibling   int32 [T] out        next larger-index node with the same parent, -1 if none
 *  status         int32 [batch] out    OVERWRITTEN: TV_ST_BAD_SIZE / _BAD_ROOT / _BAD_PARENT
 *                                      or 0. Starts the step's per-request status.
 */
int tv_tree_build(const int32_t* parents, const int32_t* cu_nodes, const int32_t* prompt_len,
                  int32_t batch, int32_t max_nodes, uint32_t* mask_bits, int32_t* depth,
                  int32_t* positions, int32_t* retrieve_index, int32_t* next_token,
                  int32_t* next_sibling, int32_t* status, void* stream);

/*
 * Dense export of the tree mask ([GLOSSARY] "Packed tree attention": the
 * [N, P+N] mask, bool or additive -inf, in which a node sees the whole prefix
 * plus its ancestor chain and itself; [ATLAS] §3: the FULL_MASK and QLEN_ONLY
 * modes beside bit-packing), for attention code that takes a dense mask.
 *
 *  mask_bits, cu_nodes, prompt_len, max_nodes   as for tv_tree_build
 *  status     int32 [batch] in: requests with non-zero status are not written
 *  mode       TV_MASK_FULL: request b's block is [N_b][P_b + N_b] (prompt
 *             columns first); TV_MASK_QLEN_ONLY: [N_b][N_b] (tree columns only)
 *  dtype      TV_MASK_BOOL: uint8, 1 visible / 0 masked;
 *             TV_MASK_ADDITIVE_F32: float32, 0 visible / -inf masked
 *             (out 4-byte aligned)
 *  out        the requests' blocks back to back, row-major, no padding:
 *             sum_b N_b (max(P_b, 0) + N_b) elements (FULL), sum_b N_b^2 (QLEN_ONLY)
 */
#define TV_MASK_FULL 0
#define TV_MASK_QLEN_ONLY 1
#define TV_MASK_BOOL 0
#define TV_MASK_ADDITIVE_F32 1
int tv_tree_mask_dense(const uint32_t* mask_bits, const int32_t* cu_nodes,
                       const int32_t* prompt_len, const int32_t* status, int32_t batch,
                       int32_t max_nodes, int32_t mode, int32_t dtype, void* out, void* stream);

/*
 * Packed tree attention with depth RoPE and the tentative KV write
 * ([GLOSSARY] "Packed tree attention" and its packed-vs-branch experiment:
 * softmax(q k^T * scale) v over the committed prefix plus the node's ancestor
 * chain, RoPE at the node's depth position; [ATLAS] §3; [WIBLOG]
 * "实现中的 KV Cache 与批处理约束": the tree's tentative KV occupies a contiguous
 * region in node order).
 *
 *  q              bf16 [T][Hq][D]      raw (un-rotated) queries of the tree nodes
 *  k_new, v_new   bf16 [T][Hkv][D]     raw keys / values of the tree nodes
 *  cu_nodes       int32 [batch+1]
 *  positions      int32 [T]            from tv_tree_build
 *  mask_bits      uint32 [T][W]        from tv_tree_build (W = ceil(max_nodes/32))
 *  prompt_len     int32 [batch]
 *  block_table    int32 [batch][max_blocks_per_req], n_blocks int32 [batch]
 *  k_cache,v_cache bf16 pools (see conventions). Slots [0, P_b) are read
 *                 (already rotated); slots [P_b, P_b + N_b) receive the
 *                 rotated k_new and the raw v_new of node i at slot P_b + i.
 *                 Every block covering slots [0, P_b + N_b) must be held.
 *  out            bf16 [T][Hq][D] out  attention output per node and query head
 *  workspace      device scratch of tv_workspace_bytes() bytes (256-byte aligned)
 *  status         int32 [batch] in/out requests whose status carries a tree
 *                 flag are skipped; TV_ST_BAD_BLOCK / TV_ST_TIMEOUT are OR-ed in.
 * Rotated K is rounded to bf16 (round-to-nearest-even) after an fp32
 * rotation; scores and the softmax run in fp32 with bf16 tensor-core operands.
 */
int tv_tree_attention_verify(const tv_geom* geom, int32_t batch, int32_t max_nodes,
                             const void* q, const void* k_new, const void* v_new,
                             const int32_t* cu_nodes, const int32_t* positions,
                             const uint32_t* mask_bits, const int32_t* prompt_len,
                             const int32_t* block_table, const int32_t* n_blocks,
                             int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                             int32_t num_blocks, void* out, void* workspace,
                             size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Allocation-free variant of tv_tree_attention_verify. The published tree
 * verification methods have no counterpart to this call: it exists for callers that cannot obtain device
 * memory - a plugin inside a host framework that only receives a stream and
 * tensors, code running while another component owns the whole device memory
 * pool, or a latency-critical loop that must not call cudaMalloc (which can
 * synchronise the device). Same arguments and results as
 * tv_tree_attention_verify, without the workspace.
 *
 *  - Scratch comes from a static device array of TV_NOALLOC_SCRATCH_BYTES
 *    (64 MiB) inside the library. The runtime reserves it on a GPU the first
 *    time this call runs there and keeps it until the process exits.
 *  - The first call on each device looks up that array's device address (with
 *    the device current); make that first call before any stream capture.
 *  - Every call on a device shares the one array (nothing in it needs to
 *    start at zero: a call writes each record before reading it). Calls that
 *    overlap on the GPU (other streams, other threads) race on it: serialise
 *    them.
 *  - A batch or tree that needs more scratch than TV_NOALLOC_SCRATCH_BYTES
 *    (see tv_workspace_bytes) is rejected with TV_ERR_WORKSPACE and nothing
 *    is launched.
 *  - Calls no cudaMalloc/cudaFree or any allocating routine.
 */
#define TV_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int tv_tree_attention_verify_noalloc(const tv_geom* geom, int32_t batch, int32_t max_nodes,
                                     const void* q, const void* k_new, const void* v_new,
                                     const int32_t* cu_nodes, const int32_t* positions,
                                     const uint32_t* mask_bits, const int32_t* prompt_len,
                                     const int32_t* block_table, const int32_t* n_blocks,
                                     int32_t max_blocks_per_req, void* k_cache, void* v_cache,
                                     int32_t num_blocks, void* out, int32_t* status,
                                     void* stream);

/*
 * Greedy acceptance walk ([ATLAS] §4: from the root, move to the child whose
 * token equals the target's choice, stop at the first miss, the target's
 * token there is the correction / bonus; [GLOSSARY] three-part experiment
 * verify_tree; [DDTREE] §6-§7.2). Among several matching children the
 * smallest index wins.
 *
 *  target_ids     int32 [T]   target's greedy token after each node's prefix
 *  draft_tokens   int32 [T]   token of each node (root: the previous bonus)
 *  cu_nodes, next_token, next_sibling   as produced by tv_tree_build
 *  max_nodes      as for tv_tree_build
 *  max_depth      capacity of a path: accept_path rows hold max_depth + 1 entries
 *  accept_path    int32 [batch][max_depth+1] out  local node indices from the root
 *                 (entry 0 = 0), -1 after the last accepted node
 *  accept_len     int32 [batch] out  accepted draft nodes a (path length a + 1)
 *  bonus          int32 [batch] out  next step's root token
 *  status         in/out: requests with non-zero status are skipped;
 *                 TV_ST_PATH_OVERFLOW when a > max_depth (outputs untouched)
 */
int tv_greedy_accept(const int32_t* target_ids, const int32_t* draft_tokens,
                     const int32_t* cu_nodes, const int32_t* next_token,
                     const int32_t* next_sibling, int32_t batch, int32_t max_nodes,
                     int32_t max_depth, int32_t* accept_path, int32_t* accept_len,
                     int32_t* bonus, int32_t* status, void* stream);

/*
 * Per-node sampling with the Gumbel-max trick ([DECODE] "高效离散采样" /
 * "Gumbel Max技巧": argmax_v (h_v + g_v) with Gumbel noise g is a draw from
 * softmax(h); [DDTREE] §7.2: the target picks each node's token with its own
 * rule, greedy or temperature sampling).
 *
 * For node t of request b with temperature T = temperature[b]:
 *   T == 0: token[t] = first argmax_v logits[t][v]            (greedy)
 *   T >  0: token[t] = first argmax_v fl(fl(logits[t][v] * fl(1/T)) + gumbel[t][v])
 * in float32 with each operation rounded (no fused multiply-add). A NaN
 * counts as the largest value, +0 and -0 tie; ties go to the smallest v.
 *
 *  logits         float32 [T][logits_ld], row t holds node t's vocab entries
 *                 0..vocab-1; 16-byte aligned, logits_ld % 4 == 0, >= vocab
 *  gumbel         float32 [T][gumbel_ld] noise g = -log(-log(u)), u ~ U(0,1),
 *                 drawn by the caller; same alignment rules. May be NULL when
 *                 every temperature is 0 (a request with T > 0 then gets
 *                 TV_ST_BAD_TEMPERATURE). Not read for greedy requests.
 *  cu_nodes       int32 [batch+1]
 *  temperature    float32 [batch] (device)
 *  max_nodes      largest node count of a request (1..1024)
 *  vocab          entries per row (1 .. 2^30)
 *  tokens         int32 [T] out
 *  status         in/out: requests with non-zero status are skipped;
 *                 TV_ST_BAD_SIZE (node count > max_nodes) and
 *                 TV_ST_BAD_TEMPERATURE are OR-ed in (outputs untouched)
 */
int tv_sample_tokens(const float* logits, int64_t logits_ld, const float* gumbel,
                     int64_t gumbel_ld, const int32_t* cu_nodes, const float* temperature,
                     int32_t batch, int32_t max_nodes, int32_t vocab, int32_t* tokens,
                     int32_t* status, void* stream);

/*
 * The verifier walk with the target sampling itself ([DDTREE] §7.2: from the
 * root, pick a token at the current node with the target's rule; if a child
 * of the node carries it, move there, else stop with it as the next bonus;
 * §7.3: the output then follows the target's own autoregressive sampling,
 * whatever the drafter proposed). The token at a visited node is decided
 * exactly as tv_sample_tokens decides it, so the result equals
 * tv_sample_tokens followed by tv_greedy_accept; only the visited nodes'
 * rows are read (one row of logits, and of noise when sampling, per step).
 *
 *  logits, logits_ld, gumbel, gumbel_ld, cu_nodes, temperature, vocab
 *                 as for tv_sample_tokens
 *  parents        int32 [T] local parent lists, validated by tv_tree_build
 *                 (run it first: requests it flagged are skipped)
 *  draft_tokens   int32 [T]
 *  max_nodes, max_depth, accept_path, accept_len, bonus
 *                 as for tv_greedy_accept (among several children carrying
 *                 the token the smallest index wins)
 *  status         in/out: requests with non-zero status are skipped;
 *                 TV_ST_BAD_SIZE, TV_ST_BAD_TEMPERATURE or TV_ST_PATH_OVERFLOW
 *                 are OR-ed in (outputs untouched)
 */
int tv_sampled_accept(const float* logits, int64_t logits_ld, const float* gumbel,
                      int64_t gumbel_ld, const int32_t* cu_nodes, const float* temperature,
                      const int32_t* parents, const int32_t* draft_tokens, int32_t batch,
                      int32_t max_nodes, int32_t max_depth, int32_t vocab,
                      int32_t* accept_path, int32_t* accept_len, int32_t* bonus,
                      int32_t* status, void* stream);

/*
 * Rejection-sampling verification along one chosen path ([ATLAS] §4: the
 * target's logits at every node come from the one forward; one best path is
 * chosen by its log-probability and accepted from the root edge by edge with
 * the min(1, p/q) rule; a rejection ends the walk with a correction token
 * sampled at the current node, a fully accepted path with the bonus token
 * sampled at its last node; [DECODE] "Gumbel Max技巧" for the draws).
 *
 * For request b with temperature T = temperature[b]:
 *   path   root to the leaf with the largest sum of draft_logp over its nodes
 *          (float64 sums, node 0 contributes 0; the smallest leaf index on ties)
 *   p_u    softmax(logits[u] / T) (T == 0: all mass on the first argmax)
 *   q_u    softmax(draft_logits[u]), the distribution u's children were drawn from
 *   edge u -> c on the path is accepted when uniforms[c] < p_u(x_c) / q_u(x_c),
 *          x_c = draft_tokens[c] (p_u(x_c) == 0 rejects, else
 *          q_u(x_c) == 0 accepts; x_c outside [0, vocab) rejects); the first
 *          rejection at u stops the walk
 *   bonus  after a rejection at u: Gumbel-max draw over max(0, p_u - q_u)
 *          (over p_u when that is zero everywhere) with noise row gumbel[u];
 *          after the whole path: draw over p at the last node; T == 0: the
 *          first argmax of the stop node's logits.
 * The path sums are float64 (exact choice); log-sum-exps, per-edge ratios
 * and the residual keys log(p_v - q_v) + g_v are float32, so a sampled
 * decision can differ from an exact evaluation only where the exact margin
 * is within float32 rounding. Greedy requests read only the target rows and
 * decide exactly.
 *
 *  logits, logits_ld   float32 [T][logits_ld] target logits, row per node
 *                      (logits_ld >= vocab)
 *  draft_logits, draft_ld
 *                      float32 [T][draft_ld] drafter logits at each node
 *  gumbel, gumbel_ld   float32 [T][gumbel_ld] noise, as for tv_sample_tokens;
 *                      may be NULL when every temperature is 0
 *  uniforms            float32 [T], r_c ~ U(0, 1) for the edge into node c
 *  cu_nodes, temperature, vocab
 *                      as for tv_sample_tokens
 *  parents             int32 [T] local parent lists (parent[0] = -1,
 *                      0 <= parent[i] < i; TV_ST_BAD_ROOT / TV_ST_BAD_PARENT)
 *  draft_tokens        int32 [T]
 *  draft_logp          float32 [T] draft log-probability of each node's token
 *  max_nodes, max_depth, accept_path, accept_len, bonus
 *                      as for tv_greedy_accept (accept_path lists the
 *                      accepted prefix of the chosen path)
 *  status              in/out: requests with non-zero status are skipped;
 *                      TV_ST_BAD_SIZE, _BAD_ROOT, _BAD_PARENT,
 *                      _BAD_TEMPERATURE or _PATH_OVERFLOW are OR-ed in
 *                      (outputs untouched)
 * All arrays are device memory; nothing is allocated. Returns TV_OK, or
 * TV_ERR_BAD_SIZE / TV_ERR_NULL_POINTER / TV_ERR_CUDA without launching.
 */
int tv_rejection_accept(const float* logits, int64_t logits_ld, const float* draft_logits,
                        int64_t draft_ld, const float* gumbel, int64_t gumbel_ld,
                        const float* uniforms, const int32_t* cu_nodes,
                        const float* temperature, const int32_t* parents,
                        const int32_t* draft_tokens, const float* draft_logp, int32_t batch,
                        int32_t max_nodes, int32_t max_depth, int32_t vocab,
                        int32_t* accept_path, int32_t* accept_len, int32_t* bonus,
                        int32_t* status, void* stream);

/*
 * Nodes (root included) of the trees tv_ddtree_build makes: 1 + min(budget,
 * sum_{d=1..L} k^d). Returns that count, or TV_ERR_BAD_SIZE when depth_L < 1,
 * k < 1 or budget outside [1, 1023].
 */
int tv_ddtree_nodes(int32_t depth_L, int32_t k, int32_t budget);

/*
 * Per-position top-K of a block drafter's logits ([DDTREE] §4.3, Lemma 1:
 * only each depth's top K = min(B, |V|) tokens can enter the optimal tree;
 * §3-§4.1: q_i = softmax of position i's logits).
 *
 *  logits         float32 [rows][logits_ld], row r holds vocab logits;
 *                 16-byte aligned, logits_ld % 4 == 0, logits_ld >= vocab.
 *                 Rows of a batch of requests with L positions each are
 *                 row = request * L + position. Logits must not be NaN; -inf
 *                 is allowed (a row with no finite logit gets log q = -inf).
 *  vocab          entries per row (1 .. 2^30), k in [1, min(vocab, 1024)]
 *  top_tokens     int32 [rows][k] out  tokens by logit descending, equal
 *                 logits by token id ascending
 *  top_logq       float32 [rows][k] out  log softmax(row)[token]: the logit
 *                 minus the row's log-sum-exp (accumulated in float32 per
 *                 thread, combined in float64; absolute error about 1e-6)
 */
int tv_ddtree_topk(const float* logits, int64_t logits_ld, int32_t rows, int32_t vocab,
                   int32_t k, int32_t* top_tokens, float* top_logq, void* stream);

/*
 * DDTree best-first construction ([DDTREE] §5, Algorithm 1; §4.2,
 * Proposition 2: the budget most probable prefixes form a prefix-closed,
 * optimal tree; §6-§7.1: flattened depth by depth after the root).
 *
 *  top_logq       float32 [batch][depth_L][k], top_tokens int32 [batch][depth_L][k]:
 *                 per depth, the k candidates in rank order (tv_ddtree_topk)
 *  budget         prefixes to select, 1..1023; every tree gets
 *                 n = tv_ddtree_nodes(depth_L, k, budget) nodes
 *  root_tokens    int32 [batch] token of each root (the previous bonus), or
 *                 NULL for -1
 *  parents        int32 [batch * n] out  local parent index, -1 for the root
 *  tokens         int32 [batch * n] out
 *  cu_nodes       int32 [batch + 1] out  b * n
 * A prefix's score is its parent's score plus its own log-probability, added
 * in float32; equal scores take the shallower prefix, then the one whose
 * parent was selected first. Nodes are ordered root first, then by depth,
 * selection order within a depth, so parents precede children and the
 * output feeds tv_tree_build directly. Shared memory: 4 L k + 20 n bytes
 * (at most 200 KB, else TV_ERR_BAD_SIZE).
 */
int tv_ddtree_build(const float* top_logq, const int32_t* top_tokens, int32_t batch,
                    int32_t depth_L, int32_t k, int32_t budget, const int32_t* root_tokens,
                    int32_t* parents, int32_t* tokens, int32_t* cu_nodes, void* stream);

/*
 * Candidates of an EAGLE-style expansion, shared by the two calls below.
 * Request b owns candidates [b * max_cands, b * max_cands + cand_count[b]) in
 * generation order (a parent before its children):
 *  logp     float32  drafter log-probability of the candidate's token under
 *                    its parent (<= 0)
 *  parent   int32    index of the parent candidate within the request, -1 for
 *                    the root's children (TV_ST_BAD_PARENT if outside [-1, c))
 *  token    int32
 * A candidate's score is its parent's score plus its own log-probability
 * (float32, in that order) - the log of its prefix survival probability;
 * its depth is its parent's plus one (root's children: 1). max_cands <= 4096.
 */

/*
 * Layer expansion ([ATLAS] §3: each step expands the top-k nodes of the
 * current layer): the k candidates of depth `layer` with the largest scores,
 * earlier generated first on ties.
 *  selected   int32 [batch][k] out  candidate indices, best first, -1 when the
 *             layer has fewer than k candidates
 *  status     in/out: requests with non-zero status are skipped
 */
int tv_eagle_expand_select(const float* logp, const int32_t* parent, const int32_t* cand_count,
                           int32_t batch, int32_t max_cands, int32_t layer, int32_t k,
                           int32_t* selected, int32_t* status, void* stream);

/*
 * Global rerank ([ATLAS] §5: EAGLE-2 keeps the N_tree nodes with the largest
 * prefix survival probability): the n_keep best candidates (score
 * descending, then shallower, then earlier generated), packed breadth first
 * (depth, parent's packed index, generation order) after the root.
 *  root_tokens  int32 [batch] or NULL (-1)
 *  parents, tokens  int32 [batch * (n_keep + 1)] out; cu_nodes int32 [batch + 1] out
 *  status     in/out: requests with non-zero status are skipped; TV_ST_BAD_SIZE
 *             when cand_count < n_keep or the kept set is not prefix-closed
 *             (a positive log-probability), TV_ST_BAD_PARENT (outputs untouched)
 * n_keep in [1, 1023].
 */
int tv_eagle_rerank(const float* logp, const int32_t* parent, const int32_t* token,
                    const int32_t* cand_count, int32_t batch, int32_t max_cands, int32_t n_keep,
                    const int32_t* root_tokens, int32_t* parents, int32_t* tokens,
                    int32_t* cu_nodes, int32_t* status, void* stream);

/*
 * Commit / rollback of the tentative KV ([GLOSSARY] "Tree/Self Speculation":
 * [10,11] becomes [10,11,4,7] and the other tentative nodes are released;
 * [ATLAS] §4: the chosen path's KV is committed, the rest is discarded and
 * pages are reclaimed; [WIBLOG]: with a paged cache reclaiming frees pages).
 *
 * For k = 1..a the K and V rows (all KV heads) of slot P+accept_path[k] move
 * to slot P+k; every source row is read before any destination row of the
 * same request is written. The bytes move unchanged: the row already carries
 * RoPE at position P + k. new_len = P + 1 + a (the root is always kept).
 * Held blocks with logical index >= ceil(new_len / 16) are released in
 * ascending logical order: block_table entries become -1, n_blocks shrinks.
 *
 *  accept_path, accept_len    from tv_greedy_accept
 *  block_table, n_blocks      in/out
 *  new_len        int32 [batch] out
 *  released       int32 [batch][max_blocks_per_req] out  released block ids,
 *                 -1 after the last
 *  released_count int32 [batch] out
 *  status         in/out: requests with non-zero status are skipped;
 *                 TV_ST_BAD_BLOCK / TV_ST_BAD_SIZE (invalid path) are OR-ed in.
 */
int tv_kv_commit(const tv_geom* geom, int32_t batch, const int32_t* accept_path,
                 const int32_t* accept_len, int32_t max_depth, const int32_t* prompt_len,
                 int32_t* block_table, int32_t* n_blocks, int32_t max_blocks_per_req,
                 void* k_cache, void* v_cache, int32_t num_blocks, int32_t* new_len,
                 int32_t* released, int32_t* released_count, int32_t* status, void* stream);

/*
 * tv_greedy_accept followed by tv_kv_commit in one kernel launch (the
 * accepted path stays on chip between the two): the union of their arguments
 * (max_depth is the path capacity, accept_path rows hold max_depth + 1
 * entries), the same outputs and status flags as the two calls in sequence.
 */
int tv_accept_commit(const tv_geom* geom, const int32_t* target_ids, const int32_t* draft_tokens,
                     const int32_t* cu_nodes, const int32_t* next_token,
                     const int32_t* next_sibling, int32_t batch, int32_t max_nodes,
                     int32_t max_depth, int32_t* accept_path, int32_t* accept_len, int32_t* bonus,
                     const int32_t* prompt_len, int32_t* block_table, int32_t* n_blocks,
                     int32_t max_blocks_per_req, void* k_cache, void* v_cache, int32_t num_blocks,
                     int32_t* new_len, int32_t* released, int32_t* released_count,
                     int32_t* status, void* stream);

/* Name of a TV_ERR_* code or of a single TV_ST_* flag. */
const char* tv_status_string(int code);

/* Library interface version (increments when a signature changes). */
int tv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H_ */
