/*
 * eagle.h — C ABI of the GB300 (sm_103a) implementation of one EAGLE-2
 * tree-speculative decoding step.
 *
 * The step has four stages, each an entry point below:
 *   eagle_draft_topk  per-row softmax statistics and top-k of the draft logits
 *   eagle_tree_build  global scores, top-k frontier expansion, top-m rerank,
 *                     node order (and, optionally, the attention mask)
 *   eagle_tree_mask   ancestor-only attention mask from parent pointers
 *   eagle_tree_attn   tree-masked attention of the tree nodes over the KV prefix
 *   eagle_verify      greedy or speculative-sampling verification walk
 * and eagle_step runs the four in order (or replays them as one graph).
 *
 * Sources (the pages the method is taken from):
 *   [EAGLE-2] "論文解説: EAGLE-2 - 動的ドラフトツリーによるLLM推論の高速化"
 *             (0h-n0.github.io, paper 2406.16858)
 *   [EAGLE-1] abeam.tech explainer of "EAGLE: Speculative Sampling Requires
 *             Rethinking Feature Uncertainty" (ICML 2024)
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  Scratch memory is passed in as
 *     `workspace` (size from the matching *_workspace_size query; a size of
 *     0 means the call needs none).  A workspace needs no initialisation and
 *     keeps no state between calls: a call writes every byte of it that it
 *     reads.  One workspace must not be used by two calls that may overlap
 *     on the GPU.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream).  The return value reports argument and launch errors only:
 *     EAGLE_OK, EAGLE_ERR_INVALID (bad argument, nothing launched),
 *     EAGLE_ERR_UNSUPPORTED (valid but not implemented, nothing launched),
 *     EAGLE_ERR_WORKSPACE (workspace too small), EAGLE_ERR_CUDA (a CUDA error
 *     was reported while launching).
 *   - Errors found on the device (inputs outside the documented domain) are
 *     written to an optional device `status` word as a nonzero eagle_status;
 *     the word is never written on success, so the caller zeroes it first.
 *     No kernel traps or aborts.
 *   - Layouts are dense row-major in the index order given, unless a leading
 *     dimension `ld` (in elements) is given.  Pointers to 16-bit or 32-bit
 *     logits and to attention tensors must be 16-byte aligned.
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *eagle_stream_t;

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID = -1,
  EAGLE_ERR_UNSUPPORTED = -2,
  EAGLE_ERR_CUDA = -3,
  EAGLE_ERR_WORKSPACE = -4,
  EAGLE_ERR_TIMEOUT = -5
} eagle_status;

typedef enum { EAGLE_F32 = 0, EAGLE_BF16 = 1 } eagle_dtype;

typedef enum { EAGLE_GREEDY = 0, EAGLE_SAMPLE = 1 } eagle_mode;

/* Human-readable name of a status code (static string, never NULL). */
const char *eagle_status_string(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
int eagle_version(void);

/* ------------------------------------------------------------------------
 * Self test of the bounded device waits (failure detection).
 * The pages describe no failure handling; this call checks the library's
 * own.  Every wait inside the step's kernels (on an mbarrier completed by a
 * copy, an MMA or another CTA of a cluster) gives up after a wall-time
 * limit, and the kernel then reports EAGLE_ERR_TIMEOUT in the status word
 * instead of hanging.  This launches one warp that initialises an mbarrier
 * nothing will ever complete and waits on it with the same helper the
 * kernels use, for `limit_ns` nanoseconds:
 *   which       0: the CTA-local wait; 1: the polling wait used for
 *               barriers that other CTAs of a cluster arrive on
 *   status      device int32 (required): EAGLE_ERR_TIMEOUT when the wait
 *               gave up as designed, EAGLE_ERR_INVALID if it returned as
 *               though the barrier had completed
 *   elapsed_ns  device uint64 (out; may be NULL): the wall time waited
 * Nothing else is in flight, so the context stays usable afterwards.
 * Limits: 1000 <= limit_ns <= 100000000 (1 us to 100 ms).
 * ------------------------------------------------------------------------ */
int eagle_selftest_wait(uint64_t limit_ns, int which, int32_t *status,
                        uint64_t *elapsed_ns, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 1 — draft softmax statistics and top-k.
 * [EAGLE-2] section "ドラフトモデルのキャリブレーション": a draft token's
 * confidence is the probability the draft model assigns it; it approximates
 * the token's acceptance rate.  For each USED row x of the draft logits:
 *   M = max_t x_t,  Z = sum_t exp(x_t - M),
 *   tok[0..k-1] = the k largest logits, in order (ties -> lower token id),
 *   conf[r] = exp(x_tok[r] - M) / Z,  stats = (M, ln Z).
 * Used rows: [b, 0, 0] (the root's distribution) and [b, d, j] for
 * d = 1..D-1, j = 0..k-1 (the j-th expanded node of tree layer d).  Rows
 * [b, 0, 1..k-1] are neither read nor written.
 *
 *   logits  device, dtype `dtype`, row [b, d, j] starts at element
 *           ((b*D + d)*k + j) * ld; 16-byte aligned; V*elemsize and
 *           ld*elemsize multiples of 16 bytes.  Values finite or -inf, at
 *           least k finite per used row, no NaN.
 *   tok     device int32 [B, D, k, k]     (out)
 *   conf    device float [B, D, k, k]     (out)
 *   stats   device float [B, D, k, 2]     (out; may be NULL)
 *   status  device int32 (out; may be NULL): EAGLE_ERR_TIMEOUT if the
 *           bounded wait of a row's merge gave up (the row is then not
 *           written)
 * Workspace: none (the size is 0); a row split over several CTAs merges
 * through the shared memory of their thread-block cluster.
 * Limits: 1 <= k <= 32, k <= V, D >= 1, B >= 1.
 * ------------------------------------------------------------------------ */
size_t eagle_draft_topk_workspace_size(int B, int D, int k, int V);

int eagle_draft_topk(const void *logits, int dtype, int B, int D, int k, int V,
                     int64_t ld, int32_t *tok, float *conf, float *stats,
                     int32_t *status, void *workspace, size_t workspace_bytes,
                     eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 2 — dynamic draft tree.
 * [EAGLE-2] section "動的ドラフトツリーの構築アルゴリズム": V_i = product of
 * the confidences on the root path (V_i equation); at every depth the k
 * nodes with the largest V are expanded with their own top-k tokens; the m
 * candidates with the largest V are kept; ancestors are added so the set is
 * a connected tree.
 * Computation (exactly): root = gid 0, V = 1.  Depth-1 candidates are the
 * root row's tokens (gids 1..k).  For d = 1..D-1 the k depth-d candidates
 * greatest in the key order (V desc, parent gid asc, token asc) are the
 * expanded set E_d; E_d[j] takes row [d, j]; its children get
 * V = fl32(V_parent * conf) (IEEE float multiply, round to nearest, no
 * flush to zero) and gids numbered depth by depth, by j, then by child rank.
 * The m candidates greatest in key order are kept.  With 0 <= conf <= 1 every
 * ancestor precedes its descendants in key order, so the kept set is
 * already connected (the ancestor step adds nothing).
 * Output order: node 0 = root, nodes 1..m = kept candidates in key order, so
 * parent index < node index.
 *
 *   tok, conf    device int32 / float [B, D, k, k], as written by stage 1
 *                (tokens of one row distinct, 0 <= token < 2^20,
 *                 0 <= conf <= 1)
 *   root_tok     device int32 [B] or NULL (root token reported as -1)
 *   node_tok     device int32 [B, m+1]  (out)
 *   node_parent  device int32 [B, m+1]  (out; root -1)
 *   node_depth   device int32 [B, m+1]  (out; may be NULL)
 *   node_score   device float [B, m+1]  (out; V; may be NULL)
 *   node_src     device int32 [B, m+1]  (out; candidate gid; may be NULL)
 *   node_row     device int32 [B, m+1]  (out; d*k + j if the node was
 *                expanded with row [d, j], root 0, else -1; may be NULL)
 *   mask         device uint64 [B, m+1, W], W = ceil((m+1)/64) (out; may be
 *                NULL) — the same words eagle_tree_mask writes
 *   status       device int32 (out; may be NULL): EAGLE_ERR_INVALID when a
 *                token or confidence is outside its range above.  Repeated
 *                tokens within a row are not checked (stage 1 never writes
 *                them): the tree is then unspecified, but every output
 *                index stays in range and nothing is read or written out of
 *                bounds.
 * Limits: 1 <= k <= 32, D >= 1, 1 <= m <= k + (D-1)k^2 <= 4095.
 * ------------------------------------------------------------------------ */
int eagle_tree_build(const int32_t *tok, const float *conf, int B, int D, int k,
                     int m, const int32_t *root_tok, int32_t *node_tok,
                     int32_t *node_parent, int32_t *node_depth,
                     float *node_score, int32_t *node_src, int32_t *node_row,
                     uint64_t *mask, int32_t *status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 2, ablation variants of the tree build.
 * [EAGLE-2] section "実験結果", ablation table: the method without the global
 * acceptance probability ("confidence only") and without reranking.  Same
 * arguments, outputs and limits as eagle_tree_build, plus `flags`, a bitwise
 * OR of:
 *   EAGLE_TREE_CONFIDENCE_ONLY  rank a candidate by its own confidence c
 *       instead of V (node_score then holds c).  The expansion takes each
 *       layer's k greatest keys as before; the rerank grows the tree
 *       best-first, repeatedly adding the greatest key whose parent is
 *       already in the tree (with V keys this is exactly the top-m set), so
 *       node order is the order of selection and every parent precedes its
 *       children.
 *   EAGLE_TREE_NO_RERANK  no rerank: the tree is the layers' selections
 *       E_1, E_2, ..., E_D (each layer's k greatest keys; E_D chosen the
 *       same way although never expanded), in depth order and rank order
 *       within a depth, truncated to m nodes.  Requires m <= D*k.
 * flags = 0 is eagle_tree_build.  Other bits: EAGLE_ERR_INVALID.
 * ------------------------------------------------------------------------ */
#define EAGLE_TREE_CONFIDENCE_ONLY 1
#define EAGLE_TREE_NO_RERANK 2
int eagle_tree_build_variant(const int32_t *tok, const float *conf, int B, int D,
                             int k, int m, int flags, const int32_t *root_tok,
                             int32_t *node_tok, int32_t *node_parent,
                             int32_t *node_depth, float *node_score,
                             int32_t *node_src, int32_t *node_row,
                             uint64_t *mask, int32_t *status,
                             eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 2 for the EAGLE-1 static draft tree.
 * [EAGLE-2] sections "背景" and "EAGLE-1からの変更点": EAGLE-1 places its draft
 * tokens on a tree shape fixed in advance and applies it to every input;
 * only the tokens come from the draft.  The shape is an input template:
 *   tree_parent  device int32 [n]: -1 for node 0 (the root), else the parent
 *                index, which must be smaller than the node's own
 *   tree_rank    device int32 [n]: node i is the tree_rank[i]-th of its
 *                parent's top-k draft tokens (0 <= rank < k, distinct among
 *                siblings; entry 0 ignored)
 * Draft rows: the root's distribution is row [0, 0]; the j-th node of depth
 * d >= 1 that has children (in node order) uses row [d, j], so a depth may
 * hold at most k such nodes and none at depth D.  Inputs tok/conf/root_tok
 * and the outputs are those of eagle_tree_build with m = n - 1: node order is
 * the template's, node_src = the template index, node_score = the float32
 * product of the confidences on the root path, node_row = d*k + j for nodes
 * with children (root 0), else -1; mask optional.
 * Device errors: a template that breaks the rules above sets
 * EAGLE_ERR_INVALID in *status (when given) and leaves the outputs unwritten.
 * Limits: 1 <= k <= 32, 1 <= D <= 32, 1 <= n <= 1024.
 * ------------------------------------------------------------------------ */
int eagle_static_tree(const int32_t *tok, const float *conf, int B, int D, int k,
                      const int32_t *tree_parent, const int32_t *tree_rank, int n,
                      const int32_t *root_tok, int32_t *node_tok,
                      int32_t *node_parent, int32_t *node_depth,
                      float *node_score, int32_t *node_src, int32_t *node_row,
                      uint64_t *mask, int32_t *status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Ancestor-only attention mask.
 * [EAGLE-2] section "注意マスクの調整": each token attends only to its
 * ancestors.  Bit (j % 64) of word j / 64 of row i is set iff j == i or j is
 * an ancestor of i (the root is an ancestor of every node).
 *   node_parent  device int32 [B, n] (root -1, parent index < node index)
 *   mask         device uint64 [B, n, ceil(n/64)] (out)
 * Limits: 1 <= n <= 4096.
 * ------------------------------------------------------------------------ */
int eagle_tree_mask(const int32_t *node_parent, int B, int n, uint64_t *mask,
                    eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 3 — tree attention.
 * [EAGLE-1] sections "用語解説" (Tree Attention) and "Tree Attention の役割":
 * the target scores every branch of the tree in one forward pass; with the
 * [EAGLE-2] mask each tree node attends to the prefix and to its own
 * ancestors.  For node i (0..n-1, n = m+1), query head h, KV head
 * g = h / (Hq/Hkv):
 *   keys = k_cache[b, g, 0:kv_len[b]]  ++  { k_tree[b, g, j] : mask bit j of row i }
 *   s = scale * <q[b, i, h], key>,  out[b, i, h] = softmax(s) . values,
 *   lse[b, i, h] = ln sum exp(s).
 *   q          [B, n, Hq, dh]        dtype
 *   k_cache    [B, Hkv, Lmax, dh]    dtype   (v_cache alike)
 *   kv_len     device int32 [B], 0 <= kv_len[b] <= Lmax
 *   k_tree     [B, Hkv, n, dh]       dtype   (v_tree alike)
 *   mask       device uint64 [B, n, ceil(n/64)] (as eagle_tree_mask writes)
 *   out        [B, n, Hq, dh]        dtype   (out)
 *   lse        device float [B, n, Hq]  (out; may be NULL)
 *   status     device int32 (out; may be NULL): EAGLE_ERR_TIMEOUT if a
 *              bounded wait inside the kernel gave up
 * Arithmetic: fp32 accumulation and softmax.  bf16 inputs run on the tensor
 * cores (tcgen05, operands staged by TMA, accumulators in tensor memory,
 * probabilities rounded to bf16 for the P.V product); fp32 inputs run on the
 * CUDA cores.  Cache rows at or beyond kv_len[b] are never read; every row
 * of k_tree / v_tree must hold finite values.
 * Workspace (bf16): a launch that splits the KV prefix of a head over
 * several CTAs needs one slot per CTA (fp32 O rows and (m, l) per row); each
 * CTA leaves its partial results there.  When every CTA of the launch is
 * resident at once (one wave) the splits of a head are one thread-block
 * cluster and merge from L2 after a cluster barrier; otherwise a second
 * kernel merges them.  An unsplit launch needs none (size 0).  fp32:
 * partial results and weights.
 * Limits: Hq % Hkv == 0, dh in {64, 128}, 1 <= n <= 4096, B*Hkv <= 65535.
 * ------------------------------------------------------------------------ */
size_t eagle_tree_attn_workspace_size(int dtype, int B, int n, int Hq, int Hkv,
                                      int dh, int Lmax);

/* Kernels one eagle_tree_attn call with these arguments launches (1 or 2:
 * the attention, and the merge of a split launch of several waves, or the
 * fp32 combine); 0 for invalid arguments.  Host only. */
int eagle_tree_attn_kernel_count(int dtype, int B, int n, int Hq, int Hkv,
                                 int dh, int Lmax);

int eagle_tree_attn(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *kv_len, const void *k_tree,
                    const void *v_tree, const uint64_t *mask, int dtype, int B,
                    int n, int Hq, int Hkv, int dh, int Lmax, float scale,
                    void *out, float *lse, int32_t *status, void *workspace,
                    size_t workspace_bytes, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 3 over a paged KV prefix (block-table attention).
 * Same computation as eagle_tree_attn; the prefix K/V live in page pools
 *   k_pages, v_pages  bf16 [num_pages, Hkv, page_size, dh]
 *   block_table       device int32 [B, max_pages]: logical page p of
 *                     sequence b is physical page block_table[b, p]
 * so prefix position L of sequence b is row L % page_size of page
 * block_table[b, L / page_size] (entries for pages at or beyond kv_len are
 * not read).  kv_len[b] is clamped to max_pages * page_size.  Other
 * arguments as in eagle_tree_attn.  Workspace from
 * eagle_tree_attn_paged_workspace_size.
 * Device errors: a block-table entry outside [0, num_pages) for a page the
 * prefix uses sets EAGLE_ERR_INVALID (page 0 is read in its place).
 * Limits: bf16 only (other dtypes EAGLE_ERR_UNSUPPORTED); dh in {64, 128};
 * page_size a power of two in [16, 4096]; max_pages * page_size <= 2^24.
 * ------------------------------------------------------------------------ */
size_t eagle_tree_attn_paged_workspace_size(int dtype, int B, int n, int Hq,
                                            int Hkv, int dh, int max_pages,
                                            int page_size);

int eagle_tree_attn_paged(const void *q, const void *k_pages,
                          const void *v_pages, const int32_t *block_table,
                          int max_pages, int page_size, int num_pages,
                          const int32_t *kv_len, const void *k_tree,
                          const void *v_tree, const uint64_t *mask, int dtype,
                          int B, int n, int Hq, int Hkv, int dh, float scale,
                          void *out, float *lse, int32_t *status,
                          void *workspace, size_t workspace_bytes,
                          eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 4 — verification walk.
 * [EAGLE-1] section "検証方法": each draft token is accepted or rejected by
 * the ratio of target and draft distributions; after a rejection the rest is
 * discarded and a token resampled; the output follows the target exactly
 * ([EAGLE-2]: lossless, rejection sampling as in EAGLE-1; temp=0 greedy).
 * Row i of the target logits is the target's distribution after node i.
 *   GREEDY: from the root, a = argmax of the current row (ties -> lower
 *     token); move to the child carrying a while one exists; a is the bonus.
 *   SAMPLE (temperature T > 0): children are point-mass drafts.  With
 *     e_t = exp(x_t/T - max), Z = sum e, S = tokens rejected at this node:
 *     child x (token t) is accepted iff u[b,x,0] * (Z - sum_S e) < e_t;
 *     otherwise t joins S.  With no child accepted, the bonus is the
 *     smallest t not in S whose cumulative residual mass exceeds
 *     u[b,cur,1] * (Z - sum_S e).  Children are tried in node-index order.
 *   target     dtype, row (b, i) starts at element (b*(m+1) + i) * ld
 *   node_tok, node_parent   device int32 [B, m+1] (as stage 2 writes)
 *   uniforms   device float [B, m+1, 2] in [0, 1) (SAMPLE; NULL for GREEDY)
 *   accept_len device int32 [B]            (out; accepted draft tokens)
 *   path_nodes device int32 [B, D+1]       (out; root first; -1 padded)
 *   out_tokens device int32 [B, D+1]       (out; accepted tokens, then the
 *                                           bonus token; -1 padded)
 *   status     device int32 (out; may be NULL): EAGLE_ERR_INVALID when the
 *              walk meets a row with no finite logit (greedy: no argmax) or
 *              with no residual mass (sampling), or a child token outside
 *              [0, V) (sampling); the bonus token is then -1
 * D bounds the tree depth.  Limits: V*elemsize and ld*elemsize multiples of
 * 16 bytes; 1 <= m+1 <= 4096; D >= 1.
 * ------------------------------------------------------------------------ */
size_t eagle_verify_workspace_size(int B, int m, int V);

int eagle_verify(const void *target, int dtype, int64_t ld,
                 const int32_t *node_tok, const int32_t *node_parent, int B,
                 int m, int D, int V, int mode, float temperature,
                 const float *uniforms, int32_t *accept_len,
                 int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                 void *workspace, size_t workspace_bytes,
                 eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 4 without caller scratch: eagle_verify_noalloc.
 * The paper has no counterpart to this entry point.  It serves callers that
 * cannot allocate device memory for a workspace: a plugin or custom-op hook
 * inside a host runtime that owns every device buffer and hands the op only
 * its inputs and outputs; a serving loop that must not call cudaMalloc once
 * it is running (cudaMalloc can synchronise the device and stall the work
 * in flight); a process whose device memory is all handed to its own pool.
 * Same arguments, results and device errors as eagle_verify, without the
 * workspace arguments.  The per-chunk statistics records that eagle_verify
 * keeps in its workspace live instead in one array inside the library
 * (a file-scope __device__ array of EAGLE_VERIFY_NOALLOC_SCRATCH_BYTES
 * bytes), which every GPU that loads the library holds until the process
 * exits.  Nothing is allocated by the call itself.
 *   - A request whose records exceed the array (eagle_verify_workspace_size
 *     > EAGLE_VERIFY_NOALLOC_SCRATCH_BYTES) returns EAGLE_ERR_WORKSPACE and
 *     launches nothing.  8 MiB covers B * (m+1) * ceil(V/2048) <= 524288
 *     records, e.g. B = 64, m = 60, V = 201088.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and keeps it; make that first call before any
 *     stream capture.
 *   - Every call shares the one array, and it keeps the last call's
 *     records.  No record needs clearing: each call writes every record it
 *     reads.  Two calls that may overlap on the GPU (on different streams
 *     without an ordering between them, or on one device from two threads
 *     through unordered streams) race on the array and give wrong results.
 * ------------------------------------------------------------------------ */
#define EAGLE_VERIFY_NOALLOC_SCRATCH_BYTES (8u << 20)

int eagle_verify_noalloc(const void *target, int dtype, int64_t ld,
                         const int32_t *node_tok, const int32_t *node_parent,
                         int B, int m, int D, int V, int mode,
                         float temperature, const float *uniforms,
                         int32_t *accept_len, int32_t *path_nodes,
                         int32_t *out_tokens, int32_t *status,
                         eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * Stage 4 with draft distributions — speculative-sampling verification of a
 * tree whose tokens were drawn from the draft's distribution q.
 * [EAGLE-1] section "検証方法": a drafted token t is accepted with
 * probability min(1, p(t)/q(t)); after a rejection the target distribution is
 * replaced by the residual norm(max(0, p - q)) and a token is finally drawn
 * from it, so the output follows the target exactly.  Tree form: at node cur
 * the children (node-index order, all drafted from q = softmax(draft row of
 * cur / T)) are tested in turn against the current residual R = max(0, p -
 * C q) with normaliser S (C = 0, S = 1 before any rejection; a rejection
 * adds S to C and S becomes sum over the vocabulary of the new R):
 *   child x with token t is accepted iff u[b,x,0] * S * q(t) < R(t);
 * with no child accepted (or at a leaf) the bonus is the smallest token
 * whose cumulative R exceeds u[b,cur,1] * sum(R).  A residual that sums to 0
 * is replaced by p.  p = softmax(target row / T).
 *   target     dtype, row (b, i) at element (b*(m+1) + i) * ld_t
 *   draft      dtype, draft logits [B, D, k, V], row (b, d, j) at element
 *              ((b*D + d)*k + j) * ld_d (the rows eagle_draft_topk reads)
 *   node_tok, node_parent, node_row   device int32 [B, m+1] as stage 2
 *              writes them; node_row[b, i] = d*k + j names the draft row of
 *              every node that has children
 *   uniforms   device float [B, m+1, 2] in [0, 1)
 *   accept_len, path_nodes, out_tokens, status   as in eagle_verify
 * No workspace: the CTAs of a sequence (one thread-block cluster of up to
 * 8, each over a slice of the vocabulary) keep their state in shared memory
 * and exchange their partial sums through distributed shared memory.
 * Device errors: a node with children whose node_row is outside [0, D*k),
 * a token outside [0, V) or no residual mass set EAGLE_ERR_INVALID.
 * Limits: temperature > 0; V*elemsize, ld_t*elemsize and ld_d*elemsize
 * multiples of 16 bytes; 16-byte aligned logits; 1 <= m+1 <= 4096;
 * 1 <= D; 1 <= k <= 32; B <= 65535 (else EAGLE_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------ */
int eagle_verify_draft(const void *target, const void *draft, int dtype,
                       int64_t ld_t, int64_t ld_d, const int32_t *node_tok,
                       const int32_t *node_parent, const int32_t *node_row,
                       int B, int m, int D, int k, int V, float temperature,
                       const float *uniforms, int32_t *accept_len,
                       int32_t *path_nodes, int32_t *out_tokens,
                       int32_t *status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * After verification — commit the accepted path's keys and values.
 * [EAGLE-1] section "検証方法" / [EAGLE-2]: the accepted draft tokens become
 * part of the sequence; everything after a rejection is discarded.  The
 * root's K/V is already the last prefix position.  For each sequence b with
 * a = accept_len[b], nodes path_nodes[b, 1..a] (as eagle_verify writes them)
 * have their rows of k_tree/v_tree [B, Hkv, n, dh] copied, in path order, to
 * positions kv_len[b] .. kv_len[b]+a-1 of the cache, and kv_len[b] becomes
 * kv_len[b] + a (updated in place).
 *   cache        block_table == NULL: contiguous k_cache/v_cache
 *                [B, Hkv, Lmax, dh]; otherwise page pools [num_pages, Hkv,
 *                page_size, dh] addressed through block_table [B, max_pages]
 *                (the caller has mapped the pages the new positions need)
 *   slot_mapping device int32 [B, n] (out, may be NULL): node i's position
 *                after the commit (root kv_len-1), -1 for nodes not kept
 * Device errors: a path node outside [1, n), a = accept_len outside [0, D],
 * kv_len < 1, or new positions beyond the cache (Lmax, or an unmapped page)
 * set EAGLE_ERR_INVALID and leave that sequence unchanged.
 * Limits: dh*elemsize a multiple of 16 bytes; 1 <= D <= 64; n <= 4096; page
 * rules as for eagle_tree_attn_paged.
 * ------------------------------------------------------------------------ */
int eagle_kv_commit(const void *k_tree, const void *v_tree, int dtype, int B,
                    int n, int Hkv, int dh, const int32_t *accept_len,
                    const int32_t *path_nodes, int D, void *k_cache,
                    void *v_cache, int Lmax, const int32_t *block_table,
                    int max_pages, int page_size, int num_pages,
                    int32_t *kv_len, int32_t *slot_mapping, int32_t *status,
                    eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole step in one call, and as one recorded graph.
 * [EAGLE-2] section "動的ドラフトツリーの構築アルゴリズム" (draft confidences,
 * then the tree), [EAGLE-1] sections "Tree Attention の役割" (the target
 * scores the tree in one pass) and "検証方法" (then verification): the
 * stages run in that order, each on the previous one's results:
 *   eagle_draft_topk -> eagle_tree_build (with the mask) -> eagle_tree_attn
 *   -> eagle_verify
 * on one stream, each kernel chained to the previous one.  The target
 * logits are an input: the target's layers between the attention and its
 * logits are not part of the library.
 *
 * eagle_step_args names every buffer of the four calls; each field means
 * what the argument of the same name means there (n = m + 1 tree nodes):
 *   draft_logits, draft_ld            eagle_draft_topk's logits, ld
 *   tok, conf, stats                  its outputs (stats may be NULL)
 *   root_tok, node_tok ... node_row   eagle_tree_build's (root_tok,
 *                                     node_depth, node_score, node_src and
 *                                     node_row may be NULL)
 *   mask                              required: the attention reads it
 *   q, k_cache, v_cache, kv_len, k_tree, v_tree, scale, attn_out, lse
 *                                     eagle_tree_attn's (attn_out is its
 *                                     `out`; lse may be NULL)
 *   target, target_ld, uniforms, accept_len, path_nodes, out_tokens
 *                                     eagle_verify's (uniforms only for
 *                                     EAGLE_SAMPLE)
 *   status                            one word shared by every stage (may
 *                                     be NULL)
 * dtype applies to the draft logits, the attention tensors and the target
 * logits alike.
 * ------------------------------------------------------------------------ */
typedef struct eagle_step_args {
  int dtype;
  int B, D, k, m, V;
  int Hq, Hkv, dh, Lmax;
  int mode;
  float temperature;
  float scale;
  const void *draft_logits;
  int64_t draft_ld;
  int32_t *tok;
  float *conf;
  float *stats;
  const int32_t *root_tok;
  int32_t *node_tok, *node_parent, *node_depth;
  float *node_score;
  int32_t *node_src, *node_row;
  uint64_t *mask;
  const void *q, *k_cache, *v_cache;
  const int32_t *kv_len;
  const void *k_tree, *v_tree;
  void *attn_out;
  float *lse;
  const void *target;
  int64_t target_ld;
  const float *uniforms;
  int32_t *accept_len, *path_nodes, *out_tokens;
  int32_t *status;
} eagle_step_args;

/* Bytes of the one workspace a step needs (the stages' workspaces, each at
 * a 256-byte aligned offset); 0 for invalid arguments.  Host only. */
size_t eagle_step_workspace_size(const eagle_step_args *args);

/* The four calls in order on `stream`.  Returns the first nonzero status
 * of a call (the calls after it are not made); the arguments of each call
 * are checked by that call. */
int eagle_step(const eagle_step_args *args, void *workspace,
               size_t workspace_bytes, eagle_stream_t stream);

/* A step recorded once into a CUDA graph; each launch replays all of its
 * kernels with one call.  The graph holds the buffers' addresses (and the
 * tensor maps built from them), so every buffer and the workspace must stay
 * allocated, at the same address, until the graph is destroyed; their
 * contents (inputs, kv_len) may change between launches.
 * eagle_step_graph_create first runs the step once on a stream of its own
 * (work that produces the inputs on other streams must have completed) and
 * waits for it (one-time kernel set-up happens outside the recording; the
 * outputs are then those of that run), then records the step on that
 * stream (capture mode local to the calling thread) and instantiates the
 * graph.  Unlike the other calls it allocates (the stream and the graph)
 * and synchronises; the launches do neither.  On failure *graph is NULL.
 * Destroy a graph only after the launches made with it have completed. */
typedef struct eagle_step_graph_s *eagle_step_graph_t;

int eagle_step_graph_create(const eagle_step_args *args, void *workspace,
                            size_t workspace_bytes, eagle_step_graph_t *graph);
int eagle_step_graph_launch(eagle_step_graph_t graph, eagle_stream_t stream);
int eagle_step_graph_destroy(eagle_step_graph_t graph);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE_H */
