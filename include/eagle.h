/*
 * eagle.h -- C-ABI of the GB300 (sm_103a) EAGLE speculative-decoding hot path.
 *
 * One tree-verify round of EAGLE-family speculative decoding is served by
 * six calls (plus eagle_lmhead_verify_stats / eagle_tree_verify_stats, which
 * serve stochastic verification without materialised logits, eagle_tree_commit
 * which publishes the accepted path, and the drafter step: eagle_draft_input,
 * the token-embedding input FC, and eagle_draft_layer, its decoder layer,
 * built on eagle_linear):
 *   eagle_fuse_proj             EAGLE-3 fused feature g = W_proj [h_low; h_mid; h_high]
 *   eagle_tree_attn             tree-masked attention vs a paged KV cache + the tree rows
 *   eagle_lmhead_topk           LM-head GEMM with fused per-row top-k and log-softmax
 *   eagle_tree_expand           one EAGLE-2 dynamic-tree expansion step
 *                               (eagle_tree_expand_static: one depth of a fixed EAGLE-1 tree)
 *   eagle_tree_expand_finalize  EAGLE-2 global rerank + flatten (rows, mask, positions)
 *   eagle_tree_verify           lossless verification (greedy / rejection sampling)
 *
 * Sources (web pages cited by title and section):
 *   [E3]   "EAGLE-3: Scaling up Inference Acceleration of Large Language Models
 *          via Training-Time Test" (paper summary)
 *   [E1]   "EAGLE: Speculative Sampling Requires Rethinking Feature Uncertainty"
 *          (paper summary)
 *   [M7.5] "M7.5 - EAGLE Feature Drafting: Uncertainty, Dynamic Trees, HASS,
 *          and EAGLE-3"
 *   [BLOG] "EAGLE-3: Why the Best Draft Models Stopped Predicting Features"
 *
 * Conventions shared by every call
 *   - All array arguments are DEVICE pointers to contiguous row-major arrays
 *     owned by the caller.  The library never allocates or frees memory;
 *     scratch space comes from a caller buffer `ws` of at least the size
 *     returned by the matching *_workspace_size() query.
 *   - Matrix operands read by TMA (weights, activations) must be 16-byte
 *     aligned; leading dimensions are given by the shapes.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous, never synchronise, keep no state between calls, and may be
 *     issued from several host threads on different streams and buffers.
 *   - Kernels are launched with programmatic stream serialization: one may be
 *     scheduled while the previous kernel on the stream is finishing, but it
 *     reads and writes no global memory before that kernel has completed, so
 *     stream order is unchanged for the caller -- with one exception: the
 *     weight matrices (w_lm of the LM-head calls, w_proj of eagle_fuse_proj,
 *     w_in of eagle_draft_input) may be read earlier.  They are constants of
 *     the model; do not write them with a kernel on the same stream right
 *     before the call.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned as eagle_status.  Errors that only the device can see (a
 *     malformed tree, a non-finite value, a timed-out wait) are written to the
 *     optional `dev_status` word (first error wins; 0 = OK); pass NULL to skip.
 *     A timed-out wait never hangs the device: the kernel records
 *     EAGLE_ERR_TIMEOUT, drains its in-flight copies, frees its tensor memory
 *     and returns.
 */
#ifndef EAGLE_GB300_EAGLE_H
#define EAGLE_GB300_EAGLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum ...     */
  EAGLE_ERR_UNSUPPORTED = 2, /* shape or dtype outside the kernels' limits     */
  EAGLE_ERR_WORKSPACE = 3,   /* ws too small or misaligned                      */
  EAGLE_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed     */
  EAGLE_ERR_BAD_TREE = 5,    /* device: non-topological parents, duplicate
                                sibling token, sibling mass > 1, too deep      */
  EAGLE_ERR_BAD_KV = 6,      /* device: page id out of range                    */
  EAGLE_ERR_NONFINITE = 7,   /* device: NaN / +inf where a probability is read */
  EAGLE_ERR_TIMEOUT = 8      /* device: a bounded wait ran out                  */
} eagle_status;

typedef enum { EAGLE_FP32 = 0, EAGLE_BF16 = 1 } eagle_dtype;

typedef enum {
  EAGLE_PROPOSAL_DETERMINISTIC = 0, /* children are deterministic top-k       */
  EAGLE_PROPOSAL_SAMPLED = 1        /* children are i.i.d. draws from q       */
} eagle_proposal;

/* Human-readable name of a status code (static string). */
const char* eagle_status_string(int status);

/* Synchronises `stream`, copies *dev_status to *host_status and returns it
 * as an eagle_status (test helper; the only call that synchronises). */
int eagle_read_status(const int32_t* dev_status, void* stream, int32_t* host_status);

/* Number of kernels this library has launched in this process (counter for
 * benchmarks; incremented on every launch, never reset). */
uint64_t eagle_launch_count(void);

/* Self-test of the bounded waits (no counterpart in the pages): launches one
 * CTA whose thread 0 waits on an mbarrier that nothing ever completes, with a
 * limit of `limit_us` microseconds (1 .. 1,000,000), through the same bounded
 * wait every kernel of the library uses.  Expected device result:
 * dev_status[0] = EAGLE_ERR_TIMEOUT (the wait gave up) and dev_status[1] = 1
 * (a second waiter of the CTA, on the ordinary 2 s limit, ended early through
 * the abort flag the first one raised).  dev_status: [2] int32, zeroed by the
 * caller.  The device stays usable; nothing else is touched. */
int eagle_selftest_wait_timeout(unsigned int limit_us, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_fuse_proj -- EAGLE-3 multi-layer feature fusion.
 *   g[i, o] = sum_c W[o, c] h_low[i, c] + W[o, d+c] h_mid[i, c]
 *             + W[o, 2d+c] h_high[i, c]  (+ bias[o])
 * [E3] section 3.4 "Change 2: The fusion FC layer" (concatenate l, m, h into
 * 3k and project back to k; bias optional); [M7.5] section 0x08B
 * "Multi-Layer Feature Fusion" (r_t = W_R [f_low; f_mid; f_high],
 * W_R in R^{d x 3d}); [BLOG] "What EAGLE-3 changes" (g_t = W_proj @ concat).
 *
 *   h_low, h_mid, h_high : [M, d]   activations of dtype `dtype`
 *   w_proj               : [d, 3d]  row o = output feature o (out x in)
 *   bias                 : [d] fp32, or NULL
 *   g                    : [M, d]   output, dtype `dtype`
 * The concatenation is never materialised: the K loop walks the three inputs.
 * bf16 runs on the tensor cores with fp32 accumulation; fp32 runs on the CUDA
 * cores in exact fp32 arithmetic.
 * Limits: 1 <= M <= 4096, d % 128 == 0, d <= 16384.
 * ---------------------------------------------------------------------- */
size_t eagle_fuse_proj_workspace_size(int M, int d, int dtype);
int eagle_fuse_proj(const void* h_low, const void* h_mid, const void* h_high,
                    const void* w_proj, const float* bias, void* g, int M, int d,
                    int dtype, void* ws, size_t ws_bytes, int32_t* dev_status,
                    void* stream);

/* ------------------------------------------------------------------------
 * eagle_fuse_proj_accepted -- the fusion of eagle_fuse_proj over the accepted
 * rows only.
 * [M7.5] section 0x05D "Feature And KV Commit" (only the verified path is
 * published: its target features are gathered for the next draft round, every
 * other tree row is discarded); [E3] "Stage 2: Verification" with section 3.4
 * "Change 2: The fusion FC layer" (the next round's drafter input is the fused
 * feature of those rows).  The accepted rows of request b are
 * path_rows[b, 0 .. accept_len[b]] in path order -- the rows
 * eagle_tree_commit publishes.
 *   g[b, j, :] = W_proj [h_low[r]; h_mid[r]; h_high[r]] (+ bias),
 *                r = b * R + path_rows[b, j], for j <= accept_len[b];
 *   g[b, j, :] = 0 for accept_len[b] < j <= max_depth.
 *
 *   h_low, h_mid, h_high : [B*R, d] verify-row features, dtype `dtype`
 *   w_proj, bias         : as eagle_fuse_proj
 *   path_rows, accept_len: outputs of eagle_tree_verify ([B, max_depth+1], [B])
 *   g                    : [B, max_depth+1, d] output, dtype `dtype`
 * bf16: a gather kernel packs the accepted rows (and their output slots) into
 * `ws`, and the tensor-core projection runs on the packed rows only: its
 * stream-K split is planned on the device from the accepted-row count, so
 * rejected tree rows cost neither weight traffic nor MMAs.  fp32: CUDA cores,
 * exact fp32.  Unlike eagle_fuse_proj, w_proj is not read before the previous
 * kernel on the stream has completed.
 * Device-detected: accept_len[b] outside [0, max_depth] or a path row outside
 * [0, R) -> EAGLE_ERR_BAD_TREE; that request projects no row (all its slots
 * are zeroed).
 * Limits: B * (max_depth + 1) <= 4096, d % 128 == 0, d <= 16384; 16-byte
 * aligned arrays.
 * ---------------------------------------------------------------------- */
size_t eagle_fuse_proj_accepted_workspace_size(int B, int max_depth, int d, int dtype);
int eagle_fuse_proj_accepted(const void* h_low, const void* h_mid, const void* h_high,
                             const void* w_proj, const float* bias, const int32_t* path_rows,
                             const int32_t* accept_len, int B, int R, int max_depth, int d,
                             int dtype, void* g, void* ws, size_t ws_bytes, int32_t* dev_status,
                             void* stream);

/* ------------------------------------------------------------------------
 * eagle_draft_input -- drafter input FC with the token-embedding lookup fused.
 *   u[i, o] = sum_c W[o, c] r[i, c] + W[o, d+c] embed[token_ids[i], c]
 *             (+ bias[o])
 * [M7.5] section 0x08B (u_t = W_I [r_t; e(x_{t+1})], W_I in R^{d x 2d}: the
 * fused state joined with the embedding of the sampled token); [E3] section
 * 3.4 "Input projection FC layer" ([g; e] in R^{2k} projected back to k);
 * [E1] "Draft Model Architecture" (FC layer with bias over [f; e], embedding
 * table frozen from the target model); [M7.5] section 0x03 "EAGLE-1 Tensor
 * Path" (u_t = W_F c_t + b_F).
 *
 *   r         : [M, d]      fused feature (or the drafter's own output a_t at
 *                           drafted positions), dtype `dtype`
 *   token_ids : [M] int32   token per row, in [0, vocab)
 *   embed     : [vocab, d]  token-embedding table, dtype `dtype`
 *   w_in      : [d, 2d]     row o = output feature o (out x in)
 *   bias      : [d] fp32, or NULL
 *   u         : [M, d]      output, dtype `dtype`
 * The concatenation is never materialised: a lookup kernel over all SMs
 * copies the M embedding rows into `ws`, and the K loop of the tensor-core
 * projection then reads r and those rows through two tensor maps (weights
 * stream as in eagle_fuse_proj).  bf16 runs on the tensor cores with fp32
 * accumulation; fp32 on the CUDA cores in exact fp32 arithmetic, where the
 * lookup is fused into the dot products.
 * Device-detected: a token id outside [0, vocab) -> EAGLE_ERR_BAD_TREE (that
 * row's embedding half reads as zeros).  w_in may be read before the previous
 * kernel on the stream has completed (see the conventions above).
 * Limits: 1 <= M <= 4096, d % 128 == 0, d <= 16384.
 * ---------------------------------------------------------------------- */
size_t eagle_draft_input_workspace_size(int M, int d, int dtype);
int eagle_draft_input(const void* r, const int32_t* token_ids, const void* embed, int vocab,
                      const void* w_in, const float* bias, void* u, int M, int d, int dtype,
                      void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_linear -- y = x W^T (+ bias) (+ residual): the weight-streaming
 * tensor-core projection of eagle_fuse_proj for one input of any width.
 * The projections of the drafter's decoder layer ([E3] section 3.4 "The
 * transformer decoder layer") are made of it.
 *
 *   x        : [M, k_in]      activations, dtype `dtype` (must not alias y)
 *   w        : [n_out, k_in]  weights (out x in)
 *   bias     : [n_out] fp32, or NULL
 *   residual : [M, n_out] dtype `dtype` added to the result, or NULL; may be y
 *   y        : [M, n_out]
 * bf16 on the tensor cores (fp32 accumulation, stream-K over the SMs), fp32
 * on the CUDA cores in exact fp32.  w may be read before the previous kernel
 * on the stream has completed (see the conventions above).
 * Limits: 1 <= M <= 4096, n_out % 128 == 0, k_in % 64 == 0, both <= 65536.
 * ---------------------------------------------------------------------- */
size_t eagle_linear_workspace_size(int M, int n_out, int k_in, int dtype);
int eagle_linear(const void* x, const void* w, const float* bias, const void* residual, void* y,
                 int M, int n_out, int k_in, int dtype, void* ws, size_t ws_bytes,
                 int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_attn -- attention of the tree rows against the committed prefix
 * (read through a page table) plus the visible tree rows.
 *   For tree row r of request b and query head h (kv head h / (Hq/Hkv)):
 *     keys = prefix tokens 0..ctx_lens[b]-1 followed by tree rows j whose bit
 *            j is set in tree_mask[b, r];
 *     out[b, r, h] = softmax(scale * q k^T) v over those keys;
 *     lse[b, r, h] = natural-log sum of exp(scale * q k^T) over those keys.
 * [M7.5] section 0x08C "Training-Time Test": A(u, v) = 1 iff v is in
 * TargetPrefix(u), DraftAncestors(u) or {u}; [E1] "Tree-Structured Draft
 * Generation": each node attends only to its ancestors; [E3] "The Attention
 * Mechanism Modifications": never to tokens in other branches.
 *
 *   q            : [B, R, Hq, D]       (positions already applied)
 *   k_tree, v_tree : [B, R, Hkv, D]    the tree's own K/V rows
 *   k_cache, v_cache : [P, page_size, Hkv, D]  paged committed prefix
 *   num_pages    : P (pool size), for page-id range checks (EAGLE_ERR_BAD_KV)
 *   block_table  : [B, max_pages] int32 page ids (entries past the prefix unused)
 *   ctx_lens     : [B] int32, 0 <= ctx_lens[b] <= max_pages * page_size
 *   tree_mask    : [B, R] uint64, bit j = row j visible (self bit required)
 *   out          : [B, R, Hq, D] dtype `dtype`;  lse: [B, R, Hq] fp32 or NULL
 *   scale        : score scale (pass 1/sqrt(D) for the standard one)
 *   num_splits   : schedule.  0 = automatic: with many 64-key blocks per SM
 *                  (>= 16, counted with the block table's width) the stream
 *                  schedule -- one persistent CTA per SM, the key blocks of
 *                  every (request, kv head, query-tile group) split evenly
 *                  over the SMs from the real ctx_lens, planned on the device,
 *                  and the pieces of a split unit merged by a second kernel;
 *                  otherwise the split schedule -- one CTA per (query-tile
 *                  group, KV range, request x kv head) with the KV-range count
 *                  chosen from the SM count, the ranges merged by a second
 *                  kernel.  n > 0 = the split schedule with n KV ranges;
 *                  -1 = the stream schedule.
 * The workspace size depends on the schedule: query it with the same
 * num_splits.
 * Limits: R <= 64, D in {64, 128}, page_size == 16, Hq % Hkv == 0,
 * Hq / Hkv <= 16, num_splits >= -1.
 * ---------------------------------------------------------------------- */
size_t eagle_tree_attn_workspace_size(int B, int R, int Hq, int Hkv, int D,
                                      int max_pages, int page_size, int num_splits,
                                      int dtype);
int eagle_tree_attn(const void* q, const void* k_tree, const void* v_tree,
                    const void* k_cache, const void* v_cache, int num_pages,
                    const int32_t* block_table, int max_pages, const int32_t* ctx_lens,
                    const uint64_t* tree_mask, void* out, float* lse, int B, int R,
                    int Hq, int Hkv, int D, int page_size, float scale, int num_splits,
                    int dtype, void* ws, size_t ws_bytes, int32_t* dev_status,
                    void* stream);

/* ------------------------------------------------------------------------
 * eagle_draft_layer -- the drafter's decoder layer over the W new tree nodes
 * of one depth of each of B requests (one pass for the whole depth).
 * [E3] section 3.4 "The transformer decoder layer" (self-attention and a
 * feed-forward sublayer, each with a residual connection and normalisation);
 * the form is that of the LLaMA-family targets ([E3] section 6, Limitation 6:
 * pre-normalisation, SwiGLU, rotary embeddings, grouped-query attention);
 * the attention is tree attention over the drafter's own K/V ([M7.5]
 * sections 0x03C, 0x05B).  With m = b * W + j:
 *   h     = RMSNorm(x) * w_norm1             (x / sqrt(mean(x^2) + eps))
 *   q,k,v = split(h W_qkv^T); q, k rotated (rotate-half RoPE: pair (i, i+D/2)
 *           by positions[m] * theta^(-2i/D))
 *   q_tree[b, r0+j], k_tree[b, r0+j], v_tree[b, r0+j] = q, k, v
 *   a     = tree attention of row r0+j over the prefix (paged cache) and the
 *           tree rows its mask row shows (as eagle_tree_attn, R = Rmax,
 *           scale 1/sqrt(D))
 *   x1    = x + a W_o^T
 *   h2    = RMSNorm(x1) * w_norm2
 *   out   = x1 + (silu(h2 Wg^T) * (h2 Wu^T)) W_down^T,  W_gu = [Wg; Wu]
 *
 *   x        : [B*W, d] dtype `dtype` (must not alias out)
 *   w_norm1, w_norm2 : [d];  w_qkv : [(Hq + 2 Hkv) D, d] (q heads, k heads,
 *              v heads);  w_o : [d, Hq D];  w_gu : [2 I, d] (gate rows then up
 *              rows);  w_down : [d, I]; all dtype `dtype`, out x in
 *   positions: [B, W] int32 (the nodes' positions: prefix length + depth)
 *   k_cache, v_cache, num_pages, block_table, max_pages, ctx_lens: the
 *              drafter's committed prefix, as for eagle_tree_attn
 *   q_tree   : [B, Rmax, Hq, D], k_tree / v_tree : [B, Rmax, Hkv, D]: the
 *              drafter's tree rows, owned by the caller for the whole round;
 *              rows r0 .. r0+W-1 are written, the others are read (rows no
 *              call has written yet must hold finite values: zero them once)
 *   tree_mask: [B, Rmax] uint64, bit i of row r = row i visible to row r
 *              (the new rows: their ancestors' rows and themselves)
 *   out      : [B*W, d]
 * Limits: B*W <= 4096, r0 + W <= Rmax <= 64, D in {64, 128}, Hq % Hkv == 0,
 * d % 128 == 0, (Hq + 2 Hkv) D % 128 == 0, Hq D % 128 == 0, I % 64 == 0.
 * ---------------------------------------------------------------------- */
/* ------------------------------------------------------------------------
 * eagle_draft_rows -- bookkeeping of one drafter pass of a draft round:
 * which draft-KV row each node of the depth takes, the rows it sees, its
 * position, token and feature input, for eagle_draft_input and
 * eagle_draft_layer.  [M7.5] section 0x05B (the nodes of a depth are expanded
 * in one pass; each keeps its token, parent, position and draft-KV row);
 * [E3] section 3.4 "Input representation" (a drafted node's feature is the
 * drafter's own output at its parent; the target feature only at the root).
 *   step 0 : the root: row 0, position ctx_lens[b], token root_token[b],
 *            feature prev[b] (the target's fused feature g, [B, d]); also
 *            starts the round (node_row = -1 except node 0, every row of
 *            row_mask sees only itself).
 *   step s : frontier slot j of request b (the nodes eagle_tree_expand step
 *            s - 1 chose) takes row 1 + (s - 1) * width + j, row_mask[b, row]
 *            = row_mask[b, row(parent)] | (1 << row), position = ctx + depth,
 *            token = node_token, feature = prev[b * W_prev + slot of the
 *            parent] where prev = the previous pass's eagle_draft_layer
 *            output [B * W_prev, d] (W_prev = 1 after step 0, else width).
 *            Slots past n_frontier[b]: token 0, position ctx, zero feature,
 *            a row that sees only itself.
 *   node_row : [B, max_nodes] int32 state; row_mask : [B, Rmax] uint64 state
 *   r_in     : [B * W, d] out (dtype `dtype`), tokens : [B * W] int32 out,
 *   positions: [B, W] int32 out, W = 1 at step 0, else width.
 * The layer call of the pass then uses r0 = 0 (step 0) or
 * 1 + (step - 1) * width, and R = Rmax.
 * Device-detected: a node whose parent the previous pass did not process,
 * or a node id out of range -> EAGLE_ERR_BAD_TREE (the slot reads as empty).
 * Limits: width <= 64, 1 + step * width <= Rmax <= 64, d * element size a
 * multiple of 16 bytes.
 * ---------------------------------------------------------------------- */
int eagle_draft_rows(int B, int step, int width, int Rmax, int max_nodes, int d, int dtype,
                     const int32_t* root_token, const int32_t* frontier,
                     const int32_t* n_frontier, const int32_t* node_parent,
                     const int32_t* node_token, const int32_t* node_depth,
                     const int32_t* ctx_lens, int32_t* node_row, uint64_t* row_mask,
                     const void* prev, void* r_in, int32_t* tokens, int32_t* positions,
                     int32_t* dev_status, void* stream);

size_t eagle_draft_layer_workspace_size(int B, int W, int d, int Hq, int Hkv, int D, int I,
                                        int Rmax, int max_pages, int dtype);
int eagle_draft_layer(const void* x, const void* w_norm1, const void* w_qkv, const void* w_o,
                      const void* w_norm2, const void* w_gu, const void* w_down, float eps,
                      float theta, const int32_t* positions, const void* k_cache,
                      const void* v_cache, int num_pages, const int32_t* block_table,
                      int max_pages, const int32_t* ctx_lens, void* q_tree, void* k_tree,
                      void* v_tree, const uint64_t* tree_mask, int r0, int Rmax, void* out,
                      int B, int W, int d, int Hq, int Hkv, int D, int I, int dtype, void* ws,
                      size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_lmhead_topk -- vocabulary logits and per-row top-k, fused.
 *   z[i, v] = sum_c W_U[v, c] x[i, c] (+ bias[v])
 *   topk_ids[i, :]      = the k ids of largest z (z descending, ties to the
 *                         lower id)
 *   topk_logprobs[i, j] = z[i, id_j]/T - logsumexp_v(z[i, v]/T)
 *   row_max[i]          = max_v z[i, v]/T;  row_sumexp[i] = sum_v exp(z/T - row_max)
 * Full-vocabulary logits are never written to memory.
 * [E3] "Output path to LM head" (logits = W_LM a + b_LM, bias if present);
 * [E1] "Tree-Structured Draft Generation" (greedy: top-k tokens become the
 * children); [M7.5] section 0x06B (confidence = conditional token probability
 * under the parent's prefix; omitted vocabulary mass allowed).
 *
 *   x            : [M, d] dtype `dtype`;  w_lm: [V, d] dtype `dtype`
 *   bias         : [V] fp32 or NULL
 *   topk_ids     : [M, k] int32;  topk_logprobs: [M, k] fp32
 *   row_max, row_sumexp : [M] fp32 or NULL
 * bf16 runs on the tensor cores with fp32 accumulation; fp32 runs on the CUDA
 * cores in exact fp32 arithmetic.
 * Limits: 1 <= M <= 2048, 1 <= k <= 32, k <= V, d % 64 == 0,
 * V % 16 == 0, temperature > 0.
 * ---------------------------------------------------------------------- */
size_t eagle_lmhead_topk_workspace_size(int M, int d, int V, int k, int dtype);
int eagle_lmhead_topk(const void* x, const void* w_lm, const float* bias, int M, int d,
                      int V, int k, float temperature, int32_t* topk_ids,
                      float* topk_logprobs, float* row_max, float* row_sumexp, int dtype,
                      void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* The same call in two halves (same arguments, same `ws`, in stream order):
 * eagle_lmhead_topk_partial runs the GEMM and leaves each CTA's partial
 * lists and log-sum-exp terms in `ws`; eagle_lmhead_topk_merge turns them
 * into topk_ids / topk_logprobs / row_max / row_sumexp.  Together they launch
 * exactly the kernels of eagle_lmhead_topk (lets a caller time or overlap the
 * GEMM on its own). */
int eagle_lmhead_topk_partial(const void* x, const void* w_lm, const float* bias, int M, int d,
                              int V, int k, float temperature, int dtype, void* ws,
                              size_t ws_bytes, int32_t* dev_status, void* stream);
int eagle_lmhead_topk_merge(int M, int d, int V, int k, float temperature, int32_t* topk_ids,
                            float* topk_logprobs, float* row_max, float* row_sumexp, int dtype,
                            void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_expand -- one EAGLE-2 expansion step for B requests.
 * [M7.5] section 0x06A "Path Value Derivation" and 0x06B "Expansion And
 * Reranking": every child of an expanded parent is stored with
 *   log V(child) = log V(parent) + log max(c, 1e-12)     (fp32)
 * (c = exp(logprob), logprob clamped to <= 0), depth = parent depth + 1 and a
 * creation-ordered node id; only the new nodes form the next frontier, and
 * the next nodes to expand are its top `width` by the key
 * (-log V, depth, node_id).
 *
 *   step          : 0 initialises the store with the seed (node 0: parent -1,
 *                   token root_token[b], log V 0, depth 0) and expands it.
 *   cand_ids      : [B, P, k] int32 top-k ids per expanded parent, P = 1 at
 *                   step 0, else `width`; row j belongs to frontier[b, j]
 *                   (rows j >= n_frontier[b] are ignored); an id < 0 marks a
 *                   missing alternative (no node is created).
 *   cand_logprobs : [B, P, k] fp32 log conditional probabilities.
 *   root_token    : [B] int32 (read at step 0 only)
 *   node_parent, node_token, node_depth : [B, max_nodes] int32 tree store
 *   node_logv     : [B, max_nodes] fp32
 *   node_count    : [B] int32 nodes stored (seed included)
 *   frontier      : [B, width] int32 in/out: parents expanded by this step on
 *                   entry, the next parents to expand (key order) on exit
 *   n_frontier    : [B] int32 in/out: valid entries of frontier
 * Device-detected: duplicate id under one parent, sibling probability mass
 * above 1 (+1e-4 slack for fp32) -> EAGLE_ERR_BAD_TREE; NaN or +inf
 * log-prob -> EAGLE_ERR_NONFINITE (the request's step is then skipped).
 * Limits: width <= 64, k <= 32, width*k <= 1024, max_nodes <= 2048, and
 * max_nodes >= 1 + k + step*width*k (checked on the host).
 * ---------------------------------------------------------------------- */
int eagle_tree_expand(int B, int step, int width, int k, int max_nodes,
                      const int32_t* cand_ids, const float* cand_logprobs,
                      const int32_t* root_token, int32_t* node_parent,
                      int32_t* node_token, float* node_logv, int32_t* node_depth,
                      int32_t* node_count, int32_t* frontier, int32_t* n_frontier,
                      int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_expand_lmhead -- eagle_tree_expand whose candidate lists come
 * straight from an LM-head call's partial results.
 * [M7.5] sections 0x06A, 0x06B (as eagle_tree_expand) with [E1]
 * "Tree-Structured Draft Generation" (the children are the top-k tokens of
 * the parent's drafter row).  The call follows an eagle_lmhead_topk_partial
 * over M = B * P drafter rows (P = 1 at step 0, else width; row b * P + j =
 * parent slot j of request b) with the same k, d, V, dtype and temperature,
 * and takes its workspace `lm_ws`: each parent row's top-k ids and log-probs
 * are merged from the LM head's per-CTA partial lists inside the expansion
 * kernel, so no merge kernel and no [M, k] candidate arrays sit between the
 * LM head and the expansion.  The merged lists equal those of
 * eagle_lmhead_topk_merge bit for bit, and the tree state equals that of
 * eagle_lmhead_topk_merge followed by eagle_tree_expand.
 * Limits: those of eagle_tree_expand and eagle_lmhead_topk (M <= 2048).
 * ---------------------------------------------------------------------- */
int eagle_tree_expand_lmhead(int B, int step, int width, int k, int max_nodes,
                             const void* lm_ws, size_t lm_ws_bytes, int d, int V,
                             float temperature, int dtype, const int32_t* root_token,
                             int32_t* node_parent, int32_t* node_token, float* node_logv,
                             int32_t* node_depth, int32_t* node_count, int32_t* frontier,
                             int32_t* n_frontier, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_expand_static -- one depth of a static (EAGLE-1) draft tree.
 * [E1] "Tree-Structured Draft Generation" and its note on the tree used: a
 * fixed tree whose root branches into its top-4 tokens and whose deeper
 * nodes branch into fewer.  The shape is given depth by depth: node j of the
 * current depth (frontier[b, j], creation order) keeps its top-fanout[j]
 * candidates (ranks 0 .. fanout[j]-1).  Values, depths, node ids, validation
 * and every argument are as for eagle_tree_expand, except that the next
 * frontier is all the new nodes in creation order (no reranking), `width`
 * is the frontier capacity (the widest depth), and
 *   fanout : [P] int32 device, the same for every request (P = 1 at step 0,
 *            else width), each in [0, k].
 * Flatten a finished static tree with eagle_tree_expand_finalize and a
 * budget of all its nodes.
 * Device-detected: a fan-out outside [0, k], or more new nodes than `width`
 * -> EAGLE_ERR_BAD_TREE (plus the checks of eagle_tree_expand).
 * ---------------------------------------------------------------------- */
int eagle_tree_expand_static(int B, int step, int width, int k, int max_nodes,
                             const int32_t* fanout, const int32_t* cand_ids,
                             const float* cand_logprobs, const int32_t* root_token,
                             int32_t* node_parent, int32_t* node_token, float* node_logv,
                             int32_t* node_depth, int32_t* node_count, int32_t* frontier,
                             int32_t* n_frontier, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_expand_finalize -- EAGLE-2 rerank, then flatten for verification.
 * [M7.5] section 0x06B: selected = the first `budget` non-seed nodes in
 * (-log V, depth, node_id) order; since a child never outranks its parent
 * the selection is ancestor-closed with no repair.  [M7.5] section 0x05C
 * "Target Verification": the selection is flattened with ancestry-aware
 * positions and a tree mask; section 0x09: a retrieve map ties rows to nodes.
 *
 *   Output rows per request: R (>= 1 + budget, <= 64).  Row 0 = seed,
 *   row i = i-th selected node.  Rows >= n_rows[b] are padding (token -1,
 *   parent_row -1, depth 0, mask = own bit, node_id -1, position ctx).
 *   token, parent_row, depth, node_id, position : [B, R] int32
 *   mask        : [B, R] uint64 (bit j = row j is the row itself or an ancestor)
 *   n_rows      : [B] int32 = 1 + min(budget, node_count[b] - 1)
 *   ctx_lens    : [B] int32 (positions = ctx_lens[b] + depth), or NULL (0)
 * Device-detected: a selected node whose parent is not selected before it
 * -> EAGLE_ERR_BAD_TREE.  Limits: max_nodes <= 2048.
 * ---------------------------------------------------------------------- */
int eagle_tree_expand_finalize(int B, int max_nodes, int budget, int R,
                               const int32_t* node_parent, const int32_t* node_token,
                               const float* node_logv, const int32_t* node_depth,
                               const int32_t* node_count, const int32_t* ctx_lens,
                               int32_t* token, int32_t* parent_row, int32_t* depth,
                               uint64_t* mask, int32_t* node_id, int32_t* position,
                               int32_t* n_rows, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_verify -- lossless acceptance of a flattened draft tree.
 * [E1] "Verification Phase: Multi-Round Speculative Sampling on Trees"
 * (Algorithm 1): candidates under a node are tried in order, t_i accepted
 * when r < p(t_i)/p_hat_i(t_i); after a rejection p <- norm(max(0, p -
 * p_hat_i)); if all are rejected a token is drawn from the final p.  [E3]
 * "Stage 2: Verification".  The target logits of row r give the distribution
 * p of the children of row r (softmax of z/T).
 *   temperature == 0 : greedy; p = one-hot(argmax z) (ties to the lower id),
 *                      i.e. accept the child whose token is the argmax.
 *   DETERMINISTIC    : the children are deterministic top-k (EAGLE-2); the
 *                      proposal of a child is the point mass on its token, so
 *                      accept iff u < p(t), and a rejected token is removed
 *                      from p, which is renormalised.
 *   SAMPLED          : Algorithm 1 with p_hat = softmax(draft logits / T)
 *                      (children i.i.d. from it): accept iff u < p(t)/q(t);
 *                      after a rejection p <- norm(max(0, p - q)) (unchanged
 *                      when that mass is 0); the bonus is drawn from the
 *                      final p.  Needs draft_logits [B, R, V] fp32 and T > 0.
 * The final draw is an exponential race argmax_y (z_y/T - log(-log u_y)) over
 * the ids not rejected at the stop row.
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11), key = seed; accept test of
 * row i of request b = word 0 at counter (i, b, 2*offset_hi, offset_lo); race
 * uniform of id y = word (y & 3) at counter (y >> 2, b, 2*offset_hi + 1,
 * offset_lo); u = (2*(x >> 9) + 1) * 2^-24.  `uniforms_override` [B, R]
 * replaces the accept-test uniforms when non-NULL.
 *
 *   parent_row, token : [B, R] int32 (row 0 = seed with parent -1;
 *                       0 <= parent_row[i] < i), n_rows: [B] int32 or NULL (= R)
 *   target_logits     : [B, R, V] fp32 (may be NULL when temperature == 0 and
 *                       target_argmax is given)
 *   target_argmax     : [B, R] int32 or NULL
 *   accept_len        : [B] int32 accepted drafted nodes
 *   path_rows         : [B, max_depth+1] int32, row 0 then the accepted rows
 *   out_tokens        : [B, max_depth+1] int32, accepted tokens then the
 *                       bonus token; unused entries -1
 * Device-detected: non-topological parents, path deeper than max_depth ->
 * EAGLE_ERR_BAD_TREE; NaN in a read logit row -> EAGLE_ERR_NONFINITE.
 * Limits: R <= 1024, V >= 2, max_depth <= 64, offset < 2^63.
 * ---------------------------------------------------------------------- */
size_t eagle_tree_verify_workspace_size(int B, int R, int V);
int eagle_tree_verify(int B, int R, int V, const int32_t* parent_row, const int32_t* token,
                      const int32_t* n_rows, const float* target_logits,
                      const int32_t* target_argmax, const float* draft_logits,
                      float temperature, int proposal_mode, uint64_t seed, uint64_t offset,
                      const float* uniforms_override, int max_depth, int32_t* accept_len,
                      int32_t* path_rows, int32_t* out_tokens, void* ws, size_t ws_bytes,
                      int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_lmhead_verify_stats -- the verification LM head for stochastic
 * verification: everything the deterministic-proposal walk of [E1]
 * "Verification Phase: Multi-Round Speculative Sampling on Trees" reads from
 * the target logits z = W_U a (+ b) of the B*R verify rows, without ever
 * writing the [B, R, V] logits.  Rows are request-major (row = b*R + r).
 *   row_max[row]    = max_v z/T;  row_sumexp[row] = sum_v exp(z/T - row_max)
 *   child_logit[row]= z[b*R + parent_row(row)][token(row)] for tree rows
 *                     1 <= r < n_rows[b]; 0 for the root and unused rows
 *   race_ids / race_keys [row, race_k]: the race_k ids of largest
 *                     key_y = z_y/T - log(-log u_{b,y}) (ties to the lower
 *                     id), sorted, with their keys; u as in eagle_tree_verify
 *                     (Philox word (y & 3) at counter (y >> 2, b,
 *                     2*offset_hi + 1, offset_lo), key = seed).  The
 *                     renormalisation of the race is common to all ids, so
 *                     the stop row's bonus token is its first candidate not
 *                     rejected there: race_k must exceed the number of
 *                     children of any row (top-k trees: race_k = k + 1).
 * No counterpart call on the pages: it fuses what [E1]'s verification reads
 * into the LM head that produces the logits.
 *   x : [B*R, d], w_lm : [V, d] (dtype `dtype`), bias : [V] fp32 or NULL
 *   parent_row, token : [B, R] int32;  n_rows : [B] int32 or NULL (= R)
 *   race_ids : [B*R, race_k] int32; race_keys : [B*R, race_k] fp32
 *   row_max, row_sumexp, child_logit : [B*R] fp32
 *   ws : eagle_lmhead_topk_workspace_size(B*R, d, V, race_k, dtype) bytes
 * Device-detected: a parent or token out of range -> EAGLE_ERR_BAD_TREE;
 * NaN logits -> EAGLE_ERR_NONFINITE.
 * Limits: those of eagle_lmhead_topk with M = B*R and k = race_k; T > 0;
 * offset < 2^63.
 * ---------------------------------------------------------------------- */
int eagle_lmhead_verify_stats(const void* x, const void* w_lm, const float* bias, int B, int R,
                              int d, int V, const int32_t* parent_row, const int32_t* token,
                              const int32_t* n_rows, float temperature, uint64_t seed,
                              uint64_t offset, int race_k, int32_t* race_ids, float* race_keys,
                              float* row_max, float* row_sumexp, float* child_logit, int dtype,
                              void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_verify_stats -- eagle_tree_verify for T > 0 with deterministic
 * proposals, reading the outputs of eagle_lmhead_verify_stats instead of
 * target logits.  Same walk, same accept uniforms (and uniforms_override),
 * same outputs: child c of the current row r is accepted when
 * u_c < p / (1 - mass of the distinct tokens already rejected at r), with
 * p = exp(child_logit[c]/T - row_max[r]) / row_sumexp[r]; the bonus token at
 * the stop row is its first race candidate not rejected there.  Needs no
 * workspace (one kernel).
 * Device-detected: as eagle_tree_verify; every race candidate of the stop row
 * rejected (race_k too small) -> EAGLE_ERR_INVALID_ARG and bonus -1.
 * Limits: R <= 1024, max_depth <= 64, T > 0, offset < 2^63.
 * ---------------------------------------------------------------------- */
int eagle_tree_verify_stats(int B, int R, int V, const int32_t* parent_row, const int32_t* token,
                            const int32_t* n_rows, const float* row_max, const float* row_sumexp,
                            const float* child_logit, const int32_t* race_ids, int race_k,
                            float temperature, uint64_t seed, uint64_t offset,
                            const float* uniforms_override, int max_depth, int32_t* accept_len,
                            int32_t* path_rows, int32_t* out_tokens, int32_t* dev_status,
                            void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_commit -- publish the verified path.
 * [M7.5] section 0x05D "Feature And KV Commit" (publish_verified_path):
 * the target K/V of the accepted rows are appended to the committed prefix
 * and their target features gathered for the next draft round; every other
 * tree row is discarded.  Rows are taken by the flat row index of the
 * verified path, never by token id.  The accepted rows of request b are
 * path_rows[b, 0 .. accept_len[b]] (the root row -- the previous frontier
 * token, computed by this verify forward -- then the accepted drafted rows);
 * row i lands at position ctx_lens[b] + i (page block_table[b, pos / 16],
 * slot pos % 16) and ctx_lens[b] grows by accept_len[b] + 1.  The new
 * frontier token is not a verified row and needs a later target append.
 *   k_tree, v_tree : [B, R, Hkv, D] dtype `dtype` (the verify forward's rows)
 *   path_rows, accept_len : outputs of eagle_tree_verify ([B, max_depth+1], [B])
 *   k_cache, v_cache : [num_pages, 16, Hkv, D], written in place
 *   block_table : [B, max_pages] (the caller has mapped pages for the new
 *                 positions);  ctx_lens : [B] int32, updated in place
 *   features : [B*R, F] or NULL; features_out : [B, max_depth+1, F] or NULL
 *                 (rows past accept_len are zeroed)
 * Device-detected: accept_len or a path row out of range -> EAGLE_ERR_BAD_TREE;
 * no room in the block table or a page id out of range -> EAGLE_ERR_BAD_KV;
 * such a request is left untouched (nothing written, ctx_lens unchanged).
 * Limits: max_depth <= 64; Hkv * D * element size and F * element size
 * multiples of 16 bytes; 16-byte aligned arrays; num_pages <= 2^26.
 * ---------------------------------------------------------------------- */
int eagle_tree_commit(int B, int R, int Hkv, int D, int max_depth, int dtype, const void* k_tree,
                      const void* v_tree, const int32_t* path_rows, const int32_t* accept_len,
                      void* k_cache, void* v_cache, int num_pages, const int32_t* block_table,
                      int max_pages, int32_t* ctx_lens, const void* features, int F,
                      void* features_out, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * eagle_tree_verify_noalloc -- eagle_tree_verify without a workspace.
 * The pages have no counterpart of this call: it exists for callers that
 * cannot allocate device memory, such as a plugin whose host framework owns
 * every device allocation and passes it only its input and output tensors,
 * or a latency-critical loop that must not call cudaMalloc (which can
 * synchronise the whole device).  Arguments, outputs and semantics are those
 * of eagle_tree_verify minus `ws` / `ws_bytes`; the scratch that
 * eagle_tree_verify keeps in `ws` lives in a fixed buffer inside the library
 * instead.
 *   Capacity: B * R <= 65536 rows and, when temperature > 0,
 *   B * ceil(V / 4096) <= 65536 race chunks; larger calls return
 *   EAGLE_ERR_WORKSPACE without launching anything.  The buffer (2.5 MB:
 *   row statistics, argmax, rejected tokens, per-request walk results and
 *   race partials) is a static device
 *   array: every GPU that loads the library holds one copy until the process
 *   exits, and no call allocates or frees memory.
 *   The buffer's device address is looked up in the current CUDA context
 *   (with cudaGetSymbolAddress) on every call made outside stream capture,
 *   and kept per context.  A call made while `stream` is capturing uses the
 *   address an earlier call in the same context looked up, and returns
 *   EAGLE_ERR_INVALID_ARG, launching nothing, if no such call has run: make
 *   the first call in each context (and the first after cudaDeviceReset,
 *   which replaces the context) outside capture.  A failed lookup returns
 *   EAGLE_ERR_CUDA and clears the runtime's last error.
 *   All calls on a device share the buffer and it keeps the last call's
 *   contents (no field needs to start at zero); calls whose kernels overlap
 *   on the same device race on it, so serialise them (e.g. one stream).
 * ---------------------------------------------------------------------- */
int eagle_tree_verify_noalloc(int B, int R, int V, const int32_t* parent_row,
                              const int32_t* token, const int32_t* n_rows,
                              const float* target_logits, const int32_t* target_argmax,
                              const float* draft_logits, float temperature, int proposal_mode,
                              uint64_t seed, uint64_t offset, const float* uniforms_override,
                              int max_depth, int32_t* accept_len, int32_t* path_rows,
                              int32_t* out_tokens, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_GB300_EAGLE_H */
