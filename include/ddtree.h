/*
 * ddtree.h - C ABI of the DDTree tree-verify step on one GB300 (sm_103a).
 *
 * The step has four calls, taken in this order for one speculative-decoding
 * step of a batch of B requests, after an optional fifth that prepares the
 * first one's input on the device:
 *
 *   ddtree_draft_topk     draft logits -> per-depth top-k tokens + log-probs
 *   ddtree_build          per-depth top-k  -> best-first tree, mask, positions
 *   tree_verify_attn      tree rows attend to their context (paged KV, read
 *                         once per request and KV head) plus visible tree rows
 *   ddtree_accept_greedy  longest root path matching the target argmax + bonus
 *   ddtree_accept_sample  the same at temperature, by recursive rejection
 *                         sampling over siblings + a bonus from the residual
 *                         (ddtree_accept_sample_ratio: the draft-ratio rule)
 *
 * and ddtree_commit_kv appends the committed path's K/V to the paged cache;
 * ddtree_step_* records build -> attention -> walk -> commit as one graph.
 *
 * Sources (page titles; sections named at each call):
 *   [Arch]   "The Architecture of Speculative Decoding: Dissecting DDTree's
 *            Tree-Parallel Evaluation Strategy"
 *   [Verify] "The Architecture of Speculative Verification: Implementing
 *            Temperature-Aware Tree Sampling for DDTree"
 *   [Pivot]  "The Pivot Point: Strategic Decision-Making in Speculative
 *            Decoding Optimization"
 *   [Branch] "The Tree That Couldn't Branch: Diagnosing a 2x Acceptance
 *            Regression in DDTree Speculative Decoding"
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every array pointer is DEVICE memory owned by the caller; the library
 *   allocates nothing, keeps no pointer after the call returns, and writes
 *   only the outputs (and the caller-provided workspace) it documents.
 * - Arrays are dense, row-major (C order), with the shapes given; no strides.
 * - bf16 arrays hold raw bfloat16 bit patterns (ddtree_bf16).
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *   stream). Calls are asynchronous on it, never synchronise the host and
 *   allocate nothing, so a sequence of calls with fixed sizes can be captured
 *   in a CUDA graph.
 * - Return value: DDT_OK, or a negative ddtree_status. Argument checks happen
 *   on the host before any launch; on an argument error nothing is launched
 *   and no output is written.
 * - `dev_status` (nullable, one int32 in device memory): data errors found on
 *   the device (a page id outside the pool, a token outside the vocabulary,
 *   a malformed tree, a bad temperature) are OR-ed into it as DDT_DEV_* bits;
 *   the library never clears it. The affected rows get defined, harmless
 *   outputs (zeros or -1) and no out-of-bounds access is made. Nothing traps.
 * - N = budget + 1 tree rows per request, W = (N + 31) / 32 mask words.
 * - Sizes are plain int; every element count must fit in int64.
 */
#ifndef DDTREE_H
#define DDTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ddtree_bf16;

enum ddtree_status {
    DDT_OK = 0,
    DDT_EINVAL = -1,      /* null pointer or bad scalar argument              */
    DDT_ESHAPE = -2,      /* sizes outside the supported range                */
    DDT_ECUDA = -3,       /* a CUDA runtime call or launch failed             */
    DDT_ETIMEOUT = -4,    /* reserved: a bounded device wait gave up          */
    DDT_EWORKSPACE = -6,  /* workspace pointer null or smaller than required  */
    DDT_ESCRATCH = -7     /* sizes need more scratch than the fixed array of  */
                          /* tree_verify_attn_noalloc holds                   */
};

/* bits OR-ed into *dev_status by the device */
enum ddtree_device_error {
    DDT_DEV_BAD_PAGE = 1,         /* page_table entry < 0 or >= num_pages       */
    DDT_DEV_BAD_CTX = 2,          /* ctx_len < 0 or > max_pages * page_size     */
    DDT_DEV_BAD_TREE = 4,         /* tree arrays inconsistent (child index out  */
                                  /* of range, walk longer than D, n_nodes > N) */
    DDT_DEV_BAD_TEMPERATURE = 8,  /* temperature <= 0 or not finite             */
    DDT_DEV_BAD_TOKEN = 16,       /* token id outside [0, V)                    */
    DDT_DEV_TIMEOUT = 32          /* a bounded wait inside a kernel gave up; the */
                                  /* affected outputs are undefined             */
};

/* Limits checked on the host (DDT_ESHAPE beyond them). */
#define DDT_MAX_TOPK 32           /* K                                         */
#define DDT_MAX_DEPTH 64          /* D                                         */
#define DDT_MAX_NODES 128         /* N = budget + 1                            */

/* Human-readable name of a status code (static string). */
const char* ddtree_status_string(int status);

/* Text of the last CUDA error seen by a call that returned DDT_ECUDA on this
 * host thread ("" if none). */
const char* ddtree_last_error(void);

/*
 * ddtree_draft_topk - per-depth top-K of the draft, with log-probs.
 *
 * [Arch] Section 1 (The Five-Step Flow of DDTree), step 1: the draft runs once
 * over the block and, at each depth position, its top-k tokens are kept with
 * their log-probs. [Branch] Hypothesis 4: one distribution per depth, shared
 * by every node of that depth. The output is exactly ddtree_build's input.
 *
 * Inputs
 *   draft_logits  fp32 [B, D, V]  the draft's logits, depth d's row for the
 *                                 tokens at depth d+1
 * Outputs
 *   topk_logp     fp32  [B, D, K] log-probs, descending along K
 *   topk_tok      int32 [B, D, K] their token ids
 * Ranking is by the logit (the same order as the log-prob), ties to the lower
 * token id, NaN below every number (-0 equals +0). The log-prob is the logit
 * minus the row's log-sum-exp (max + log of an fp32 exp-sum), formed in fp64
 * and rounded to fp32; the error against the exact value is within
 * (V/512 + 64) * 2^-22 + 2^-23 |log-prob| (about 1e-6 measured). A row
 * holding a NaN or +inf, or only -inf, has a NaN log-sum-exp: its K tokens
 * are still ranked and its log-probs are NaN.
 * 1 <= K <= min(32, V), 1 <= D <= 64, B * D < 2^31. Rows are read with 16-byte
 * loads when V % 4 == 0 and draft_logits is 16-byte aligned, else 4-byte.
 * No device errors.
 */
int ddtree_draft_topk(const float* draft_logits, int B, int D, int V, int K,
                      float* topk_logp, int32_t* topk_tok, void* stream);

/*
 * ddtree_build - best-first draft tree from the per-depth top-k.
 *
 * [Arch] Section 1 (The Five-Step Flow of DDTree), steps 2-3: a heap keyed by
 * cumulative log-prob; pop the best node and add it; push its best child and
 * its next sibling; stop after `budget` nodes (budget + 1 with the root). The
 * mask lets each node see its ancestors and itself (and, implicitly, the whole
 * context). [Branch] Context section: the cap K bounds the children of a node;
 * Hypothesis 3: a node at depth d sits at position ctx_len + d, so siblings
 * share a position; Hypothesis 4: every node of depth d takes its children
 * from the same depth-(d+1) top-k.
 *
 * Inputs
 *   topk_logp  fp32  [B, D, K]  log-probs of depth d+1's top-K, sorted
 *                               descending along K (d = 0..D-1)
 *   topk_tok   int32 [B, D, K]  their token ids (distinct along K)
 *   root_tok   int32 [B]        the anchor token (tree row 0)
 *   ctx_len    int32 [B]        tokens already in the KV cache
 * Outputs, [B, N] unless stated; row 0 is the root, rows are in pop order so a
 * parent always precedes its children; rows >= n_nodes[b] are pads:
 *   parent       int32   root -1, pad -1
 *   depth        int32   root 0,  pad -1
 *   token        int32   root root_tok, pad -1
 *   rank         int32   rank within its depth's top-k; root 0, pad -1
 *   pos          int32   ctx_len + depth; pad -1
 *   score        float64 cumulative log-prob (fp64 sums of the fp32 inputs in
 *                        path order); root 0, pad -inf
 *   first_child  int32   first child in index (= rank) order, -1 if none
 *   next_sibling int32   next child of the same parent, -1 if none
 *   vis          uint32 [B, N, W]  bit (j % 32) of word j / 32 set iff row j
 *                        is row i or an ancestor of it; pads all zero
 *   n_nodes      int32 [B]   1 + nodes chosen (< N only if the candidates run
 *                        out, e.g. K = 1 and budget > D)
 * Ties in score go to the earlier push; a popped node pushes its child before
 * its sibling. 1 <= K <= 32, 1 <= D <= 64, 0 <= budget <= 127.
 * Device errors: ctx_len < 0 sets DDT_DEV_BAD_CTX (pos is still written).
 */
int ddtree_build(const float* topk_logp, const int32_t* topk_tok,
                 const int32_t* root_tok, const int32_t* ctx_len,
                 int B, int D, int K, int budget,
                 int32_t* parent, int32_t* depth, int32_t* token, int32_t* rank,
                 int32_t* pos, double* score, int32_t* first_child,
                 int32_t* next_sibling, uint32_t* vis, int32_t* n_nodes,
                 int32_t* dev_status, void* stream);

/*
 * tree_verify_attn - attention of all tree rows in one pass.
 *
 * [Arch] Section 1, step 4: all budget+1 nodes go through the target at once
 * with the tree mask; Section 2 (Context Loading): every node sees the whole
 * prefix, whose KV is read once and shared by all nodes. [Pivot] The Design
 * Constraint (Load Contexts Once).
 *
 * For request b, row i < n_nodes[b] and query head h (kv head h / (Hq/Hkv)):
 *   out[b,i,h,:] = softmax_j(scale * q[b,i,h,:] . k_j) v_j
 * over the ctx_len[b] context keys (all visible) followed by the tree keys j
 * whose bit is set in vis[b,i,:]. Rows i >= n_nodes[b] get zeros.
 *
 * Inputs
 *   q           bf16  [B, N, Hq, Dh]
 *   k_tree      bf16  [B, N, Hkv, Dh]   K of the tree rows (row 0 = root)
 *   v_tree      bf16  [B, N, Hkv, Dh]
 *   k_cache     bf16  [num_pages, page_size, Hkv, Dh]  paged context K
 *   v_cache     bf16  [num_pages, page_size, Hkv, Dh]
 *   page_table  int32 [B, max_pages]  token t of request b is slot
 *               t % page_size of page page_table[b, t / page_size]; only
 *               the first ceil(ctx_len[b] / page_size) entries are read
 *   ctx_len     int32 [B]
 *   vis         uint32 [B, N, W]   as written by ddtree_build
 *   n_nodes     int32 [B]
 * Outputs
 *   out         bf16  [B, N, Hq, Dh]
 *   lse         fp32  [B, N, Hq] (nullable): natural-log softmax denominator
 *               (log-sum-exp of the scaled scores); -inf for pad rows
 * Workspace: `workspace` (device, >= tree_verify_attn_workspace_size(...)
 * bytes, 256-byte aligned) holds split-KV partial results; its contents on
 * entry do not matter. Slots of a page at or beyond ctx_len[b] are never used
 * (their values may be anything, NaN included).
 * Supported: Dh in {64, 128}; 1 <= Hkv <= Hq, Hq % Hkv == 0; N <= 128;
 * page_size a multiple of 16 in [16, 1024]; ctx_len[b] <= max_pages * page_size.
 * Kernels: Dh 128 with G = Hq / Hkv <= 128 and a page size that divides or is
 * a multiple of 64 runs the tensor-core kernel (any number of rows N * G, in
 * row groups); other supported shapes run a warp-MMA kernel, slower, with
 * results within the same tolerance.
 * Overlap with ddtree_build: the tensor-core kernel is launched as a
 * programmatic dependent of the work before it on the stream. Directly after
 * ddtree_build it starts while the build finishes (loading Q, the tree K/V
 * and the paged context, which the build does not write) and reads n_nodes
 * and vis only once the build's grid has completed; after any other work it
 * starts when that work has completed, as an ordinary launch.
 * Device errors: DDT_DEV_BAD_PAGE (that page's slots are read as zeros),
 * DDT_DEV_BAD_CTX (the request's rows are zeros).
 */
int tree_verify_attn(const ddtree_bf16* q, const ddtree_bf16* k_tree,
                     const ddtree_bf16* v_tree, const ddtree_bf16* k_cache,
                     const ddtree_bf16* v_cache, int num_pages, int page_size,
                     const int32_t* page_table, int max_pages,
                     const int32_t* ctx_len, const uint32_t* vis,
                     const int32_t* n_nodes, int B, int N, int Hq, int Hkv, int Dh,
                     float scale, ddtree_bf16* out, float* lse, void* workspace,
                     size_t workspace_bytes, int32_t* dev_status, void* stream);

/* Bytes of workspace tree_verify_attn needs for these sizes when every
 * context is at most max_ctx tokens (max_ctx = max_pages * page_size covers
 * any page table). Returns 0 for unsupported sizes. The split-KV plan is
 * sized in waves of the current device's SM count (queried once per
 * device), so ask with the device current that will run the call. */
size_t tree_verify_attn_workspace_size(int B, int N, int Hq, int Hkv, int Dh,
                                       int max_ctx);

/*
 * ddtree_accept_greedy - the greedy verify walk.
 *
 * [Arch] Section 1, step 5: from the root, follow the target's argmax at the
 * current node into the child carrying that token; stop when no child
 * matches; the accepted chain plus one bonus token (the argmax at the last
 * node) is committed. [Verify] Context section: on a chain this is the linear
 * rule (draft i is accepted while the argmax at position i-1 equals it).
 *
 * Inputs
 *   logits        fp32 [B, N, V]  row u = target prediction for the token
 *                                 after node u; only rows on the walk are read
 *   token, first_child, next_sibling  int32 [B, N]  from ddtree_build
 *   n_nodes       int32 [B]
 * Outputs
 *   accept_len    int32 [B]       accepted draft tokens (bonus excluded)
 *   out_tokens    int32 [B, D+1]  accepted tokens then the bonus; -1 after
 *   out_nodes     int32 [B, D+1]  row 0 then the accepted rows; -1 after
 *   bonus         int32 [B]
 *   walk_stats    int32 [B, 4]    (nullable) per request: accepted depth
 *                                 (= accept_len), nodes built (n_nodes as
 *                                 read), tokens emitted (the commit length:
 *                                 accepted tokens plus the bonus) and the
 *                                 children compared without a match.
 *                                 [Branch] Output Knowledge Created, item 5:
 *                                 node counts, accepted depths and commit
 *                                 lengths as debug metrics.
 * Argmax ties go to the lowest index; NaN ranks below every number (an
 * all-NaN row gives 0). Device errors: DDT_DEV_BAD_TREE (walk stops).
 */
int ddtree_accept_greedy(const float* logits, int V, const int32_t* token,
                         const int32_t* first_child, const int32_t* next_sibling,
                         const int32_t* n_nodes, int B, int N, int D,
                         int32_t* accept_len, int32_t* out_tokens,
                         int32_t* out_nodes, int32_t* bonus, int32_t* walk_stats,
                         int32_t* dev_status, void* stream);

/*
 * ddtree_accept_sample - verify at temperature by recursive rejection
 * sampling over siblings.
 *
 * [Arch] Section 3 (Temperature Support), tree case: at each node reject-
 * sample the children in turn, descend on an acceptance, and once all are
 * rejected draw the bonus from the residual and stop. [Verify] Path B and
 * item 3 of the knowledge list: target q = softmax(logits / T), accept with
 * min(1, q/p), renormalise q on rejection. A DDTree child is a deterministic
 * top-k token (a point-mass proposal), so child j of a node, token x_j, is
 * accepted when u_j * (1 - sum_{i<j} q(x_i)) < q(x_j); the bonus is sampled
 * from q with the node's children removed (Gumbel-max). Emitted tokens are
 * distributed exactly as the target.
 *
 * Inputs: as ddtree_accept_greedy, plus
 *   temperature  fp32   [B]   T > 0 per request
 *   seed         uint64 [B]   Philox key per request
 *   philox_offset             advance per decoding step; < 2^56
 * Randomness: Philox4x32-10 with key (seed lo32, seed hi32) and counter
 * (purpose | (offset >> 32) << 8, node, index, offset lo32): purpose 0 =
 * child test (index = child slot, word 0), purpose 1 = Gumbel noise for vocab
 * entry v (index = v >> 2, word v & 3); uniform = ((w >> 8) + 0.5) * 2^-24.
 * The noise g = -log(-log U) is formed in fp32 within 2e-6 of its exact value
 * for every uniform (ddtree_testing_gumbel in ddtree_testing.h returns it).
 * Outputs: as ddtree_accept_greedy (walk_stats column 3 counts the child
 * tests that rejected), plus
 *   margin_stats  fp32 [B] (nullable): the smallest decision margin on the
 *                 request's path: |u_j - q(x_j) / R| over the child tests
 *                 (R = 1 - sum_{i<j} q(x_i)) and, for the bonus, the gap
 *                 between the best and the runner-up perturbed score
 *                 logits/T + g; +inf when no decision was taken, NaN for a
 *                 bad temperature. The kernel's fp32 q values carry a
 *                 relative error of about 1e-5 at most, which moves a child
 *                 test's threshold by about 1e-5 / R: a decision whose
 *                 margin is below that could go the other way in exact
 *                 arithmetic, and this output lets a caller see such
 *                 near-threshold requests. [Branch] Output Knowledge
 *                 Created, item 5 (debug metrics).
 * Logits must be finite.
 * Device errors: DDT_DEV_BAD_TEMPERATURE (that request emits nothing:
 * accept_len 0, bonus -1), DDT_DEV_BAD_TREE.
 */
int ddtree_accept_sample(const float* logits, int V, const int32_t* token,
                         const int32_t* first_child, const int32_t* next_sibling,
                         const int32_t* n_nodes, int B, int N, int D,
                         const float* temperature, const uint64_t* seed,
                         uint64_t philox_offset, int32_t* accept_len,
                         int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus,
                         float* margin_stats, int32_t* walk_stats,
                         int32_t* dev_status, void* stream);

/*
 * ddtree_accept_greedy_sample - ddtree_accept_greedy and ddtree_accept_sample
 * of the same tree and logits in one launch.
 *
 * [Arch] Section 1 step 5 and Section 3: the two walks are the ones the two
 * calls above make; this entry point runs them side by side, one round per
 * tree level, so that both share each round's synchronisation and, while
 * they stand on the same node, its logits row. The pages have no such call:
 * it exists because a verify step that needs both results (a serving loop
 * that verifies greedy and sampled requests of one batch, or a caller that
 * reports both) would otherwise pay two latency-bound launches that do not
 * overlap on the GPU.
 *
 * Inputs: as ddtree_accept_sample (temperature, seed and philox_offset are
 * used by the temperature walk only).
 * Outputs: greedy_* as ddtree_accept_greedy's outputs, sample_* as
 * ddtree_accept_sample's (both *_walk_stats and sample_margin_stats
 * nullable); every output is bit-identical to the one the separate call
 * writes for the same inputs. Device errors: the union of the two calls'.
 * Errors: as the two calls (the same argument checks, applied to both output
 * sets).
 * The kernel is launched as a programmatic dependent of the work before it
 * on the stream and reads nothing until that work's grid has completed, so
 * only its launch overlaps (the split-KV merge of tree_verify_attn lets it
 * start early).
 */
int ddtree_accept_greedy_sample(const float* logits, int V, const int32_t* token,
                                const int32_t* first_child, const int32_t* next_sibling,
                                const int32_t* n_nodes, int B, int N, int D,
                                const float* temperature, const uint64_t* seed,
                                uint64_t philox_offset,
                                int32_t* greedy_accept_len, int32_t* greedy_out_tokens,
                                int32_t* greedy_out_nodes, int32_t* greedy_bonus,
                                int32_t* greedy_walk_stats,
                                int32_t* sample_accept_len, int32_t* sample_out_tokens,
                                int32_t* sample_out_nodes, int32_t* sample_bonus,
                                float* sample_margin_stats, int32_t* sample_walk_stats,
                                int32_t* dev_status, void* stream);

/*
 * ddtree_accept_sample_ratio - the temperature walk with the draft-ratio rule.
 *
 * [Arch] Section 3 (linear case: accept draft token t with probability
 * min(1, p_target(t) / p_draft(t)), else resample from the residual; tree
 * case: reject-sample the children, bonus from the residual); [Verify] The
 * Knowledge Required, item 3; [Arch] Mistakes and Incorrect Assumptions (the
 * rule needs the draft's full distribution): this call takes the draft
 * logits. At node u (depth d): q = softmax(logits[b, u] / T),
 * p = softmax(draft_logits[b, d] / T) (the row the children were taken from).
 * Children are tested in rank order against a residual r that starts at q:
 * child j (token x) is accepted when U_j * p(x) < r(x), i.e. with probability
 * min(1, r(x) / p(x)); after a rejection r <- normalise(max(r - p, 0)). Once
 * every child is rejected (or at a node without children) the bonus is drawn
 * from r by Gumbel-max; if a rejection leaves r without mass, from q. With
 * candidates drawn independently from p the emitted tokens follow q; a
 * top-k-1 tree is linear speculative sampling. Cost: one pass over the
 * target and draft rows per visited node, one more per rejection.
 *
 * Inputs and outputs as ddtree_accept_sample, plus
 *   draft_logits  fp32 [B, D, V]   as given to ddtree_draft_topk
 * Randomness: the counters of ddtree_accept_sample (child test: purpose 0,
 * node u, slot j, word 0; Gumbel noise of token v: purpose 1, node u, index
 * v >> 2, word v & 3). A child whose token is outside [0, V) sets
 * DDT_DEV_BAD_TOKEN and is skipped. margin_stats (nullable, [B]) is the
 * smallest |U_j - r(x_j) / p(x_j)| over the child tests and the bonus's
 * top-2 gap of log r + g; walk_stats (nullable, [B, 4]) as
 * ddtree_accept_sample. Precision: q and p are fp32, c and R fp64, and each
 * residual max(q - c p, 0) is one fused multiply-add; after rejections the
 * threshold r(x)/p(x) inherits the fp32 error of q and p amplified by
 * (1 + c) / R (measured at most 6e-6 (1 + c) / R). Device errors as
 * ddtree_accept_sample.
 */
int ddtree_accept_sample_ratio(const float* logits, const float* draft_logits, int V,
                               const int32_t* token, const int32_t* first_child,
                               const int32_t* next_sibling, const int32_t* n_nodes,
                               int B, int N, int D, const float* temperature,
                               const uint64_t* seed, uint64_t philox_offset,
                               int32_t* accept_len, int32_t* out_tokens,
                               int32_t* out_nodes, int32_t* bonus, float* margin_stats,
                               int32_t* walk_stats, int32_t* dev_status, void* stream);

/*
 * ddtree_commit_kv - append the committed path's K/V to the paged cache.
 *
 * [Arch] Section 1, step 5: only the single longest verified path is
 * committed; the other tree nodes are dropped. [Branch] Hypothesis 3: a node
 * of depth d was verified at position ctx_len + d. Path row i (i = 0 is the
 * root, whose K/V this verify pass computed, then the accepted nodes) is
 * written to token position t = ctx_len[b] + i, i.e. slot t % page_size of
 * page page_table[b, t / page_size]. The bonus token is not written: it is
 * the next step's root. Then new_ctx_len[b] = ctx_len[b] + accept_len[b] + 1.
 *
 * Inputs
 *   k_tree, v_tree  bf16 [B, N, Hkv, Dh]   as given to tree_verify_attn
 *   out_nodes       int32 [B, D+1]         from either accept walk
 *   accept_len      int32 [B]
 *   page_table      int32 [B, max_pages]   must already map the positions up
 *                                          to ctx_len + accept_len
 *   ctx_len         int32 [B]
 * In/out
 *   k_cache, v_cache bf16 [num_pages, page_size, Hkv, Dh]: only the slots of
 *                   the committed positions are written
 * Outputs
 *   new_ctx_len     int32 [B]; may be the same array as ctx_len (advanced in
 *                   place: each request's length is read before it is
 *                   written)
 * The four K/V pointers must be 16-byte aligned; Hkv * Dh % 8 == 0.
 * Device errors: accept_len outside [0, D] or a path row outside [0, N) sets
 * DDT_DEV_BAD_TREE; ctx_len < 0 or ctx_len + accept_len + 1 beyond
 * max_pages * page_size sets DDT_DEV_BAD_CTX; a page id outside the pool sets
 * DDT_DEV_BAD_PAGE. Such a request writes no slot and keeps its length.
 */
int ddtree_commit_kv(const ddtree_bf16* k_tree, const ddtree_bf16* v_tree,
                     const int32_t* out_nodes, const int32_t* accept_len,
                     int B, int N, int D, int Hkv, int Dh,
                     ddtree_bf16* k_cache, ddtree_bf16* v_cache, int num_pages,
                     int page_size, const int32_t* page_table, int max_pages,
                     const int32_t* ctx_len, int32_t* new_ctx_len,
                     int32_t* dev_status, void* stream);

/*
 * ddtree_step_* - the whole verify step as one CUDA graph.
 *
 * [Arch] Section 1, steps 2-5 (build, one target pass over the tree, walk,
 * commit) as a single launch. [Pivot] The Strategic Decision: the verify
 * path is to run under CUDA graphs; [Verify] its CUDA-graph considerations:
 * the walk stays on the GPU so that the step can be captured. Capture needs
 * fixed shapes and no allocation or synchronisation inside, which every call
 * here keeps. ddtree_step_create records, on a stream of its
 * own, the calls
 *   ddtree_build -> tree_verify_attn -> ddtree_accept_greedy (walk = 0) or
 *   ddtree_accept_sample (walk = 1) -> ddtree_commit_kv
 * with the arguments below (each call checks them as it does alone; the
 * first failure is returned and no graph is kept), and instantiates the
 * graph. ddtree_step_launch replays it on `stream`: every launch reads the
 * arrays' current contents (the pointers are fixed at creation). The commit
 * writes new_ctx_len, or advances ctx_len in place when new_ctx_len is NULL,
 * so that consecutive launches decode consecutive steps.
 * ddtree_step_create allocates the graph (host and driver memory, no device
 * buffer); launches allocate nothing. ddtree_step_destroy frees it (NULL is
 * ignored). A step object may be launched from one host thread at a time.
 */
typedef struct ddtree_step_args {
    /* sizes */
    int B, D, K, budget, V, Hq, Hkv, Dh, num_pages, page_size, max_pages;
    float scale;                 /* attention scale                          */
    int walk;                    /* 0 greedy, 1 sampled, 2 draft-ratio walk  */
    uint64_t philox_offset;      /* sampled walk only                        */
    /* inputs (device) */
    const float* topk_logp;      /* [B, D, K]        ddtree_build            */
    const int32_t* topk_tok;     /* [B, D, K]                                */
    const int32_t* root_tok;     /* [B]                                      */
    int32_t* ctx_len;            /* [B]              read; advanced in place */
                                 /*                  if new_ctx_len is NULL  */
    const ddtree_bf16* q;        /* [B, N, Hq, Dh]   tree_verify_attn        */
    const ddtree_bf16* k_tree;   /* [B, N, Hkv, Dh]                          */
    const ddtree_bf16* v_tree;   /* [B, N, Hkv, Dh]                          */
    ddtree_bf16* k_cache;        /* [num_pages, page_size, Hkv, Dh]          */
    ddtree_bf16* v_cache;        /* [num_pages, page_size, Hkv, Dh]          */
    const int32_t* page_table;   /* [B, max_pages]                           */
    const float* logits;         /* [B, N, V]        the walk                */
    const float* temperature;    /* [B]              sampled walk only       */
    const uint64_t* seed;        /* [B]              sampled walk only       */
    const float* draft_logits;   /* [B, D, V]        draft-ratio walk only   */
    /* tree (ddtree_build outputs) */
    int32_t* parent; int32_t* depth; int32_t* token; int32_t* rank; int32_t* pos;
    double* score; int32_t* first_child; int32_t* next_sibling;
    uint32_t* vis; int32_t* n_nodes;
    /* attention */
    ddtree_bf16* attn_out;       /* [B, N, Hq, Dh]                           */
    float* lse;                  /* [B, N, Hq] or NULL                       */
    void* workspace;             /* tree_verify_attn_workspace_size(...)     */
    size_t workspace_bytes;      /*   with max_ctx = max_pages * page_size   */
    /* walk */
    int32_t* accept_len; int32_t* out_tokens; int32_t* out_nodes; int32_t* bonus;
    /* commit */
    int32_t* new_ctx_len;        /* [B] or NULL (in place)                   */
    int32_t* dev_status;         /* nullable                                 */
} ddtree_step_args;

typedef struct ddtree_step ddtree_step;

/* sizeof(ddtree_step_args), for bindings that mirror the struct */
size_t ddtree_step_args_size(void);
int ddtree_step_create(const ddtree_step_args* args, ddtree_step** out);
int ddtree_step_launch(ddtree_step* step, void* stream);
void ddtree_step_destroy(ddtree_step* step);

/*
 * The verify walks for a request split over GPUs by KV head (tensor
 * parallelism): ddtree_shard_walk_*.
 *
 * [Pivot] The Strategic Decision: TP8 (one request spread over the GPUs of a
 * node). [Arch] Section 1 step 1: the head is vocabulary-parallel, so each
 * rank holds the logits of its own vocabulary slice [v0, v0 + Vs) only. The
 * attention of such a request needs no exchange (each rank runs
 * tree_verify_attn on its own KV heads and their query heads); the walk needs
 * the argmax, the softmax denominator and the Gumbel-max over the whole
 * vocabulary at each visited node. These calls split each of those
 * reductions into a per-rank partial and a merge that every rank performs
 * identically, so all ranks take the same decisions; between them the
 * caller exchanges a few words per request (an all-gather over the ranks).
 * One level of the walk:
 *
 *   ddtree_shard_walk_partial   this rank's record per request (36 int32
 *                               words: the packed argmax key over the slice,
 *                               the slice's (max, sum of exp(logit/T - max)),
 *                               the logits of the current node's children
 *                               that lie in the slice, -inf for the others)
 *   all-gather of the records   -> [world, B, 36] on every rank
 *   ddtree_shard_walk_advance   merge in rank order; greedy: follow the child
 *                               matching the argmax, else emit the bonus;
 *                               sampled: the child tests of
 *                               ddtree_accept_sample, else mark the bonus due
 *   (sampled) ddtree_shard_walk_bonus   this rank's Gumbel-max key over its
 *                               slice for requests whose bonus is due
 *   all-gather of the keys      -> [world, B] int64
 *   (sampled) ddtree_shard_walk_finish  the bonus is the largest key
 *
 * D + 1 levels finish every request. ddtree_shard_walk_begin resets the state
 * and the outputs first. The results equal those of ddtree_accept_greedy /
 * ddtree_accept_sample on the whole vocabulary: bit for bit for the greedy
 * walk (the argmax key carries the global index, ties to the lowest), and for
 * the sampled walk with the same Philox counters (global vocabulary indices)
 * up to the fp32 rounding of the softmax denominator, which is merged over
 * ranks instead of over the walk kernel's thread-block cluster.
 *
 * Arguments: the tree arrays and outputs as ddtree_accept_greedy (token,
 * first_child, next_sibling, n_nodes [B, N]; accept_len [B], out_tokens and
 * out_nodes [B, D+1], bonus [B]); logits_shard fp32 [B, N, Vs] (this rank's
 * slice of every row); V the whole vocabulary; state int32 [B, 4] (current
 * node, accepted length, phase, child tests that did not accept) kept on the
 * device between calls; temperature NULL selects the greedy walk.
 * Device errors as the unsplit walks.
 */
int ddtree_shard_walk_begin(int B, int D, int32_t* state, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* out_nodes, int32_t* bonus, void* stream);
int ddtree_shard_walk_partial(const float* logits_shard, int Vs, int v0, int V, const int32_t* token,
                              const int32_t* first_child, const int32_t* next_sibling,
                              const int32_t* n_nodes, int B, int N, const float* temperature,
                              const int32_t* state, int32_t* record, void* stream);
int ddtree_shard_walk_advance(const int32_t* records, int world, int V, const int32_t* token,
                              const int32_t* first_child, const int32_t* next_sibling,
                              const int32_t* n_nodes, int B, int N, int D, const float* temperature,
                              const uint64_t* seed, uint64_t philox_offset, int32_t* state,
                              int32_t* accept_len, int32_t* out_tokens, int32_t* out_nodes, int32_t* bonus,
                              int32_t* dev_status, void* stream);
int ddtree_shard_walk_bonus(const float* logits_shard, int Vs, int v0, int V, const int32_t* token,
                            const int32_t* first_child, const int32_t* next_sibling, const int32_t* n_nodes,
                            int B, int N, const float* temperature, const uint64_t* seed,
                            uint64_t philox_offset, const int32_t* state, int64_t* key, void* stream);
int ddtree_shard_walk_finish(const int64_t* keys, int world, int B, int D, int32_t* state,
                             int32_t* accept_len, int32_t* out_tokens, int32_t* bonus, void* stream);

/*
 * tree_verify_attn_noalloc - tree_verify_attn without a caller workspace.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory at run time (for example a serving engine
 * that reserves nearly all of HBM for its own KV pool at start-up and gives
 * plugins no allocator, or a hot loop where a cudaMalloc would stall the
 * device). Arguments, outputs and results are those of tree_verify_attn
 * minus the workspace. The split-KV scratch comes from one fixed device array
 * inside the library, of tree_verify_attn_noalloc_max_scratch() bytes
 * (64 MiB), which every GPU that loads the library holds until the process
 * exits. The call allocates nothing and frees nothing.
 *
 * - Sizes whose scratch need (tree_verify_attn_workspace_size) exceeds the
 *   array are rejected with DDT_ESCRATCH before anything is launched.
 * - The first call on each device looks up the array's device address with
 *   that device current and caches it with the id of the current CUDA
 *   context; a call under another context (after cudaDeviceReset, say)
 *   looks it up again. Make the first call on a device, and the first after
 *   a reset, before any stream capture.
 * - All calls share the array and it keeps the last call's contents; every
 *   scratch word a call reads is written earlier in the same call, so nothing
 *   is cleared. Calls that overlap on the GPU (unordered streams, or several
 *   host threads) race on the array and must be serialised by the caller.
 */
int tree_verify_attn_noalloc(const ddtree_bf16* q, const ddtree_bf16* k_tree,
                             const ddtree_bf16* v_tree, const ddtree_bf16* k_cache,
                             const ddtree_bf16* v_cache, int num_pages, int page_size,
                             const int32_t* page_table, int max_pages,
                             const int32_t* ctx_len, const uint32_t* vis,
                             const int32_t* n_nodes, int B, int N, int Hq, int Hkv,
                             int Dh, float scale, ddtree_bf16* out, float* lse,
                             int32_t* dev_status, void* stream);

/* Size in bytes of the fixed scratch array behind tree_verify_attn_noalloc. */
size_t tree_verify_attn_noalloc_max_scratch(void);

#ifdef __cplusplus
}
#endif

#endif /* DDTREE_H */
