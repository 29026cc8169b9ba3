/*
 * specverify.h -- C ABI of the GB300 (sm_103a) one-pass tree-verification library.
 *
 * The library implements the target model's verification step of EAGLE-style
 * speculative decoding, as stated on these pages:
 *   - "EAGLE 演化史 (1 → 2 → 3) 与 DFlash 的回答", § Tree Verification 详解:
 *       A  one target forward pass verifies a whole draft tree;
 *       B  the tree is flattened in BFS order and given an attention mask in
 *          which a node sees the cached prefix, its ancestors and itself;
 *       C  the walk from the root: children in order, the rejection test,
 *          the residual after each rejected sibling, sampling from the
 *          residual when every child is rejected, the longest accepted path;
 *       G  the worked 7-node example.
 *   - "Eagle vs DFlash", § Target-model decoding is serial: accept x_i with
 *       probability min(1, p_i(x_i)/q_i(x_i)); on rejection sample from the
 *       normalised residual max(0, p_i - q_i); the bonus token.
 *   - "EAGLE-4 Technical Deepdive", § EAGLE-4 verification trees and harness:
 *       each token attends to the shared prefix, its ancestors and itself.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller; the
 *     library allocates no memory and keeps no pointer after a call returns.
 *   - Every call is asynchronous on the caller's CUDA stream (NULL = the
 *     legacy default stream). Nothing synchronises with the host.
 *   - Arrays are dense and row-major in the order their shapes are written.
 *   - The tree of sequence b is given by parent[b][0..N): node 0 is the root
 *     (parent -1) and 0 <= parent[i] < i for i >= 1 (BFS order). N counts the
 *     root. Node i's K/V sits at logical token position seq_lens[b] + i.
 *   - The host return code reports argument and launch errors only
 *     (svf_status). Data errors found on the device (a bad parent[], a token
 *     outside the vocabulary, a page id outside the cache) set bits in the
 *     caller's int32 status[B] array (SVF_DEV_*); that sequence's outputs are
 *     then written as defined "no result" values and the other sequences are
 *     unaffected. Each call overwrites status[0..B).
 *   - B == 0 is a valid empty call: nothing is launched and SVF_OK returned.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without the CUDA headers. */
typedef struct CUstream_st *svf_stream_t;

/* Element types of q, K, V and the attention output. */
enum svf_dtype { SVF_F32 = 0, SVF_BF16 = 1 };

/* Host return codes. */
enum svf_status {
    SVF_OK = 0,
    SVF_ERR_ARG = -1,         /* null pointer, negative size, bad alignment */
    SVF_ERR_UNSUPPORTED = -2, /* sizes outside the limits stated per call */
    SVF_ERR_LAUNCH = -3,      /* a CUDA launch or driver call failed */
    SVF_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
    SVF_ERR_SCRATCH_LIMIT = -5 /* request larger than svf_spec_accept_noalloc's fixed scratch */
};

/* Device-side status bits, OR-ed into status[b]. */
enum svf_device_status {
    SVF_DEV_BAD_PARENT = 1, /* parent[b] is not a BFS-flattened tree */
    SVF_DEV_BAD_TOKEN = 2,  /* a draft token (node >= 1) outside [0, V) */
    SVF_DEV_BAD_PAGE = 4,   /* a needed page id outside [0, num_pages) */
    SVF_DEV_BAD_LENGTH = 8, /* seq_lens[b] < 0 or the sequence overflows its page table */
    SVF_DEV_TIMEOUT = 16,   /* an internal wait gave up (the outputs of b are undefined) */
    SVF_DEV_BAD_PATH = 32,  /* accept_len or path[b] is not a root path in BFS order */
    SVF_DEV_BAD_CLUSTER = 64 /* a kernel ran without the thread-block cluster it was
                                launched for (e.g. re-launched by a tool that drops the
                                cluster attribute); it did no work, outputs undefined */
};

/* ------------------------------------------------------------------------
 * svf_tree_mask_build -- ancestor bitmasks of BFS-flattened draft trees.
 *
 * Follows "EAGLE 演化史", § Tree Verification 详解, B: each node may attend
 * only to its ancestors and itself. With W = ceil(N / 64):
 *   anc[b][i][w] bit k  set  <=>  node 64*w + k is node i or an ancestor of i
 *   depth[b][i]              =  number of edges from the root to node i
 *
 *   parent  [B, N] int32     in
 *   anc     [B, N, W] uint64 out
 *   depth   [B, N] int32     out, may be NULL
 *   status  [B] int32        out; SVF_DEV_BAD_PARENT if parent[b][0] != -1 or
 *                            some parent[b][i] is outside [0, i). Then every
 *                            node of b gets only its own bit and depth 0.
 * Limits: 1 <= N <= 1024.
 * ---------------------------------------------------------------------- */
int svf_tree_mask_build(const int32_t *parent, int B, int N, uint64_t *anc, int32_t *depth,
                        int32_t *status, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_tree_verify_attn -- attention of a flattened draft tree against a
 * cached KV prefix, one target layer, grouped-query heads.
 *
 * Follows "EAGLE 演化史", § Tree Verification 详解, A-B (one forward pass
 * over prefix + tree; ancestor-only mask; the output of node i equals running
 * prompt + root->i path as an ordinary causal sequence) and "EAGLE-4
 * Technical Deepdive" (prefix, ancestors and self are visible). For sequence
 * b, query head h, node i, with G = Hq / Hkv and KV head g = h / G, the
 * visible tokens are t < L_b = seq_lens[b] and t = L_b + j for every j whose
 * bit is set in anc[b][i]:
 *   s_t = sm_scale * <q[b][i][h], K_b,g(t)>
 *   out[b][i][h] = sum_t softmax(s)_t V_b,g(t),   lse[b][i][h] = log sum_t e^{s_t}
 *
 *   q          [B, N, Hq, D]                      dtype (post-RoPE)
 *   k_cache,   [num_pages, page_size, Hkv, D]     dtype; token t of sequence
 *   v_cache                                        b lives in page
 *                                                  page_table[b][t / page_size],
 *                                                  slot t % page_size. The
 *                                                  tree's K/V must already be
 *                                                  written at t = L_b .. L_b+N-1.
 *   page_table [B, max_pages] int32               entries past the sequence's
 *                                                  last page are not read
 *   seq_lens   [B] int32                          L_b, the prefix length
 *   anc        [B, N, 1] uint64                   from svf_tree_mask_build
 *   sm_scale   <= 0 selects 1/sqrt(D)
 *   out        [B, N, Hq, D] dtype                out
 *   lse        [B, N, Hq] float32                 out, may be NULL (natural log)
 *   workspace  device scratch of svf_tree_verify_attn_workspace_size(...)
 *              bytes, ZERO-FILLED once before its first use. For SVF_BF16
 *              with Hq / Hkv a power of two it holds the pieces of the units
 *              that the persistent kernel splits between SMs (two slots per
 *              SM) and a pair of counters per unit, which every call leaves
 *              at zero again; a workspace that is large enough for one shape
 *              is reused as is by any call whose size fits in it. Calls that
 *              may overlap on the GPU need workspaces of their own. NULL (or
 *              fewer bytes) selects the kernel that merges a unit's KV chunks
 *              on chip, inside a thread-block cluster, which needs none;
 *              SVF_F32 needs none.
 *   status     [B] int32                          out; SVF_DEV_BAD_LENGTH,
 *                                                  SVF_DEV_BAD_PAGE. A bad
 *                                                  sequence's out and lse are 0.
 * A contiguous cache is page_size = capacity, num_pages = B, page_table[b][0] = b.
 * Limits: N <= 64; D in {64, 128} for SVF_F32, D == 128 for SVF_BF16;
 * Hq % Hkv == 0; for SVF_BF16 page_size in {16, 32, 64} or a multiple of 128,
 * q / k_cache / v_cache 16-byte aligned. Bytes past a sequence's last token
 * inside its last page may hold anything.
 * ---------------------------------------------------------------------- */
size_t svf_tree_verify_attn_workspace_size(int B, int N, int Hq, int Hkv, int D, int dtype,
                                           int max_pages, int page_size);
int svf_tree_verify_attn(const void *q, const void *k_cache, const void *v_cache, int num_pages,
                         int page_size, const int32_t *page_table, int max_pages,
                         const int32_t *seq_lens, const uint64_t *anc, int B, int N, int Hq,
                         int Hkv, int D, int dtype, float sm_scale, void *out, float *lse,
                         void *workspace, size_t workspace_bytes, int32_t *status,
                         svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_tree_mask_attn -- svf_tree_mask_build and svf_tree_verify_attn in one
 * call: the ancestor masks are built from parent[] where the attention needs
 * them ("EAGLE 演化史", § Tree Verification 详解, B: a node sees its
 * ancestors and itself; A: one pass verifies the whole tree).
 *
 * Arguments are those of the two calls: parent [B, N] int32 in; anc
 * [B, N, 1] uint64, depth [B, N] int32 and mask_status [B] int32 get exactly
 * what svf_tree_mask_build writes (for SVF_BF16 each may be NULL; for
 * SVF_F32 anc and mask_status are required, since that path reads the masks
 * from memory); the attention arguments and outputs are svf_tree_verify_attn's
 * (its anc argument is replaced by parent; workspace sizes are the same).
 * For SVF_BF16 one kernel does both: its prologue checks the tree and walks
 * every node's parent links in shared memory. Limits: those of
 * svf_tree_verify_attn (N <= 64).
 * ---------------------------------------------------------------------- */
int svf_tree_mask_attn(const int32_t *parent, uint64_t *anc, int32_t *depth,
                       int32_t *mask_status, const void *q, const void *k_cache,
                       const void *v_cache, int num_pages, int page_size,
                       const int32_t *page_table, int max_pages, const int32_t *seq_lens, int B,
                       int N, int Hq, int Hkv, int D, int dtype, float sm_scale, void *out,
                       float *lse, void *workspace, size_t workspace_bytes, int32_t *status,
                       svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept -- lossless acceptance walk over the verified tree.
 *
 * Follows "Eagle vs DFlash" (accept x with probability min(1, p(x)/q(x));
 * on rejection, sample from normalize(max(0, p - q))) and "EAGLE 演化史",
 * § Tree Verification 详解, C and G (walk from the root; try children in
 * order, after each rejected child replace the target side by the residual
 * and test the next sibling; when all are rejected sample there; the bonus
 * token is drawn at the last accepted node). With p_j = softmax(target[b][j])
 * and q_j = softmax(draft[b][j]) (temperature 1):
 *   - start at the root with p~ = p_0;
 *   - for each child c of the current node j in ascending index order, with
 *     x = tokens[b][c]: accept iff u_accept[b][c] * q_j(x) < p~(x). On accept
 *     move to c with p~ = p_c. On reject set p~ = normalize(max(0, p~ - q_j))
 *     (left unchanged if that has no mass) and try the next sibling;
 *   - when the current node has no child left, the bonus token is the
 *     smallest k with sum_{v<=k} p~(v) > u_bonus[b] * sum_v p~(v).
 *
 *   target_logits, draft_logits [B, N, V] float32   rows of leaves in draft
 *                                                    are not read
 *   tokens     [B, N] int32   node i's draft token (the root's is not read)
 *   parent     [B, N] int32
 *   u_accept   [B, N] float32 in [0, 1)   u_accept[b][c] tests node c
 *   u_bonus    [B] float32 in [0, 1)
 *   accept_len [B] int32      out: accepted draft tokens (root excluded)
 *   path       [B, N] int32   out: 0, then the accepted nodes, then -1
 *   out_tokens [B, N] int32   out: accepted draft tokens, the bonus, then -1
 *   ratio      [B, N] float32 out, may be NULL: p~(x)/q_j(x) for every tested
 *                             node, NaN for nodes never tested
 *   workspace  at least svf_spec_accept_workspace_size(B, N, V) bytes; that
 *              size is 0 (workspace may be NULL) for V <= 262144, whose
 *              rows the walk holds on chip. Larger vocabularies stream
 *              their rows from memory after a statistics pre-pass that
 *              keeps per-(row, chunk) results in the workspace.
 *   status     [B] int32      out: SVF_DEV_BAD_PARENT, SVF_DEV_BAD_TOKEN; a
 *                             bad sequence gets accept_len 0 and -1 in path
 *                             and out_tokens (ratio NaN).
 * Limits: 1 <= N <= 1024, 1 <= V <= 786432.
 * ---------------------------------------------------------------------- */
size_t svf_spec_accept_workspace_size(int B, int N, int V);
int svf_spec_accept(const float *target_logits, const float *draft_logits, const int32_t *tokens,
                    const int32_t *parent, const float *u_accept, const float *u_bonus, int B,
                    int N, int V, int32_t *accept_len, int32_t *path, int32_t *out_tokens,
                    float *ratio, void *workspace, size_t workspace_bytes, int32_t *status,
                    svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept_noalloc -- svf_spec_accept for callers that cannot provide
 * device scratch memory.
 *
 * The pages have no counterpart to this call. It is here for users of the
 * library who have no way to allocate device memory where they run the
 * acceptance step: an inference runtime that gives a plugin only its input
 * and output buffers, or a serving loop that reserved all device memory at
 * start-up and must not allocate (or risk an allocation's implicit
 * synchronisation) afterwards.
 *
 * Arguments, layouts, results and status bits are those of svf_spec_accept,
 * without the workspace. Vocabularies up to 262144 need no scratch at all;
 * for larger ones the streaming kernels' scratch lives in one 4 MiB array
 * that the library itself defines in device memory; every GPU that loads
 * the library holds it until the process exits. The call allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - Limits: those of svf_spec_accept, and a request whose scratch
 *     (svf_spec_accept_workspace_size(B, N, V)) exceeds 4 MiB returns
 *     SVF_ERR_SCRATCH_LIMIT without launching anything.
 *   - The first call on a device looks up that array's device address (once
 *     per device and context, with the device current), and a new context
 *     on the device (after cudaDeviceReset, say) gets a new lookup. With
 *     lazy module loading that first call may be where the library's device
 *     code, and with it the 4 MiB array, is loaded: it can reserve that
 *     memory and synchronise. The guarantee of no allocation and no
 *     implicit synchronisation holds from the second call on a device. Make
 *     that first call before any stream capture begins.
 *   - Every call shares the one array. Calls that overlap on the GPU (on
 *     different streams, or from different host threads without ordering)
 *     race on it and corrupt each other's results; order them. Nothing in
 *     the array needs to start at zero: each call writes every entry it
 *     reads.
 * ---------------------------------------------------------------------- */
int svf_spec_accept_noalloc(const float *target_logits, const float *draft_logits,
                            const int32_t *tokens, const int32_t *parent, const float *u_accept,
                            const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                            int32_t *path, int32_t *out_tokens, float *ratio, int32_t *status,
                            svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept_bf16 -- svf_spec_accept on bf16 logits.
 *
 * The same walk, rule and outputs as svf_spec_accept ("Eagle vs DFlash" and
 * "EAGLE 演化史", § C); the logits rows are bf16 (raw bits, [B, N, V]) and
 * are widened exactly to fp32 as they are read, so the result is
 * svf_spec_accept's on the widened values. Reads half the bytes per visited
 * row. No workspace.
 * Limits: 1 <= N <= 1024, 1 <= V <= 262144 (rows held on chip); both logits
 * arrays 8-byte aligned when V % 4 == 0.
 * ---------------------------------------------------------------------- */
int svf_spec_accept_bf16(const void *target_logits, const void *draft_logits,
                         const int32_t *tokens, const int32_t *parent, const float *u_accept,
                         const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                         int32_t *path, int32_t *out_tokens, float *ratio, int32_t *status,
                         svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept_greedy -- temperature-0 acceptance over the tree.
 *
 * "Eagle vs DFlash", § A fair evaluation protocol: greedy speculative
 * decoding must reproduce a target-only greedy run. From the root, let a be
 * the argmax of the current node's target logits (equal maxima: the lowest
 * token id); accept the first child, in ascending node index, whose token is
 * a and continue there; stop when no child carries a. The bonus token is the
 * last a. Only the target rows of visited nodes are read.
 *   target_logits [B, N, V] float32, tokens / parent [B, N] int32 (as for
 *   svf_spec_accept); outputs accept_len [B], path [B, N], out_tokens [B, N]
 *   and status [B] as for svf_spec_accept (same status bits and "no result"
 *   values).
 * Limits: 1 <= N <= 1024, 1 <= V <= 786432 (up to 262144 a cluster holds
 * the visited node's row in registers; above that each CTA streams its
 * slice of the row from memory on every pass: one per visited node, and
 * for the one-hot bonus one more plus the crossing group's); target_logits
 * 16-byte aligned when V % 4 == 0. No workspace.
 * ---------------------------------------------------------------------- */
int svf_spec_accept_greedy(const float *target_logits, const int32_t *tokens,
                           const int32_t *parent, int B, int N, int V, int32_t *accept_len,
                           int32_t *path, int32_t *out_tokens, int32_t *status,
                           svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept_onehot -- the sampling rule with one-hot draft
 * distributions, for deterministic (top-k) sibling candidates.
 *
 * "Eagle vs DFlash" gives the rule (accept x with probability
 * min(1, p(x)/q(x)); on rejection continue from normalize(max(0, p - q))).
 * With the draft's q shared by siblings it is exact only when the siblings
 * are independent draws from q; this call takes q = one-hot(candidate) for
 * every child instead, which keeps the output distributed as the target's
 * for any fixed candidate set. Child c with token x is accepted iff
 * u_accept[b][c] < p~(x); a rejection gives p~ <- normalize(max(0, p~ -
 * one-hot(x))), i.e. x loses its mass; when every child of the current node
 * is rejected, or at a leaf, the bonus token is the inverse CDF of p~ at
 * u_bonus[b] (smallest k whose cumulative p~ exceeds u * sum p~). Only the
 * target rows of visited nodes are read.
 *   Arguments and outputs as for svf_spec_accept without draft_logits and
 *   workspace; ratio [B, N] (may be NULL) gets p~(x) = p~(x)/q(x) for every
 *   tested child, NaN otherwise.
 * Limits: 1 <= N <= 1024, 1 <= V <= 786432 (up to 262144 a cluster holds
 * the visited node's row in registers; above that each CTA streams its
 * slice of the row from memory on every pass: one per visited node, and
 * for the one-hot bonus one more plus the crossing group's); target_logits
 * 16-byte aligned when V % 4 == 0. No workspace.
 * ---------------------------------------------------------------------- */
int svf_spec_accept_onehot(const float *target_logits, const int32_t *tokens,
                           const int32_t *parent, const float *u_accept, const float *u_bonus,
                           int B, int N, int V, int32_t *accept_len, int32_t *path,
                           int32_t *out_tokens, float *ratio, int32_t *status,
                           svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept_greedy_bf16, svf_spec_accept_onehot_bf16 -- the same two
 * rules on bf16 target logits (target_logits [B, N, V] bf16, each value
 * widened exactly to fp32 on load; the arithmetic and the outputs are those
 * of the fp32 calls on the widened logits). Limits as for the fp32 calls,
 * with target_logits 8-byte aligned when V % 4 == 0.
 * ---------------------------------------------------------------------- */
int svf_spec_accept_greedy_bf16(const void *target_logits, const int32_t *tokens,
                                const int32_t *parent, int B, int N, int V, int32_t *accept_len,
                                int32_t *path, int32_t *out_tokens, int32_t *status,
                                svf_stream_t stream);
int svf_spec_accept_onehot_bf16(const void *target_logits, const int32_t *tokens,
                                const int32_t *parent, const float *u_accept,
                                const float *u_bonus, int B, int N, int V, int32_t *accept_len,
                                int32_t *path, int32_t *out_tokens, float *ratio,
                                int32_t *status, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * EAGLE-2 dynamic draft-tree construction.
 *
 * "EAGLE 演化史", § E.2-E.3, and "The EAGLE Family" (EAGLE-2): a node's value
 * is the product of the draft confidences on its root path, a confidence
 * being the draft softmax probability of the node's own token. Each round
 * expands the k most valuable nodes of the previous round into their k most
 * probable draft tokens; rerank keeps the N most valuable nodes (a connected
 * subtree) and flattens them in BFS order for verification. The drafter runs
 * between rounds, so the build is a sequence of calls on a node pool per
 * sequence, all on one stream:
 *   svf_eagle2_init      root (pool id 0, value 1, depth 0); count = 1
 *   svf_eagle2_expand    one round; round 1 expands frontier {0}
 *   svf_eagle2_finalize  rerank + BFS numbering -> parent[] / tokens
 *
 * Pool (device, caller-owned, [B, capacity] each, row b for sequence b;
 * capacity >= 1 + k + (rounds - 1) k^2 holds every node; the node with pool
 * id c is "creation id" c): pool_parent int32 (parent's id, -1 for the root),
 * pool_depth int32, pool_token int32, pool_value float64; pool_count [B]
 * int32 = nodes created so far.
 *
 * svf_eagle2_expand: draft_rows [B, R, V] float32, row r = the drafter's
 * logits at node frontier[b][r] (frontier [B, R] int32 pool ids, -1 entries
 * only after the valid ones; their rows are not read). For every valid
 * frontier node f, in order, its k most probable tokens (ties to the lower
 * id) become children with ids pool_count[b] + r k + i (i = rank), value
 * value(f) * softmax(row)[token]; pool_count advances by k per valid row
 * (capped at capacity; children past it are dropped). next_frontier [B, k]
 * int32 gets the ids of the k most valuable new children (value desc, id
 * asc), -1 padded: the nodes to draft from next. V <= 1048576 (else
 * SVF_ERR_UNSUPPORTED). status [B] int32 (device, may be NULL) is
 * overwritten: 0, or SVF_DEV_TIMEOUT when a wait of the row kernel gave up
 * (that sequence's new nodes are then undefined).
 *
 * svf_eagle2_finalize: keeps the root and the n_nodes - 1 most valuable other
 * nodes (value desc, depth asc, id asc) and numbers them level by level, a
 * level ordered by (parent's new index, value desc, id asc). Outputs
 * [B, n_nodes]: parent (new indices, -1 for the root), tokens, values
 * (float64), cids (pool ids); entries past n_out[b] (when the pool holds
 * fewer nodes) are -1 / 0.
 *
 * Limits: 1 <= k <= 16, k <= V; capacity <= 2048; 1 <= n_nodes <= 1024.
 * Confidences are computed in fp32 statistics with an fp64 final step; values
 * within ~1e-6 relative of each other may order differently from an exact
 * computation.
 * ---------------------------------------------------------------------- */
int svf_eagle2_init(const int32_t *root_tokens, int B, int capacity, int32_t *pool_parent,
                    int32_t *pool_depth, int32_t *pool_token, double *pool_value,
                    int32_t *pool_count, svf_stream_t stream);
int svf_eagle2_expand(const float *draft_rows, int B, int R, int V, int k,
                      const int32_t *frontier, int capacity, int32_t *pool_parent,
                      int32_t *pool_depth, int32_t *pool_token, double *pool_value,
                      int32_t *pool_count, int32_t *next_frontier, int32_t *status,
                      svf_stream_t stream);
int svf_eagle2_finalize(int B, int capacity, const int32_t *pool_parent,
                        const int32_t *pool_depth, const int32_t *pool_token,
                        const double *pool_value, const int32_t *pool_count, int n_nodes,
                        int32_t *parent, int32_t *tokens, double *values, int32_t *cids,
                        int32_t *n_out, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_kv_commit -- keep the accepted path's K/V and roll back the rejected
 * nodes' entries.
 *
 * Follows "EAGLE-4 Technical Deepdive", § EAGLE-4 verification trees and
 * harness (after verification the accepted continuation is kept and the
 * KV-cache entries of rejected nodes are freed) and "EAGLE 演化史", § D.2
 * (every tree node writes its own K/V in the verification pass; entries of
 * nodes that fail must not stay in the cache, which is rolled back page by
 * page). For every layer l, sequence b and k = 0 .. accept_len[b]:
 *   token L_b + k  <-  token L_b + path[b][k]     (K and V, all heads)
 * with every source read before its destination is written, so tokens
 * L_b .. L_b + accept_len[b] hold the root and the accepted nodes in path
 * order. Tokens before L_b and past L_b + accept_len[b] are not written.
 *
 *   k_cache,    layer l at k_cache + l * layer_stride elements, each layer
 *   v_cache     [num_pages, page_size, Hkv, D] dtype, paged as in
 *               svf_tree_verify_attn (token t of b in page
 *               page_table[b][t / page_size], slot t % page_size); 16-byte
 *               aligned; updated in place
 *   layer_stride  elements between layers, >= num_pages * page_size * Hkv * D
 *               when num_layers > 1 (ignored for one layer)
 *   seq_lens   [B] int32    L_b, the prefix length before the tree
 *   path       [B, N] int32, accept_len [B] int32: svf_spec_accept's outputs
 *   new_seq_lens [B] int32  out: L_b + accept_len[b] + 1 (root + accepted)
 *   freed_pages [B, max_free] int32  out, may be NULL when max_free is 0: ids
 *               of the pages that held tree entries and hold no committed
 *               token now (page-table indices ceil(new_len / page_size) ..
 *               ceil((L_b + N) / page_size) - 1, in order), -1 after them;
 *               max_free >= ceil(N / page_size) holds every case
 *   n_freed    [B] int32    out, may be NULL: that count
 *   status     [B] int32    out; SVF_DEV_BAD_PATH (accept_len outside
 *               [0, N-1], path[0] != 0, or path not strictly increasing
 *               inside [0, N)), SVF_DEV_BAD_LENGTH (L_b < 0 or L_b + N past
 *               the page table), SVF_DEV_BAD_PAGE (a page of tokens
 *               [L_b, L_b + N) outside [0, num_pages)). A flagged sequence's
 *               cache is not written, new_seq_lens[b] = L_b and nothing is
 *               freed.
 * The pages of tokens [L_b, L_b + N) must be distinct and belong to b alone;
 * otherwise the cache contents are undefined (nothing faults).
 * Limits: 1 <= N <= 1024, 1 <= num_layers <= 65535, Hkv * D * element size a
 * multiple of 16 bytes, dtype SVF_F32 or SVF_BF16.
 * ---------------------------------------------------------------------- */
int svf_kv_commit(void *k_cache, void *v_cache, int num_layers, long long layer_stride,
                  int num_pages, int page_size, const int32_t *page_table, int max_pages,
                  const int32_t *seq_lens, const int32_t *path, const int32_t *accept_len, int B,
                  int N, int Hkv, int D, int dtype, int32_t *new_seq_lens, int32_t *freed_pages,
                  int max_free, int32_t *n_freed, int32_t *status, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_selftest_wait_timeout -- a diagnostic: make a bounded wait run out.
 *
 * Every wait of this library's kernels on an mbarrier (for a TMA copy, a
 * tensor-core commit, another warp or another CTA of a cluster) gives up
 * after a deadline (2 s in the product kernels); the waiting CTA then leaves
 * its loops, releases what it holds and sets SVF_DEV_TIMEOUT in the
 * caller's status word, and the CUDA context stays usable. This call runs
 * the same wait helpers, with deadline_ns (1 us .. 1 s), on mbarriers that
 * nothing ever completes: one inside a CTA and one that a peer CTA of a
 * two-CTA cluster would complete. result [4] int32 (device): status of the
 * CTA wait, its elapsed microseconds, status of the cluster wait, its
 * elapsed microseconds; both statuses are SVF_DEV_TIMEOUT when the waits
 * are bounded. Nothing faults or traps.
 * ---------------------------------------------------------------------- */
int svf_selftest_wait_timeout(int32_t *result, long long deadline_ns, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_lm_head -- target logits of every tree node from its hidden state.
 *
 * "The EAGLE Family", § Why predict features instead of tokens?: the target
 * distribution at a node is softmax(W_LM h), h the node's last hidden
 * state; "EAGLE 演化史", § Tree Verification 详解, D.2 places the verify
 * pass's bandwidth cost in this LM head and the softmax over N·|V|.
 *   logits[r][v] = sum_k hidden[r][k] * weight[v][k]
 * bf16 operands, products accumulated in fp32 on the tensor cores, fp32
 * results; the weight is read from memory once per call.
 *   hidden  [R, H] bf16 (raw bits), row-major, 16-byte aligned   in
 *   weight  [V, H] bf16, row-major, 16-byte aligned              in
 *   logits  [R, V] fp32, row-major                               out
 *   status  [1] int32, nullable: SVF_DEV_TIMEOUT is OR-ed in if an
 *           internal wait gave up (logits are then undefined)
 * Limits: 1 <= R, V <= 2^24; H a multiple of 64, 64 <= H <= 65536.
 * Returns SVF_ERR_ARG for null or misaligned pointers, SVF_ERR_UNSUPPORTED
 * outside the limits. All memory is the caller's; nothing is allocated.
 * ---------------------------------------------------------------------- */
int svf_lm_head(const void *hidden, const void *weight, int R, int H, int V, float *logits,
                int32_t *status, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_spec_accept_lmhead -- the LM head and the acceptance walk in one call.
 *
 * The target rows of svf_spec_accept are produced here from the nodes'
 * hidden states ("The EAGLE Family", § Why predict features instead of
 * tokens?: p = softmax(W_LM h)): svf_lm_head writes every node's fp32
 * logits into target_logits, then the walk of svf_spec_accept ("Eagle vs
 * DFlash", § Target-model decoding is serial; "EAGLE 演化史", § C) reads the
 * rows of the nodes it visits. The two kernels are chained on the stream.
 *   hidden        [B, N, H] bf16 in      weight [V, H] bf16 in
 *   draft_logits  [B, N, V] fp32 in      target_logits [B, N, V] fp32 out
 *   tokens, parent, u_accept, u_bonus, accept_len, path, out_tokens,
 *   ratio, status: as svf_spec_accept.
 *   lm_status     [1] int32, nullable: the LM head's SVF_DEV_TIMEOUT bit.
 * Limits: those of svf_lm_head with R = B*N, and of svf_spec_accept with a
 * vocabulary the walk holds on chip (V <= 262144), so no workspace.
 * ---------------------------------------------------------------------- */
int svf_spec_accept_lmhead(const void *hidden, const void *weight, const float *draft_logits,
                           const int32_t *tokens, const int32_t *parent, const float *u_accept,
                           const float *u_bonus, int B, int N, int H, int V,
                           float *target_logits, int32_t *accept_len, int32_t *path,
                           int32_t *out_tokens, float *ratio, int32_t *lm_status,
                           int32_t *status, svf_stream_t stream);

/* ------------------------------------------------------------------------
 * svf_debug_set_attn_wait_ns -- test hook: the deadline of every internal
 * wait of the bf16 (tensor-core) attention kernel, for later calls in this
 * process. The pages have no counterpart; it exists so that a test can make
 * a wait of the product kernel run out without any fault: the kernel then
 * leaves its loops, waits (with the default deadline) for its copies and
 * tensor-core operations in flight, releases its tensor memory and sets
 * SVF_DEV_TIMEOUT in status[b]; outputs of such a sequence are undefined
 * (zeros when its chunks merge in a cluster). ns <= 0 restores the default
 * of 2 s. Deadlines under 1 ms poll without blocking. Returns SVF_OK.
 * ---------------------------------------------------------------------- */
int svf_debug_set_attn_wait_ns(long long ns);

/* ------------------------------------------------------------------------
 * svf_debug_set_attn_splits -- test hook: the number of KV chunks per
 * (sequence, KV head, row block) of later bf16 attention calls in this
 * process, 1..8 (the CTAs of one cluster, merged on chip); 0 restores the
 * library's own choice. It changes how the work is divided, not the result
 * (which stays within the stated tolerance). The pages have no counterpart;
 * it lets tests run every cluster size on the same inputs. Returns SVF_OK,
 * or SVF_ERR_ARG outside 0..8.
 * ---------------------------------------------------------------------- */
int svf_debug_set_attn_splits(int splits);

/* ------------------------------------------------------------------------
 * svf_debug_set_attn_kernel -- test hook: which bf16 attention kernel later
 * calls in this process run. 0: the library's choice; 1: one CTA per (unit,
 * KV chunk), the chunks of a unit merged inside a thread-block cluster (no
 * workspace); 2: one persistent CTA per SM over an equal share of all units'
 * tiles, split units merged through the workspace (SVF_ERR_WORKSPACE without
 * one). A chunk count set with svf_debug_set_attn_splits selects kernel 1.
 * The result is the same within the stated tolerance. The pages have no
 * counterpart; it lets tests run both kernels on the same inputs. Returns
 * SVF_OK, or SVF_ERR_ARG outside 0..2.
 * ---------------------------------------------------------------------- */
int svf_debug_set_attn_kernel(int which);

/* Human-readable name of a host return code or of one device status bit. */
const char *svf_status_string(int code);

/* Library version, 100 * major + minor. */
int svf_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
