/*
 * graft.h — C ABI of the GB300 hybrid-tree verify-step library (libgraft.so).
 *
 * The library computes one verify step of hybrid-tree speculative decoding
 * as described by "Draft Less, Retrieve More: Hybrid Tree Construction for
 * Speculative Decoding" (the aitrends.kr article on it, cited below as the
 * Graft article, and the chatpaper.ai abstract, cited as the Graft
 * abstract):
 *
 *   graft_build_tree      prune the draft, fill the retrieval template from M
 *                         and merge both into one Kmax-node tree
 *   graft_retrieve        the retrieval fill alone
 *   graft_tree_attention  tree-masked GQA attention for one layer
 *   graft_accept_compact  greedy longest accepted path, KV compaction
 *   graft_update_M        online update of the adjacency table M
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a caller-owned DEVICE pointer unless marked
 *   "host".  The library never allocates, frees or retains memory: scratch
 *   space comes from a caller buffer `ws` of at least the size the matching
 *   *_workspace_size function reports (pointer aligned to 256 bytes).
 * - Every call is asynchronous on the caller's CUDA stream (`stream`, a
 *   cudaStream_t; NULL is the legacy default stream).  A return value of
 *   GRAFT_OK means the work was enqueued.
 * - Arguments are validated on the host before any launch; an invalid call
 *   returns a negative code and enqueues nothing.  Errors that depend on
 *   device data (token ids out of range, a cache that would overflow) are
 *   OR-ed as GRAFT_STATUS_* bits into the caller's device word `status`
 *   (may be NULL to ignore them), readable after the stream synchronises.
 * - bf16 tensors are IEEE bfloat16 stored as 16-bit words; all layouts are
 *   dense row-major in the order written, with no padding.
 * - Token ids are int32 in [0, V).  Node indices are int32 in [0, Kmax).
 */
#ifndef GRAFT_H_
#define GRAFT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, spelled without including CUDA headers. */
typedef struct CUstream_st* graft_stream_t;

/* Return codes. */
#define GRAFT_OK 0
#define GRAFT_ERR_INVALID_ARG (-1)      /* null pointer, negative size, inconsistent config */
#define GRAFT_ERR_UNSUPPORTED_SHAPE (-2) /* a size outside what the kernels handle (limits below) */
#define GRAFT_ERR_WORKSPACE (-3)        /* ws missing, too small or misaligned */
#define GRAFT_ERR_CUDA (-4)             /* a CUDA launch or device query failed */

/* Device status bits, OR-ed into *status by the kernels. */
#define GRAFT_STATUS_TOKEN_RANGE 1    /* a token id outside [0, V) was read; the node became a pad / the pair was skipped */
#define GRAFT_STATUS_CACHE_OVERFLOW 2 /* L[b] + accepted length > Lcap; that request was not compacted */
#define GRAFT_STATUS_LENGTH 4         /* L[b] < 0 or L[b] > Lcap; that request was skipped */
#define GRAFT_STATUS_TREE 8           /* a kept draft node's parent was not kept (cannot happen for finite logits) */
#define GRAFT_STATUS_TIMEOUT 16       /* a bounded wait inside a kernel expired; that CTA's output is incomplete */
#define GRAFT_STATUS_WORKSPACE 32     /* a workspace's arrival counter was found not zeroed (graft_build_tree, graft_tree_attention) */

/* Limits. */
#define GRAFT_MAX_KMAX 64        /* tree nodes per request (one uint64 ancestor mask) */
#define GRAFT_MAX_CHECKPOINTS 4  /* pruning checkpoints */
#define GRAFT_MAX_TOPK 16        /* draft branching k */
#define GRAFT_MAX_DEPTH 16       /* drafter calls D */
#define GRAFT_MAX_W 32           /* successors per row of M */
#define GRAFT_HEAD_DIM 128       /* the only head size the attention kernel supports */

/*
 * GraftConfig — the method's parameters (host struct, passed by pointer).
 *
 * Graft article, method paragraph (first point) and architecture paragraph:
 * pruning tests a per-depth confidence c_d against a threshold tau_d at
 * checkpoints d0, d1, d5, and each stage s splits the budget as
 * Kmax = K_draft_s + K_ret_s, a smaller s giving retrieval more; the
 * retrieval templates G_ret_s are per-stage prefixes of one envelope.
 *
 *   Kmax            tree nodes per request, root included (1..64)
 *   D, k            drafter calls and top-k branching of the draft tree
 *   V               vocabulary size; W successors per row of M
 *   n_checkpoints   number of pruning checkpoints (0..4)
 *   checkpoint[s]   drafter call (0-based) after which c is tested; strictly increasing, < D
 *   tau[s]          threshold: drafting stops at the first s with c_{checkpoint[s]} < tau[s]
 *   K_draft[s]      draft nodes kept (root included) when stopped at s;
 *                   K_draft[n_checkpoints] is the unpruned stage and must equal Kmax.
 *                   A value above 1 + the stage's pool (k + checkpoint[s] k^2
 *                   candidates) keeps the whole pool and leaves the rest of
 *                   the draft slots as empty nodes (see graft_config_no_retrieval)
 *   n_tmpl          envelope size = max_s (Kmax - K_draft[s])
 *   tmpl_parent[j]  parent of envelope node j: -1 = the root, else an index < j
 *   tmpl_rank[j]    rank (0..W-1) of node j among its parent token's successors in M
 */
typedef struct GraftConfig {
    int32_t Kmax, D, k, V, W;
    int32_t n_checkpoints;
    int32_t checkpoint[GRAFT_MAX_CHECKPOINTS];
    float tau[GRAFT_MAX_CHECKPOINTS];
    int32_t K_draft[GRAFT_MAX_CHECKPOINTS + 1];
    int32_t n_tmpl;
    int32_t tmpl_parent[GRAFT_MAX_KMAX];
    int32_t tmpl_rank[GRAFT_MAX_KMAX];
} GraftConfig;

/*
 * graft_config_init — fill *cfg (host) with the default budget split and
 * retrieval envelope for the given sizes.  Checkpoints >= D are dropped.
 *   K_draft[s] = 1 + min(k + d_s k^2, floor((Kmax - 1)(d_s + 1) / D)), K_draft[last] = Kmax;
 *   envelope = rank paths (r_1..r_m), m <= D, r_i < W, ordered by
 *   (prod(r_i + 1), m, lexicographic), first n_tmpl of them.
 * Host only; no CUDA call.  Returns GRAFT_ERR_INVALID_ARG /
 * GRAFT_ERR_UNSUPPORTED_SHAPE for sizes outside the limits or a draft too
 * small to fill Kmax.
 */
int graft_config_init(GraftConfig* cfg, int Kmax, int D, int k, int V, int W,
                      int n_checkpoints, const int32_t* checkpoints /* host */,
                      const float* tau /* host */);

/* graft_config_validate — check a (possibly hand-edited) config. Host only. */
int graft_config_validate(const GraftConfig* cfg);

/*
 * graft_config_no_retrieval — turn a valid *cfg (host) into the "w/o
 * retrieval" ablation of the Graft article's results paragraph: the
 * retrieval budget is zero at every stage (K_ret_s = 0), so the whole
 * budget goes to the draft, K_draft[s] = Kmax, and the envelope is empty
 * (n_tmpl = 0).  Pruning is unchanged.  A stage whose candidate pool holds
 * fewer than Kmax - 1 nodes (a prune at d0 with k < Kmax - 1) keeps all of
 * them; the draft slots it cannot fill are EMPTY NODES: token
 * GRAFT_EMPTY_TOKEN (-1), parent 0 (the root), depth 1.  No target token
 * equals -1, so graft_accept_compact never accepts an empty node, and
 * graft_update_M adds no pair for it.  Host only; no CUDA call.
 */
#define GRAFT_EMPTY_TOKEN (-1)
int graft_config_no_retrieval(GraftConfig* cfg);

/*
 * graft_build_tree — stages 1 to 3 of the step for B requests
 * (Graft article, step summary and method paragraph, first three points;
 * Graft abstract: "prune-then-graft").
 *
 *   draft_logits [B][D][k][V] f32  drafter logits; row (b, d, f) belongs to
 *                                  the f-th frontier node of drafter call d
 *                                  (call 0 reads only slot f = 0, the root).
 *                                  Rows past the pruning point are not read.
 *   root_tok [B] i32               last emitted token of each request
 *   M_succ [V][W] i32              successor table (-1 = empty slot)
 *   L [B] i32                      tokens already in each request's KV cache
 * Outputs, [B][Kmax] unless noted:
 *   tree_tok, tree_parent (root -1), tree_depth, tree_pos (= L[b] + depth) i32,
 *   tree_mask u64 (bit j of node i set iff j is i or an ancestor of i),
 *   stage [B] i32 (pruning stage; n_checkpoints = not pruned).
 * Tree order: root; kept draft nodes by (depth asc, score desc); empty
 * nodes if the pool ran short of K_draft (graft_config_no_retrieval); then
 * the stage's first K_ret envelope nodes (empty M slots give pad token 0).
 * Workspace: graft_build_tree_workspace_size bytes, 256-byte aligned,
 * ZERO-FILLED once before its first use: the call is one cooperative launch
 * (all CTAs resident, so it fails with GRAFT_ERR_CUDA where the device cannot
 * host a cooperative grid) whose phases meet at a grid barrier kept in the
 * workspace; every completed call leaves that barrier's count at zero again.
 * A barrier wait is bounded (half a second): one that runs out sets
 * GRAFT_STATUS_TIMEOUT and the outputs are incomplete; zero the workspace
 * again before the next call.  A barrier count found out of its range sets
 * GRAFT_STATUS_WORKSPACE (that call's output is unreliable).  Workspaces
 * must not be shared by calls that may run concurrently.
 */
int graft_build_tree_workspace_size(const GraftConfig* cfg, int B, size_t* bytes);
int graft_build_tree(const GraftConfig* cfg, int B, const float* draft_logits,
                     const int32_t* root_tok, const int32_t* M_succ, const int32_t* L,
                     int32_t* tree_tok, int32_t* tree_parent, int32_t* tree_depth,
                     int32_t* tree_pos, uint64_t* tree_mask, int32_t* stage,
                     int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream);

/*
 * graft_build_tree_block — graft_build_tree for a block drafter (Graft
 * abstract and results paragraph: grafting applied to DFlash-style block
 * drafting).  A block drafter emits one distribution per depth in a single
 * pass, not one per frontier node, so
 *
 *   block_logits [B][D][V] f32   row (b, d) is the drafter's distribution at
 *                                depth d + 1, shared by every frontier node
 *                                of drafter call d
 *
 * and the tree is assembled exactly as graft_build_tree would from drafter
 * logits whose k slot rows of each depth all equal that row: per-position
 * top-k, cumulative scores, pruning at the checkpoints and the retrieval
 * graft.  Same outputs, workspace and errors as graft_build_tree.
 *
 * Ablations of the method need no entry point of their own: without
 * pruning, set every tau to 0 (the confidence never drops below it, so the
 * dense tree of stage n_checkpoints is built); without retrieval, apply
 * graft_config_no_retrieval to the config (K_ret_s = 0 at every stage).
 */
int graft_build_tree_block(const GraftConfig* cfg, int B, const float* block_logits,
                           const int32_t* root_tok, const int32_t* M_succ, const int32_t* L,
                           int32_t* tree_tok, int32_t* tree_parent, int32_t* tree_depth,
                           int32_t* tree_pos, uint64_t* tree_mask, int32_t* stage,
                           int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream);

/*
 * graft_retrieve — the retrieval fill alone (Graft article, step summary:
 * retrieval starts from the root token through the GPU-resident adjacency
 * matrix; method paragraph, second point).
 *   ret_tok [B][n_tmpl] i32: envelope node j's token = M_succ[parent token][tmpl_rank[j]],
 *   -1 where the slot is empty or the parent is already -1.
 * No workspace.
 */
int graft_retrieve(const GraftConfig* cfg, int B, const int32_t* root_tok, const int32_t* M_succ,
                   int32_t* ret_tok, int32_t* status, graft_stream_t stream);

/*
 * graft_tree_attention — tree-masked GQA attention of one layer (Graft
 * article, architecture paragraph: the hybrid tree is verified on the
 * standard tree-attention path in one target forward).
 *
 *   Q  [B][Kmax][Hq][128] bf16     queries of the tree nodes (rotary already applied)
 *   Kc, Vc [B][Lcap][Hkv][128] bf16 this layer's KV cache; rows 0..L[b]-1 are read
 *   Kt, Vt [B][Kmax][Hkv][128] bf16 the tree nodes' own KV
 *   L [B] i32, tree_mask [B][Kmax] u64 as produced by graft_build_tree
 *   O  [B][Kmax][Hq][128] bf16     output (round to nearest even)
 * O[b,i,h] = softmax over {prefix keys 0..L[b]-1} U {tree keys j in mask[b][i]}
 * of scale * q.k, applied to V; q head h uses KV head h / (Hq / Hkv).
 * Float32 scores and accumulation.  Requires head_dim == 128, Hq % Hkv == 0,
 * Kmax * Hq / Hkv <= 1024.  Workspace: graft_tree_attention_workspace_size
 * (depends on the current device's SM count).
 *
 * The workspace must be ZERO-FILLED before its first use (cudaMemset): when
 * the items' key blocks are split evenly over persistent CTAs
 * (GraftAttnTuning.split), an item cut between two CTAs is merged by
 * whichever piece finishes last, and the arrival counters that decide it
 * live at the start of the workspace.  Every call that completes leaves the
 * counters at zero again, so one zero fill per buffer suffices; after a call
 * that reported GRAFT_STATUS_TIMEOUT, zero the buffer again.  Counters found
 * non-zero set GRAFT_STATUS_WORKSPACE (that call's output is unreliable).
 * Calls sharing a workspace must not run at the same time.
 */
int graft_tree_attention_workspace_size(int B, int Hq, int Hkv, int head_dim, int Kmax,
                                        int64_t Lcap, size_t* bytes);
int graft_tree_attention(int B, int Hq, int Hkv, int head_dim, int Kmax, const void* Q,
                         const void* Kc, const void* Vc, int64_t Lcap, const void* Kt,
                         const void* Vt, const int32_t* L, const uint64_t* tree_mask,
                         float scale, void* O, int32_t* status, void* ws, size_t ws_bytes,
                         graft_stream_t stream);

/*
 * GraftAttnTuning — explicit overrides of graft_tree_attention's launch plan
 * (host struct, passed by pointer; NULL or an all-zero struct keeps the
 * default plan).  The default plan depends only on the call's shape and the
 * current device's SM count; these fields let tests drive every kernel
 * variant on small shapes and let tuning runs compare plans.  The result is
 * the same attention whatever the plan (up to float32 summation order).
 *
 *   tiles         0 = default; 1 or 2 = 128-row query tiles per CTA on the
 *                 tensor-core path (group sizes dividing 128)
 *   min_chunk     0 = default (256); else the fewest prefix keys a key chunk
 *                 may hold (rounded up to whole 128-key blocks): large values
 *                 give one chunk per request
 *   persist_ctas  0 = default (the persistent two-tile kernel with one CTA
 *                 per SM when the two-tile grid exceeds one wave); -1 = never
 *                 persistent; n > 0 = persistent with n CTAs whenever the
 *                 two-tile kernel runs with an even tile count (at most one
 *                 per work item when requests are split into key chunks)
 *   split         0 = default: a persistent launch deals whole items to
 *                 its CTAs in turn; 1 = with one key chunk per request and at
 *                 most 256 requests, split the items' key blocks evenly over
 *                 the CTAs instead (an item cut between CTAs is merged by
 *                 its last piece through the workspace's arrival counters)
 *   wait_ns       0 = default (0.5 s); n > 0 = bound, in nanoseconds, on
 *                 every pipeline wait inside the tensor-core kernels.  A
 *                 wait that runs out sets GRAFT_STATUS_TIMEOUT; the CTA then
 *                 stops issuing work, waits (with fixed bounds) for the loads
 *                 and products it issued, frees its tensor memory and exits,
 *                 so the device stays usable.  A bound under 1000 ns
 *                 means no waiting at all (a wait succeeds only if its phase
 *                 has already completed), so the first waits run out: the
 *                 failure path, for tests
 *   reserved      must be zero
 *
 * graft_tree_attention_workspace_size_ex / graft_tree_attention_ex take the
 * same arguments as the plain entry points plus `tuning`; a workspace must be
 * sized with the same tuning it is used with.  Invalid fields return
 * GRAFT_ERR_INVALID_ARG.
 */
typedef struct GraftAttnTuning {
    int32_t tiles;
    int32_t min_chunk;
    int32_t persist_ctas;
    int32_t split;
    int32_t wait_ns;
    int32_t reserved[3];
} GraftAttnTuning;

int graft_tree_attention_workspace_size_ex(int B, int Hq, int Hkv, int head_dim, int Kmax,
                                           int64_t Lcap, const GraftAttnTuning* tuning,
                                           size_t* bytes);
int graft_tree_attention_ex(int B, int Hq, int Hkv, int head_dim, int Kmax, const void* Q,
                            const void* Kc, const void* Vc, int64_t Lcap, const void* Kt,
                            const void* Vt, const int32_t* L, const uint64_t* tree_mask,
                            float scale, void* O, int32_t* status,
                            const GraftAttnTuning* tuning, void* ws, size_t ws_bytes,
                            graft_stream_t stream);

/*
 * graft_accept_compact — greedy lossless acceptance and KV compaction
 * (Graft article, architecture paragraph: retrieved nodes are ordinary
 * proposals and the final distribution stays lossless).
 *
 *   target_logits [B][Kmax][V] f32 the target's logits at every tree node
 *   tree_tok, tree_parent, tree_depth [B][Kmax] i32 from graft_build_tree
 *   Kc_layers, Vc_layers  device arrays of n_layers device pointers, each a
 *                         [B][Lcap][Hkv][head_dim] bf16 cache (written)
 *   Kt_layers, Vt_layers  device arrays of n_layers device pointers, each a
 *                         [B][Kmax][Hkv][head_dim] bf16 tree KV (read)
 *   L [B] i32             in: cache lengths; out: L[b] + acc_len[b]
 * Outputs: argmax [B][Kmax] (target argmax per node, ties to the lower id),
 *   acc_len [B] (accepted path length, root included), path [B][Kmax]
 *   (accepted node indices from the root, -1 past acc_len), out_tok [B][Kmax]
 *   (emitted tokens: the path after the root then the bonus, -1 past
 *   acc_len), bonus [B] (target argmax at the deepest accepted node).
 * Node i is accepted iff every node on its root path carries the target's
 * argmax at its parent; the deepest accepted node wins, lower index on ties.
 * Cache row L[b] + t receives tree row path[b][t] for t < acc_len[b] in every
 * layer.  A request whose cache would overflow sets
 * GRAFT_STATUS_CACHE_OVERFLOW and is left uncompacted with L unchanged.
 * target_logits may be NULL: argmax [B][Kmax] is then an INPUT holding the
 * target's argmax per node (as graft_lm_head_argmax writes it; ids outside
 * [0, V) set GRAFT_STATUS_TOKEN_RANGE and are treated as 0) and only the
 * acceptance and compaction run.
 * Workspace: graft_accept_compact_workspace_size.
 */
int graft_accept_compact_workspace_size(int B, int Kmax, int V, size_t* bytes);
int graft_accept_compact(int B, int Kmax, int V, int n_layers, const float* target_logits,
                         const int32_t* tree_tok, const int32_t* tree_parent,
                         const int32_t* tree_depth, void* const* Kc_layers,
                         void* const* Vc_layers, const void* const* Kt_layers,
                         const void* const* Vt_layers, int Hkv, int head_dim, int64_t Lcap,
                         int32_t* L, int32_t* argmax, int32_t* acc_len, int32_t* path,
                         int32_t* out_tok, int32_t* bonus, int32_t* status, void* ws,
                         size_t ws_bytes, graft_stream_t stream);

/*
 * graft_lm_head_argmax — the target's greedy token at every tree node
 * straight from its final hidden states (Graft article, architecture
 * paragraph: the tree is verified in one target forward; greedy acceptance
 * needs only the argmax at each node).  g[n] = argmax_v sum_k H[n][k]
 * W_lm[v][k] with ties to the lower id, computed on the tensor cores (bf16
 * in, fp32 accumulation) without writing the [N][V] logits.
 *
 *   H [N][d_model] bf16      final hidden states of the N = B * Kmax nodes
 *   W_lm [V][d_model] bf16   output embedding (lm_head) rows
 * Outputs: argmax [N] i32; max_logit [N] f32 (the winning logit; may be
 *   NULL).  d_model must be a multiple of 8; H and W_lm 16-byte aligned.
 *   Rows whose two best logits differ by less than the fp32 rounding of the
 *   sum may pick either (the rounding order is the kernel's).
 * Feed argmax to graft_accept_compact with target_logits == NULL.
 * Workspace: graft_lm_head_argmax_workspace_size (8 bytes per row).
 */
int graft_lm_head_argmax_workspace_size(int N, size_t* bytes);
int graft_lm_head_argmax(int N, int d_model, int V, const void* H, const void* W_lm, int32_t* argmax,
                         float* max_logit, int32_t* status, void* ws, size_t ws_bytes,
                         graft_stream_t stream);

/*
 * graft_sample_tokens — the target's sample at every tree node, for lossless
 * sampling acceptance at temperature > 0 (Graft article, architecture
 * paragraph, and Graft abstract: verification is lossless).  Every proposal
 * in a Graft tree is deterministic (the drafter's top-k, retrieved tokens);
 * for such proposals the speculative-sampling rule over a node's children
 * (accept child i with its residual probability, renormalise on rejection)
 * has the law of drawing one sample y ~ softmax(logits / T) per node and
 * accepting the first child whose token is y.  Feed the samples to
 * graft_accept_compact as its argmax input (target_logits NULL).
 *
 *   target_logits [B][Kmax][V] f32, tree_pos [B][Kmax] i32 (graft_build_tree)
 *   temperature > 0; seed: 64-bit stream key
 * Output: sampled [B][Kmax] = argmax_v(logits[v] / T + G_v), G Gumbel noise
 *   from Philox-4x32-10 (Salmon et al., SC 2011) with counter (v / 4,
 *   tree_pos + 1, b, 0) and key (seed low, seed high) words, draw x = word
 *   v % 4, u = ((x >> 9) + 1/2) / 2^23, G = -log(-log u).  Nodes at the same
 *   position see the same noise, so tree decoding emits exactly what
 *   autoregressive sampling with this noise emits.
 * Workspace: graft_sample_tokens_workspace_size.
 */
int graft_sample_tokens_workspace_size(int B, int Kmax, int V, size_t* bytes);
int graft_sample_tokens(int B, int Kmax, int V, const float* target_logits, const int32_t* tree_pos,
                        float temperature, uint64_t seed, int32_t* sampled, void* ws, size_t ws_bytes,
                        graft_stream_t stream);

/*
 * graft_lm_head_sample — graft_sample_tokens fused into the lm_head product
 * of graft_lm_head_argmax: rows n = b * Kmax + i of H are the nodes of the
 * B trees, tree_pos [N] their positions; the logits are never written.
 * N must be a multiple of Kmax.  Workspace: graft_lm_head_argmax_workspace_size.
 */
int graft_lm_head_sample(int N, int d_model, int V, const void* H, const void* W_lm, int Kmax,
                         const int32_t* tree_pos, float temperature, uint64_t seed, int32_t* sampled,
                         int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream);

/*
 * graft_update_M — online update of the adjacency table from verified
 * pairs (Graft article, method paragraph, fourth point: M is updated
 * continuously from the verified tree's logits).
 *
 *   M_succ, M_cnt [V][W] i32 (in place); row t ranks up to W successors of
 *   token t by (count desc, token asc), empty slots (-1, 0) last.
 *   src, dst [n] i32: the multiset of pairs (src -> dst) to add.
 * Each pair already in its row adds 1 to that count (an atomic increment);
 * new successors enter with their multiplicity; each touched row keeps its
 * top W by (count desc, token asc).  The result depends only on the
 * multiset, not on pair order, and is bit-exact.  A pair whose src is -1
 * (an empty slot, or an empty tree node of graft_config_no_retrieval) is
 * skipped silently; any other id outside [0, V) is skipped and flagged.
 * Workspace: graft_update_M_workspace_size.
 * To seed M from a prompt's evidence, pass its bigrams: src = tokens,
 * dst = tokens + 1, n = length - 1.
 */
int graft_update_M_workspace_size(int64_t n, size_t* bytes);
int graft_update_M(int32_t* M_succ, int32_t* M_cnt, int V, int W, const int32_t* src,
                   const int32_t* dst, int64_t n, int32_t* status, void* ws, size_t ws_bytes,
                   graft_stream_t stream);

/*
 * graft_update_M_emitted — refresh M from the bigrams of the tokens a verify
 * step emitted (Graft article, method paragraph: retrieval draws on the
 * evidence of the context itself; seeding M from the prompt's bigrams at
 * prefill and adding each step's emitted bigrams keeps it current for long
 * contexts).
 *
 *   tree_tok [B][Kmax] i32   the step's tree (node 0 = the last token
 *                            emitted before the step)
 *   out_tok [B][Kmax], acc_len [B] i32   graft_accept_compact's outputs
 * Adds, as one multiset under graft_update_M's rule, the acc_len[b] pairs
 * (tree_tok[b][0] -> out_tok[b][0]), (out_tok[b][t-1] -> out_tok[b][t]) for
 * 0 < t < acc_len[b].  Workspace: graft_update_M_emitted_workspace_size.
 */
int graft_update_M_emitted_workspace_size(int B, int Kmax, size_t* bytes);
int graft_update_M_emitted(int32_t* M_succ, int32_t* M_cnt, int V, int W, int B, int Kmax,
                           const int32_t* tree_tok, const int32_t* out_tok, const int32_t* acc_len,
                           int32_t* status, void* ws, size_t ws_bytes, graft_stream_t stream);

/*
 * graft_update_M_noalloc — graft_update_M without a workspace argument.
 *
 * The Graft pages have no counterpart to this entry point; it exists for
 * callers that cannot provide device scratch memory: a plug-in that only sees
 * the tensors its host framework passes in and has no allocator of its own,
 * or a serving loop that must not call cudaMalloc because it synchronises the
 * whole device.  Arguments and results are those of graft_update_M.
 *
 * Scratch lives in one static device array of the library (1 MiB, kept on
 * every GPU that loads the library until the process exits), enough for
 * n <= GRAFT_NOALLOC_MAX_PAIRS pairs; larger n returns
 * GRAFT_ERR_UNSUPPORTED_SHAPE and enqueues nothing.  The call allocates and
 * frees nothing.  Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  The address is kept for the life of the
 * process, so resetting a device (cudaDeviceReset) after that first call is
 * not supported.  Device ordinals 0 to 63 are supported; a current device
 * beyond them returns GRAFT_ERR_UNSUPPORTED_SHAPE.  All calls on a device share the array
 * (each call clears the parts it reads), so calls that may run at the same
 * time on the GPU — different streams with no ordering between them — race
 * and corrupt each other's result: order them on one stream or with events.
 */
#define GRAFT_NOALLOC_MAX_PAIRS 16384
int graft_update_M_noalloc(int32_t* M_succ, int32_t* M_cnt, int V, int W, const int32_t* src,
                           const int32_t* dst, int64_t n, int32_t* status, graft_stream_t stream);

/* Human-readable text for a return code (static string). */
const char* graft_status_string(int code);

/* Library version as an integer (major * 10000 + minor * 100 + patch). */
int graft_version(void);

/*
 * graft_launch_count — number of kernel launches this process has enqueued
 * through the library so far (host-side counter, all devices, all threads).
 * Launches recorded into a CUDA graph count once, at capture time.
 */
uint64_t graft_launch_count(void);

/*
 * graft_last_cuda_error — name of the most recent CUDA runtime error that an
 * entry point of this library observed on the calling host thread (the cause
 * behind a GRAFT_ERR_CUDA return), or "cudaSuccess" if there was none.  The
 * string is static; the caller does not free it.
 */
const char* graft_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GRAFT_H_ */
