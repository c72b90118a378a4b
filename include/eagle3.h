/*
 * eagle3.h -- C ABI of one EAGLE-3 draft-and-verify round on a single B300.
 *
 * The operations follow the pages' statement of the problem:
 *   - multi-layer feature fusion and the one-layer draft decoder
 *     ("EAGLE-3 精读" §1 为什么推翻 feature regression, paragraph 2; abstract
 *     of "EAGLE-3: Scaling up Inference Acceleration of Large Language Models
 *     via Training-Time Test");
 *   - the draft's own states fed back along draft paths with a tree attention
 *     mask ("EAGLE-3 精读" §2 Training-Time Test);
 *   - the EAGLE-2 confidence-value dynamic tree ("EAGLE-3 精读" 核心变化, and
 *     §2 last paragraph), confidence = product of draft probabilities (EAGLE-4
 *     blog, 几条技术路线正在收敛, second trend);
 *   - strict verification, greedy and sampling with residual correction
 *     ("EAGLE-3 精读" §5 正确性、复现与风险);
 *   - the two-stage "Efficient LM Head" (EAGLE-4 blog, sections on the
 *     Efficient LM Head): low-rank recall, exact rerank.
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must be device memory of the current
 *     CUDA device; the caller owns them and keeps them alive until the work on
 *     `stream` has finished.  The library never frees caller memory.
 *   - Weights are borrowed, never copied: row-major [out, in] matrices in the
 *     storage type of the config (fp32 or bf16).  They must stay valid and
 *     unchanged for the life of the context.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  Outputs
 *     are valid once the stream has reached the call's end.  Nothing inside a
 *     call synchronises with the host.
 *   - Arguments are checked on the host before any launch; a bad argument
 *     returns a status and launches nothing.  EAGLE3_ERR_CUDA wraps a launch
 *     error.  Device-side checks (page index in range, ancestor closure of a
 *     supplied pool, ...) raise a flag read by eagle3_check().
 *   - A context is not thread-safe; use one context per host thread.
 */
#ifndef EAGLE3_H
#define EAGLE3_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct eagle3_ctx eagle3_ctx;
typedef struct CUstream_st* eagle3_stream; /* same handle as cudaStream_t */

typedef enum {
  EAGLE3_OK = 0,
  EAGLE3_ERR_INVALID_ARG = 1,   /* null pointer, value out of range */
  EAGLE3_ERR_SHAPE = 2,         /* sizes inconsistent with the config or capacity */
  EAGLE3_ERR_UNSUPPORTED = 3,   /* valid request this build does not implement */
  EAGLE3_ERR_OOM = 4,           /* workspace allocation failed at create time */
  EAGLE3_ERR_CUDA = 5,          /* a CUDA call or kernel launch failed */
  EAGLE3_ERR_TIMEOUT = 6,       /* a bounded device wait gave up */
  EAGLE3_ERR_DEVICE_ASSERT = 7, /* a device-side check failed (see eagle3_last_error) */
  EAGLE3_ERR_STATE = 8          /* call order violated (e.g. verify before any draft round) */
} eagle3_status;

enum { EAGLE3_FP32 = 0, EAGLE3_BF16 = 1 };

/* Drafter variants (eagle3_config.variant, bits).  The EAGLE-4 blog (section
 * 在EAGLE4中) states that its one-layer drafter keeps EAGLE-3.1's "FC Norm" and
 * "Post-norm"; the pages give no formula, so the plainest readings are used:
 *   EAGLE3_FC_NORM:   g = rms(W_fc [low; mid; high]) * g_fc (an RMSNorm with
 *                     gain g_fc on the fused feature, before it enters the
 *                     decoder input and its residual stream);
 *   EAGLE3_POST_NORM: each residual sum is normalised after the add:
 *                     r = rms(hid + W_o attn) * g_post,
 *                     s = rms(r + W_down(silu(W_gate r) * W_up r)) * g_final,
 *                     and s is both the LM head's input and the state fed to
 *                     the node's children (no separate final norm).
 * 0 is the EAGLE-3 pre-norm drafter: z = rms(r) feeds the FFN, h = rms(s). */
enum { EAGLE3_FC_NORM = 1, EAGLE3_POST_NORM = 2, EAGLE3_SAMPLED_DRAFT = 4 };
/* EAGLE3_SAMPLED_DRAFT (single-stage head only): a node's k children are drawn
 * from the draft distribution q without replacement -- the k largest
 * log q(x) + G(x), G Gumbel noise from Philox stream 2 at (round id, b,
 * node slot) keyed by the seed of eagle3_draft_noise -- in draw order, with
 * their true log q.  The i-th draw's score is its parent's score plus
 * min(log max q, log q of draws 1..i-1): it depends only on the draws before
 * it, never on the draw itself, and is non-increasing in draw order, so a
 * kept sibling set is always the first draws and is chosen by a stopping
 * rule -- the condition under which eagle3_verify mode 2 (recursive
 * rejection over the kept draws; see there) keeps the target distribution.
 * The pass's logits are written to the workspace (rows x V fp32). */

/* Shapes of the draft model and of the round.  All sizes in elements. */
typedef struct {
  int d;           /* model width */
  int n_q_heads;   /* query heads Hq */
  int n_kv_heads;  /* key/value heads Hkv (Hq % Hkv == 0) */
  int head_dim;    /* dh, even, <= 128 */
  int ffn;         /* SwiGLU inner width F */
  int vocab;       /* V */
  int lr_rank;     /* two-stage head: rank r of U [V, r] V_lr [r, d], r % 8 == 0; 0 = single-stage head */
  int lr_cand;     /* two-stage head: candidates C rescored by the exact head, k <= C <= 128, C <= V;
                      log q is normalised over C */
  float rope_theta;
  float rms_eps;
  int dtype;       /* EAGLE3_FP32 or EAGLE3_BF16: weights, features, KV cache */
  int depth;       /* D: sequential decoder passes per round, 1..16 */
  int topk;        /* k: children per expanded node and frontier width, 1..16 */
  int n_verify;    /* M: nodes kept for verification, 1..128 and <= pool size */
  int page_size;   /* 0 = contiguous cache, else rows per KV page */
  int max_batch;   /* largest B of any call */
  int max_prefix;  /* rows one request may hold in the cache (contiguous layout stride) */
  int max_new;     /* largest n_new of a draft round */
  int variant;     /* EAGLE3_FC_NORM | EAGLE3_POST_NORM bits, 0 = EAGLE-3 pre-norm */
} eagle3_config;

/* Device pointers of the draft weights (row-major [out, in], config dtype).
 *   w_fc [d, 3d]; embed [V, d]; w_q [Hq*dh, 2d]; w_k, w_v [Hkv*dh, 2d];
 *   w_o [d, Hq*dh]; w_gate, w_up [F, d]; w_down [d, F];
 *   g_emb, g_hid, g_post, g_final [d] RMSNorm gains;
 *   w_lm [V, d] draft LM head; w_target [V, d] synthetic target head used by
 *   eagle3_verify; lr_u [V, r], lr_v [r, d] the two-stage head (else NULL);
 *   g_fc [d] gain of the FC norm (EAGLE3_FC_NORM only, else NULL). */
typedef struct {
  const void *w_fc, *embed, *w_q, *w_k, *w_v, *w_o, *w_gate, *w_up, *w_down;
  const void *g_emb, *g_hid, *g_post, *g_final;
  const void *w_lm, *w_target, *lr_u, *lr_v;
  const void* g_fc;
} eagle3_weights;

/* Draft KV cache, caller-owned, config dtype, K after RoPE.
 *   contiguous (page_size == 0): k, v are [max_batch, max_prefix, Hkv, dh];
 *   paged: k, v are [n_pages, page_size, Hkv, dh] and page_table [B, max_pages]
 *   (int32, device) maps request b's logical page j to a physical page.
 * seq_lens [B] (int32, device): rows already committed per request.  No entry
 * point changes seq_lens: the caller advances it after committing rows. */
typedef struct {
  void *k, *v;
  const int* page_table;
  const int* seq_lens;
  int max_pages;
  int n_pages;
} eagle3_kv;

/* The kept tree, device arrays.  Node 0 of request b is the root (the newest
 * row), nodes 1..M the kept draft nodes in canonical order (depth ascending,
 * then selection rank).  Shapes [B, M+1]; mask [B, M+1, W] with
 * W = (M + 32) / 32 words: bit j of row i is set iff node j is an ancestor of
 * node i or i itself.  parent of the root is -1; pool_index is the node's index
 * in the round's pool (-1 for the root). */
typedef struct {
  int *tokens, *parent, *depth, *pos, *pool_index;
  float* score;
  uint32_t* mask;
} eagle3_tree;

/* Every node the round created, device arrays [B, pool_n] with
 * pool_n = k + (D-1) k^2, in creation order (depth, parent's frontier rank,
 * child rank).  parent is a pool index (-1 = root); fwd is the node's frontier
 * slot if it was expanded, else -1; score = cumulative log q.
 * cand (two-stage head only, may be NULL): [B, 1 + (D-1) k, lr_cand] int32,
 * the candidate tokens of every expanded node in low-rank order (score desc,
 * token asc): the root first, then the frontier slots (depth, rank). */
typedef struct {
  int *tok, *parent, *depth, *fwd;
  float *score, *logq;
  int* cand;
} eagle3_pool;

/* Optional per-node verification details, device arrays [B, M+1]:
 * z_max / z_argmax: largest target logit and its token (ties: lowest token);
 * lse: log-sum-exp of z / T (of z when greedy); g_argmax: Gumbel-argmax of
 * z / T over the tokens that are not children of the node (sampling only).
 * Any of the four may be NULL.  Cost: without g_argmax a sampling pass draws
 * the Gumbel noise only at the node where each request's walk stops (the bf16
 * head stores the target logits in the context's workspace meanwhile); with
 * g_argmax it draws it at every node, as the walk's own draw at the stop node
 * would be, which for wide passes costs most of the verify head's time. */
typedef struct {
  float *z_max, *lse;
  int *z_argmax, *g_argmax;
} eagle3_verify_stats;

/* Per-request control of the round: caps and the cost-aware rules of the
 * EAGLE-4 blog's "EAGLE-Harness" paragraph (a warm-up measures draft and
 * verify times into a lookup table; each round then asks, in three places,
 * whether the expected extra accepted tokens per extra time clear a
 * threshold: another draft layer, how many nodes to verify, and how many
 * branches a node expands -- 8 under light load, 4 under heavy load) and of
 * its remark that confidence is the product of draft probabilities with a
 * threshold that rises with depth.  Readings (the blog gives no formula):
 *   depth:   pass t (t >= 1) runs for request b only while the confidence
 *            mass of its frontier, sum of exp(score), is at least
 *            tau_depth * depth_growth^t * pass_us[t];
 *   verify:  the kept set is the longest prefix of the score order whose i-th
 *            node has exp(score_i) >= tau_verify * (verify_us[i] -
 *            verify_us[i-1]), at least one node;
 *   branch:  a node makes at most k_light children when B <= light_batch,
 *            else k_heavy.
 * The caps depth_cap / topk_cap / verify_cap ([max_batch] int32 device arrays,
 * read when the round runs; NULL = the config's D, k, M) bound each request as
 * well, so one batch can mix requests of different D, k and M.  A pool node
 * that is not created has token -1, parent -1 and score / log q -inf; tree
 * slots past a request's kept count have token -1, parent -1, depth 0, score
 * -inf and only their own mask bit, and verification ignores them.  A rule is
 * off while its threshold is 0 (light_batch 0: no branch rule).  When no
 * request takes part in a pass, its GEMMs, attention and LM head return at
 * once. */
typedef struct {
  const int *depth_cap, *topk_cap, *verify_cap;
  float tau_depth, depth_growth, tau_verify;
  int light_batch, k_light, k_heavy;
  const float* pass_us;   /* host [D]: cost of draft pass t in microseconds (tau_depth > 0) */
  const float* verify_us; /* host [M+1]: cost of verifying m nodes, verify_us[0] = 0 (tau_verify > 0) */
} eagle3_control;

/* Set (ctl != NULL) or clear (NULL) the control of later rounds and tree
 * builds.  The cost arrays are copied (the call synchronizes the device); the
 * cap arrays are borrowed.  A captured graph keeps the control it was
 * captured with: capture again after a change. */
eagle3_status eagle3_set_control(eagle3_ctx* ctx, const eagle3_control* ctl);

/* The warm-up's lookup table: times on ascending grids of batch size B,
 * prefix length P and tokens per request n (rows of a draft pass, or nodes
 * verified), [n_batch][n_prefix][n_tokens] row-major, microseconds. */
typedef struct {
  int n_batch, n_prefix, n_tokens;
  const int *batch, *prefix, *tokens;
  const float *draft_us, *verify_us;
} eagle3_latency_table;

/* Costs of one round at (B, P) from the table, by trilinear interpolation
 * (clamped at the grid's ends): pass_us[0] = draft(B, P, 1) (the root pass),
 * pass_us[t] = draft(B, P, topk) for t = 1..depth-1; verify_us[0] = 0 and
 * verify_us[m] = verify(B, P, m) for m = 1..n_verify.  Host-only; no GPU. */
eagle3_status eagle3_latency_costs(const eagle3_latency_table* table, int B, int P, int depth,
                                   int topk, int n_verify, float* pass_us, float* verify_us);

/* Seed and round id of the sampled draft's noise (EAGLE3_SAMPLED_DRAFT), for
 * the next draft rounds on `stream` (the round id is written in stream order;
 * a graph replay uses its own round id). */
eagle3_status eagle3_draft_noise(eagle3_ctx* ctx, unsigned long long seed,
                                 unsigned long long round_id, eagle3_stream stream);

/* Create a context: checks the config, borrows the weights, allocates the
 * workspace for max_batch requests once (nothing is allocated later) and
 * prepares the kernels' tensor maps.  It synchronizes the device first: the
 * weights must be fully written before the call and stay unchanged while the
 * context exists (kernels start reading weight tiles before the preceding
 * kernel on their stream has finished).  Returns EAGLE3_ERR_OOM if the workspace
 * does not fit, EAGLE3_ERR_UNSUPPORTED for shapes outside the limits above. */
eagle3_status eagle3_create(const eagle3_config* cfg, const eagle3_weights* w, eagle3_ctx** out);

/* Free the workspace.  The caller must have finished all work on the context. */
void eagle3_destroy(eagle3_ctx* ctx);

/* Prefix rows into the draft KV cache ("EAGLE-3 精读" §1: g from the target's
 * low/mid/high features, then the decoder input [rms(E[y]); rms(g)]).
 * cu_rows [B+1] (int32, device) splits the packed rows by request; row r of
 * request b gets position seq_lens[b] + (r - cu_rows[b]).  feats [total_rows, 3d]
 * (low, mid, high concatenated), tokens [total_rows] (the token emitted after
 * each row's position).  Only K and V are produced: in a one-layer drafter a
 * prefix row's layer output feeds nothing. */
eagle3_status eagle3_prefill(eagle3_ctx* ctx, int B, int total_rows, const int* cu_rows,
                             const void* feats, const int* tokens, const eagle3_kv* kv,
                             eagle3_stream stream);

/* One draft round ("EAGLE-3 精读" §1, paragraph 2: the drafter fuses the
 * target's low/mid/high features into g and runs one decoder layer over g, its
 * own state and the token embedding; §2 Training-Time Test: deeper draft steps
 * are fed the draft's own states; scholarfeed "EAGLE-3" page, the quote that
 * each added tree depth costs one more sequential drafter pass; "EAGLE-3 精读"
 * 核心变化 and the EAGLE-4 blog, 几条技术路线正在收敛, second trend: the
 * EAGLE-2 confidence tree, confidence = product of draft probabilities).
 * It appends n_new rows per request at positions
 * seq_lens[b] .. seq_lens[b] + n_new - 1 (the last is the tree's root), runs D
 * decoder passes (root, then one per tree depth), builds the pool of
 * k + (D-1) k^2 nodes and keeps the global top-M as `out`.
 * feats_new [B, n_new, 3d], tokens_new [B, n_new] (device).  pool_out may be
 * NULL.  The round keeps its node states in the context for eagle3_verify. */
eagle3_status eagle3_draft_round(eagle3_ctx* ctx, int B, int n_new, const void* feats_new,
                                 const int* tokens_new, const eagle3_kv* kv, eagle3_tree* out,
                                 eagle3_pool* pool_out, eagle3_stream stream);

/* The same round with a different number of new rows per request, as in
 * steady-state decoding ("EAGLE-3 精读" §1 and §2 as for eagle3_draft_round;
 * §2: after a verification the drafter continues from the target's accepted
 * sequence, whose features arrive as several new rows): request b's new rows are rows cu_new[b] ..
 * cu_new[b+1] - 1 of feats_new [total_new, 3d] / tokens_new [total_new]
 * (device), at positions seq_lens[b] onward; the last is the request's root.
 * cu_new [B+1] (int32, device) with cu_new[0] = 0, cu_new[B] = total_new and
 * 1 <= cu_new[b+1] - cu_new[b] <= max_new.  A count outside that range is
 * clamped and raises a device flag (EAGLE3_ERR_DEVICE_ASSERT from eagle3_check). */
eagle3_status eagle3_draft_round_ragged(eagle3_ctx* ctx, int B, int total_new, const int* cu_new,
                                        const void* feats_new, const int* tokens_new,
                                        const eagle3_kv* kv, eagle3_tree* out, eagle3_pool* pool_out,
                                        eagle3_stream stream);

/* The token rows of the next round from a verification, without a host round
 * trip ("EAGLE-3 精读" §2: the drafter continues from the target's accepted
 * sequence).  Request b contributes accept_len[b] + 1 rows: its accepted
 * tokens then the bonus token, out_tokens[b][0 .. accept_len[b]] of
 * eagle3_verify.  Writes cu_new [B+1] and tokens_new [sum of rows] (int32,
 * device) for eagle3_draft_round_ragged.  The caller supplies the rows'
 * target features and, once the previous round's rows are committed,
 * advances seq_lens by that round's row counts.  B <= 1024; max_new should be
 * at least D + 1. */
eagle3_status eagle3_next_rows(eagle3_ctx* ctx, int B, const int* accept_len, const int* out_tokens,
                               int* cu_new, int* tokens_new, eagle3_stream stream);

/* Tree builder alone (for tests and outside drafters).  "EAGLE-3 精读"
 * 核心变化: EAGLE-3 keeps EAGLE-2's confidence-value dynamic draft tree; the
 * EAGLE-4 blog, 几条技术路线正在收敛, second trend: a node's confidence is the
 * product of its draft probabilities.  It keeps the top-M of a pool by (score
 * desc, depth asc, pool index asc) -- score = cumulative log q -- and writes
 * the canonical tree.  pool arrays [B, pool_n] (device; parent = pool index or -1), root_tok
 * and root_pos [B] (device).  pool_n <= 4096.  The kept set must be
 * ancestor-closed (child score <= parent score); otherwise the device flag
 * EAGLE3_ERR_DEVICE_ASSERT is raised and the tree is left partial. */
eagle3_status eagle3_build_tree(eagle3_ctx* ctx, int B, int pool_n, const int* pool_tok,
                                const int* pool_parent, const float* pool_score,
                                const int* pool_depth, const int* root_tok, const int* root_pos,
                                eagle3_tree* out, eagle3_stream stream);

/* Strict verification of the tree of the last eagle3_draft_round on this
 * context ("EAGLE-3 精读" §5).  The synthetic target reruns the decoder over
 * the M kept nodes with the tree mask and applies w_target.  mode 0: greedy
 * (walk while the target argmax is a child's token); mode 1: sampling at
 * `temperature` > 0 with sequential point-mass acceptance and a Gumbel draw
 * from the residual, using Philox4x64-10 with key (seed, 0) and counter
 * (round_id, b * 2^32 + node, idx, stream); mode 2 (EAGLE3_SAMPLED_DRAFT only):
 * sampling at `temperature` with the q-ratio test -- the node's draws in draw
 * order, the i-th accepted when U q_i(c) < p_i(c), on rejection p_{i+1} =
 * norm(max(0, p_i - q_i)) and q_{i+1} = q_i without c, the bonus drawn from
 * the last residual (q = softmax of the draft logits at the node, recomputed
 * over the kept nodes).  Outputs (device): accept_len [B],
 * path [B, D] (tree indices, -1 padded), out_tokens [B, D+1] (accepted tokens
 * then the bonus token, -1 padded).  stats may be NULL. */
eagle3_status eagle3_verify(eagle3_ctx* ctx, int B, const eagle3_tree* tree, const eagle3_kv* kv,
                            int mode, float temperature, unsigned long long seed,
                            unsigned long long round_id, int* accept_len, int* path,
                            int* out_tokens, eagle3_verify_stats* stats, eagle3_stream stream);

/* Strict verification of a kept tree against target logits that the caller
 * supplies ("EAGLE-3 精读" §5 正确性、复现与风险: greedy keeps the target's
 * greedy sequence; sampling keeps the target's distribution when the residual
 * correction is done).  This is the form a real target model drives: it
 * scores every tree node in one forward pass and passes its logits here, in
 * place of eagle3_verify's synthetic target.
 *   tree: a kept tree in the layout of eagle3_draft_round's output (device;
 *     node 0 the root, parents before children, padding slots token -1); at
 *     most `topk` children per node and depth at most `depth` (the walk
 *     accepts at most `depth` tokens).  The tree need not come from this
 *     context's last round.
 *   logits: [B, M+1, ld] device array (caller-owned) in logits_dtype
 *     (EAGLE3_FP32 or EAGLE3_BF16): row (b, u) holds the target's logits of
 *     the token after node u's root-to-node path; only the first `vocab`
 *     entries of a row are read, and padding rows are not read.  ld >= vocab
 *     elements; the base address and ld * element size must be multiples of
 *     16 bytes (EAGLE3_ERR_INVALID_ARG otherwise).
 *   mode 0: greedy -- walk from the root while the target's argmax (ties:
 *     lowest token) is a child's token, then emit that argmax as the bonus;
 *   mode 1: sampling at `temperature` > 0 -- point-mass acceptance of the
 *     children in tree order and a Gumbel draw from the residual, with the
 *     Philox4x64-10 counter layout of eagle3_verify mode 1 (identical logits
 *     give identical draws); mode 2 returns EAGLE3_ERR_UNSUPPORTED.
 * Outputs as eagle3_verify: accept_len [B], path [B, D], out_tokens [B, D+1],
 * stats (may be NULL).  A node with more than topk children, a parent index
 * out of range or a token outside [0, vocab) raises the device flag that
 * eagle3_check reports.  The logits are read once, from HBM. */
eagle3_status eagle3_verify_logits(eagle3_ctx* ctx, int B, const eagle3_tree* tree, const void* logits,
                                   int logits_dtype, long long ld, int mode, float temperature,
                                   unsigned long long seed, unsigned long long round_id,
                                   int* accept_len, int* path, int* out_tokens,
                                   eagle3_verify_stats* stats, eagle3_stream stream);

/* Record one whole step -- eagle3_draft_round followed, if with_verify, by
 * eagle3_verify, with the same arguments as those two calls (no pool or stats
 * outputs; the verify arguments are ignored without with_verify) -- into a
 * CUDA graph kept by the context, replacing any earlier one.  The step's
 * pointers (new rows, KV descriptor, tree and verification outputs) are fixed
 * in the graph: refill the same buffers before each replay.  The round id is
 * not: each eagle3_graph_launch passes its own.  Needs one eager draft round
 * on the context first (one-time kernel set-up runs there), and a stream
 * other than the legacy default stream.  Nothing runs during the capture. */
eagle3_status eagle3_graph_capture(eagle3_ctx* ctx, int B, int n_new, const void* feats_new,
                                   const int* tokens_new, const eagle3_kv* kv, eagle3_tree* out,
                                   int with_verify, int mode, float temperature,
                                   unsigned long long seed, int* accept_len, int* path,
                                   int* out_tokens, eagle3_stream stream);

/* Replay the captured step on `stream` with the given round id (the Philox
 * counter of the sampling draws).  EAGLE3_ERR_STATE if nothing was captured.
 * The replay's results equal those of the eager calls with that round id. */
eagle3_status eagle3_graph_launch(eagle3_ctx* ctx, unsigned long long round_id, eagle3_stream stream);

/* The draft LM head alone on R given rows h [R, d] (config dtype, device):
 * per row the top-k (token, log q) and the log-sum-exp of the logits (for the
 * two-stage head: normalised over the candidate set).  tok [R, k] int32,
 * logq [R, k] fp32, lse [R] fp32 (may be NULL).  R <= max_batch * topk. */
eagle3_status eagle3_lm_head_topk(eagle3_ctx* ctx, int R, const void* h, int* tok, float* logq,
                                  float* lse, eagle3_stream stream);

/* The draft LM head and top-k of eagle3_lm_head_topk without a context, for
 * callers that cannot allocate device memory: a server runtime that has
 * reserved all of HBM for its own pools, a plugin restricted to its host
 * framework's allocator, or a latency-critical path that cannot afford
 * cudaMalloc's implicit synchronisation.  (The pages have no counterpart: this
 * is a deployment variant of the same computation.)
 *   w_lm [vocab, d] and h [R, d] in `dtype` (EAGLE3_FP32 or EAGLE3_BF16),
 *   device, caller-owned; tok [R, topk] int32, logq [R, topk] fp32 and lse [R]
 *   fp32 (may be NULL) are written as by eagle3_lm_head_topk.  dev_status
 *   (device int, may be NULL) receives the device error flags of this call
 *   (0 = none) in stream order.
 * Scratch: the per-tile partials live in one 16 MiB array in the library's
 * device global memory (held on every GPU that loads the library until exit).
 * Calls needing more -- 256 + P*R*(2 + 2*topk)*4 bytes, 256-byte aligned per
 * part, with P = 4*ceil(vocab/128) (bf16) or ceil(vocab/64) (fp32) -- return
 * EAGLE3_ERR_SHAPE and launch nothing.  bf16 also needs d % 8 == 0, 16-byte
 * aligned w_lm and h, and R <= 256 (EAGLE3_ERR_INVALID_ARG / _SHAPE).
 * No call allocates or calls an allocating routine, but the first call on a
 * device looks up the array's device address (with that device current) and
 * caches it, and under CUDA's default lazy module loading that lookup is what
 * loads the library module holding the array onto the device: the 16 MiB are
 * placed then (the load may synchronise the device, and fails with
 * EAGLE3_ERR_CUDA if 16 MiB are not free).  Make the first call on each device
 * before reserving memory pools and before capturing any stream; later calls
 * allocate nothing.  Every call shares the array and it keeps the last call's
 * contents: calls whose work may overlap on the GPU race and must be ordered
 * by the caller.  EAGLE3_ERR_CUDA also reports a driver that refuses the
 * tensor-map encode or a failed launch. */
eagle3_status eagle3_lm_head_topk_noalloc(int dtype, int vocab, int d, int topk, const void* w_lm,
                                          int R, const void* h, int* tok, float* logq, float* lse,
                                          int* dev_status, eagle3_stream stream);

/* One of the context's weight matrices applied to R given rows, for kernel
 * tests: Y [R, N] (fp32, device) = X [R, K] (config dtype, device) W^T, with
 * which = 0 w_fc, 1 w_q, 2 w_k, 3 w_v, 4 w_o, 5 w_gate, 6 w_up, 7 w_down,
 * 8 w_lm, 9 w_target.  Runs the same GEMM kernel as the round (tcgen05 for
 * bf16 storage).  R <= the context's row capacity. */
eagle3_status eagle3_linear(eagle3_ctx* ctx, int which, int R, const void* X, float* Y,
                            eagle3_stream stream);

/* Wait for the context's last stream, then report and clear the device flag. */
eagle3_status eagle3_check(eagle3_ctx* ctx);

/* Text of the last error on this context ("" if none).  Valid until the next call. */
const char* eagle3_last_error(const eagle3_ctx* ctx);

/* Bytes of device workspace the context holds. */
size_t eagle3_workspace_bytes(const eagle3_ctx* ctx);

/* Kernel launches issued by the last call on this context. */
int eagle3_last_launch_count(const eagle3_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE3_H */
