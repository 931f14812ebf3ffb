/*
 * dartree.h -- C ABI of the GB300 (sm_103a) DARTree supertree builder.
 *
 * What it computes.  DARTree builds a speculative draft tree with a causal
 * correction head: level by level, ONE batched head call scores every kept
 * path, each path is expanded by its top-k children, candidates are scored by
 * accumulated (corrected) path log-probability and the best W are kept; after
 * D levels exactly D head calls have been made and a pool of scored nodes is
 * cached.  Pruning is deferred: one global Top-B over the pool (with a depth
 * bonus beta <= 0, which by Lemma 1 equals sequential best-first max-heap
 * pruning) selects the verification tree, emitted with its tree-attention
 * (ancestor) mask.
 *   Sources: "DARTree: Teaching a Chain-Trained Corrector to Think in Trees"
 *   -- Core Mechanism; "Technische Samenvatting: DARTree" -- Methodologie
 *   1 (Depth-Wise Parallel AR Expansie) and 2 (Deferred Best-First Pruning,
 *   Lemma 1); "Accelerating Language Models with Diffusion Draft Trees" --
 *   Summary & Methodology Analysis.
 *
 * The pages do not give the correction head's architecture; this library
 * uses a fixed stand-in:
 *     state after committing token t :  s' = q(tanh(A s + E[t]))
 *     corrected logits at depth d    :  l  = z_d + s Wout^T
 * where z_d are the drafter's base logits for depth d and q() rounds to bf16
 * (nearest-even) when the weights are bf16.  The root state is q(state0).
 *
 * Conventions used by every entry point:
 *   - All array pointers are DEVICE pointers unless a function says "host".
 *     Matrices are row-major and densely packed.
 *   - Weights (A [H,H], E [V,H], Wout [V,H]) have the context's dtype: fp32
 *     or bf16 (raw 16-bit patterns).  Base logits and scores are fp32.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream).
 *     Calls are asynchronous on that stream unless stated otherwise; device
 *     checks are collected by dartree_sync_status().
 *   - Selections are total orders: top-K by (logit desc, token asc), top-W
 *     by (score desc, candidate index i*K+j asc), Top-B by (key desc, pool
 *     index asc) with key = score + beta*depth (fp32 ops in that order).
 *   - The caller owns every input and output buffer; the context owns its
 *     workspace.  No call except dartree_create allocates device memory.
 *   - Thread safety: a context is used by one host thread at a time.
 */
#ifndef DARTREE_H
#define DARTREE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dartree_status {
  DARTREE_OK = 0,
  DARTREE_ERR_INVALID_ARG = 1,  /* bad argument; nothing was launched */
  DARTREE_ERR_UNSUPPORTED = 2,  /* valid but outside this build's limits */
  DARTREE_ERR_CUDA = 3,         /* a CUDA runtime call failed (see last_error) */
  DARTREE_ERR_DEVICE_CHECK = 4, /* a kernel flagged bad data (non-finite logits,
                                   empty row, broken ancestor closure) */
  DARTREE_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up */
  DARTREE_ERR_OOM = 6           /* workspace allocation failed */
} dartree_status;

typedef enum dartree_wdtype { DARTREE_W_F32 = 0, DARTREE_W_BF16 = 1 } dartree_wdtype;

/* Build limits of this library. */
#define DARTREE_MAX_K 32     /* children per node */
#define DARTREE_MAX_ROWS 256 /* R * W: head rows per call */
#define DARTREE_MAX_D 32     /* depth */
#define DARTREE_MAX_B 1024   /* verification budget */

/* Fixed shape and capacity of a context.
 *   V, H          vocabulary size, head width.  bf16: H % 64 == 0; fp32: H % 8 == 0.
 *   max_D/W/K/B   largest per-call D, W, K, B (K <= 32, D <= 32, B <= 1024).
 *   max_requests  largest R; R * max_W must stay <= 256.
 *   wdtype        dartree_wdtype of A, E and Wout. */
typedef struct dartree_config {
  int32_t V, H, max_D, max_W, max_K, max_B, max_requests, wdtype;
} dartree_config;

/* Head weights (device, context dtype): A [H,H] (row h = output unit),
 * E [V,H] (token embeddings), Wout [V,H] (output projection). */
typedef struct dartree_head {
  const void *A, *E, *Wout;
} dartree_head;

/* Verification trees of R requests (device or, for dartree_build_host, host).
 * Request r uses parent/token/depth/score[r*B .. r*B+B), mask words
 * [r*B*ceil(B/32) ..), n_out[r].  Node i (canonical order, parents first):
 * parent rank (-1 at depth 1), token, depth (1-based), cumulative score
 * (fp32 log-prob without beta); mask row i has bit j%32 of word j/32 set iff
 * node j is i or an ancestor of i.  Rows >= n_out[r] = min(B, pool size) are
 * parent/token -1, depth 0, score 0, mask 0. */
typedef struct dartree_tree {
  int32_t *parent, *token, *depth;
  float *score;
  uint32_t *mask;
  int32_t *n_out;
} dartree_tree;

typedef struct dartree_ctx dartree_ctx;

/* Pool size of one request: sum_{d=1..D} |F_d|, |F_0| = 1,
 * |F_d| = min(W, K |F_{d-1}|).  Returns -1 on bad arguments. */
int32_t dartree_pool_size(int32_t D, int32_t W, int32_t K);

/* Creates a context on the current CUDA device and allocates all workspace
 * (the only allocating call).  Fails with UNSUPPORTED on a device other than
 * compute capability 10.3.
 * Tuning (environment, read here; defaults in brackets): the head call runs
 * the vocabulary-on-M kernel below DARTREE_ROWS_MIN head rows [64] and the
 * row-major kernel from there, in vocabulary tiles of DARTREE_ROWS_NV
 * entries [256; or 128], with more than 128 rows on CTA pairs unless
 * DARTREE_ROWS_PAIR=0, and with at most 64 rows on one CTA streaming 64-row
 * state boxes unless DARTREE_ROWS_HALF_S=0; DARTREE_TC_MAX_STAGES caps the
 * pipeline depth and DARTREE_TC_CTAS_PER_SM=2 puts two vocabulary-on-M CTAs
 * on an SM; the row merge keeps only the list keys that reach the head
 * call's row bound unless DARTREE_MERGE_BOUND=0, with the row blocks of a
 * request (at most 16) as one thread-block cluster that hands the rows to
 * the selection in shared memory unless DARTREE_MERGE_CLUSTER=0; the Top-B
 * of pools of 512 or more nodes is a block radix select (DARTREE_RADIX=0:
 * never, =1: the top-W and every Top-B as well); the top-W of at most
 * DARTREE_RANK_MAX
 * candidates [512, at most 1024] is picked by rank counting; fp32 head calls
 * of at most 16 rows use four threads per weight row unless
 * DARTREE_F32_SPLIT=0, and also compute the next state contraction unless
 * DARTREE_F32_FOLD=0.  Results are the same under every setting (up to the
 * order of fp32 additions). */
dartree_status dartree_create(const dartree_config *cfg, dartree_ctx **out);

/* Releases the context and its workspace (synchronises the device). */
void dartree_destroy(dartree_ctx *ctx);

/* One supertree build for R independent requests sharing one head.
 *   base_logits [R, D, V] fp32 : drafter logits z_d per request and depth.
 *   state0      [R, H]    fp32 : head state at each request's prefix.
 *   Requires 1 <= D, W, K, B, R within the context's limits, K <= V,
 *   beta <= 0 (Lemma 1 needs a non-positive depth bonus), and with bf16
 *   weights A, E and Wout 16-byte aligned (INVALID_ARG otherwise).
 * Runs D batched head calls (dartree_head_calls() reports them), then the
 * deferred Top-B and the mask; writes `out`.  Asynchronous; never allocates
 * device memory.  On a created stream (not the legacy NULL stream, not one
 * being captured by the caller) the launches of a build are captured once
 * into a CUDA graph; a later call with the same arguments (sizes, pointers,
 * stream) replays it, reading the buffers' current contents.  Set
 * DARTREE_GRAPH=0 to launch eagerly, DARTREE_PDL=0 to turn off programmatic
 * dependent launch between the kernels. */
dartree_status dartree_build(dartree_ctx *ctx, const float *base_logits, const float *state0,
                             const dartree_head *head, int32_t R, int32_t D, int32_t W, int32_t K,
                             int32_t B, float beta, const dartree_tree *out, void *stream);

/* Build variants (dartree_build_ex).  All zeros = dartree_build.
 *
 * head_kind
 *   DARTREE_HEAD_RECURRENT  s' = q(tanh(A s + E[tok])) (A required).
 *   DARTREE_HEAD_MARKOV     s' = q(tanh(E[tok])): the state after a token
 *       depends on that token alone (the A = 0 case; head->A may be NULL and
 *       is not read).  "Technische Samenvatting: DARTree", Experimentele
 *       Resultaten, Ablatie: DARTree applied to the DSpark drafter, whose
 *       correction head is Markov.
 * candidates
 *   DARTREE_CAND_CORRECTED  each branch's children are the top-K of its own
 *       corrected distribution over the whole vocabulary ("DARTree: Teaching
 *       a Chain-Trained Corrector to Think in Trees", Core Mechanism).
 *   DARTREE_CAND_BASE       the K candidates of depth d are the top-K of the
 *       base logits z_d (z desc, token asc), shared by every branch of the
 *       request; each branch scores them with its corrected logits
 *       z_d[c] + s . Wout[c], normalised over the K candidates (log-softmax
 *       restricted to them).  "Technische Samenvatting: DARTree",
 *       Methodologie 1 (Kandidaat Selectie from the base logits; Gebatchte
 *       Correctie of the candidates of all branches in one batch).
 * expansion
 *   DARTREE_EXPAND_DEPTHWISE   the DARTree build: D batched head calls, then
 *       the deferred Top-B.
 *   DARTREE_EXPAND_BESTFIRST   the sequential baseline that DARTree replaces:
 *       node-by-node best-first growth with one head call per expanded node
 *       (B calls).  "Technische Samenvatting: DARTree", Probleemstelling
 *       (Causale Correctie: pop one node, correct it, push its children) and
 *       Experimentele Resultaten, Ablatie (latency of the sequential
 *       heap build).  The tree, in pop order, goes to `out` in the same
 *       layout; W is ignored; candidates must be CORRECTED. */
typedef enum dartree_head_kind {
  DARTREE_HEAD_RECURRENT = 0,
  DARTREE_HEAD_MARKOV = 1
} dartree_head_kind;
typedef enum dartree_cand_kind { DARTREE_CAND_CORRECTED = 0, DARTREE_CAND_BASE = 1 } dartree_cand_kind;
typedef enum dartree_expand_kind {
  DARTREE_EXPAND_DEPTHWISE = 0,
  DARTREE_EXPAND_BESTFIRST = 1
} dartree_expand_kind;
typedef struct dartree_options {
  int32_t head_kind, candidates, expansion;
} dartree_options;

/* dartree_build with options (NULL = all zeros).  Same arguments, errors,
 * graph capture and output layout as dartree_build.  INVALID_ARG for an
 * unknown option value; UNSUPPORTED for BESTFIRST with BASE candidates. */
dartree_status dartree_build_ex(dartree_ctx *ctx, const float *base_logits, const float *state0,
                                const dartree_head *head, int32_t R, int32_t D, int32_t W,
                                int32_t K, int32_t B, float beta, const dartree_options *opt,
                                const dartree_tree *out, void *stream);

/* Same as dartree_build with HOST base_logits, state0 and outputs (weights
 * stay on the device): copies the inputs into the context's staging buffers,
 * builds, copies the tree back and synchronises the stream.  Depth 1's base
 * logits and state0 are copied on `stream`; the later depths' on a context
 * stream, overlapping the first head call (the head call of depth 2 waits
 * for them).  The host buffers should be pinned (page-locked) for the copies
 * to overlap.  Returns the folded device status like dartree_sync_status. */
dartree_status dartree_build_host(dartree_ctx *ctx, const float *base_logits_host,
                                  const float *state0_host, const dartree_head *head, int32_t R,
                                  int32_t D, int32_t W, int32_t K, int32_t B, float beta,
                                  const dartree_tree *out_host, void *stream);

/* Synchronises `stream`, reads and clears the device check word and returns
 * OK, DEVICE_CHECK or TIMEOUT (or CUDA if the synchronisation failed).  After
 * a device error it also resets the context's arrival counters, so the
 * context can be used again; the failed build's outputs are undefined.
 * With ctx == NULL it reports the context-free state step instead
 * (dartree_state_step_noalloc on the current device): the flags its calls
 * gathered since the last such report, cleared on read; OK when no call has
 * run on the device (reason text in dartree_last_error(NULL)).
 * Test knob: DARTREE_WAIT_LIMIT_CYCLES (read at dartree_create, and at every
 * dartree_state_step_noalloc call) shortens the kernels' pipeline waits to
 * provoke the TIMEOUT path. */
dartree_status dartree_sync_status(dartree_ctx *ctx, void *stream);

/* Number of head calls made by the last build: D for a depth-wise build,
 * B for a best-first one (one per step, including steps whose node cannot
 * be expanded). */
int64_t dartree_head_calls(const dartree_ctx *ctx);

/* Layout of the output projection Wout that a bf16 context's later calls
 * read (dartree_build, _build_ex, _build_host, _head_topk; A and E stay
 * row-major):
 *   DARTREE_LAYOUT_ROWS   [V][H] row-major (the default);
 *   DARTREE_LAYOUT_BLOCKS blocks of 128 rows x 64 columns: block (b, k) --
 *                         rows 128 b .. 128 b + 127, columns 64 k .. 64 k +
 *                         63 -- at element (b * H/64 + k) * 8192, row-major
 *                         inside (64 elements per row); rows past V are zero.
 * Each head call streams the projection in exactly these blocks, so with
 * the blocked layout every 16 KB piece is one contiguous read instead of 128
 * strided 128-byte pieces (measured: q8b 3.151 -> 3.088 ms per build, q4b
 * 2.057 -> 1.965).  Results are bit-identical in both layouts.  Convert once
 * with dartree_block_weights (the weights do not change between builds).
 * Base-logit candidates (DARTREE_CAND_BASE) gather K whole rows per head
 * row, which only the row-major layout keeps contiguous: that variant runs
 * about 5 % slower blocked.
 * Returns INVALID_ARG for a NULL context or an unknown layout and
 * UNSUPPORTED for BLOCKS on an fp32 context. */
#define DARTREE_LAYOUT_ROWS 0
#define DARTREE_LAYOUT_BLOCKS 1
dartree_status dartree_set_weight_layout(dartree_ctx *ctx, int32_t layout);

/* Bytes of a [V][H] bf16 matrix in the blocked layout: ceil(V/128) * 128 *
 * H * 2 (0 for H not a multiple of 64 or a size below 1). */
size_t dartree_blocked_weight_bytes(int32_t V, int32_t H);

/* Writes the blocked layout of the row-major bf16 matrix W [V][H] (device
 * memory, 16-byte aligned; H a multiple of 64) into W_blocked
 * (dartree_blocked_weight_bytes(V, H) bytes of device memory, 16-byte
 * aligned, not overlapping W).  Context-free, asynchronous on `stream`, no
 * allocation; INVALID_ARG on bad sizes, pointers or alignment. */
dartree_status dartree_block_weights(const void *W, int32_t V, int32_t H, void *W_blocked,
                                     void *stream);

/* Text of the last error recorded by this context ("" if none); with a NULL
 * context, why the last failed context-free call on this thread
 * (dartree_create or dartree_state_step_noalloc) failed. */
const char *dartree_last_error(const dartree_ctx *ctx);

/* Per-kernel timing.  When enabled, every launch of a build is bracketed by
 * CUDA events on the build's stream; dartree_sync_status() adds the elapsed
 * times to per-kind totals.  Kinds: 0 head call (fused logits + log-softmax
 * + top-K partials; with base candidates the candidate logits), 1 state
 * step, 2 row merge, 3 top-W select, 4 Top-B + mask, 5 root rows, 6 base
 * candidates (top-K of the base logits), 7 best-first step (node append +
 * pop).  Enabling creates the events (no device memory). */
#define DARTREE_KERNEL_KINDS 8
dartree_status dartree_set_timing(dartree_ctx *ctx, int32_t enable);
/* Totals since the last reset: milliseconds and launch count per kind. */
dartree_status dartree_get_timing(const dartree_ctx *ctx, int32_t kind, double *total_ms,
                                  int64_t *launches);
dartree_status dartree_reset_timing(dartree_ctx *ctx);

/* Debug: copy the last depth-wise build's pool ([R, P] each, pool index
 * depth-major, rank order within a depth, parent = pool index or -1) into
 * any memory (host or device).  Asynchronous on `stream`. */
dartree_status dartree_get_pool(dartree_ctx *ctx, int32_t *parent, int32_t *token,
                                int32_t *depth, float *score, void *stream);

/* Debug: the last build's per-row head results at depth d (1-based) for its
 * R*|F_{d-1}| head rows: lse [rows] fp64, top-K tokens [rows, K] and their
 * log-probs [rows, K].  After a best-first build, d = 1..B selects head call
 * d-1 and rows = R (one per request; call 0 expands the root, call q+1 the
 * node popped at rank q when its depth is below D, otherwise its results
 * are unused).  Any memory; asynchronous. */
dartree_status dartree_get_rows(dartree_ctx *ctx, int32_t d, double *lse, int32_t *tok,
                                float *logp, void *stream);

/* Debug: the head states used by head call d (1-based) of the last build,
 * [R*|F_{d-1}|, H] in the context's dtype (bf16 bits or fp32), row order as
 * dartree_get_rows (best-first: [R, H], the states of call d-1).  Any
 * memory; asynchronous. */
dartree_status dartree_get_states(dartree_ctx *ctx, int32_t d, void *states, void *stream);

/* One batched head call (corrected logits fused with log-softmax and top-K)
 * for M head rows with states S [M, H] (context dtype: bf16 bits or fp32).
 * Row m belongs to request m / rows_per_req and uses base logits
 * z + (m / rows_per_req) * z_req_stride (fp32 [V]).  Outputs: lse [M] fp64,
 * tok [M, K] int32, logp [M, K] fp32 (= logit - lse), sorted by (logit desc,
 * token asc).  M <= 256, K <= max_K, K <= V.  Asynchronous. */
dartree_status dartree_head_topk(dartree_ctx *ctx, const void *S, const float *z,
                                 int64_t z_req_stride, int32_t rows_per_req, const void *Wout,
                                 int32_t M, int32_t K, double *lse, int32_t *tok, float *logp,
                                 void *stream);

/* Head state step for M rows: S_out[m] = q(tanh(A S_par[m] + E[tok[m]])).
 * S_par, S_out [M, H] in the context dtype; tok [M] int32 in [0, V).
 * M <= 256; bf16 A and E 16-byte aligned (INVALID_ARG otherwise).
 * Asynchronous. */
dartree_status dartree_state_step(dartree_ctx *ctx, const void *S_par, const int32_t *tok,
                                  const void *A, const void *E, int32_t M, void *S_out,
                                  void *stream);

/* Deferred Top-B + compaction + mask over given pools (pool arrays [R, P],
 * layout as dartree_get_pool).  R <= max_requests, P <= R-independent pool
 * capacity of the context, B <= max_B, beta <= 0.  Asynchronous. */
dartree_status dartree_prune(dartree_ctx *ctx, const int32_t *pool_parent,
                             const int32_t *pool_token, const int32_t *pool_depth,
                             const float *pool_score, int32_t R, int32_t P, int32_t B, float beta,
                             const dartree_tree *out, void *stream);

/* Head state step that allocates no device memory, for callers that cannot
 * create a context: code whose device heap belongs to someone else (an
 * inference server or framework whose caching allocator has reserved the
 * GPU's memory, a plugin that may only use the buffers it is handed) and
 * latency-critical paths that cannot pay for cudaMalloc/cudaFree, which
 * synchronise the device.  The paper has no counterpart; this is a library
 * convenience.
 *   Computes S_out[m] = bf16(tanh(A S_par[m] + E[tok[m]])) for m < M, like
 *   dartree_state_step, with bf16 weights: S_par, S_out [M, H] bf16 bits,
 *   tok [M] int32 in [0, V), A [H, H], E [V, H] bf16 bits (A and E 16-byte
 *   aligned, else INVALID_ARG).  Device pointers; asynchronous on `stream`.
 *   Limits: M <= 256, H <= 4096 and H % 64 == 0; larger sizes return
 *   DARTREE_ERR_UNSUPPORTED (reason in dartree_last_error(NULL)) and launch
 *   nothing.
 *   Scratch: about 12 MiB of statically allocated device memory, held by
 *   every GPU that loads the library until the process exits.  The first
 *   call on a device sets that device up (symbol lookup, a small synchronous
 *   copy): make it before any stream capture.  All calls share the scratch,
 *   so calls that overlap on the GPU race; order them on one stream.  Each
 *   call zeroes only the padding rows of its staging array (rows M up to
 *   the MMA's padded row count); every other scratch byte it reads was
 *   written earlier in the same call.
 *   Device checks (a pipeline wait that ran out, a bad index) gather in a
 *   per-device word until dartree_sync_status(NULL, stream) synchronises,
 *   reports them as TIMEOUT / DEVICE_CHECK and clears the word; S_out of a
 *   call that failed is undefined. */
dartree_status dartree_state_step_noalloc(const void *S_par, const int32_t *tok, const void *A,
                                          const void *E, int32_t H, int32_t M, void *S_out,
                                          void *stream);

/* ------------------------------------------------------------------
 * Verification consumer of a built tree ("DARTree: Teaching a Chain-Trained
 * Corrector to Think in Trees", Core Mechanism: with the tree and its mask a
 * single target forward verifies all branches, and the longest prefix the
 * target agrees with is kept; "Technische
 * Samenvatting: DARTree", Methodologie 2, Verificatie).  Context-free,
 * asynchronous on `stream`, no allocation.  Errors are INVALID_ARG /
 * UNSUPPORTED before any launch; dartree_last_error(NULL) has the text.
 * ------------------------------------------------------------------ */

/* One attention layer of the target over the prefix and the tree of R
 * requests (all device memory, bf16 bits unless stated):
 *   Q    [R][B+1][Hq][dh]  queries; row 0 = the root (the last verified
 *                          token, already at prefix position Lp-1), rows
 *                          1..B = the tree nodes in canonical order;
 *   K    [R][Hkv][L][dh]  the key cache, L = Lp + B: per key/value head the
 *                          Lp prefix keys, then the B tree nodes' keys in
 *                          canonical order;
 *   Vt   [R][Hkv][ceil(L/64)][dh][64]  the value cache in blocks of 64 keys,
 *                          each block transposed (keys innermost; same key
 *                          order; entries past L are ignored);
 *   mask [R][B][ceil(B/32)] the build's ancestor mask (dartree_tree.mask);
 *   O    [R][B+1][Hq][dh] fp32 out; O_bf16 the same rounded to bf16 (or NULL).
 * Row 0 attends to the Lp prefix keys; node i attends to the prefix and to
 * the nodes j of mask row i-1.  Query head h reads key/value head
 * h / (Hq/Hkv).  O = softmax(scale * q.k) v with fp32 accumulation on the
 * tensor cores; the softmax weights are rounded to bf16 for the P.V
 * product and its normaliser.  A row with no visible key gives 0.  dh must
 * be 128 (UNSUPPORTED otherwise); Hq % Hkv == 0, B <= 1024,
 * (B+1) (Hq/Hkv)^2 < 2^32 (UNSUPPORTED otherwise); Q, K, Vt, O 16-byte
 * aligned.
 * When a launch would leave SMs idle the keys are split over up to 8 CTAs
 * per query tile (a thread-block cluster that combines its partial rows in
 * distributed shared memory).  work / work_bytes: unused (the splits need
 * no scratch; kept for the interface, may be NULL).
 * err: optional device word; a bounded pipeline wait that runs out ORs
 * 2 (timeout) into it (NULL: a library-internal word). */
dartree_status dartree_tree_attention(const void *Q, const void *K, const void *Vt,
                                      const uint32_t *mask, int32_t R, int32_t Lp, int32_t B,
                                      int32_t Hq, int32_t Hkv, int32_t dh, float scale, float *O,
                                      void *O_bf16, void *work, size_t work_bytes, int32_t *err,
                                      void *stream);

/* Scratch bytes dartree_tree_attention needs: 0 (the key splits combine in
 * distributed shared memory). */
size_t dartree_tree_attention_workspace(int32_t R, int32_t Lp, int32_t B, int32_t Hq,
                                        int32_t Hkv);

/* Longest accepted prefix of each request's tree (device memory):
 *   parent, token [R][B], n_out [R]  the build's output;
 *   pred [R][B+1]  the target's token after the root (0) and after node i (i+1).
 * From the root, the child whose token equals the current node's prediction
 * is accepted and becomes the current node (siblings carry distinct tokens).
 * Out: accept_len [R] (number of accepted draft tokens), accept_nodes
 * [R][max_len] (their ranks in order, -1 after the end; a longer path keeps
 * only its first max_len ranks), bonus [R] (the prediction at the last
 * accepted node, the root's when none). */
dartree_status dartree_accept(const int32_t *parent, const int32_t *token, const int32_t *n_out,
                              const int32_t *pred, int32_t R, int32_t B, int32_t max_len,
                              int32_t *accept_len, int32_t *accept_nodes, int32_t *bonus,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DARTREE_H */
