// Kernel parameter blocks and launchers (host <-> device, internal).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <string>

namespace dt {

// Batched head contraction (tensor-core bf16 path and SIMT fp32 path).
struct TcParams {
  int pdl;             // launch with programmatic dependent launch (host only)
  int rows;            // rows of the weight matrix: V (logits) or H (state)
  int H;               // contraction length
  int M;               // valid head rows (GEMM columns)
  int n_tiles;         // ceil(rows / 128)
  int stages;          // pipeline depth (set by the launcher)
  int max_stages;      // launcher cap on the pipeline depth (0: default)
  int ctas_per_sm;     // CTAs sharing one SM's shared memory (0: 1)
  int* err;            // device error word
  long long wait_limit;  // pipeline wait limit in cycles (0: the full ~2 s)
  int V_tok;           // vocabulary size (bound of state-step tokens)
  int w_tiled;         // logits: the weights in blocks of 128 rows x 64 columns
                       // (DARTREE_LAYOUT_BLOCKS), block (tile, k step) at row
                       // (tile * w_nk + k step) * 128 of a [rows][64] tensor map
  int w_nk;            // k steps of 64 per weight row (H / 64)
  int s_rows;          // row-major head kernel: state rows per TMA box of tmap_s (64: one
                       // CTA with at most 64 live rows and 256-entry tiles; else 128)
  // logits epilogue
  const float* z;      // base logits of this depth, request 0
  long long z_req_stride;
  int rows_per_req;    // head rows per request (|F_{d-1}|)
  int K;
  float* pm;           // [rows_max][cta_stride] running max per CTA
  float* ps;           // [rows_max][cta_stride] sum exp(x - max) per CTA
  uint64_t* ptop;      // [rows_max][list_stride][K] per-CTA top-K keys
  unsigned long long* gth;  // [rows_max] per-row global bound of the K-th key (zero
                            // between launches)
  unsigned long long* gmx;  // [rows_max][32] per row, the best key of each CTA group
                            // (CTA % K); zero between launches
  int cta_stride;
  int list_stride;
  // state epilogue: U = A S_in for the M input rows, then output row q
  // (q < M_out) is q(tanh(U[:, slot[q]] + E[tok[q]])); rows M_out .. pad
  // are written as zeros.
  int M_out;
  const int32_t* slot;       // [M_out] input row (parent) of each output row
  const int32_t* tok;        // [M_out] committed token of each output row
  const uint16_t* E_bf16;    // [V][H]
  uint16_t* S_out_bf16;      // [rows_max][H]
  int n_split;               // contraction split across CTAs (tensor-core path)
  int early_operands;        // the weights and S_in were complete before the previous
                             // kernel started: stream them before waiting for it
                             // (only slot / tok / scratch come from that kernel)
  float* part;               // [n_split][256][H] fp32 partial sums of U = A S_in
                             // (split-K; finished by k_state_finish)
  // SIMT operands (fp32 path)
  const float* W_f32;        // [rows][H]
  const float* S_f32;        // [rows_max][H]
  // k_head_f32 with the next depth's state contraction folded in: tiles
  // n_tiles .. n_tiles + ceil(H / 128) - 1 take A's rows and write
  // U = A S_in (row-major [M][H]) instead of logits
  const float* A_f32;        // [H][H], 16-byte aligned, or null
  float* U_f32;              // [M][H]
};

// One object file per MMA N (16, 32, 64, 128, 256) defines these.
#define DT_DECLARE_N(NN)                                                                    \
  cudaError_t init_head_tc_attrs_##NN();                                                    \
  cudaError_t launch_head_tc_##NN(bool logits, const CUtensorMap& tw, const CUtensorMap& ts, \
                                  const TcParams& p, int grid, cudaStream_t st);            \
  cudaError_t init_head_simt_attrs_##NN();                                                  \
  cudaError_t launch_head_simt_##NN(const TcParams& p, int grid, cudaStream_t st);
DT_DECLARE_N(16)
DT_DECLARE_N(32)
DT_DECLARE_N(64)
DT_DECLARE_N(128)
DT_DECLARE_N(256)
#undef DT_DECLARE_N

inline cudaError_t launch_head_tc(int n_pad, bool logits, const CUtensorMap& tw,
                                  const CUtensorMap& ts, const TcParams& p, int grid,
                                  cudaStream_t st) {
  switch (n_pad) {
    case 16: return launch_head_tc_16(logits, tw, ts, p, grid, st);
    case 32: return launch_head_tc_32(logits, tw, ts, p, grid, st);
    case 64: return launch_head_tc_64(logits, tw, ts, p, grid, st);
    case 128: return launch_head_tc_128(logits, tw, ts, p, grid, st);
    case 256: return launch_head_tc_256(logits, tw, ts, p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// Logits head call with the head rows on the MMA M side (head_rows.cu):
// M in [1, 256] rows (one or two 128-row halves), vocabulary tiles of nv
// (128 or 256) entries; ts is the state map with 128-row boxes.  pair: M in
// [129, 256] with the two-CTA MMA over CTA pairs (nv = 256).  `units` CTAs
// (pairs) requested; units_used receives the count launched (= the number
// of partial slots per row).
cudaError_t init_head_rows_attrs();
cudaError_t launch_head_rows(int M, int nv, bool pair, const CUtensorMap& tw, const CUtensorMap& ts,
                             const TcParams& p, int units, cudaStream_t st, int* units_used);

// Logits head call with fp32 weights and at most 16 head rows, four threads
// per weight row (head_f32.cu; W_f32 16-byte aligned).  head_f32_fits says
// which calls it takes.
bool head_f32_fits(int M, int H, int K);
cudaError_t init_head_f32_attrs();
cudaError_t launch_head_f32(const TcParams& p, int grid, cudaStream_t st);

inline cudaError_t launch_head_simt(int n_pad, const TcParams& p, int grid, cudaStream_t st) {
  switch (n_pad) {
    case 16: return launch_head_simt_16(p, grid, st);
    case 32: return launch_head_simt_32(p, grid, st);
    case 64: return launch_head_simt_64(p, grid, st);
    case 128: return launch_head_simt_128(p, grid, st);
    case 256: return launch_head_simt_256(p, grid, st);
    default: return cudaErrorInvalidValue;
  }
}

// Finish of a split-K state step: output row q (q < n_out, zeros from
// M_out on) is q(tanh(sum_s part[s][slot[q]][:] + E[tok[q]][:])).
struct StateFinishParams {
  int pdl;             // launch with programmatic dependent launch (host only)
  int H, M_in, M_out, n_out, n_split, V_tok;
  const float* part;   // [n_split][256][H]
  const int32_t* slot; // [M_out] input row (parent) of each output row
  const int32_t* tok;  // [M_out]
  const uint16_t* E;   // [V][H] bf16
  uint16_t* S_out;     // [256][H] bf16
  int* err;
};
cudaError_t launch_state_finish(const StateFinishParams& p, cudaStream_t st);

// State step with fp32 weights: S_out[q] = tanh(A S_in[slot[q]] + E[tok[q]])
// for q < M_out, zeros up to n_out.
struct StateF32Params {
  int pdl;             // launch with programmatic dependent launch (host only)
  int H, M_in, M_out, n_out, V_tok;
  const float* A;      // [H][H]
  const float* S_in;   // [M_in][H]
  const int32_t* slot; // [M_out] input row (parent) of each output row
  const int32_t* tok;  // [M_out]
  const float* E;      // [V][H]
  float* S_out;        // [n_out][H]
  int* err;
};
cudaError_t launch_state_f32(const StateF32Params& p, cudaStream_t st);

// Merge of per-CTA partials into per-row lse and top-K (log-probs), and
// (select != 0) the global top-W of each request with pool append.
struct MergeParams {
  int pdl;             // launch with programmatic dependent launch (host only)
  int groups;          // blocks per row, each merging a contiguous share of the CTAs
  uint64_t* gpl;       // [256][8][32] per-group top-K lists
  float2* gls;         // [256][8] per-group (max, sum-exp)
  int* row_cnt;        // [256] group arrival counters, zero between launches
  unsigned long long* gth;  // [256] per-row top-K bounds of the head call (reset here)
  unsigned long long* gmx;  // [256][32] per-row CTA-group best keys (reset here)
  const float* pm;
  const float* ps;
  const uint64_t* ptop;
  int n_cta;
  int cta_stride;
  int list_stride;
  int K;
  int M;
  double* row_lse;     // [M]
  int32_t* row_tok;    // [M][K]
  float* row_logp;     // [M][K]
  int* err;
  // fused selection
  int select;
  int R, F, Fd, depth;       // depth is 1-based; F = rows per request
  int off_prev, off;         // pool offsets of depth-1 and depth
  int pool_stride;           // pool entries per request
  const float* score_in;     // [R*F]
  float* score_out;          // [R*Fd]
  int32_t* slot_next;        // [R*Fd] parent row (in this call) of each kept node
  int32_t* tok_next;         // [R*Fd]
  int32_t* pool_parent;
  int32_t* pool_token;
  int32_t* pool_depth;
  float* pool_score;
  int* counters;             // [R] zero between launches
  int surv_cap;              // k_merge_bound: keys at or above the bound staged in shared
                             // memory (at most 512; more go the slow way)
  int radix;                 // top-W by block radix select (else as below)
  int rank_max;              // top-W by rank counting when F K <= rank_max (else merge
                             // folds / bitonic sort)
  int cluster;               // k_merge_bound with select: the F row blocks of a request
                             // are one thread-block cluster (F <= kClusterRows); the rows
                             // reach the selection through the leader's shared memory
  // fp32 state step folded into the selection (the head call wrote U = A S
  // for its rows): the request's next rows S_next[m] = tanh(U[slot_next[m]]
  // + E[tok_next[m]])
  const float* U_f32;        // [R*F][H], or null: no state step here
  const float* E_f32;        // [V_tok][H]
  float* S_next_f32;         // [R*Fd][H]
  int H, V_tok;
};
cudaError_t launch_merge_rows(const MergeParams& p, cudaStream_t st);
// The same merge (and selection) with one block per row that keeps only the
// list keys reaching the head call's row bound (K <= 32, at most 320
// partials per row; merge_bound_fits says which).
bool merge_bound_fits(const MergeParams& p);
cudaError_t launch_merge_bound(const MergeParams& p, cudaStream_t st);
// Largest cluster of k_merge_bound blocks the device schedules (at most
// kClusterRows; 0 when clusters cannot be used).
constexpr int kClusterRows = 16;
int merge_cluster_limit();

// Deferred Top-B, compaction and the ancestor mask.
struct PruneParams {
  int pdl;             // launch with programmatic dependent launch (host only)
  int R, P, pool_stride, B, words;
  float beta;
  const int32_t* pool_parent;
  const int32_t* pool_token;
  const int32_t* pool_depth;
  const float* pool_score;
  int32_t* parent;
  int32_t* token;
  int32_t* depth;
  float* score;
  uint32_t* mask;
  int32_t* n_out;
  int* err;
  int radix;           // Top-B by block radix select (else a bitonic sort of the pool)
};
cudaError_t launch_prune(const PruneParams& p, cudaStream_t st);

// Root rows: S[r] = q(state0[r]), zero padding rows, scores 0.
struct RootParams {
  int pdl;             // launch with programmatic dependent launch (host only)
  int R, n_pad, H, bf16;
  const float* state0;
  void* S;
  float* score;
};
cudaError_t launch_root(const RootParams& p, cudaStream_t st);

// Markov head state (the state depends on the last token only):
// S_out[q] = q(tanh(E[tok[q]])) for q < M_out, zero rows up to n_out.
struct MarkovParams {
  int pdl;
  int M_out, n_out, H, V, bf16;
  const int32_t* tok;  // [M_out]
  const void* E;       // [V][H] bf16 bits or fp32
  void* S_out;         // [n_out][H]
  int* err;
};
cudaError_t launch_state_markov(const MarkovParams& p, cudaStream_t st);

// Base-logit candidates: the top-K of every row of z ([rows][V], a row per
// (request, depth)) by (z desc, token asc).  Grid (chunks, rows); the last
// chunk block of a row merges the chunk lists.
struct BaseTopkParams {
  int pdl;
  int rows, V, K, n_chunks;
  const float* z;
  uint64_t* part;   // [rows][n_chunks][K] chunk lists
  int* cnt;         // [rows] arrival counters, zero between launches
  int32_t* cand;    // [rows][K] candidate tokens, best first
  int* err;
};
constexpr int kBaseChunk = 8192;  // vocabulary entries per chunk block
cudaError_t launch_base_topk(const BaseTopkParams& p, cudaStream_t st);

// Corrected logits of the K base candidates of each head row, written as the
// row's single partial (n_cta = 1) of the row merge: one (max, sum-exp) pair
// over the K candidates and the K keys sorted.
struct CandParams {
  int pdl;
  int M, H, K, rows_per_req, bf16;
  const float* z;           // this depth's base logits, request 0
  long long z_req_stride;
  const int32_t* cand;      // this depth's candidates, request 0
  long long cand_req_stride;
  const void* S;            // [M][H] head states (bf16 bits or fp32)
  const void* Wout;         // [V][H], or blocks of 128 x 64 (w_tiled, bf16)
  int w_tiled, w_nk;        // (w_nk = H / 64)
  float* pm;
  float* ps;
  uint64_t* ptop;
  int cta_stride, list_stride;
  int* err;
};
cudaError_t launch_cand_logits(const CandParams& p, cudaStream_t st);

// Row-major bf16 W [V][H] (H a multiple of 64) -> blocks of 128 rows x 64
// columns (DARTREE_LAYOUT_BLOCKS), rows past V zero.
cudaError_t launch_block_weights(const uint16_t* W, int V, int H, uint16_t* out,
                                 cudaStream_t st);

// Sequential best-first baseline: requests advance in lockstep, one head
// call (one row per request) per step.  Per request a node table holds every
// created node; `st` = {nodes created, nodes popped, node expanded by the
// current call (-1 root), expand flag}.
struct BestFirstParams {
  int pdl;
  int R, B, K, D, H, words, bf16;
  float beta;
  int max_nodes;                 // node table entries per request (B * K)
  int32_t* node_par;             // [R][max_nodes] parent node (-1: root)
  int32_t* node_tok;
  int32_t* node_dep;
  int32_t* node_rank;            // popped rank, -1 while in the heap
  float* node_score;
  int* st;                       // [R][4]
  const int32_t* row_tok;        // [R][K] this call's children
  const float* row_logp;         // [R][K]
  const void* S_call;            // [256][H] this call's head states
  void* S_pop;                   // [R][B][H] state of each popped rank
  void* S_stage;                 // [256][H] parent state of the next expansion
  const void* S_root;            // [256][H] root states
  int32_t* tok_next;             // [R] token of the next expansion
  int32_t* z_row;                // [R] depth of the next expanded node (z row of its children)
  int V;
  const float* z;                // [R][D][V] base logits
  float* z_stage;                // [R][V] the base logits of the next call
  int32_t* parent;               // outputs, as dartree_tree
  int32_t* token;
  int32_t* depth;
  float* score;
  uint32_t* mask;
  int32_t* n_out;
  int* err;
};
cudaError_t launch_bestfirst_init(const BestFirstParams& p, cudaStream_t st);
cudaError_t launch_bestfirst_step(const BestFirstParams& p, cudaStream_t st);
cudaError_t launch_bestfirst_z(const BestFirstParams& p, cudaStream_t st);

// Records why the last context-free call on this thread failed; read back
// through dartree_last_error(NULL).
void set_context_free_error(const std::string& why);
// Flags gathered by dartree_state_step_noalloc on the current device (read
// and cleared after synchronising `st`); -1 if no call set the device up.
int noalloc_take_status(cudaStream_t st, cudaError_t* err);

// One-time kernel attribute setup (dynamic shared memory opt-in).
cudaError_t init_select_attrs();
inline cudaError_t init_head_attrs() {
  cudaError_t e;
  if ((e = init_head_tc_attrs_16()) != cudaSuccess) return e;
  if ((e = init_head_tc_attrs_32()) != cudaSuccess) return e;
  if ((e = init_head_tc_attrs_64()) != cudaSuccess) return e;
  if ((e = init_head_tc_attrs_128()) != cudaSuccess) return e;
  if ((e = init_head_tc_attrs_256()) != cudaSuccess) return e;
  if ((e = init_head_rows_attrs()) != cudaSuccess) return e;
  if ((e = init_head_f32_attrs()) != cudaSuccess) return e;
  if ((e = init_head_simt_attrs_16()) != cudaSuccess) return e;
  if ((e = init_head_simt_attrs_32()) != cudaSuccess) return e;
  if ((e = init_head_simt_attrs_64()) != cudaSuccess) return e;
  if ((e = init_head_simt_attrs_128()) != cudaSuccess) return e;
  return init_head_simt_attrs_256();
}

}  // namespace dt
