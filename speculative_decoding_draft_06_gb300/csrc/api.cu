// C ABI of the DARTree supertree builder: context, argument checks, tensor
// maps, and the depth loop that chains the kernels on the caller's stream.
//
// Per build (R requests, depth D):
//   root rows -> for d = 1..D { [d >= 2] state step (A) ; head call (Wout,
//   fused log-softmax + top-K partials) ; merge rows ; top-W select + pool
//   append + state gather } -> Top-B + compaction + mask.
// That is exactly D head calls ("DARTree: Teaching a Chain-Trained Corrector
// to Think in Trees", Core Mechanism and Framework Shift: head calls =
// O(depth), not O(nodes)).  Frontier sizes are a closed form, so every launch
// shape is known on the host and no data-dependent control flow is needed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/dartree.h"
#include "common.cuh"
#include "kernels.h"

using dt::pad_rows;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kNumPads = 5;  // N = 16, 32, 64, 128, 256
int pad_index(int n) { return n == 16 ? 0 : n == 32 ? 1 : n == 64 ? 2 : n == 128 ? 3 : 4; }

int frontier_after(int F, int W, int K) {
  const long long f = static_cast<long long>(K) * F;
  return f < W ? static_cast<int>(f) : W;
}

}  // namespace

struct dartree_ctx {
  dartree_config cfg{};
  int device = 0;
  int num_sms = 0;
  bool bf16 = false;
  size_t elem = 4;
  int pool_cap = 0;   // pool entries per request
  int max_cta = 0;    // partial slots per row
  EncodeTiledFn encode = nullptr;

  // workspace (device)
  void* S_all = nullptr;  // [n_slots][256][H]: slot d-1 = states of head call d
  int n_slots = 0;
  float* score[2] = {nullptr, nullptr};
  int32_t* tok_next = nullptr;      // [256] token of each next-depth row
  int32_t* slot_next = nullptr;     // [256] parent row of each next-depth row
  int32_t* iota = nullptr;          // [256] 0, 1, 2, ...
  int* counters = nullptr;          // [256] per-request arrival counters (select)
  int* row_cnt = nullptr;           // [256] per-row group arrival counters (merge)
  uint64_t* gpl = nullptr;          // [256][8][32] per-group top-K lists (merge)
  float2* gls = nullptr;            // [256][8] per-group (max, sum-exp) (merge)
  unsigned long long* gth = nullptr;  // [256] per-row top-K bound of a head call, then
                                      // [256][32] per-row CTA-group best keys
  float* part = nullptr;            // split-K partial sums of the state step
  int state_split = 1;
  int tc_max_stages = 0;   // tuning: pipeline depth cap of the head call (0: default)
  bool pdl = true;         // programmatic dependent launch between the kernels of a build
  long long wait_limit = 0;  // test knob: pipeline wait limit in cycles (0: full)
  bool use_graph = true;   // capture each build shape once into a CUDA graph
  // selection by block radix select: -1 (default) for the Top-B of pools of at
  // least 512 nodes only (where it beats the bitonic sort of the pool; the
  // top-W stays a merge of the already sorted child lists, which is faster),
  // 1 for the top-W and the Top-B, 0 never
  int radix = -1;
  bool f32_split = true;   // fp32 head calls of <= 16 rows: four threads per weight row
  bool f32_fold = true;    // ... which also compute the next state contraction
  int rank_max = 512;      // top-W by rank counting for at most this many candidates
  bool merge_cluster = true;  // the row blocks of a request as one cluster (k_merge_bound)
  int cluster_limit = 0;   // the largest such cluster the device schedules

  // the captured build and the arguments it was captured with
  struct GraphKey {
    const float *z, *s0;
    const void *A, *E, *Wout;
    int R, D, W, K, B;
    float beta;
    dartree_options opt;
    int32_t z_late;  // base logits of depth >= 2 arrive on the copy stream (dartree_build_host):
                     // 1 all before head call 2, 2 each before its own head call
    int32_t w_layout;  // the layout Wout's tensor map was encoded for
    dartree_tree out;
    cudaStream_t st;
    bool operator==(const GraphKey& o) const { return std::memcmp(this, &o, sizeof o) == 0; }
  };
  cudaGraphExec_t gexec = nullptr;
  GraphKey gkey{};
  int tc_ctas_per_sm = 1;  // tuning: head-call CTAs per SM
  int rows_min = 64;       // head calls with at least this many rows put the rows on the MMA M side
  int rows_nv = 256;       // ... in vocabulary tiles of this many entries (128 or 256)
  bool rows_pair = true;   // ... and with more than 128 rows on CTA pairs (two-CTA MMA)
  bool rows_half_s = true;  // ... and with at most 64 rows on one CTA, 64-row state boxes
  bool merge_bound = true;  // row merge through the head call's row bound (k_merge_bound)
  bool w_tiled = false;     // Wout in blocks of 128 x 64 (dartree_set_weight_layout)
  int merge_surv_cap = 512;  // ... staging at most this many keys (test knob)
  float* pm = nullptr;
  float* ps = nullptr;
  uint64_t* ptop = nullptr;
  double* rows_lse = nullptr;   // [max_D][256]
  int32_t* rows_tok = nullptr;  // [max_D][256][max_K]
  float* rows_logp = nullptr;
  int32_t* pool_parent = nullptr;
  int32_t* pool_token = nullptr;
  int32_t* pool_depth = nullptr;
  float* pool_score = nullptr;
  int* d_err = nullptr;
  // base-logit candidates (dartree_build_ex, DARTREE_CAND_BASE)
  int32_t* cand = nullptr;          // [max_requests * max_D][max_K]
  uint64_t* base_part = nullptr;    // [max_requests * max_D][base_chunks][max_K]
  int* base_cnt = nullptr;          // [max_requests * max_D]
  int base_chunks = 0;
  // sequential best-first baseline (DARTREE_EXPAND_BESTFIRST)
  int bf_nodes = 0;                 // node table entries per request (max_B * max_K)
  int32_t* bf_par = nullptr;        // [max_requests][bf_nodes]
  int32_t* bf_tok = nullptr;
  int32_t* bf_dep = nullptr;
  int32_t* bf_rank = nullptr;
  float* bf_score = nullptr;
  int* bf_st = nullptr;             // [max_requests][4]
  int32_t* bf_tok_next = nullptr;   // [max_requests]
  int32_t* bf_zrow = nullptr;       // [max_requests]
  float* bf_z = nullptr;            // [max_requests][V] base logits of the next call
  void* bf_S = nullptr;             // [max_requests][max_B][H] state per popped rank
  double* bf_lse = nullptr;         // [max_B][max_requests] rows of each call
  int32_t* bf_rtok = nullptr;       // [max_B][max_requests][max_K]
  float* bf_rlogp = nullptr;
  int last_expansion = DARTREE_EXPAND_DEPTHWISE;
  int last_B = 0;
  // staging for dartree_build_host; its base logits past depth 1 are copied
  // on copy_st while the first head call runs (z_ready: done, z_order: the
  // previous work on the build stream is done with the staging)
  cudaStream_t copy_st = nullptr;
  cudaEvent_t z_order = nullptr;
  std::vector<cudaEvent_t> z_ready;  // [max_D + 1]: depth d's base logits are complete
  float* z_stage = nullptr;
  float* s0_stage = nullptr;
  // the tree of a host build, laid out contiguously for its (R, B) so that
  // one copy brings it back (o_all), and its pinned host image with the
  // device check word after it (h_stage)
  uint8_t* o_all = nullptr;
  uint8_t* h_stage = nullptr;
  size_t o_bytes = 0;

  std::vector<CUtensorMap> tm_S;  // [n_slots * kNumPads]
  void* S(int slot) const {
    return static_cast<uint8_t*>(S_all) + static_cast<size_t>(slot) * dt::kMaxRows * cfg.H * elem;
  }
  const CUtensorMap& tmS(int slot, int n_pad) const { return tm_S[slot * kNumPads + pad_index(n_pad)]; }
  CUtensorMap tm_A{}, tm_Wout{};
  const void* tm_A_ptr = nullptr;
  const void* tm_Wout_ptr = nullptr;

  // per-kernel timing (events around launches; see dartree_set_timing)
  bool timing = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<std::pair<int, size_t>> ev_marks;  // (kind, index of start event)
  double t_ms[DARTREE_KERNEL_KINDS] = {0};
  int64_t t_n[DARTREE_KERNEL_KINDS] = {0};

  // last build
  int last_R = 0, last_D = 0, last_W = 0, last_K = 0, last_P = 0;
  int64_t head_calls = 0;
  std::string last_error;

  dartree_status fail(dartree_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    last_error = buf;
    return s;
  }
  dartree_status cuda_fail(cudaError_t e, const char* what) {
    return fail(DARTREE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  }
};

namespace {

// Why the last dartree_create on this thread failed (no context exists then).
thread_local std::string g_create_error;

dartree_status create_fail(dartree_status s, const char* what, cudaError_t e = cudaSuccess) {
  g_create_error = what;
  if (e != cudaSuccess) {
    g_create_error += ": ";
    g_create_error += cudaGetErrorString(e);
  }
  return s;
}

dartree_status encode_2d(dartree_ctx* c, CUtensorMap* m, const void* ptr, uint64_t rows,
                         uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(dt::kTileH), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = c->encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return c->fail(DARTREE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return DARTREE_OK;
}

// Launch bracketing for dartree_set_timing: start()/stop() record a pair of
// events around one kernel launch of the given kind.
struct KernelTimer {
  dartree_ctx* c;
  cudaStream_t st;
  int kind;
  size_t idx = 0;
  bool on = false;
  KernelTimer(dartree_ctx* c_, cudaStream_t st_, int kind_) : c(c_), st(st_), kind(kind_) {
    if (c->timing && c->ev_used + 2 <= c->ev_pool.size()) {
      idx = c->ev_used;
      c->ev_used += 2;
      on = cudaEventRecord(c->ev_pool[idx], st) == cudaSuccess;
    }
  }
  ~KernelTimer() {
    if (on && cudaEventRecord(c->ev_pool[idx + 1], st) == cudaSuccess)
      c->ev_marks.emplace_back(kind, idx);
  }
};

void flush_timing(dartree_ctx* c) {
  for (auto& m : c->ev_marks) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, c->ev_pool[m.second], c->ev_pool[m.second + 1]) == cudaSuccess) {
      c->t_ms[m.first] += ms;
      c->t_n[m.first] += 1;
    }
  }
  c->ev_marks.clear();
  c->ev_used = 0;
}

// Offsets of the six tree arrays of R requests of B nodes in one region
// (each 16-byte aligned): parent, token, depth, score, mask, n_out.  Returns
// the region's size.
size_t tree_layout(size_t R, size_t B, size_t* off) {
  const size_t nb = R * B, nw = nb * ((B + 31) / 32);
  const size_t sz[6] = {nb * 4, nb * 4, nb * 4, nb * 4, nw * 4, R * 4};
  size_t at = 0;
  for (int i = 0; i < 6; ++i) {
    if (off) off[i] = at;
    at += (sz[i] + 15) & ~static_cast<size_t>(15);
  }
  return at;
}

template <typename T>
cudaError_t alloc(T** p, size_t count) {
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T) + 16);
}

// Head call for M rows whose states are in state slot `sbuf` (rows >= M up to the
// padded count are zero or finite): fused logits + partials, then the row
// merge (+ the request's top-W selection when sel != nullptr).
dartree_status run_merge(dartree_ctx* c, int n_cta, int M, int K, double* lse, int32_t* tok,
                         float* logp, const dt::MergeParams* sel, cudaStream_t st);

// fp32 head call by k_head_f32 (at most 16 rows, 16-byte rows)
bool head_f32_path(const dartree_ctx* c, int M, int K) {
  return !c->bf16 && c->f32_split && dt::head_f32_fits(M, c->cfg.H, K) &&
         (reinterpret_cast<uintptr_t>(c->tm_Wout_ptr) & 15) == 0;
}

// A_fold (fp32 k_head_f32 calls only): the call also writes U = A S for its
// rows to c->part, which the selection (sel->U_f32) turns into the next states.
dartree_status run_head(dartree_ctx* c, int sbuf, const float* z, long long z_req_stride,
                        int rows_per_req, int M, int K, double* lse, int32_t* tok, float* logp,
                        const dt::MergeParams* sel, cudaStream_t st,
                        const float* A_fold = nullptr) {
  const int V = c->cfg.V, H = c->cfg.H;
  const int N = pad_rows(M);
  dt::TcParams p{};
  p.rows = V;
  p.H = H;
  p.M = M;
  p.n_tiles = (V + dt::kTileV - 1) / dt::kTileV;
  p.w_tiled = c->bf16 && c->w_tiled;
  p.w_nk = H / dt::kTileH;
  p.err = c->d_err;
  p.z = z;
  p.z_req_stride = z_req_stride;
  p.rows_per_req = rows_per_req;
  p.K = K;
  p.pm = c->pm;
  p.ps = c->ps;
  p.ptop = c->ptop;
  p.gth = c->gth;
  p.gmx = c->gth + dt::kMaxRows;
  p.cta_stride = c->max_cta;
  p.list_stride = c->max_cta;
  p.pdl = c->pdl;
  p.wait_limit = c->wait_limit;
  int grid;
  cudaError_t e;
  {
    KernelTimer tk(c, st, 0);
    if (c->bf16 && M >= c->rows_min) {  // head rows on the MMA M side
      // more than 128 rows: CTA pairs with the two-CTA MMA (256-entry tiles)
      const bool pair = M > 128 && c->rows_pair;
      const int nv = pair ? 256 : c->rows_nv;
      const int tiles = (V + nv - 1) / nv;
      int units = pair ? c->num_sms / 2 : c->num_sms;
      if (units > tiles) units = tiles;
      p.max_stages = c->tc_max_stages;
      p.s_rows = !pair && M <= 64 && nv == 256 && c->rows_half_s ? 64 : 128;
      e = dt::launch_head_rows(M, nv, pair, c->tm_Wout, c->tmS(sbuf, p.s_rows), p, units, st,
                               &grid);
    } else if (c->bf16) {
      const int slots = c->num_sms * c->tc_ctas_per_sm;
      grid = p.n_tiles < slots ? p.n_tiles : slots;
      p.max_stages = c->tc_max_stages;
      p.ctas_per_sm = c->tc_ctas_per_sm;
      e = dt::launch_head_tc(N, true, c->tm_Wout, c->tmS(sbuf, N), p, grid, st);
    } else if (head_f32_path(c, M, K)) {
      int tiles = p.n_tiles;
      if (A_fold) {  // the state tiles after the vocabulary's
        p.A_f32 = A_fold;
        p.U_f32 = c->part;
        tiles += (H + dt::kTileV - 1) / dt::kTileV;
      }
      grid = tiles < c->num_sms ? tiles : c->num_sms;
      p.W_f32 = static_cast<const float*>(c->tm_Wout_ptr);
      p.S_f32 = static_cast<const float*>(c->S(sbuf));
      e = dt::launch_head_f32(p, grid, st);
    } else {
      grid = p.n_tiles < c->max_cta ? p.n_tiles : c->max_cta;
      p.W_f32 = static_cast<const float*>(c->tm_Wout_ptr);
      p.S_f32 = static_cast<const float*>(c->S(sbuf));
      e = dt::launch_head_simt(N, p, grid, st);
    }
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "head logits launch");
  return run_merge(c, grid, M, K, lse, tok, logp, sel, st);
}

// Row merge of n_cta partials per row (+ the request's top-W selection when
// sel != nullptr).
dartree_status run_merge(dartree_ctx* c, int n_cta, int M, int K, double* lse, int32_t* tok,
                         float* logp, const dt::MergeParams* sel, cudaStream_t st) {
  const int grid = n_cta;
  cudaError_t e;
  dt::MergeParams mp{};
  if (sel) mp = *sel;
  mp.pm = c->pm;
  mp.ps = c->ps;
  mp.ptop = c->ptop;
  mp.n_cta = grid;
  mp.cta_stride = c->max_cta;
  mp.list_stride = c->max_cta;
  mp.K = K;
  mp.M = M;
  mp.row_lse = lse;
  mp.row_tok = tok;
  mp.row_logp = logp;
  mp.err = c->d_err;
  mp.select = sel != nullptr;
  mp.pdl = c->pdl;
  // split each row's CTA partials over group blocks (at most 8, at most 160
  // partials each: 20 per warp, loaded before any is merged) until about 256
  // blocks run; the last group block of a row combines the groups
  int groups = (256 + M - 1) / M;
  const int min_groups = (grid + 159) / 160;
  const int max_groups = (grid + 19) / 20;
  if (groups > max_groups) groups = max_groups;
  if (groups < min_groups) groups = min_groups;
  mp.groups = groups < 1 ? 1 : groups > 8 ? 8 : groups;
  mp.gpl = c->gpl;
  mp.gls = c->gls;
  mp.row_cnt = c->row_cnt;
  mp.gth = c->gth;
  mp.gmx = c->gth + dt::kMaxRows;
  mp.surv_cap = c->merge_surv_cap;
  mp.radix = c->radix == 1;
  mp.rank_max = c->rank_max;
  const bool bound = c->merge_bound && dt::merge_bound_fits(mp);
  mp.cluster = bound && sel && c->merge_cluster && !mp.radix && sel->F <= c->cluster_limit &&
               K <= 32;
  {
    KernelTimer tk(c, st, 2);
    e = bound ? dt::launch_merge_bound(mp, st) : dt::launch_merge_rows(mp, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "merge launch");
  return DARTREE_OK;
}

// State step: slot src+1 row q = q(tanh(A S[slot[q]] + E[tok[q]])) for
// q < M_out (zeros up to the padded count); state slot src holds M_in rows.
dartree_status run_state(dartree_ctx* c, const void* A, const void* E, int src, int M_in,
                         const int32_t* slot, const int32_t* tok, int M_out, cudaStream_t st,
                         bool early = false) {
  const int H = c->cfg.H;
  const int N = pad_rows(M_in);
  dt::TcParams p{};
  p.rows = H;
  p.H = H;
  p.M = M_in;
  p.M_out = M_out;
  p.slot = slot;
  p.tok = tok;
  p.n_tiles = (H + dt::kTileV - 1) / dt::kTileV;
  p.err = c->d_err;
  p.pdl = c->pdl;
  p.wait_limit = c->wait_limit;
  p.V_tok = c->cfg.V;
  cudaError_t e;
  KernelTimer tk(c, st, 1);
  if (c->bf16) {
    p.E_bf16 = static_cast<const uint16_t*>(E);
    p.S_out_bf16 = static_cast<uint16_t*>(c->S(src + 1));
    p.n_split = c->state_split;
    p.part = c->part;
    p.early_operands = early && c->pdl;
    e = dt::launch_head_tc(N, false, c->tm_A, c->tmS(src, N), p,
                           p.n_tiles * p.n_split, st);
    if (e == cudaSuccess && p.n_split > 1) {
      dt::StateFinishParams f{};
      f.pdl = c->pdl;
      f.H = H;
      f.M_in = M_in;
      f.M_out = M_out;
      f.n_out = pad_rows(M_out);
      f.n_split = p.n_split;
      f.V_tok = c->cfg.V;
      f.part = c->part;
      f.slot = slot;
      f.tok = tok;
      f.E = p.E_bf16;
      f.S_out = p.S_out_bf16;
      f.err = c->d_err;
      e = dt::launch_state_finish(f, st);
    }
  } else {
    dt::StateF32Params f{};
    f.pdl = c->pdl;
    f.H = H;
    f.M_in = M_in;
    f.M_out = M_out;
    f.n_out = pad_rows(M_out);
    f.V_tok = c->cfg.V;
    f.A = static_cast<const float*>(A);
    f.S_in = static_cast<const float*>(c->S(src));
    f.slot = slot;
    f.tok = tok;
    f.E = static_cast<const float*>(E);
    f.S_out = static_cast<float*>(c->S(src + 1));
    f.err = c->d_err;
    e = dt::launch_state_f32(f, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "state step launch");
  return DARTREE_OK;
}

// Markov head state step: slot src+1 row q = q(tanh(E[tok[q]])) for
// q < M_out, zeros up to the padded count.
dartree_status run_state_markov(dartree_ctx* c, const void* E, int src, const int32_t* tok,
                                int M_out, cudaStream_t st) {
  dt::MarkovParams p{};
  p.pdl = c->pdl;
  p.M_out = M_out;
  p.n_out = pad_rows(M_out);
  p.H = c->cfg.H;
  p.V = c->cfg.V;
  p.bf16 = c->bf16;
  p.tok = tok;
  p.E = E;
  p.S_out = c->S(src + 1);
  p.err = c->d_err;
  cudaError_t e;
  {
    KernelTimer tk(c, st, 1);
    e = dt::launch_state_markov(p, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "Markov state launch");
  return DARTREE_OK;
}

// Base-candidate head call for M rows in state slot `sbuf`: the corrected
// logits of each row's K candidates as one partial per row, then the row
// merge (+ selection).
dartree_status run_cand(dartree_ctx* c, int sbuf, const float* z, long long z_req_stride,
                        const int32_t* cand, long long cand_req_stride, int rows_per_req, int M,
                        int K, const void* Wout, double* lse, int32_t* tok, float* logp,
                        const dt::MergeParams* sel, cudaStream_t st) {
  dt::CandParams p{};
  p.pdl = c->pdl;
  p.M = M;
  p.H = c->cfg.H;
  p.K = K;
  p.rows_per_req = rows_per_req;
  p.bf16 = c->bf16;
  p.z = z;
  p.z_req_stride = z_req_stride;
  p.cand = cand;
  p.cand_req_stride = cand_req_stride;
  p.S = c->S(sbuf);
  p.Wout = Wout;
  p.w_tiled = c->bf16 && c->w_tiled;
  p.w_nk = c->cfg.H / dt::kTileH;
  p.pm = c->pm;
  p.ps = c->ps;
  p.ptop = c->ptop;
  p.cta_stride = c->max_cta;
  p.list_stride = c->max_cta;
  p.err = c->d_err;
  cudaError_t e;
  {
    KernelTimer tk(c, st, 0);
    e = dt::launch_cand_logits(p, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "candidate logits launch");
  return run_merge(c, 1, M, K, lse, tok, logp, sel, st);
}

dartree_status bind_weights(dartree_ctx* c, const void* A, const void* Wout) {
  if (!c->bf16) {
    c->tm_A_ptr = A;
    c->tm_Wout_ptr = Wout;
    return DARTREE_OK;
  }
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(Wout)) & 15)
    return c->fail(DARTREE_ERR_INVALID_ARG, "bf16 weights must be 16-byte aligned");
  // (A is null for the Markov head)
  dartree_status s;
  if (A != nullptr && A != c->tm_A_ptr) {
    if ((s = encode_2d(c, &c->tm_A, A, c->cfg.H, c->cfg.H, dt::kTileV)) != DARTREE_OK) return s;
    c->tm_A_ptr = A;
  }
  if (Wout != nullptr && Wout != c->tm_Wout_ptr) {
    const uint64_t vt = (static_cast<uint64_t>(c->cfg.V) + dt::kTileV - 1) / dt::kTileV;
    if ((s = c->w_tiled ? encode_2d(c, &c->tm_Wout, Wout,
                                    vt * (c->cfg.H / dt::kTileH) * dt::kTileV, dt::kTileH,
                                    dt::kTileV)
                        : encode_2d(c, &c->tm_Wout, Wout, c->cfg.V, c->cfg.H, dt::kTileV)) !=
        DARTREE_OK)
      return s;
    c->tm_Wout_ptr = Wout;
  }
  return DARTREE_OK;
}

dartree_status check_build_args(dartree_ctx* c, const void* z, const void* s0,
                                const dartree_head* head, int R, int D, int W, int K, int B,
                                float beta, const dartree_tree* out,
                                const dartree_options& o = dartree_options{}) {
  if (o.head_kind != DARTREE_HEAD_RECURRENT && o.head_kind != DARTREE_HEAD_MARKOV)
    return c->fail(DARTREE_ERR_INVALID_ARG, "unknown head kind %d", o.head_kind);
  if (o.candidates != DARTREE_CAND_CORRECTED && o.candidates != DARTREE_CAND_BASE)
    return c->fail(DARTREE_ERR_INVALID_ARG, "unknown candidate kind %d", o.candidates);
  if (o.expansion != DARTREE_EXPAND_DEPTHWISE && o.expansion != DARTREE_EXPAND_BESTFIRST)
    return c->fail(DARTREE_ERR_INVALID_ARG, "unknown expansion kind %d", o.expansion);
  if (o.expansion == DARTREE_EXPAND_BESTFIRST && o.candidates != DARTREE_CAND_CORRECTED)
    return c->fail(DARTREE_ERR_UNSUPPORTED, "best-first growth takes corrected candidates only");
  const bool need_A = o.head_kind == DARTREE_HEAD_RECURRENT;
  if (!z || !s0 || !head || (need_A && !head->A) || !head->E || !head->Wout || !out ||
      !out->parent || !out->token || !out->depth || !out->score || !out->mask || !out->n_out)
    return c->fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  const dartree_config& g = c->cfg;
  if (R < 1 || R > g.max_requests) return c->fail(DARTREE_ERR_INVALID_ARG, "R=%d out of [1,%d]", R, g.max_requests);
  if (D < 1 || D > g.max_D) return c->fail(DARTREE_ERR_INVALID_ARG, "D=%d out of [1,%d]", D, g.max_D);
  if (W < 1 || W > g.max_W) return c->fail(DARTREE_ERR_INVALID_ARG, "W=%d out of [1,%d]", W, g.max_W);
  if (K < 1 || K > g.max_K) return c->fail(DARTREE_ERR_INVALID_ARG, "K=%d out of [1,%d]", K, g.max_K);
  if (K > g.V) return c->fail(DARTREE_ERR_INVALID_ARG, "K=%d exceeds V=%d", K, g.V);
  if (B < 1 || B > g.max_B) return c->fail(DARTREE_ERR_INVALID_ARG, "B=%d out of [1,%d]", B, g.max_B);
  if (!(beta <= 0.0f)) return c->fail(DARTREE_ERR_INVALID_ARG, "beta must be <= 0 (Lemma 1)");
  // the state finish reads bf16 embedding rows with 8-byte loads
  if (c->bf16 && (reinterpret_cast<uintptr_t>(head->E) & 15))
    return c->fail(DARTREE_ERR_INVALID_ARG, "bf16 weights must be 16-byte aligned");
  const int rows = o.expansion == DARTREE_EXPAND_BESTFIRST ? R : R * W;  // head rows per call
  if (rows > dt::kMaxRows) return c->fail(DARTREE_ERR_UNSUPPORTED, "%d head rows > 256", rows);
  // the vocabulary-on-M head kernel (fewer than rows_min rows) keeps its
  // rows' lists in shared memory next to a deep pipeline
  if (c->bf16 && o.candidates == DARTREE_CAND_CORRECTED && rows < c->rows_min &&
      pad_rows(rows) * K > 2048)
    return c->fail(DARTREE_ERR_UNSUPPORTED, "padded rows x K = %d > 2048", pad_rows(rows) * K);
  return DARTREE_OK;
}

dartree_status run_bestfirst(dartree_ctx* c, const float* z, const float* s0,
                             const dartree_head* head, int R, int D, int K, int B, float beta,
                             const dartree_options& o, const dartree_tree* out, cudaStream_t st);

// z_wait (or null): z_wait[d], where not null, is complete once the base
// logits the head call of depth d reads are (depth 1's are complete on st).
dartree_status run_build(dartree_ctx* c, const float* z, const float* s0, const dartree_head* head,
                         int R, int D, int W, int K, int B, float beta, const dartree_options& o,
                         const dartree_tree* out, cudaStream_t st,
                         const cudaEvent_t* z_wait = nullptr) {
  if (o.expansion == DARTREE_EXPAND_BESTFIRST)
    return run_bestfirst(c, z, s0, head, R, D, K, B, beta, o, out, st);
  const bool markov = o.head_kind == DARTREE_HEAD_MARKOV;
  const bool base = o.candidates == DARTREE_CAND_BASE;
  dartree_status s = bind_weights(c, markov ? nullptr : head->A, head->Wout);
  if (s != DARTREE_OK) return s;
  const int V = c->cfg.V, H = c->cfg.H;
  const int P = dartree_pool_size(D, W, K);
  dt::RootParams rp{};
  rp.R = R;
  rp.n_pad = pad_rows(R);
  rp.H = H;
  rp.bf16 = c->bf16;
  rp.state0 = s0;
  rp.S = c->S(0);
  rp.score = c->score[0];
  rp.pdl = c->pdl;
  cudaError_t e;
  {
    KernelTimer tk(c, st, 5);
    e = dt::launch_root(rp, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "root launch");
  if (base) {
    // the candidates of every (request, depth): top-K of the base logits
    dt::BaseTopkParams bp{};
    bp.pdl = c->pdl;
    bp.rows = R * D;
    bp.V = V;
    bp.K = K;
    bp.n_chunks = c->base_chunks;
    bp.z = z;
    bp.part = c->base_part;
    bp.cnt = c->base_cnt;
    bp.cand = c->cand;
    bp.err = c->d_err;
    {
      KernelTimer tk(c, st, 6);
      e = dt::launch_base_topk(bp, st);
    }
    if (e != cudaSuccess) return c->cuda_fail(e, "base candidates launch");
  }
  int F = 1, F_prev = 1, off_prev = 0, off = 0, cur = 0, sbuf = 0;
  int64_t calls = 0;
  bool folded = false;  // this depth's states came with the previous selection
  for (int d = 1; d <= D; ++d) {
    const int M = R * F;
    if (d >= 2 && folded) {
      ++sbuf;
    } else if (d >= 2) {
      // states of this depth's rows from their parents (the rows of call d-1)
      // A and the parent states (written three kernels back) are complete
      // before the merge that precedes this step starts: the step streams
      // them while that merge runs
      s = markov ? run_state_markov(c, head->E, sbuf, c->tok_next, M, st)
                 : run_state(c, head->A, head->E, sbuf, R * F_prev, c->slot_next, c->tok_next,
                             M, st, /*early=*/true);
      if (s != DARTREE_OK) return s;
      ++sbuf;  // each depth keeps its own state slot
    }
    const int Fd = frontier_after(F, W, K);
    dt::MergeParams sel{};
    sel.R = R;
    sel.F = F;
    sel.Fd = Fd;
    sel.depth = d;
    sel.off_prev = off_prev;
    sel.off = off;
    sel.pool_stride = P;
    sel.score_in = c->score[cur];
    sel.score_out = c->score[cur ^ 1];
    sel.slot_next = c->slot_next;
    sel.tok_next = c->tok_next;
    sel.pool_parent = c->pool_parent;
    sel.pool_token = c->pool_token;
    sel.pool_depth = c->pool_depth;
    sel.pool_score = c->pool_score;
    sel.counters = c->counters;
    // fp32 k_head_f32 call with a next depth: it computes U = A S for its
    // rows, and the selection finishes the next depth's states (c->part is
    // the bf16 state step's scratch, unused on this path)
    const bool fold = !markov && !base && d < D && c->f32_fold && head_f32_path(c, M, K) &&
                      (reinterpret_cast<uintptr_t>(head->A) & 15) == 0;
    if (fold) {
      sel.U_f32 = c->part;
      sel.E_f32 = static_cast<const float*>(head->E);
      sel.S_next_f32 = static_cast<float*>(c->S(sbuf + 1));
      sel.H = H;
      sel.V_tok = V;
    }
    const size_t ro = static_cast<size_t>(d - 1) * dt::kMaxRows;
    if (base)
      s = run_cand(c, sbuf, z + static_cast<size_t>(d - 1) * V, static_cast<long long>(D) * V,
                   c->cand + static_cast<size_t>(d - 1) * K, static_cast<long long>(D) * K, F, M,
                   K, head->Wout, c->rows_lse + ro, c->rows_tok + ro * K, c->rows_logp + ro * K,
                   &sel, st);
    else {
      if (z_wait && z_wait[d]) {  // this depth's base logits come from the copy stream
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) cs = cudaStreamCaptureStatusNone;
        const cudaError_t ew = cudaStreamWaitEvent(
            st, z_wait[d], cs == cudaStreamCaptureStatusActive ? cudaEventWaitExternal : 0);
        if (ew != cudaSuccess) return c->cuda_fail(ew, "base-logit copy wait");
      }
      s = run_head(c, sbuf, z + static_cast<size_t>(d - 1) * V, static_cast<long long>(D) * V,
                   F, M, K, c->rows_lse + ro, c->rows_tok + ro * K, c->rows_logp + ro * K, &sel,
                   st, fold ? static_cast<const float*>(head->A) : nullptr);
    }
    if (s != DARTREE_OK) return s;
    folded = fold;
    ++calls;
    cur ^= 1;
    off_prev = off;
    off += Fd;
    F_prev = F;
    F = Fd;
  }
  dt::PruneParams pp{};
  pp.R = R;
  pp.P = P;
  pp.pool_stride = P;
  pp.B = B;
  pp.words = (B + 31) / 32;
  pp.beta = beta;
  pp.pool_parent = c->pool_parent;
  pp.pool_token = c->pool_token;
  pp.pool_depth = c->pool_depth;
  pp.pool_score = c->pool_score;
  pp.parent = out->parent;
  pp.token = out->token;
  pp.depth = out->depth;
  pp.score = out->score;
  pp.mask = out->mask;
  pp.n_out = out->n_out;
  pp.err = c->d_err;
  pp.radix = c->radix == 1 || (c->radix < 0 && P >= 512);
  pp.pdl = c->pdl;
  {
    KernelTimer tk(c, st, 4);
    e = dt::launch_prune(pp, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "prune launch");
  c->last_R = R;
  c->last_D = D;
  c->last_W = W;
  c->last_K = K;
  c->last_P = P;
  c->last_B = B;
  c->last_expansion = DARTREE_EXPAND_DEPTHWISE;
  c->head_calls = calls;
  return DARTREE_OK;
}

// Sequential best-first growth: B steps, each one head call with one row per
// request (call 0 on the root states, call q+1 on the node popped at rank q),
// then the step kernel that appends the children and pops the next node.
// State slots: 0 root states, 1 staged parent states, 2 the call's states.
dartree_status run_bestfirst(dartree_ctx* c, const float* z, const float* s0,
                             const dartree_head* head, int R, int D, int K, int B, float beta,
                             const dartree_options& o, const dartree_tree* out, cudaStream_t st) {
  const bool markov = o.head_kind == DARTREE_HEAD_MARKOV;
  dartree_status s = bind_weights(c, markov ? nullptr : head->A, head->Wout);
  if (s != DARTREE_OK) return s;
  const int V = c->cfg.V, H = c->cfg.H;
  dt::RootParams rp{};
  rp.R = R;
  rp.n_pad = pad_rows(R);
  rp.H = H;
  rp.bf16 = c->bf16;
  rp.state0 = s0;
  rp.S = c->S(0);
  rp.score = c->score[0];
  rp.pdl = c->pdl;
  cudaError_t e;
  {
    KernelTimer tk(c, st, 5);
    e = dt::launch_root(rp, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "root launch");
  dt::BestFirstParams bp{};
  bp.pdl = c->pdl;
  bp.R = R;
  bp.B = B;
  bp.K = K;
  bp.D = D;
  bp.H = H;
  bp.words = (B + 31) / 32;
  bp.bf16 = c->bf16;
  bp.beta = beta;
  bp.max_nodes = c->bf_nodes;
  bp.node_par = c->bf_par;
  bp.node_tok = c->bf_tok;
  bp.node_dep = c->bf_dep;
  bp.node_rank = c->bf_rank;
  bp.node_score = c->bf_score;
  bp.st = c->bf_st;
  bp.S_pop = c->bf_S;
  bp.S_stage = c->S(1);
  bp.S_root = c->S(0);
  bp.tok_next = c->bf_tok_next;
  bp.z_row = c->bf_zrow;
  bp.V = V;
  bp.z = z;
  bp.z_stage = c->bf_z;
  bp.parent = out->parent;
  bp.token = out->token;
  bp.depth = out->depth;
  bp.score = out->score;
  bp.mask = out->mask;
  bp.n_out = out->n_out;
  bp.err = c->d_err;
  {
    KernelTimer tk(c, st, 7);
    e = dt::launch_bestfirst_init(bp, st);
  }
  if (e != cudaSuccess) return c->cuda_fail(e, "best-first init launch");
  for (int call = 0; call < B; ++call) {
    {
      KernelTimer tk(c, st, 7);
      e = dt::launch_bestfirst_z(bp, st);
    }
    if (e != cudaSuccess) return c->cuda_fail(e, "best-first base logits launch");
    if (call >= 1) {
      s = markov ? run_state_markov(c, head->E, 1, c->bf_tok_next, R, st)
                 : run_state(c, head->A, head->E, 1, R, c->iota, c->bf_tok_next, R, st);
      if (s != DARTREE_OK) return s;
    }
    const int sbuf = call == 0 ? 0 : 2;
    const size_t ro = static_cast<size_t>(call) * c->cfg.max_requests;
    s = run_head(c, sbuf, c->bf_z, V, 1, R, K, c->bf_lse + ro, c->bf_rtok + ro * K,
                 c->bf_rlogp + ro * K, nullptr, st);
    if (s != DARTREE_OK) return s;
    bp.row_tok = c->bf_rtok + ro * K;
    bp.row_logp = c->bf_rlogp + ro * K;
    bp.S_call = c->S(sbuf);
    {
      KernelTimer tk(c, st, 7);
      e = dt::launch_bestfirst_step(bp, st);
    }
    if (e != cudaSuccess) return c->cuda_fail(e, "best-first step launch");
  }
  c->last_R = R;
  c->last_D = D;
  c->last_W = 1;
  c->last_K = K;
  c->last_P = 0;
  c->last_B = B;
  c->last_expansion = DARTREE_EXPAND_BESTFIRST;
  c->head_calls = B;
  return DARTREE_OK;
}

// One build: replay the captured graph when the arguments match the last
// capture, else capture the launches of run_build into a new graph (eager
// launches on the legacy stream and while kernel timing is on).
dartree_status build_dispatch(dartree_ctx* c, const float* z, const float* s0,
                              const dartree_head* head, int R, int D, int W, int K, int B,
                              float beta, const dartree_options& o, const dartree_tree* out,
                              cudaStream_t st, const cudaEvent_t* z_wait = nullptr,
                              int z_late = 0) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (st != nullptr && cudaStreamIsCapturing(st, &cap) != cudaSuccess) cap = cudaStreamCaptureStatusNone;
  if (!c->use_graph || c->timing || st == nullptr || cap != cudaStreamCaptureStatusNone)
    return run_build(c, z, s0, head, R, D, W, K, B, beta, o, out, st, z_wait);
  dartree_ctx::GraphKey key{};
  key.z_late = z_late;
  key.w_layout = c->w_tiled ? DARTREE_LAYOUT_BLOCKS : DARTREE_LAYOUT_ROWS;
  key.opt = o;
  key.z = z;
  key.s0 = s0;
  key.A = head->A;
  key.E = head->E;
  key.Wout = head->Wout;
  key.R = R;
  key.D = D;
  key.W = W;
  key.K = K;
  key.B = B;
  key.beta = beta;
  key.out = *out;
  key.st = st;
  if (c->gexec == nullptr || !(key == c->gkey)) {
    if (c->gexec) {
      cudaGraphExecDestroy(c->gexec);
      c->gexec = nullptr;
    }
    cudaError_t e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return c->cuda_fail(e, "begin capture");
    dartree_status s = run_build(c, z, s0, head, R, D, W, K, B, beta, o, out, st, z_wait);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(st, &g);
    if (s != DARTREE_OK) {
      if (g) cudaGraphDestroy(g);
      return s;
    }
    if (e != cudaSuccess) return c->cuda_fail(e, "end capture");
    e = cudaGraphInstantiate(&c->gexec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      c->gexec = nullptr;
      return c->cuda_fail(e, "graph instantiate");
    }
    c->gkey = key;
  } else {
    const bool bf = o.expansion == DARTREE_EXPAND_BESTFIRST;
    c->last_R = R;
    c->last_D = D;
    c->last_W = bf ? 1 : W;
    c->last_K = K;
    c->last_P = bf ? 0 : dartree_pool_size(D, W, K);
    c->last_B = B;
    c->last_expansion = o.expansion;
    c->head_calls = bf ? B : D;
  }
  cudaError_t e = cudaGraphLaunch(c->gexec, st);
  if (e != cudaSuccess) return c->cuda_fail(e, "graph launch");
  return DARTREE_OK;
}

void free_events(dartree_ctx* c) {
  for (cudaEvent_t ev : c->ev_pool) cudaEventDestroy(ev);
  c->ev_pool.clear();
  c->ev_marks.clear();
  c->ev_used = 0;
}

void free_all(dartree_ctx* c) {
  free_events(c);
  if (c->gexec) cudaGraphExecDestroy(c->gexec);
  c->gexec = nullptr;
  for (cudaEvent_t ev : c->z_ready)
    if (ev) cudaEventDestroy(ev);
  c->z_ready.clear();
  if (c->z_order) cudaEventDestroy(c->z_order);
  if (c->copy_st) cudaStreamDestroy(c->copy_st);
  c->z_order = nullptr;
  c->copy_st = nullptr;
  if (c->h_stage) cudaFreeHost(c->h_stage);
  c->h_stage = nullptr;
  void* ptrs[] = {c->S_all,     c->score[0],    c->score[1],   c->tok_next,
                  c->slot_next, c->iota,       c->counters,    c->part,
                  c->row_cnt,   c->gpl,        c->gls,         c->gth,
                  c->pm,        c->ps,         c->ptop,        c->rows_lse,   c->rows_tok,
                  c->rows_logp, c->pool_parent, c->pool_token, c->pool_depth, c->pool_score,
                  c->d_err,     c->z_stage,    c->s0_stage,    c->o_all,      c->cand,
                  c->base_part, c->base_cnt,   c->bf_par,      c->bf_tok,     c->bf_dep,
                  c->bf_rank,   c->bf_score,   c->bf_st,       c->bf_tok_next, c->bf_zrow,
                  c->bf_S,      c->bf_lse,     c->bf_rtok,     c->bf_rlogp,   c->bf_z};
  for (void* p : ptrs)
    if (p) cudaFree(p);
}

}  // namespace

void dt::set_context_free_error(const std::string& why) { g_create_error = why; }

extern "C" {

int32_t dartree_pool_size(int32_t D, int32_t W, int32_t K) {
  if (D < 1 || W < 1 || K < 1) return -1;
  long long f = 1, p = 0;
  for (int d = 0; d < D; ++d) {
    f = f * K < W ? f * K : W;
    p += f;
  }
  return p > 0x7FFFFFFF ? -1 : static_cast<int32_t>(p);
}

dartree_status dartree_create(const dartree_config* cfg, dartree_ctx** out) {
  if (!cfg || !out) return create_fail(DARTREE_ERR_INVALID_ARG, "null argument");
  *out = nullptr;
  g_create_error.clear();
  const dartree_config g = *cfg;
  if (g.wdtype != DARTREE_W_F32 && g.wdtype != DARTREE_W_BF16)
    return create_fail(DARTREE_ERR_INVALID_ARG, "unknown weight dtype");
  if (g.V < 1 || g.H < 1 || g.max_D < 1 || g.max_W < 1 || g.max_K < 1 || g.max_B < 1 ||
      g.max_requests < 1)
    return create_fail(DARTREE_ERR_INVALID_ARG, "sizes must be >= 1");
  if (g.max_K > DARTREE_MAX_K || g.max_D > DARTREE_MAX_D || g.max_B > DARTREE_MAX_B ||
      g.max_W > DARTREE_MAX_ROWS || static_cast<long long>(g.max_requests) * g.max_W > DARTREE_MAX_ROWS)
    return create_fail(DARTREE_ERR_UNSUPPORTED, "capacity beyond the build limits");
  if (g.wdtype == DARTREE_W_BF16 ? (g.H % 64 != 0) : (g.H % 8 != 0))
    return create_fail(DARTREE_ERR_UNSUPPORTED, "H must be a multiple of 64 (bf16) or 8 (fp32)");

  dartree_ctx* c = new (std::nothrow) dartree_ctx();
  if (!c) return DARTREE_ERR_OOM;
  c->cfg = g;
  c->bf16 = g.wdtype == DARTREE_W_BF16;
  c->elem = c->bf16 ? 2 : 4;
  cudaError_t e = cudaGetDevice(&c->device);
  cudaDeviceProp prop{};
  if (e == cudaSuccess) e = cudaGetDeviceProperties(&prop, c->device);
  if (e != cudaSuccess) {
    delete c;
    return create_fail(DARTREE_ERR_CUDA, "device query", e);
  }
  if (prop.major != 10 || prop.minor != 3) {
    delete c;
    return create_fail(DARTREE_ERR_UNSUPPORTED, "needs a compute capability 10.3 device");
  }
  c->num_sms = prop.multiProcessorCount;
  c->max_cta = 2 * c->num_sms;
  // tuning knobs of the head-call pipeline (defaults when unset)
  if (const char* v = getenv("DARTREE_TC_MAX_STAGES")) c->tc_max_stages = atoi(v);
  if (const char* v = getenv("DARTREE_PDL")) c->pdl = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_WAIT_LIMIT_CYCLES")) c->wait_limit = atoll(v);
  if (const char* v = getenv("DARTREE_GRAPH")) c->use_graph = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_RADIX")) c->radix = atoi(v) != 0 ? 1 : 0;
  if (const char* v = getenv("DARTREE_F32_SPLIT")) c->f32_split = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_F32_FOLD")) c->f32_fold = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_RANK_MAX")) c->rank_max = atoi(v);
  if (const char* v = getenv("DARTREE_MERGE_CLUSTER")) c->merge_cluster = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_ROWS_MIN")) c->rows_min = atoi(v);
  if (const char* v = getenv("DARTREE_ROWS_NV")) c->rows_nv = atoi(v) == 128 ? 128 : 256;
  if (const char* v = getenv("DARTREE_ROWS_PAIR")) c->rows_pair = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_ROWS_HALF_S")) c->rows_half_s = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_MERGE_BOUND")) c->merge_bound = atoi(v) != 0;
  if (const char* v = getenv("DARTREE_MERGE_SURV_CAP")) c->merge_surv_cap = atoi(v);
  if (const char* v = getenv("DARTREE_TC_CTAS_PER_SM")) {
    const int n = atoi(v);
    c->tc_ctas_per_sm = n == 2 ? 2 : 1;
  }
  c->pool_cap = dartree_pool_size(g.max_D, g.max_W, g.max_K);

  cudaDriverEntryPointQueryResult q;
  void* fn = nullptr;
  e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    delete c;
    return create_fail(DARTREE_ERR_CUDA, "cuTensorMapEncodeTiled entry point", e);
  }
  c->encode = reinterpret_cast<EncodeTiledFn>(fn);

  const size_t rows = dt::kMaxRows;
  const size_t Rc = static_cast<size_t>(g.max_requests);
  const size_t B = static_cast<size_t>(g.max_B), words = (B + 31) / 32;
  const int h_tiles = (g.H + dt::kTileV - 1) / dt::kTileV;
  const int nk = g.H / dt::kTileH;
  c->state_split = c->num_sms / h_tiles;
  if (c->state_split > nk) c->state_split = nk;
  if (c->state_split < 1) c->state_split = 1;
  c->n_slots = g.max_D > 3 ? g.max_D : 3;
  c->base_chunks = (g.V + dt::kBaseChunk - 1) / dt::kBaseChunk;
  c->bf_nodes = g.max_B * g.max_K;
  const size_t RD = Rc * g.max_D;
  const size_t bfn = Rc * c->bf_nodes;
  const size_t slot_bytes = rows * g.H * c->elem;
  c->o_bytes = tree_layout(Rc, B, nullptr);
  bool ok = alloc(reinterpret_cast<uint8_t**>(&c->S_all), c->n_slots * slot_bytes) == cudaSuccess &&
            alloc(&c->score[0], rows) == cudaSuccess && alloc(&c->score[1], rows) == cudaSuccess &&
            alloc(&c->tok_next, rows) == cudaSuccess && alloc(&c->slot_next, rows) == cudaSuccess &&
            alloc(&c->iota, rows) == cudaSuccess && alloc(&c->counters, rows) == cudaSuccess &&
            alloc(&c->part, static_cast<size_t>(h_tiles) * c->state_split * rows * dt::kTileV) ==
                cudaSuccess &&
            alloc(&c->row_cnt, rows) == cudaSuccess && alloc(&c->gpl, rows * 8 * 32) == cudaSuccess &&
            alloc(&c->gls, rows * 8) == cudaSuccess && alloc(&c->gth, rows * 33) == cudaSuccess &&
            alloc(&c->pm, rows * c->max_cta) == cudaSuccess &&
            alloc(&c->ps, rows * c->max_cta) == cudaSuccess &&
            alloc(&c->ptop, rows * c->max_cta * dt::kEpiWarps * g.max_K) == cudaSuccess &&
            alloc(&c->rows_lse, static_cast<size_t>(g.max_D) * rows) == cudaSuccess &&
            alloc(&c->rows_tok, static_cast<size_t>(g.max_D) * rows * g.max_K) == cudaSuccess &&
            alloc(&c->rows_logp, static_cast<size_t>(g.max_D) * rows * g.max_K) == cudaSuccess &&
            alloc(&c->pool_parent, Rc * c->pool_cap) == cudaSuccess &&
            alloc(&c->pool_token, Rc * c->pool_cap) == cudaSuccess &&
            alloc(&c->pool_depth, Rc * c->pool_cap) == cudaSuccess &&
            alloc(&c->pool_score, Rc * c->pool_cap) == cudaSuccess &&
            alloc(&c->d_err, 1) == cudaSuccess &&
            alloc(&c->z_stage, Rc * g.max_D * static_cast<size_t>(g.V)) == cudaSuccess &&
            alloc(&c->s0_stage, Rc * g.H) == cudaSuccess &&
            alloc(&c->o_all, c->o_bytes) == cudaSuccess &&
            cudaMallocHost(reinterpret_cast<void**>(&c->h_stage), c->o_bytes + 16) == cudaSuccess &&
            alloc(&c->cand, RD * g.max_K) == cudaSuccess &&
            alloc(&c->base_part, RD * c->base_chunks * g.max_K) == cudaSuccess &&
            alloc(&c->base_cnt, RD) == cudaSuccess &&
            alloc(&c->bf_par, bfn) == cudaSuccess && alloc(&c->bf_tok, bfn) == cudaSuccess &&
            alloc(&c->bf_dep, bfn) == cudaSuccess && alloc(&c->bf_rank, bfn) == cudaSuccess &&
            alloc(&c->bf_score, bfn) == cudaSuccess && alloc(&c->bf_st, Rc * 4) == cudaSuccess &&
            alloc(&c->bf_tok_next, Rc) == cudaSuccess && alloc(&c->bf_zrow, Rc) == cudaSuccess &&
            alloc(&c->bf_z, Rc * g.V) == cudaSuccess &&
            alloc(reinterpret_cast<uint8_t**>(&c->bf_S), Rc * B * g.H * c->elem) == cudaSuccess &&
            alloc(&c->bf_lse, B * Rc) == cudaSuccess &&
            alloc(&c->bf_rtok, B * Rc * g.max_K) == cudaSuccess &&
            alloc(&c->bf_rlogp, B * Rc * g.max_K) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return create_fail(DARTREE_ERR_OOM, "workspace allocation");
  }
  e = cudaMemset(c->S_all, 0, c->n_slots * slot_bytes);
  if (e == cudaSuccess) e = cudaMemset(c->d_err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->counters, 0, rows * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->row_cnt, 0, rows * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->gth, 0, rows * 33 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(c->base_cnt, 0, RD * sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->bf_tok_next, 0, Rc * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(c->bf_zrow, 0, Rc * sizeof(int32_t));
  if (e == cudaSuccess) {
    int32_t h_iota[dt::kMaxRows];
    for (int i = 0; i < dt::kMaxRows; ++i) h_iota[i] = i;
    e = cudaMemcpy(c->iota, h_iota, sizeof h_iota, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->copy_st, cudaStreamNonBlocking);
  c->z_ready.assign(static_cast<size_t>(g.max_D) + 1, nullptr);
  for (size_t d = 2; d < c->z_ready.size() && e == cudaSuccess; ++d)
    e = cudaEventCreateWithFlags(&c->z_ready[d], cudaEventDisableTiming);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->z_order, cudaEventDisableTiming);
  if (e == cudaSuccess) e = dt::init_head_attrs();
  if (e == cudaSuccess) e = dt::init_select_attrs();
  if (e == cudaSuccess) c->cluster_limit = dt::merge_cluster_limit();
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_all(c);
    delete c;
    return create_fail(DARTREE_ERR_CUDA, "workspace initialisation", e);
  }
  if (c->bf16) {
    c->tm_S.resize(static_cast<size_t>(c->n_slots) * kNumPads);
    for (int sl = 0; sl < c->n_slots; ++sl)
    for (int i = 0; i < kNumPads; ++i) {
      const uint32_t n = 16u << i;
      if (encode_2d(c, &c->tm_S[sl * kNumPads + i], c->S(sl), rows, g.H, n) != DARTREE_OK) {
        free_all(c);
        delete c;
        return create_fail(DARTREE_ERR_CUDA, "state tensor map");
      }
    }
  }
  *out = c;
  return DARTREE_OK;
}

void dartree_destroy(dartree_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  free_all(ctx);
  delete ctx;
}

dartree_status dartree_build(dartree_ctx* ctx, const float* base_logits, const float* state0,
                             const dartree_head* head, int32_t R, int32_t D, int32_t W, int32_t K,
                             int32_t B, float beta, const dartree_tree* out, void* stream) {
  return dartree_build_ex(ctx, base_logits, state0, head, R, D, W, K, B, beta, nullptr, out,
                          stream);
}

dartree_status dartree_build_ex(dartree_ctx* ctx, const float* base_logits, const float* state0,
                                const dartree_head* head, int32_t R, int32_t D, int32_t W,
                                int32_t K, int32_t B, float beta, const dartree_options* opt,
                                const dartree_tree* out, void* stream) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  const dartree_options o = opt ? *opt : dartree_options{};
  dartree_status s =
      check_build_args(ctx, base_logits, state0, head, R, D, W, K, B, beta, out, o);
  if (s != DARTREE_OK) return s;
  return build_dispatch(ctx, base_logits, state0, head, R, D, W, K, B, beta, o, out,
                        static_cast<cudaStream_t>(stream));
}

namespace {
dartree_status status_from_word(dartree_ctx* ctx, int h);
}  // namespace

dartree_status dartree_sync_status(dartree_ctx* ctx, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!ctx) {  // the context-free state step's check word on this device
    cudaError_t e = cudaSuccess;
    const int h = dt::noalloc_take_status(st, &e);
    if (e != cudaSuccess) {
      dt::set_context_free_error(std::string("status read: ") + cudaGetErrorString(e));
      return DARTREE_ERR_CUDA;
    }
    char msg[96];
    if (h > 0 && (h & dt::DT_ERR_TIMEOUT)) {
      snprintf(msg, sizeof msg, "device wait timed out (flags 0x%x)", h);
      dt::set_context_free_error(msg);
      return DARTREE_ERR_TIMEOUT;
    }
    if (h > 0) {
      snprintf(msg, sizeof msg, "device check failed (flags 0x%x)", h);
      dt::set_context_free_error(msg);
      return DARTREE_ERR_DEVICE_CHECK;
    }
    return DARTREE_OK;
  }
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "stream synchronize");
  flush_timing(ctx);
  int h = 0;
  e = cudaMemcpy(&h, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "error word read");
  return status_from_word(ctx, h);
}

namespace {

// The status a device check word stands for (after the stream's work is
// complete).  A failed launch may have left arrival counters part-way: a
// nonzero word also clears them and the word, so the next build starts from
// a clean workspace.
dartree_status status_from_word(dartree_ctx* ctx, int h) {
  cudaError_t e = cudaSuccess;
  if (h != 0) {
    e = cudaMemset(ctx->d_err, 0, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(ctx->counters, 0, dt::kMaxRows * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(ctx->row_cnt, 0, dt::kMaxRows * sizeof(int));
    if (e == cudaSuccess)
      e = cudaMemset(ctx->gth, 0, dt::kMaxRows * 33 * sizeof(unsigned long long));
    if (e == cudaSuccess)
      e = cudaMemset(ctx->base_cnt, 0,
                     sizeof(int) * static_cast<size_t>(ctx->cfg.max_requests) * ctx->cfg.max_D);
  }
  if (e != cudaSuccess) return ctx->cuda_fail(e, "error word read");
  if (h & dt::DT_ERR_TIMEOUT)
    return ctx->fail(DARTREE_ERR_TIMEOUT, "device wait timed out (flags 0x%x)", h);
  if (h != 0) return ctx->fail(DARTREE_ERR_DEVICE_CHECK, "device check failed (flags 0x%x)", h);
  return DARTREE_OK;
}

}  // namespace

dartree_status dartree_build_host(dartree_ctx* ctx, const float* zh, const float* s0h,
                                  const dartree_head* head, int32_t R, int32_t D, int32_t W,
                                  int32_t K, int32_t B, float beta, const dartree_tree* out_host,
                                  void* stream) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  dartree_status s = check_build_args(ctx, zh, s0h, head, R, D, W, K, B, beta, out_host);
  if (s != DARTREE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t V = ctx->cfg.V, sn = static_cast<size_t>(R) * ctx->cfg.H;
  const size_t pitch = static_cast<size_t>(D) * V * 4;  // one request's [D, V] rows
  // depth 1's base logits of every request (and the root states) on the
  // build stream; the later depths' on the copy stream, which the head call
  // of depth 2 waits for -- the copy runs under the first head call
  cudaError_t e = cudaMemcpy2DAsync(ctx->z_stage, pitch, zh, pitch, V * 4, R,
                                    cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->s0_stage, s0h, sn * 4, cudaMemcpyHostToDevice, st);
  // small per-depth slices: one copy, which the head call of depth 2
  // waits for; large ones (many requests): one copy and one event per
  // depth, so that each head call waits only for its own
  cudaEvent_t ev[DARTREE_MAX_D + 1] = {};
  const bool each = static_cast<size_t>(R) * V * 4 >= (size_t(4) << 20);
  const int z_late = D > 1 ? (each ? 2 : 1) : 0;
  if (z_late) {
    if (e == cudaSuccess) e = cudaEventRecord(ctx->z_order, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ctx->copy_st, ctx->z_order, 0);
    for (int d = 2; d <= D && e == cudaSuccess; ++d) {
      const int n = each ? 1 : D - 1;  // depths in this copy
      e = cudaMemcpy2DAsync(ctx->z_stage + (d - 1) * V, pitch, zh + (d - 1) * V, pitch,
                            n * V * 4, R, cudaMemcpyHostToDevice, ctx->copy_st);
      if (e == cudaSuccess) e = cudaEventRecord(ctx->z_ready[d], ctx->copy_st);
      ev[d] = ctx->z_ready[d];
      if (!each) break;
    }
  }
  if (e != cudaSuccess) return ctx->cuda_fail(e, "input copy");
  size_t off[6];
  const size_t bytes = tree_layout(R, B, off);
  uint8_t* o = ctx->o_all;
  dartree_tree dev{reinterpret_cast<int32_t*>(o + off[0]), reinterpret_cast<int32_t*>(o + off[1]),
                   reinterpret_cast<int32_t*>(o + off[2]), reinterpret_cast<float*>(o + off[3]),
                   reinterpret_cast<uint32_t*>(o + off[4]), reinterpret_cast<int32_t*>(o + off[5])};
  s = build_dispatch(ctx, ctx->z_stage, ctx->s0_stage, head, R, D, W, K, B, beta,
                     dartree_options{}, &dev, st, z_late ? ev : nullptr, z_late);
  if (s != DARTREE_OK) return s;
  // the tree in one copy, the check word in another, one synchronisation
  int* h_err = reinterpret_cast<int*>(ctx->h_stage + ctx->o_bytes);
  e = cudaMemcpyAsync(ctx->h_stage, o, bytes, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(h_err, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "output copy");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "stream synchronize");
  flush_timing(ctx);
  const size_t nb = static_cast<size_t>(R) * B, nw = nb * ((B + 31) / 32);
  void* dst[6] = {out_host->parent, out_host->token, out_host->depth,
                  out_host->score,  out_host->mask,  out_host->n_out};
  const size_t n[6] = {nb * 4, nb * 4, nb * 4, nb * 4, nw * 4, static_cast<size_t>(R) * 4};
  for (int i = 0; i < 6; ++i) std::memcpy(dst[i], ctx->h_stage + off[i], n[i]);
  return status_from_word(ctx, *h_err);
}

dartree_status dartree_set_timing(dartree_ctx* ctx, int32_t enable) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  if (!enable) {
    cudaDeviceSynchronize();
    free_events(ctx);
    ctx->timing = false;
    return DARTREE_OK;
  }
  if (ctx->ev_pool.empty()) {
    const size_t n = 2 * (4 * static_cast<size_t>(std::max(ctx->cfg.max_D, ctx->cfg.max_B)) + 8);
    for (size_t i = 0; i < n; ++i) {
      cudaEvent_t ev;
      cudaError_t e = cudaEventCreate(&ev);
      if (e != cudaSuccess) {
        free_events(ctx);
        return ctx->cuda_fail(e, "event create");
      }
      ctx->ev_pool.push_back(ev);
    }
  }
  ctx->timing = true;
  return DARTREE_OK;
}

dartree_status dartree_get_timing(const dartree_ctx* ctx, int32_t kind, double* total_ms,
                                  int64_t* launches) {
  if (!ctx || !total_ms || !launches || kind < 0 || kind >= DARTREE_KERNEL_KINDS)
    return DARTREE_ERR_INVALID_ARG;
  *total_ms = ctx->t_ms[kind];
  *launches = ctx->t_n[kind];
  return DARTREE_OK;
}

dartree_status dartree_reset_timing(dartree_ctx* ctx) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  for (int k = 0; k < DARTREE_KERNEL_KINDS; ++k) {
    ctx->t_ms[k] = 0.0;
    ctx->t_n[k] = 0;
  }
  return DARTREE_OK;
}

int64_t dartree_head_calls(const dartree_ctx* ctx) { return ctx ? ctx->head_calls : -1; }

namespace {
// Context-free failure: the text goes to dartree_last_error(NULL).
dartree_status free_fail(dartree_status s, const char* why) {
  dt::set_context_free_error(why);
  return s;
}
}  // namespace

dartree_status dartree_set_weight_layout(dartree_ctx* ctx, int32_t layout) {
  if (!ctx) return free_fail(DARTREE_ERR_INVALID_ARG, "null context");
  if (layout != DARTREE_LAYOUT_ROWS && layout != DARTREE_LAYOUT_BLOCKS)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "unknown weight layout %d", layout);
  if (layout == DARTREE_LAYOUT_BLOCKS && !ctx->bf16)
    return ctx->fail(DARTREE_ERR_UNSUPPORTED, "the blocked layout needs bf16 weights");
  const bool tiled = layout == DARTREE_LAYOUT_BLOCKS;
  if (tiled != ctx->w_tiled) {
    ctx->w_tiled = tiled;
    ctx->tm_Wout_ptr = nullptr;  // the next call re-encodes Wout's tensor map
  }
  return DARTREE_OK;
}

size_t dartree_blocked_weight_bytes(int32_t V, int32_t H) {
  if (V < 1 || H < 1 || H % 64 != 0) return 0;
  return (static_cast<size_t>(V) + 127) / 128 * 128 * static_cast<size_t>(H) * 2;
}

dartree_status dartree_block_weights(const void* W, int32_t V, int32_t H, void* W_blocked,
                                     void* stream) {
  const size_t bytes = dartree_blocked_weight_bytes(V, H);
  if (!W || !W_blocked || bytes == 0)
    return free_fail(DARTREE_ERR_INVALID_ARG, "bad W, W_blocked, V or H");
  if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(W_blocked)) & 15)
    return free_fail(DARTREE_ERR_INVALID_ARG, "W and W_blocked must be 16-byte aligned");
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(W), b0 = reinterpret_cast<uintptr_t>(W_blocked);
  const size_t src_bytes = static_cast<size_t>(V) * H * 2;
  if (a0 < b0 + bytes && b0 < a0 + src_bytes)
    return free_fail(DARTREE_ERR_INVALID_ARG, "W and W_blocked overlap");
  const cudaError_t e =
      dt::launch_block_weights(static_cast<const uint16_t*>(W), V, H,
                               static_cast<uint16_t*>(W_blocked), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return free_fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  return DARTREE_OK;
}

const char* dartree_last_error(const dartree_ctx* ctx) {
  return ctx ? ctx->last_error.c_str() : g_create_error.c_str();
}

dartree_status dartree_get_pool(dartree_ctx* ctx, int32_t* parent, int32_t* token, int32_t* depth,
                                float* score, void* stream) {
  if (!ctx || !parent || !token || !depth || !score) return DARTREE_ERR_INVALID_ARG;
  if (ctx->last_P == 0) return ctx->fail(DARTREE_ERR_INVALID_ARG, "no depth-wise build yet");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t n = static_cast<size_t>(ctx->last_R) * ctx->last_P * 4;
  cudaError_t e = cudaMemcpyAsync(parent, ctx->pool_parent, n, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(token, ctx->pool_token, n, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(depth, ctx->pool_depth, n, cudaMemcpyDefault, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(score, ctx->pool_score, n, cudaMemcpyDefault, st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "pool copy");
  return DARTREE_OK;
}

dartree_status dartree_get_rows(dartree_ctx* ctx, int32_t d, double* lse, int32_t* tok, float* logp,
                                void* stream) {
  if (!ctx || !lse || !tok || !logp) return DARTREE_ERR_INVALID_ARG;
  if (ctx->last_expansion == DARTREE_EXPAND_BESTFIRST) {  // rows of call d-1
    if (d < 1 || d > ctx->last_B)
      return ctx->fail(DARTREE_ERR_INVALID_ARG, "call %d not in the last build", d - 1);
    const size_t rows = ctx->last_R, K = ctx->last_K;
    const size_t ro = static_cast<size_t>(d - 1) * ctx->cfg.max_requests;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(lse, ctx->bf_lse + ro, rows * 8, cudaMemcpyDefault, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(tok, ctx->bf_rtok + ro * K, rows * K * 4, cudaMemcpyDefault, st);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(logp, ctx->bf_rlogp + ro * K, rows * K * 4, cudaMemcpyDefault, st);
    if (e != cudaSuccess) return ctx->cuda_fail(e, "rows copy");
    return DARTREE_OK;
  }
  if (ctx->last_P == 0 || d < 1 || d > ctx->last_D)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "depth %d not in the last build", d);
  int F = 1;
  for (int i = 1; i < d; ++i) F = frontier_after(F, ctx->last_W, ctx->last_K);
  const size_t rows = static_cast<size_t>(ctx->last_R) * F, K = ctx->last_K;
  const size_t ro = static_cast<size_t>(d - 1) * dt::kMaxRows;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(lse, ctx->rows_lse + ro, rows * 8, cudaMemcpyDefault, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(tok, ctx->rows_tok + ro * K, rows * K * 4, cudaMemcpyDefault, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(logp, ctx->rows_logp + ro * K, rows * K * 4, cudaMemcpyDefault, st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "rows copy");
  return DARTREE_OK;
}

dartree_status dartree_get_states(dartree_ctx* ctx, int32_t d, void* states, void* stream) {
  if (!ctx || !states) return DARTREE_ERR_INVALID_ARG;
  if (ctx->last_expansion == DARTREE_EXPAND_BESTFIRST) {  // states of call d-1
    if (d < 1 || d > ctx->last_B)
      return ctx->fail(DARTREE_ERR_INVALID_ARG, "call %d not in the last build", d - 1);
    const size_t rowb = static_cast<size_t>(ctx->cfg.H) * ctx->elem;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (d == 1)
      e = cudaMemcpyAsync(states, ctx->S(0), ctx->last_R * rowb, cudaMemcpyDefault, st);
    else
      e = cudaMemcpy2DAsync(states, rowb,
                            static_cast<const uint8_t*>(ctx->bf_S) + static_cast<size_t>(d - 2) * rowb,
                            static_cast<size_t>(ctx->last_B) * rowb, rowb, ctx->last_R,
                            cudaMemcpyDefault, st);
    if (e != cudaSuccess) return ctx->cuda_fail(e, "states copy");
    return DARTREE_OK;
  }
  if (ctx->last_P == 0 || d < 1 || d > ctx->last_D)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "depth %d not in the last build", d);
  int F = 1;
  for (int i = 1; i < d; ++i) F = frontier_after(F, ctx->last_W, ctx->last_K);
  const size_t bytes = static_cast<size_t>(ctx->last_R) * F * ctx->cfg.H * ctx->elem;
  cudaError_t e = cudaMemcpyAsync(states, ctx->S(d - 1), bytes, cudaMemcpyDefault,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ctx->cuda_fail(e, "states copy");
  return DARTREE_OK;
}

dartree_status dartree_head_topk(dartree_ctx* ctx, const void* S, const float* z,
                                 int64_t z_req_stride, int32_t rows_per_req, const void* Wout,
                                 int32_t M, int32_t K, double* lse, int32_t* tok, float* logp,
                                 void* stream) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  if (!S || !z || !Wout || !lse || !tok || !logp)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (M < 1 || M > dt::kMaxRows || rows_per_req < 1 || K < 1 || K > ctx->cfg.max_K ||
      K > ctx->cfg.V)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "bad M=%d, rows_per_req=%d or K=%d", M,
                     rows_per_req, K);
  if (ctx->bf16 && M < ctx->rows_min && pad_rows(M) * K > 2048)
    return ctx->fail(DARTREE_ERR_UNSUPPORTED, "padded rows x K > 2048");
  dartree_status s = bind_weights(ctx, ctx->tm_A_ptr, Wout);
  if (s != DARTREE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rb = static_cast<size_t>(ctx->cfg.H) * ctx->elem;
  cudaError_t e = cudaMemcpyAsync(ctx->S(0), S, M * rb, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && pad_rows(M) > M)
    e = cudaMemsetAsync(static_cast<uint8_t*>(ctx->S(0)) + M * rb, 0, (pad_rows(M) - M) * rb, st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "state copy");
  return run_head(ctx, 0, z, z_req_stride, rows_per_req, M, K, lse, tok, logp, nullptr, st);
}

dartree_status dartree_state_step(dartree_ctx* ctx, const void* S_par, const int32_t* tok,
                                  const void* A, const void* E, int32_t M, void* S_out,
                                  void* stream) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  if (!S_par || !tok || !A || !E || !S_out)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (M < 1 || M > dt::kMaxRows) return ctx->fail(DARTREE_ERR_INVALID_ARG, "bad M=%d", M);
  if (ctx->bf16 && (reinterpret_cast<uintptr_t>(E) & 15))
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "bf16 weights must be 16-byte aligned");
  dartree_status s = bind_weights(ctx, A, ctx->tm_Wout_ptr);
  if (s != DARTREE_OK) return s;
  if (!ctx->bf16) ctx->tm_A_ptr = A;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rb = static_cast<size_t>(ctx->cfg.H) * ctx->elem;
  cudaError_t e = cudaMemcpyAsync(ctx->S(0), S_par, M * rb, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && pad_rows(M) > M)
    e = cudaMemsetAsync(static_cast<uint8_t*>(ctx->S(0)) + M * rb, 0, (pad_rows(M) - M) * rb, st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "state copy");
  if ((s = run_state(ctx, A, E, 0, M, ctx->iota, tok, M, st)) != DARTREE_OK) return s;
  e = cudaMemcpyAsync(S_out, ctx->S(1), M * rb, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return ctx->cuda_fail(e, "state copy back");
  return DARTREE_OK;
}

dartree_status dartree_prune(dartree_ctx* ctx, const int32_t* pool_parent, const int32_t* pool_token,
                             const int32_t* pool_depth, const float* pool_score, int32_t R,
                             int32_t P, int32_t B, float beta, const dartree_tree* out,
                             void* stream) {
  if (!ctx) return DARTREE_ERR_INVALID_ARG;
  if (!pool_parent || !pool_token || !pool_depth || !pool_score || !out || !out->parent ||
      !out->token || !out->depth || !out->score || !out->mask || !out->n_out)
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (R < 1 || R > ctx->cfg.max_requests || P < 1 || P > ctx->pool_cap || B < 1 ||
      B > ctx->cfg.max_B || !(beta <= 0.0f))
    return ctx->fail(DARTREE_ERR_INVALID_ARG, "bad R=%d, P=%d, B=%d or beta", R, P, B);
  dt::PruneParams pp{};
  pp.R = R;
  pp.P = P;
  pp.pool_stride = P;
  pp.B = B;
  pp.words = (B + 31) / 32;
  pp.beta = beta;
  pp.pool_parent = pool_parent;
  pp.pool_token = pool_token;
  pp.pool_depth = pool_depth;
  pp.pool_score = pool_score;
  pp.parent = out->parent;
  pp.token = out->token;
  pp.depth = out->depth;
  pp.score = out->score;
  pp.mask = out->mask;
  pp.n_out = out->n_out;
  pp.err = ctx->d_err;
  pp.radix = ctx->radix == 1 || (ctx->radix < 0 && P >= 512);
  cudaError_t e = dt::launch_prune(pp, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ctx->cuda_fail(e, "prune launch");
  return DARTREE_OK;
}

}  // extern "C"
