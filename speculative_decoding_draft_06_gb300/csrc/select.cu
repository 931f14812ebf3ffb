// Selection kernels of a DARTree build: merge of the head-call partials into
// per-row log-probabilities and top-K (k_merge_rows folds every CTA list;
// k_merge_bound reads only the lists that reach the head call's row bound),
// the per-depth global top-W with pool append and state carry, the deferred
// global Top-B with compaction and the ancestor (tree-attention) mask, and
// the root rows.
//
// Every selection orders 64-bit keys (value desc, index asc; see common.cuh)
// with bitonic sorts and merges, in warps or in shared memory, or with a
// block radix select of the best keys followed by a sort of those (the Top-B
// of large pools; block.cuh), and the keys are distinct, so results are a
// deterministic total order and independent of thread timing (including the
// order in which k_merge_bound stages keys).
#include <cuda_runtime.h>

#include "block.cuh"
#include "common.cuh"
#include "kernels.h"

namespace dt {

// log(x) of a positive fp32 sum: the exponent's share e ln 2 in double, the
// mantissa's log(f), f in [0.5, 1), in fp32 (absolute error ~1e-7: the
// fp32 sum it is taken of carries more).  The double-precision log it
// replaces ran on the GPU's few fp64 units in the merge's critical path.
__device__ __forceinline__ double log_f32_exp(float x) {
  int e;
  const float f = frexpf(x, &e);
  return static_cast<double>(e) * 0.69314718055994530942 + static_cast<double>(logf(f));
}

// ------------------------------------------------ merge of rows + top-W

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;

// thread-block cluster access (the row blocks of a request, k_merge_bound)
__device__ __forceinline__ uint32_t cl_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The cluster address of `p` (this CTA's shared memory) in the CTA of rank 0.
__device__ __forceinline__ uint32_t cl_leader_addr(const void* p) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;"
               : "=r"(a)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
  return a;
}
__device__ __forceinline__ void cl_store_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cl_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split form for the start: every CTA of the cluster has begun (and its
// shared memory exists) once the wait returns.
__device__ __forceinline__ void cl_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// Global top-W of one request's candidates (run by the last merge block of
// the request).  Candidate (i, j) = child j of frontier slot i, score
// c = score_i + logp_ij (one fp32 add), index i*K + j; the best |F_d| by
// (c desc, index asc) become the new frontier in rank order ("DARTree:
// Teaching a Chain-Trained Corrector to Think in Trees", Core Mechanism:
// children ranked by cumulative path log-probability, the W best survive;
// "Accelerating Language Models with Diffusion Draft Trees", Summary: one
// global top-W per depth, whose states go on to the next depth).
// (parent row, token) of each next-depth row of the request, kept for the
// folded fp32 state step (written by write_frontier, read by state_from_u)
__shared__ int2 sh_next[kMaxRows];
// the request's candidate tokens [F][K], staged by the warp selection while
// it loads their log-probs (F K <= kTokStage)
constexpr int kTokStage = 1024;
__shared__ int32_t sh_tok[kTokStage];

// tok_sh: the request's candidate tokens in shared memory, or null (read
// them from the merged rows)
__device__ void write_frontier(const MergeParams& p, int r, int q, uint64_t k,
                               const int32_t* tok_sh = nullptr) {
  const int idx = static_cast<int>(key_index(k));
  const int i = idx / p.K, j = idx % p.K;
  const int row = r * p.F + i;
  const float c = key_value(k);
  const int32_t tok =
      tok_sh ? tok_sh[idx] : __ldcg(p.row_tok + static_cast<size_t>(row) * p.K + j);
  const size_t pi = static_cast<size_t>(r) * p.pool_stride + p.off + q;
  p.pool_parent[pi] = (p.depth == 1) ? -1 : p.off_prev + i;
  p.pool_token[pi] = tok;
  p.pool_depth[pi] = p.depth;
  p.pool_score[pi] = c;
  const int m = r * p.Fd + q;
  p.score_out[m] = c;
  p.tok_next[m] = tok;
  p.slot_next[m] = row;
  if (p.U_f32) sh_next[q] = make_int2(row, tok);
}

// The fp32 state step after request r's selection, when the head call
// computed U = A S for its rows: next row q of the request (parent row slot,
// token tok, as write_frontier kept them in shared memory) is
// tanh(U[slot] + E[tok]) ("DARTree: Teaching a Chain-Trained Corrector to
// Think in Trees", Core Mechanism: the synthetic correction head's
// recurrence).  The __syncthreads before the call makes the selection's
// entries visible.  All threads of the block call it.
__device__ void state_from_u(const MergeParams& p, int r) {
  constexpr int kB = 4;  // elements per thread whose loads go out together
  const int n = p.Fd * p.H;
  bool bad = false;
  for (int e0 = 0; e0 < n; e0 += kB * blockDim.x) {
    float u[kB], ev[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const int e = e0 + k * blockDim.x + threadIdx.x;
      u[k] = 0.f;
      ev[k] = 0.f;
      if (e < n) {
        const int q = e / p.H, h = e - q * p.H;
        int2 pt = sh_next[q];
        if (pt.x < 0 || pt.x >= p.R * p.F) pt.x = 0;  // (never, unless upstream failed)
        if (pt.y < 0 || pt.y >= p.V_tok) {            // only after an upstream failure
          bad = true;
          pt.y = 0;
        }
        u[k] = __ldcg(p.U_f32 + static_cast<size_t>(pt.x) * p.H + h);
        ev[k] = __ldg(p.E_f32 + static_cast<size_t>(pt.y) * p.H + h);
      }
    }
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const int e = e0 + k * blockDim.x + threadIdx.x;
      if (e < n) p.S_next_f32[static_cast<size_t>(r) * p.Fd * p.H + e] = tanhf(u[k] + ev[k]);
    }
  }
  if (bad) atomicOr(p.err, DT_ERR_BAD_INDEX);
}

// For |F_d| <= 32: every row's candidates are already sorted (log-probs
// descending, one fp32 add keeps the order, ties by index), so the top |F_d|
// is a fold of the F sorted lists with warp bitonic merges -- rows spread
// over the warps, then a tree across warps.  The rows' log-probs, scores and
// tokens (staged in shared memory for write_frontier) are loaded together
// before the merges.  All threads of the block call it.
__device__ void select_frontier_warp(const MergeParams& p, int r, uint64_t (*wl)[32]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int p2 = pow2_ceil32(p.Fd > p.K ? p.Fd : p.K);
  const bool stage = p.F * p.K <= kTokStage;
  constexpr int kRowsPre = 4;  // rows of this warp loaded up front (F <= 32: all of them)
  uint64_t v = 0ull;
  for (int i0 = warp; i0 < p.F; i0 += nw * kRowsPre) {
    float lp[kRowsPre], sc[kRowsPre];
#pragma unroll
    for (int u = 0; u < kRowsPre; ++u) {
      const int i = i0 + u * nw;
      const int row = r * p.F + i;
      lp[u] = 0.f;
      sc[u] = 0.f;
      if (i < p.F && lane < p.K) {
        lp[u] = __ldcg(p.row_logp + static_cast<size_t>(row) * p.K + lane);
        sc[u] = __ldcg(p.score_in + row);
        if (stage)
          sh_tok[i * p.K + lane] = __ldcg(p.row_tok + static_cast<size_t>(row) * p.K + lane);
      }
    }
#pragma unroll
    for (int u = 0; u < kRowsPre; ++u) {
      const int i = i0 + u * nw;
      if (i >= p.F) break;  // the same for the whole warp
      uint64_t cur = 0ull;
      if (lane < p.K)
        cur = make_key(__fadd_rn(sc[u], lp[u]), static_cast<uint32_t>(i * p.K + lane));
      uint64_t y = 0ull;
      if (p2 == 32) {
        y = shfl_u64(cur, 31 - lane);
      } else {
        const int src = 2 * p2 - 1 - lane;
        const uint64_t b = shfl_u64(cur, src < 0 ? 0 : src);
        v = lane < p2 ? v : (lane < 2 * p2 ? b : 0ull);
      }
      v = warp_merge_desc(v, y, p2);
    }
  }
  v = block_tree_merge(v, wl, p2);  // (its barriers also publish sh_tok)
  if (warp == 0 && lane < p.Fd) write_frontier(p, r, lane, v, stage ? sh_tok : nullptr);
}

// Best 64 of two descending 64-key lists, each held by a warp as (element
// lane, element lane + 32): the larger of A[e] and B[63 - e] for every e
// (a bitonic sequence holding the best 64), then a bitonic merge -- stride
// 32 inside the lane, strides 16 .. 1 across lanes.  Result in (a0, a1).
__device__ __forceinline__ void warp_merge64(uint64_t& a0, uint64_t& a1, uint64_t b0,
                                             uint64_t b1) {
  const int lane = threadIdx.x & 31;
  const uint64_t r0 = shfl_u64(b1, 31 - lane);  // B[63 - lane]
  const uint64_t r1 = shfl_u64(b0, 31 - lane);  // B[31 - lane]
  uint64_t c0 = a0 > r0 ? a0 : r0, c1 = a1 > r1 ? a1 : r1;
  a0 = c0 > c1 ? c0 : c1;
  a1 = c0 > c1 ? c1 : c0;
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    const uint64_t o0 = shfl_xor_u64(a0, s), o1 = shfl_xor_u64(a1, s);
    const bool lo = (lane & s) != 0;
    a0 = lo ? (a0 < o0 ? a0 : o0) : (a0 > o0 ? a0 : o0);
    a1 = lo ? (a1 < o1 ? a1 : o1) : (a1 > o1 ? a1 : o1);
  }
}

// For 32 < |F_d| <= 64: as select_frontier_warp with 64-key lists (two per
// lane).  A warp's rows (at most 8: |F_{d-1}| <= 64 over 8 warps) have their
// loads issued together; the warps' lists then fold by a pairwise tree
// through shared memory.  All threads of the block call it.
__device__ void select_frontier_warp64(const MergeParams& p, int r, uint64_t* sl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kRowsPerWarp = 64 / kMergeWarps;
  uint64_t cur[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) {
    const int i = warp + k * kMergeWarps;
    cur[k] = 0ull;
    if (i < p.F && lane < p.K) {
      const int row = r * p.F + i;
      const float lp = __ldcg(p.row_logp + static_cast<size_t>(row) * p.K + lane);
      const float c = __fadd_rn(__ldcg(p.score_in + row), lp);
      cur[k] = make_key(c, static_cast<uint32_t>(i * p.K + lane));
    }
  }
  uint64_t v0 = 0ull, v1 = 0ull;
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k) warp_merge64(v0, v1, cur[k], 0ull);
  // pairwise tree over the warps: sl[w][64]
  sl[warp * 64 + lane] = v0;
  sl[warp * 64 + 32 + lane] = v1;
  __syncthreads();
  for (int stride = 1; stride < kMergeWarps; stride <<= 1) {
    if ((warp & (2 * stride - 1)) == 0) {
      warp_merge64(v0, v1, sl[(warp + stride) * 64 + lane], sl[(warp + stride) * 64 + 32 + lane]);
      sl[warp * 64 + lane] = v0;
      sl[warp * 64 + 32 + lane] = v1;
    }
    __syncthreads();
  }
  if (warp == 0) {
    if (lane < p.Fd) write_frontier(p, r, lane, v0);
    if (lane + 32 < p.Fd) write_frontier(p, r, lane + 32, v1);
  }
}

// Radix form of the same selection: the request's F*K candidate keys in
// shared memory, a block radix select of the best |F_d| (block.cuh), then a
// bitonic sort of those |F_d| into rank order.
__device__ void select_frontier_radix(const MergeParams& p, int r, uint64_t* keys) {
  __shared__ unsigned hist[256];
  __shared__ int sh[4];
  const int n = p.F * p.K;
  const int kp2 = pow2_at_least(p.Fd);
  uint64_t* sel = keys + ((n + 1) & ~1);
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int row = r * p.F + e / p.K;
    const float lp = __ldcg(p.row_logp + static_cast<size_t>(row) * p.K + (e % p.K));
    const float c = __fadd_rn(__ldcg(p.score_in + row), lp);
    keys[e] = make_key(c, static_cast<uint32_t>(e));
  }
  for (int q = p.Fd + threadIdx.x; q < kp2; q += blockDim.x) sel[q] = 0ull;
  __syncthreads();
  block_radix_select(keys, n, p.Fd, sel, hist, sh);
  block_sort_desc(sel, kp2);
  for (int q = threadIdx.x; q < p.Fd; q += blockDim.x) write_frontier(p, r, q, sel[q]);
}

// Top-|F_d| of the request's F K candidates by rank counting (F K at most
// rank_max and kTokStage): each candidate's key (score + log-prob,
// candidate index) is staged in shared memory with its token, and goes to
// slot q = the number of keys above it when q < |F_d|.  keys: F K + |F_d|
// slots.  All threads of the block call it.
__device__ void select_frontier_rank(const MergeParams& p, int r, uint64_t* keys) {
  const int n = p.F * p.K;
  uint64_t* out = keys + n;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int i = e / p.K, j = e - i * p.K;
    const int row = r * p.F + i;
    const float lp = __ldcg(p.row_logp + static_cast<size_t>(row) * p.K + j);
    const float sc = __ldcg(p.score_in + row);
    sh_tok[e] = __ldcg(p.row_tok + static_cast<size_t>(row) * p.K + j);
    keys[e] = make_key(__fadd_rn(sc, lp), static_cast<uint32_t>(e));
  }
  __syncthreads();
  block_rank_select(keys, n, p.Fd, out);
  __syncthreads();
  for (int q = threadIdx.x; q < p.Fd; q += blockDim.x) write_frontier(p, r, q, out[q], sh_tok);
}

// The same selection from the rows' log-probs and tokens and the frontier
// scores in this CTA's shared memory (the cluster leader's): no loads.
__device__ void select_frontier_smem(const MergeParams& p, int r, uint64_t* keys,
                                     const float* logp, const int32_t* tok, const float* score) {
  const int n = p.F * p.K;
  uint64_t* out = keys + n;
  for (int e = threadIdx.x; e < n; e += blockDim.x)
    keys[e] = make_key(__fadd_rn(score[e / p.K], logp[e]), static_cast<uint32_t>(e));
  __syncthreads();
  block_rank_select(keys, n, p.Fd, out);
  __syncthreads();
  for (int q = threadIdx.x; q < p.Fd; q += blockDim.x) write_frontier(p, r, q, out[q], tok);
}

__device__ void select_frontier(const MergeParams& p, int r, uint64_t* keys,
                                uint64_t (*wl)[32]) {
  if (p.radix) {
    select_frontier_radix(p, r, keys);
    return;
  }
  if (p.F * p.K <= p.rank_max && p.F * p.K <= kTokStage) {
    select_frontier_rank(p, r, keys);
    return;
  }
  if (p.Fd <= 32) {
    select_frontier_warp(p, r, wl);
    return;
  }
  if (p.Fd <= 64 && p.F <= 64) {
    select_frontier_warp64(p, r, keys);
    return;
  }
  const int n = p.F * p.K;
  const int np2 = pow2_at_least(n);
  for (int e = threadIdx.x; e < np2; e += blockDim.x) {
    uint64_t k = 0ull;
    if (e < n) {
      const int row = r * p.F + e / p.K;
      const float lp = __ldcg(p.row_logp + static_cast<size_t>(row) * p.K + (e % p.K));
      const float c = __fadd_rn(__ldcg(p.score_in + row), lp);
      k = make_key(c, static_cast<uint32_t>(e));
    }
    keys[e] = k;
  }
  __syncthreads();
  block_sort_desc(keys, np2);
  for (int q = threadIdx.x; q < p.Fd; q += blockDim.x) write_frontier(p, r, q, keys[q]);
}

// Row merge.  Grid = (groups, M): block (g, c) merges a contiguous share of
// the per-CTA partials of head row c -- the (max, sum-exp) pairs with fp32
// log-sum-exp merges, and the sorted top-K lists by warp bitonic merges (each
// warp folds every 8th list, all of its lists' keys loaded up front, then a
// tree across the warps).  One group (up to 160 partials) finishes the row
// itself; with several, each publishes one pair and one list and the last
// group block of the row (atomic count) combines them.  The row's
//   lse = max + log(sum) (fp64 sum), top-K = best K keys, logp = fp32(logit - lse).
// With p.select set, the last row of each request then runs the request's
// top-W selection.
__global__ void __launch_bounds__(kMergeThreads) k_merge_rows(const MergeParams p) {
  extern __shared__ uint64_t dyn[];
  __shared__ uint64_t wl[kMergeWarps][32];
  __shared__ int last_flag;
  const int g = blockIdx.x, row = blockIdx.y;
  const int K = p.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int p2 = pow2_ceil32(K);
  pdl_wait();
  pdl_trigger();

  const int l0 = static_cast<int>(static_cast<long long>(g) * p.n_cta / p.groups);
  const int l1 = static_cast<int>(static_cast<long long>(g + 1) * p.n_cta / p.groups);
  // ---- this group's log-sum-exp pair (warp 0; every lane ends with it)
  float gm = -INFINITY, gs = 0.f;
  if (warp == 0) {
    for (int i = l0 + lane; i < l1; i += 32)
      lse_merge(gm, gs, p.pm[static_cast<size_t>(row) * p.cta_stride + i],
                p.ps[static_cast<size_t>(row) * p.cta_stride + i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, gm, o);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, gs, o);
      lse_merge(gm, gs, m2, s2);
    }
  }
  // ---- this group's top-K: warp w folds lists l0 + w, l0 + w + 8, ...;
  // the keys of up to kPre lists are loaded before any of them is merged
  constexpr int kPre = 20;
  const uint64_t* base = p.ptop + static_cast<size_t>(row) * p.list_stride * K;
  // the list element this lane contributes to a merge (warp_merge_desc layout)
  const int jl = p2 == 32 ? 31 - lane : 2 * p2 - 1 - lane;
  const bool takes = p2 == 32 ? jl < K : (lane >= p2 && lane < 2 * p2 && jl < K);
  uint64_t v = 0ull;
  for (int lb = l0 + warp; lb < l1; lb += kMergeWarps * kPre) {
    uint64_t pre[kPre];
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
      const int l = lb + q * kMergeWarps;
      pre[q] = (l < l1 && takes) ? __ldcg(base + static_cast<size_t>(l) * K + jl) : 0ull;
    }
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
      if (lb + q * kMergeWarps >= l1) break;  // the same for the whole warp
      if (p2 == 32) {
        v = warp_merge_desc(v, pre[q], 32);
      } else {
        v = lane < p2 ? v : pre[q];
        v = warp_merge_desc(v, 0ull, p2);
      }
    }
  }
  v = block_tree_merge(v, wl, p2);

  // ---- several groups: the last group block of the row combines them
  if (p.groups > 1) {
    if (warp == 0) {
      if (lane == 0) p.gls[row * 8 + g] = make_float2(gm, gs);
      p.gpl[(static_cast<size_t>(row) * 8 + g) * 32 + lane] = lane < p2 ? v : 0ull;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_flag = (atomicAdd(p.row_cnt + row, 1) == p.groups - 1);
    __syncthreads();
    if (!last_flag) return;
    __threadfence();
    if (threadIdx.x == 0) p.row_cnt[row] = 0;
    v = warp < p.groups ? __ldcg(p.gpl + (static_cast<size_t>(row) * 8 + warp) * 32 + lane) : 0ull;
    v = block_tree_merge(v, wl, p2);
  }
  if (threadIdx.x == 0 && p.gth) p.gth[row] = 0ull;  // the head call's bounds, ready for the next call
  if (p.gmx && threadIdx.x < 32) p.gmx[static_cast<size_t>(row) * 32 + threadIdx.x] = 0ull;
  if (warp == 0) {
    float m = -INFINITY, s = 0.f;
    if (p.groups > 1) {
      if (lane < p.groups) {
        const float2 gp = __ldcg(p.gls + row * 8 + lane);
        m = gp.x;
        s = gp.y;
      }
    } else if (lane == 0) {
      m = gm;
      s = gs;
    }
    float mx = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
    double sd = (m != -INFINITY) ? static_cast<double>(s * expf(m - mx)) : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sd += __shfl_xor_sync(0xFFFFFFFFu, sd, o);
    const double lse = (mx == -INFINITY) ? -INFINITY : static_cast<double>(mx) + log(sd);
    if (lane == 0 && mx == -INFINITY) atomicOr(p.err, DT_ERR_EMPTY_ROW);
    if (lane < K) {
      if (v == 0ull) atomicOr(p.err, DT_ERR_BAD_INDEX);  // fewer than K real entries
      const float val = key_value(v);
      p.row_tok[static_cast<size_t>(row) * K + lane] = static_cast<int32_t>(key_index(v));
      p.row_logp[static_cast<size_t>(row) * K + lane] =
          static_cast<float>(static_cast<double>(val) - lse);
    }
    if (lane == 0) p.row_lse[row] = lse;
  }
  if (!p.select) return;

  // ---- the last row of request r runs its top-W selection
  const int r = row / p.F;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_flag = (atomicAdd(p.counters + r, 1) == p.F - 1);
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  select_frontier(p, r, dyn, wl);
  if (threadIdx.x == 0) p.counters[r] = 0;
  if (p.U_f32) {
    __syncthreads();
    state_from_u(p, r);
  }
}

static size_t select_smem(const MergeParams& p);

cudaError_t launch_merge_rows(const MergeParams& p, cudaStream_t st) {
  return launch_kernel(k_merge_rows, dim3(p.groups, p.M), dim3(kMergeThreads), select_smem(p), st,
                       p.pdl != 0, p);
}

// ----------------------------------------- row merge through the row bound

// 32 keys (one per lane) sorted descending across the lanes (bitonic).
__device__ __forceinline__ uint64_t warp_sort32_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = shfl_xor_u64(v, j);
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = keep_max ? (v > o ? v : o) : (v < o ? v : o);
    }
  }
  return v;
}

// Folds up to 32 keys (one per lane, 0 = none, any order) into the running
// descending list held in lanes 0..p2-1.
__device__ __forceinline__ uint64_t fold_chunk(uint64_t v, uint64_t c, int p2) {
  const int lane = threadIdx.x & 31;
  c = warp_sort32_desc(c);
  if (p2 == 32) return warp_merge_desc(v, shfl_u64(c, 31 - lane), 32);
  const int src = 2 * p2 - 1 - lane;  // lanes p2..2p2-1: the chunk's best p2, reversed
  const uint64_t b = shfl_u64(c, src < 0 ? 0 : src > 31 ? 31 : src);
  v = lane < p2 ? v : (lane < 2 * p2 ? b : 0ull);
  return warp_merge_desc(v, 0ull, p2);
}

constexpr int kBoundParts = 320;  // CTA partials per row that k_merge_bound takes
constexpr int kSurvCap = 512;     // keys at or above the bound staged in shared memory

// Row merge through the head call's row bound.  Block = one head row.  The
// bound gth[row] never exceeds the row's K-th key (K keys of one CTA, or the
// best keys of K CTA groups, reach it), so the row's top-K are among the
// keys at or above it: in one pass over memory (every load of a round in
// flight together) the block reads every CTA's (max, sum-exp) pair and every
// list key, keeps the keys at or above the bound (typically a few K of the
// n_cta K), and sorts them.  The log-sum-exp pairs merge in fp32 in a fixed
// order (thread, lanes, warps).  With p.select set, the last row of each
// request then runs the request's top-W selection.  Shared memory stays
// small (the selection's, the survivors' 4 KB and a few more).  With
// p.cluster the F row blocks of a request are one cluster: each row's
// results also go to the leader's shared memory (distributed shared
// memory), and after one cluster barrier the leader selects -- in place of
// the global hand-over (fence, arrival count) and the selection's loads.
__global__ void __launch_bounds__(kMergeThreads) k_merge_bound(const MergeParams p) {
  extern __shared__ uint64_t dyn[];  // the selection's keys
  __shared__ uint64_t wl[kMergeWarps][32];
  __shared__ float2 wls[kMergeWarps];
  __shared__ uint64_t sv[kSurvCap];
  __shared__ int n_sv, last_flag;
  __shared__ float cl_logp[kClusterRows * 32];  // cluster leader: the rows' results
  __shared__ int32_t cl_tok[kClusterRows * 32];
  __shared__ float cl_score[kClusterRows];
  const int row = blockIdx.x, K = p.K, p2 = pow2_ceil32(K), n = p.n_cta;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) n_sv = 0;
  if (p.cluster) cl_arrive_relaxed();  // (waited on before the first remote store)
  pdl_wait();
  pdl_trigger();
  const int i_req = row % (p.F > 0 ? p.F : 1);  // this row within its request
  if (p.cluster && i_req == 0 && threadIdx.x < p.F)  // the leader: frontier scores
    cl_score[threadIdx.x] = __ldcg(p.score_in + row + threadIdx.x);
  const uint64_t th = p.gth ? __ldcg(p.gth + row) : 0ull;
  const float* pmr = p.pm + static_cast<size_t>(row) * p.cta_stride;
  const float* psr = p.ps + static_cast<size_t>(row) * p.cta_stride;
  const uint64_t* base = p.ptop + static_cast<size_t>(row) * p.list_stride * K;  // [n][K]
  // ---- the (max, sum-exp) pairs (n <= 2 x threads) and every list key at
  // or above the bound (in any order; the sort decides), loaded together
  const int i0 = threadIdx.x, i1 = threadIdx.x + kMergeThreads;
  const float m0 = i0 < n ? __ldcg(pmr + i0) : -INFINITY, s0 = i0 < n ? __ldcg(psr + i0) : 0.f;
  const float m1 = i1 < n ? __ldcg(pmr + i1) : -INFINITY, s1 = i1 < n ? __ldcg(psr + i1) : 0.f;
  const int T = n * K;
  const int cap = p.surv_cap < kSurvCap ? (p.surv_cap > 0 ? p.surv_cap : 0) : kSurvCap;
  constexpr int kPre = 8;  // keys per thread loaded before any is staged
  __syncthreads();         // n_sv
  for (int f0 = 0; f0 < T; f0 += kMergeThreads * kPre) {
    uint64_t kk[kPre];
#pragma unroll
    for (int q = 0; q < kPre; ++q) {
      const int f = f0 + q * kMergeThreads + threadIdx.x;
      kk[q] = f < T ? __ldcg(base + f) : 0ull;
    }
#pragma unroll
    for (int q = 0; q < kPre; ++q) {  // one shared atomic per warp and round
      const bool in = kk[q] != 0ull && kk[q] >= th;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
      int at = 0;
      if (lane == 0 && bal) at = atomicAdd(&n_sv, __popc(bal));
      at = __shfl_sync(0xFFFFFFFFu, at, 0);
      const int pos = at + __popc(bal & ((1u << lane) - 1u));
      if (in && pos < cap) sv[pos] = kk[q];
    }
  }
  float m = -INFINITY, s = 0.f;
  lse_merge(m, s, m0, s0);
  lse_merge(m, s, m1, s1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    lse_merge(m, s, m2, s2);
  }
  if (lane == 0) wls[warp] = make_float2(m, s);
  if (threadIdx.x < 32) wl[0][threadIdx.x] = 0ull;  // the top-K slots (fewer survivors: empty)
  __syncthreads();
  const int ns = n_sv;
  // ---- top-K of the survivors: by rank counting in shared memory; more
  // than the buffer holds: every list key, straight from memory (the ones
  // below the bound as empty), folded by every warp and a tree
  uint64_t v = 0ull;
  if (ns <= cap) {
    block_rank_select(sv, ns, K, wl[0]);
    __syncthreads();
    v = wl[0][lane];  // (warp 0 uses it: lane = rank)
  } else {
    for (int c0 = warp * 32; c0 < T; c0 += kMergeThreads * kPre) {
      uint64_t kk[kPre];
#pragma unroll
      for (int q = 0; q < kPre; ++q) {
        const int f = c0 + q * kMergeThreads + lane;
        kk[q] = f < T ? __ldcg(base + f) : 0ull;
      }
#pragma unroll
      for (int q = 0; q < kPre; ++q) v = fold_chunk(v, kk[q] >= th ? kk[q] : 0ull, p2);
    }
    v = block_tree_merge(v, wl, p2);
  }
  if (p.cluster) cl_wait();  // the leader has started: its shared memory may be written
  if (warp == 0) {
    // the warps' pairs: lanes 0..7, a fixed shuffle tree, lane 0's result to all
    float mm = lane < kMergeWarps ? wls[lane].x : -INFINITY;
    float ss = lane < kMergeWarps ? wls[lane].y : 0.f;
#pragma unroll
    for (int o = kMergeWarps / 2; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, mm, o);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, ss, o);
      lse_merge(mm, ss, m2, s2);
    }
    mm = __shfl_sync(0xFFFFFFFFu, mm, 0);
    ss = __shfl_sync(0xFFFFFFFFu, ss, 0);
    const double lse =
        (mm == -INFINITY) ? -INFINITY : static_cast<double>(mm) + log_f32_exp(ss);
    if (lane == 0 && mm == -INFINITY) atomicOr(p.err, DT_ERR_EMPTY_ROW);
    if (lane < K) {
      if (v == 0ull) atomicOr(p.err, DT_ERR_BAD_INDEX);  // fewer than K real entries
      const int32_t tk = static_cast<int32_t>(key_index(v));
      const float lp = static_cast<float>(static_cast<double>(key_value(v)) - lse);
      p.row_tok[static_cast<size_t>(row) * K + lane] = tk;
      p.row_logp[static_cast<size_t>(row) * K + lane] = lp;
      if (p.cluster) {  // the leader's copy, for its selection
        const int e = i_req * K + lane;
        cl_store_u32(cl_leader_addr(cl_tok + e), static_cast<uint32_t>(tk));
        cl_store_u32(cl_leader_addr(cl_logp + e), __float_as_uint(lp));
      }
    }
    if (lane == 0) p.row_lse[row] = lse;
    if (lane == 0 && p.gth) p.gth[row] = 0ull;  // the head call's bounds, ready for the next call
    if (p.gmx) p.gmx[static_cast<size_t>(row) * 32 + lane] = 0ull;
  }
  if (!p.select) return;
  const int r = row / p.F;
  if (p.cluster) {  // ---- one cluster per request: its leader selects
    cl_barrier();
    if (i_req != 0) return;
    select_frontier_smem(p, r, dyn, cl_logp, cl_tok, cl_score);
    if (p.U_f32) {
      __syncthreads();
      state_from_u(p, r);
    }
    return;
  }

  // ---- the last row of request r runs its top-W selection
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_flag = (atomicAdd(p.counters + r, 1) == p.F - 1);
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  select_frontier(p, r, dyn, wl);
  if (threadIdx.x == 0) p.counters[r] = 0;
  if (p.U_f32) {
    __syncthreads();
    state_from_u(p, r);
  }
}

static size_t select_smem(const MergeParams& p) {
  if (p.select && p.cluster) return static_cast<size_t>(p.F * p.K + p.Fd) * 8;
  if (p.select && p.radix) {
    int kp2 = 1;
    while (kp2 < p.Fd) kp2 <<= 1;
    return (static_cast<size_t>((p.F * p.K + 1) & ~1) + kp2) * 8;
  }
  if (p.select && p.F * p.K <= p.rank_max && p.F * p.K <= kTokStage)
    return static_cast<size_t>(p.F * p.K + p.Fd) * 8;
  if (p.select && (p.Fd > 64 || p.F > 64)) {
    int np2 = 1;
    while (np2 < p.F * p.K) np2 <<= 1;
    return static_cast<size_t>(np2) * 8;
  }
  if (p.select && p.Fd > 32) return static_cast<size_t>(kMergeWarps) * 64 * 8;  // 64-key lists
  return 0;
}

bool merge_bound_fits(const MergeParams& p) {
  return p.n_cta >= 1 && p.n_cta <= kBoundParts && p.K >= 1 && p.K <= 32;
}

cudaError_t launch_merge_bound(const MergeParams& p, cudaStream_t st) {
  if (!merge_bound_fits(p)) return cudaErrorInvalidValue;
  if (p.cluster) {
    if (!p.select || p.F < 1 || p.F > kClusterRows || p.M % p.F != 0 || p.K > 32)
      return cudaErrorInvalidValue;
    return launch_kernel_cluster(k_merge_bound, dim3(p.M), dim3(kMergeThreads), select_smem(p),
                                 st, p.pdl != 0, p.F, p);
  }
  return launch_kernel(k_merge_bound, dim3(p.M), dim3(kMergeThreads), select_smem(p), st,
                       p.pdl != 0, p);
}

int merge_cluster_limit() {
  if (cudaFuncSetAttribute(k_merge_bound, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(kClusterRows);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(kClusterRows * 32 + 256) * 8;
  int size = 0;
  if (cudaOccupancyMaxPotentialClusterSize(&size, k_merge_bound, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return size < kClusterRows ? size : kClusterRows;
}

// ------------------------------------------------- Top-B, compaction, mask

constexpr int kPruneThreads = 1024;

// One block per request.  key = score + beta * depth (two fp32 operations);
// the first min(B, P) nodes by (key desc, pool index asc) are the verification
// tree, in that (canonical) order ("Technische Samenvatting: DARTree",
// Methodologie 2: one global Top-B over all materialised prefixes with a
// non-positive depth bonus).  parent_out = rank of the pool parent; the mask
// row of node i has bit j set iff j is i or an ancestor of i ("DARTree:
// Teaching a Chain-Trained Corrector to Think in Trees", Core Mechanism:
// with this mask a single target forward verifies all branches at once).
__global__ void __launch_bounds__(kPruneThreads) k_prune(const PruneParams p) {
  extern __shared__ uint64_t keys[];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int np2 = pow2_at_least(p.P);
  const int n_sel = p.P < p.B ? p.P : p.B;
  const int sp2 = pow2_at_least(n_sel);
  // radix: keys [P] then the selection [pow2(n_sel)]; else keys [pow2(P)] sorted in place
  uint64_t* sel = p.radix ? keys + ((p.P + 1) & ~1) : keys;
  int32_t* map = reinterpret_cast<int32_t*>(p.radix ? sel + sp2 : keys + np2);  // [P] pool -> rank
  int32_t* par = map + p.P;                               // [B] parent rank
  const size_t pb = static_cast<size_t>(r) * p.pool_stride;
  const int n_keys = p.radix ? p.P : np2;
  for (int e = threadIdx.x; e < n_keys; e += blockDim.x) {
    uint64_t k = 0ull;
    if (e < p.P) {
      const float key = __fadd_rn(p.pool_score[pb + e],
                                  __fmul_rn(p.beta, static_cast<float>(p.pool_depth[pb + e])));
      k = make_key(key, static_cast<uint32_t>(e));
    }
    keys[e] = k;
  }
  for (int e = threadIdx.x; e < p.P; e += blockDim.x) map[e] = -1;
  if (p.radix)
    for (int q = n_sel + threadIdx.x; q < sp2; q += blockDim.x) sel[q] = 0ull;
  __syncthreads();
  if (p.radix) {
    __shared__ unsigned hist[256];
    __shared__ int sh[4];
    block_radix_select(keys, p.P, n_sel, sel, hist, sh);
    block_sort_desc(sel, sp2);
  } else {
    block_sort_desc(keys, np2);
  }
  for (int q = threadIdx.x; q < n_sel; q += blockDim.x) map[key_index(sel[q])] = q;
  __syncthreads();
  const size_t ob = static_cast<size_t>(r) * p.B;
  bool broken = false;
  for (int q = threadIdx.x; q < p.B; q += blockDim.x) {
    if (q < n_sel) {
      const int n = static_cast<int>(key_index(sel[q]));
      const int pp = p.pool_parent[pb + n];
      int pr = (pp < 0 || pp >= p.P) ? -1 : map[pp];
      if ((pp >= 0 && pr < 0) || pr >= q || pp >= p.P) {
        broken = true;
        pr = -1;
      }
      par[q] = pr;
      p.parent[ob + q] = pr;
      p.token[ob + q] = p.pool_token[pb + n];
      p.depth[ob + q] = p.pool_depth[pb + n];
      p.score[ob + q] = p.pool_score[pb + n];
    } else {
      par[q] = -1;
      p.parent[ob + q] = -1;
      p.token[ob + q] = -1;
      p.depth[ob + q] = 0;
      p.score[ob + q] = 0.f;
    }
  }
  if (broken) atomicOr(p.err, DT_ERR_CLOSURE);
  __syncthreads();
  const size_t mb = static_cast<size_t>(r) * p.B * p.words;
  for (int e = threadIdx.x; e < p.B * p.words; e += blockDim.x) {
    const int q = e / p.words, w = e % p.words;
    uint32_t bits = 0;
    if (q < n_sel) {
      int a = q;
      for (int steps = 0; a >= 0 && steps <= p.B; ++steps) {  // parents rank earlier
        if ((a >> 5) == w) bits |= 1u << (a & 31);
        a = par[a];
      }
    }
    p.mask[mb + e] = bits;
  }
  if (threadIdx.x == 0) p.n_out[r] = n_sel;
}

cudaError_t launch_prune(const PruneParams& p, cudaStream_t st) {
  int np2 = 1;
  while (np2 < p.P) np2 <<= 1;
  int sp2 = 1;
  while (sp2 < (p.P < p.B ? p.P : p.B)) sp2 <<= 1;
  const size_t key_bytes = p.radix ? (static_cast<size_t>((p.P + 1) & ~1) + sp2) * 8
                                   : static_cast<size_t>(np2) * 8;
  const size_t smem = key_bytes + static_cast<size_t>(p.P) * 4 + static_cast<size_t>(p.B) * 4;
  return launch_kernel(k_prune, dim3(p.R), dim3(kPruneThreads), smem, st, p.pdl != 0, p);
}

// ------------------------------------------------------------------ root

__global__ void k_root(const RootParams p) {
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  for (int h = threadIdx.x; h < p.H; h += blockDim.x) {
    const float v = m < p.R ? p.state0[static_cast<size_t>(m) * p.H + h] : 0.f;
    if (p.bf16)
      static_cast<uint16_t*>(p.S)[static_cast<size_t>(m) * p.H + h] = float_to_bf16_bits(v);
    else
      static_cast<float*>(p.S)[static_cast<size_t>(m) * p.H + h] = v;
  }
  if (threadIdx.x == 0) p.score[m] = 0.f;
}

cudaError_t launch_root(const RootParams& p, cudaStream_t st) {
  return launch_kernel(k_root, dim3(p.n_pad), dim3(256), 0, st, p.pdl != 0, p);
}

// ------------------------------------------------------- state finish

// Finish of a split-K state step ("Technische Samenvatting: DARTree",
// Methodologie 1: the kept branches carry their correction states): block
// (q, hb) = output row q, hidden units [1024 hb, 1024 hb + 1024), four per
// thread.  The splits are summed in split order, so the result does not
// depend on timing.
__global__ void __launch_bounds__(256) k_state_finish(const StateFinishParams p) {
  pdl_wait();  // the partials and the selection (slot, tok) come from earlier kernels
  pdl_trigger();
  const int q = blockIdx.x;
  const int h = (blockIdx.y * 256 + threadIdx.x) * 4;
  if (h >= p.H) return;
  uint16_t* out = p.S_out + static_cast<size_t>(q) * p.H + h;
  if (q >= p.M_out) {  // padding rows of the next head call
    *reinterpret_cast<uint2*>(out) = make_uint2(0u, 0u);
    return;
  }
  int col = __ldg(p.slot + q), tok = __ldg(p.tok + q);
  if (col < 0 || col >= p.M_in) col = 0;  // (never, unless upstream failed)
  if (tok < 0 || tok >= p.V_tok) {        // only after an upstream failure
    if (h == 0) atomicOr(p.err, DT_ERR_BAD_INDEX);
    tok = 0;
  }
  const uint2 eb = __ldg(reinterpret_cast<const uint2*>(p.E + static_cast<size_t>(tok) * p.H + h));
  float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < p.n_split; ++s) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(
        p.part + (static_cast<size_t>(s) * kMaxRows + col) * p.H + h));
    u.x += v.x;
    u.y += v.y;
    u.z += v.z;
    u.w += v.w;
  }
  const float o0 = tanhf(u.x + bf16_bits_to_float(static_cast<uint16_t>(eb.x & 0xFFFFu)));
  const float o1 = tanhf(u.y + bf16_bits_to_float(static_cast<uint16_t>(eb.x >> 16)));
  const float o2 = tanhf(u.z + bf16_bits_to_float(static_cast<uint16_t>(eb.y & 0xFFFFu)));
  const float o3 = tanhf(u.w + bf16_bits_to_float(static_cast<uint16_t>(eb.y >> 16)));
  *reinterpret_cast<uint2*>(out) =
      make_uint2(static_cast<uint32_t>(float_to_bf16_bits(o0)) |
                     (static_cast<uint32_t>(float_to_bf16_bits(o1)) << 16),
                 static_cast<uint32_t>(float_to_bf16_bits(o2)) |
                     (static_cast<uint32_t>(float_to_bf16_bits(o3)) << 16));
}

// State step with fp32 weights ("Technische Samenvatting: DARTree",
// Methodologie 1: the kept branches carry their correction states): block b
// owns hidden units [8 b, 8 b + 8), one per warp.  The warp loads its row of
// A once (lanes over j, a chunk of 256 columns at a time) and computes
// U[h][c] = sum_j A[h][j] S_in[c][j] for every input row c, four rows' loads
// in flight together, each sum finished by a butterfly; U goes to shared
// memory.  Then output row q, hidden unit 8 b + i is
// tanh(U[h][slot[q]] + E[tok[q]][h]) (zeros for the padding rows).  The step
// is a short latency chain, not a stream: few dependent load rounds per warp.
__global__ void __launch_bounds__(256) k_state_f32(const StateF32Params p) {
  extern __shared__ float sU[];  // [8][M_in]
  pdl_wait();  // the input rows and the selection (slot, tok) come from earlier kernels
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 8 + warp;
  if (h < p.H) {
    const float* a = p.A + static_cast<size_t>(h) * p.H;
    for (int j0 = 0; j0 < p.H; j0 += 256) {
      float av[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int j = j0 + lane + 32 * k;
        av[k] = j < p.H ? __ldg(a + j) : 0.f;
      }
      for (int c0 = 0; c0 < p.M_in; c0 += 4) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int c = c0 + u < p.M_in ? c0 + u : p.M_in - 1;
          const float* x = p.S_in + static_cast<size_t>(c) * p.H;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int j = j0 + lane + 32 * k;
            acc[u] = fmaf(av[k], j < p.H ? __ldcg(x + j) : 0.f, acc[u]);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc[u] += __shfl_xor_sync(kFullMask, acc[u], o);
          if (lane == 0 && c0 + u < p.M_in) {
            float* dst = sU + warp * p.M_in + c0 + u;
            *dst = (j0 == 0 ? 0.f : *dst) + acc[u];
          }
        }
      }
    }
  }
  __syncthreads();
  // outputs: thread (q, i) -> hidden unit 8 b + i of output row q
  const int i = threadIdx.x & 7;
  const int hh = blockIdx.x * 8 + i;
  if (hh >= p.H) return;
  bool bad = false;
  for (int q = threadIdx.x >> 3; q < p.n_out; q += 32) {
    float out = 0.f;
    if (q < p.M_out) {
      int col = __ldg(p.slot + q), tok = __ldg(p.tok + q);
      if (col < 0 || col >= p.M_in) col = 0;  // (never, unless upstream failed)
      if (tok < 0 || tok >= p.V_tok) {        // only after an upstream failure
        bad = true;
        tok = 0;
      }
      out = tanhf(sU[i * p.M_in + col] + __ldg(p.E + static_cast<size_t>(tok) * p.H + hh));
    }
    p.S_out[static_cast<size_t>(q) * p.H + hh] = out;
  }
  if (bad) atomicOr(p.err, DT_ERR_BAD_INDEX);
}

cudaError_t launch_state_f32(const StateF32Params& p, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(8) * p.M_in * 4;
  return launch_kernel(k_state_f32, dim3((p.H + 7) / 8), dim3(256), smem, st, p.pdl != 0, p);
}

cudaError_t launch_state_finish(const StateFinishParams& p, cudaStream_t st) {
  if (p.H % 4 != 0) return cudaErrorInvalidValue;
  const dim3 grid(p.n_out, (p.H + 1023) / 1024);
  return launch_kernel(k_state_finish, grid, dim3(256), 0, st, p.pdl != 0, p);
}

cudaError_t init_select_attrs() {
  cudaError_t e = set_max_dynamic_smem(k_merge_rows);
  if (e == cudaSuccess) e = set_max_dynamic_smem(k_merge_bound);
  if (e != cudaSuccess) return e;
  return set_max_dynamic_smem(k_prune);
}

}  // namespace dt
