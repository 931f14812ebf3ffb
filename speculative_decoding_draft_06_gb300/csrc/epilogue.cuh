// Fused epilogue of the corrected-logit contraction: per head row (a GEMM
// column) an online log-sum-exp over the vocabulary and a running top-K by
// (logit desc, token asc).  The [rows, V] logit matrix never leaves the SM.
//
// Layout: each of the 4 epilogue warps sees 32 vocabulary entries of every
// 128-entry tile (one per lane) for all head rows.  A warp keeps, per head
// row, a private sorted list of its K best 64-bit keys in shared memory;
// the CTA writes those lists and one (max, sum-exp) pair per row as
// partials, which a second kernel merges across CTAs.
//
// Softmax state: for <= 32 head rows every lane keeps a running (max, sum)
// per row in registers (columns unrolled at compile time) and lanes are
// combined once at the end; for more rows each 16-column chunk is reduced
// across the warp and the row's owner lane folds it into a per-warp running
// pair kept in shared memory.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace dt {

constexpr unsigned kFull = kFullMask;

// Bitonic sort of one key per lane; afterwards lane 0 holds the largest.
static __device__ __noinline__ uint64_t warp_sort_desc(uint64_t k) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t o = shfl_xor_u64(k, stride);
      const bool desc_block = (lane & size) == 0;
      const bool lower = (lane & stride) == 0;
      const bool keep_max = (lower == desc_block);
      k = keep_max ? (k > o ? k : o) : (k < o ? k : o);
    }
  }
  return k;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// (m, s) <- (m, s) (+) (m2, s2): log-sum-exp pairs, s = sum exp(x - m).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mx = fmaxf(m, m2);
  if (mx == -INFINITY) {
    m = -INFINITY;
    s = 0.f;
    return;
  }
  s = s * expf(m - mx) + s2 * expf(m2 - mx);
  m = mx;
}

// Insert every key of `bal` lanes (keys differ per lane) into the sorted
// list L of K keys, best first.  Warp-collective.
static __device__ __noinline__ void list_insert_lanes(uint64_t* L, int K, uint64_t key, unsigned bal) {
  const int lane = threadIdx.x & 31;
  while (bal) {
    const int src = __ffs(bal) - 1;
    bal &= bal - 1;
    const uint64_t kc = shfl_u64(key, src);
    const uint64_t e = lane < K ? L[lane] : 0ull;
    const uint64_t last = shfl_u64(e, K - 1);
    if (kc <= last) continue;  // warp-uniform
    const int pos = __popc(__ballot_sync(kFull, lane < K && e > kc));
    __syncwarp();
    if (lane >= pos && lane < K - 1) L[lane + 1] = e;
    if (lane == pos) L[pos] = kc;
    __syncwarp();
  }
}

// First tile: the list of each row is the sorted best K of the 32 lanes.
static __device__ __noinline__ void list_fill(uint64_t* L, int K, uint64_t key) {
  const uint64_t s = warp_sort_desc(key);
  if ((threadIdx.x & 31) < K) L[threadIdx.x & 31] = s;
  __syncwarp();
}

template <int N>
struct LogitsEpilogue {
  static constexpr bool kLaneLocal = N <= 32;
  float lm[kLaneLocal ? N : 1], ls[kLaneLocal ? N : 1];
  uint64_t* lists;  // this warp's lists, [N][K]
  float2* run;      // this warp's running (max, sum) per row (shared, N > 32)
  int K, M, lane;
  bool first;
  bool bad;

  __device__ __forceinline__ void init(uint64_t* warp_lists, float2* warp_run, int K_, int M_) {
    lists = warp_lists;
    run = warp_run;
    K = K_;
    M = M_;
    lane = threadIdx.x & 31;
    first = true;
    bad = false;
#pragma unroll
    for (int c = 0; c < (kLaneLocal ? N : 1); ++c) {
      lm[c] = -INFINITY;
      ls[c] = 0.f;
    }
    for (int i = lane; i < N * K_; i += 32) lists[i] = 0ull;
    for (int c = lane; c < N; c += 32) run[c] = make_float2(-INFINITY, 0.f);
    __syncwarp();
  }

  __device__ __forceinline__ void topk(int c, float xv, bool valid_v, uint32_t v) {
    const uint64_t key = (valid_v && xv == xv) ? make_key(xv, v) : 0ull;
    uint64_t* L = lists + c * K;
    if (first) {
      list_fill(L, K, key);
    } else {
      const unsigned bal = __ballot_sync(kFull, key > L[K - 1]);
      if (bal) list_insert_lanes(L, K, key, bal);
    }
  }

  // <= 32 rows: columns C0..C0+15 with compile-time indices.
  template <int C0>
  __device__ __forceinline__ void consume_static(const float (&x)[16], bool valid_v, uint32_t v) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (C0 + j >= M) break;  // uniform across the warp
      const float xv = x[j];
      if (valid_v && (xv != xv || xv == INFINITY)) bad = true;
      if (valid_v && xv > -INFINITY && xv < INFINITY) {
        const float d = xv - lm[C0 + j];
        const float e = fast_exp(-fabsf(d));
        const bool up = d > 0.f;
        ls[C0 + j] = up ? fmaf(ls[C0 + j], e, 1.f) : ls[C0 + j] + e;
        lm[C0 + j] = up ? xv : lm[C0 + j];
      }
      topk(C0 + j, xv, valid_v, v);
    }
  }

  // > 32 rows: columns c0..c0+15 (c0 a runtime multiple of 16).
  __device__ __forceinline__ void consume_dyn(const float (&x)[16], int c0, bool valid_v,
                                              uint32_t v) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int c = c0 + j;
      if (c >= M) break;
      const float xv = x[j];
      if (valid_v && (xv != xv || xv == INFINITY)) bad = true;
      const bool fin = valid_v && xv > -INFINITY && xv < INFINITY;
      const float xm = fin ? xv : -INFINITY;
      const float mx = warp_max_f(xm);
      if (mx != -INFINITY) {
        const float se = warp_sum_f(fin ? fast_exp(xm - mx) : 0.f);
        if (lane == (c & 31)) {
          float2 r = run[c];
          lse_merge(r.x, r.y, mx, se);
          run[c] = r;
        }
      }
      topk(c, xv, valid_v, v);
    }
  }

  __device__ __forceinline__ void tile_done() { first = false; }

  // Write this CTA's partials.  red = [4][N] float2 (all warps' running
  // pairs); all 128 epilogue threads must call it.
  __device__ __forceinline__ void finish(float2* red, int warp, int cta, float* pm, float* ps,
                                         int cta_stride, uint64_t* ptop, int list_stride,
                                         int* err) {
    if constexpr (kLaneLocal) {
#pragma unroll
      for (int c = 0; c < N; ++c) {
        if (c >= M) break;
        float m = lm[c], s = ls[c];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(kFull, m, o);
          const float s2 = __shfl_xor_sync(kFull, s, o);
          lse_merge(m, s, m2, s2);
        }
        if (lane == 0) red[warp * N + c] = make_float2(m, s);
      }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const int t = warp * 32 + lane;
    for (int c = t; c < M; c += 128) {
      float m = red[c].x, s = red[c].y;
#pragma unroll
      for (int w = 1; w < kEpiWarps; ++w) lse_merge(m, s, red[w * N + c].x, red[w * N + c].y);
      pm[(size_t)c * cta_stride + cta] = m;
      ps[(size_t)c * cta_stride + cta] = s;
    }
    // one list per CTA and row: warp (c % 4) folds the four warps' lists
    // (this warp's lists start at `lists`; the CTA's are [warp][N][K])
    uint64_t* all = lists - static_cast<size_t>(warp) * N * K;
    const int p2 = pow2_ceil32(K);
    for (int c = warp; c < M; c += kEpiWarps) {
      const uint64_t* L0 = all + static_cast<size_t>(c) * K;
      uint64_t v = lane < K ? L0[lane] : 0ull;
#pragma unroll
      for (int w = 1; w < kEpiWarps; ++w) {
        uint64_t y;
        merge_operands(all + (static_cast<size_t>(w) * N + c) * K, K, p2, v, y);
        v = warp_merge_desc(v, y, p2);
      }
      if (lane < K) ptop[((size_t)c * list_stride + cta) * K + lane] = v;
    }
    if (bad) atomicOr(err, DT_ERR_NONFINITE);
  }
};

}  // namespace dt
