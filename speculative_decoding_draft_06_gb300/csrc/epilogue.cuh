// Fused epilogue of the corrected-logit contraction: per head row (a GEMM
// column) an online log-sum-exp over the vocabulary and a running top-K by
// (logit desc, token asc).  The [rows, V] logit matrix never leaves the SM.
//
// Each tile holds 128 vocabulary entries x N head rows.  The producer side
// hands over 16 rows at a time, one vocabulary entry per thread (the
// tensor-memory lane layout).  The chunk is transposed through shared memory
// so that a warp owns whole head rows: row j of a chunk belongs to warp j % 4,
// which reads its 128 values, 4 per lane.  Because one warp owns a row for
// the whole kernel, the row has a single top-K list per CTA (shared memory,
// sorted, best first) and needs no cross-warp synchronisation:
//   * a value enters only if its key beats the list's K-th key and the row's
//     global bound -- the best K-th key any CTA's list has reached so far,
//     shared through a 64-bit atomicMax.  Any list's K-th key bounds the
//     row's true K-th key from below (that list alone holds K keys at or
//     above it), so no key of the final top-K is ever filtered out; the
//     bound only spares CTAs the insertions of keys that cannot make it;
//   * the common case -- no key of the row's 128 beats the threshold -- is
//     one 64-bit compare per value and one vote; rows with entrants go
//     through list_update (a tighter bound from the tile itself, then one
//     compacted batch);
//   * softmax state: for <= 64 rows each lane keeps a running (max, sum) per
//     owned row in registers and lanes are combined once at the end; for more
//     rows each chunk is reduced across the warp and folded into a per-row
//     running pair in shared memory.
// The CTA then writes one (max, sum-exp) pair and one sorted list per row as
// partials, which a second kernel merges across CTAs.
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

// Fold the candidate keys of the lanes (0 = no candidate) into the sorted
// list L: warp-sort the candidates, keep their best p2, and bitonic-merge
// with the list.  Warp-collective.
static __device__ __noinline__ void list_merge_batch(uint64_t* L, int K, uint64_t key) {
  const int lane = threadIdx.x & 31;
  const int p2 = pow2_ceil32(K);
  const uint64_t srt = warp_sort_desc(key);
  uint64_t v = lane < K ? L[lane] : 0ull;
  uint64_t y = 0ull;
  if (p2 == 32) {
    y = shfl_u64(srt, 31 - lane);
  } else {
    const int src = 2 * p2 - 1 - lane;
    const uint64_t b = shfl_u64(srt, src < 0 ? 0 : src);
    v = lane < p2 ? v : (lane < 2 * p2 ? b : 0ull);
  }
  v = warp_merge_desc(v, y, p2);
  __syncwarp();
  if (lane < K) L[lane] = v;
  __syncwarp();
}

// The entrants of one row (keys above th; cnt of this lane, total of the
// warp) into the sorted list L.  With many entrants the threshold is first
// raised to a bound from the keys themselves: split the lanes into K
// disjoint groups; the K group maxima are K distinct keys at or above their
// minimum, so no key below it is in the row's top-K.  The entrants are then
// compacted to one per lane (staging stg) and go in by single inserts or
// one batch merge.  Warp-collective.
static __device__ __forceinline__ void list_update(uint64_t* L, int K, uint64_t* stg, uint64_t th,
                                                uint64_t k0, uint64_t k1, uint64_t k2, uint64_t k3,
                                                int cnt, int total) {
  const int lane = threadIdx.x & 31;
  const uint64_t key[4] = {k0, k1, k2, k3};
  if (total > 4) {
    // K disjoint groups of gs lanes: the minimum of the group maxima
    const int gs = 1 << (31 - __clz(32 / K));
    uint64_t m = key[0] > key[1] ? key[0] : key[1];
    const uint64_t m23 = key[2] > key[3] ? key[2] : key[3];
    m = m > m23 ? m : m23;
    for (int s = 1; s < gs; s <<= 1) {
      const uint64_t o = shfl_xor_u64(m, s);
      m = m > o ? m : o;
    }
    if (lane >= K * gs) m = ~0ull;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const uint64_t o = shfl_xor_u64(m, s);
      m = m < o ? m : o;
    }
    if (m > 0ull && m - 1ull > th) {  // keys >= m may enter
      th = m - 1ull;
      cnt = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) cnt += key[i] > th ? 1 : 0;
      total = __reduce_add_sync(kFull, static_cast<unsigned>(cnt));
    }
  }
  if (total <= 32) {
    // compact: this lane's entrants go after those of the lanes below it
    const unsigned below = (1u << lane) - 1u;
    int pos = __popc(__ballot_sync(kFull, cnt & 1) & below) +
              2 * __popc(__ballot_sync(kFull, cnt & 2) & below) +
              4 * __popc(__ballot_sync(kFull, cnt & 4) & below);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (key[i] > th) stg[pos++] = key[i];
    __syncwarp();
    const uint64_t kk = lane < total ? stg[lane] : 0ull;
    __syncwarp();
    if (total <= 2)
      list_insert_lanes(L, K, kk, __ballot_sync(kFull, lane < total));
    else
      list_merge_batch(L, K, kk);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint64_t t = L[K - 1];
      t = t > th ? t : th;
      const unsigned bal = __ballot_sync(kFull, key[i] > t);
      if (bal == 0u) continue;
      if (__popc(bal) <= 2)
        list_insert_lanes(L, K, key[i], bal);
      else
        list_merge_batch(L, K, key[i] > t ? key[i] : 0ull);
    }
  }
}

// This CTA's best key of a row improved: raise its group's maximum (group =
// CTA % K), then the row's bound gth to the least of K keys of K groups --
// this CTA's best and the other groups' maxima as read at the start of the
// tile (others_min; a group's maximum only grows, so an earlier value is
// still one of its CTAs' keys).  Keys of different CTAs are different
// vocabulary entries, so these are K distinct keys of the row and their
// least bounds its K-th key from below.  Nothing waits for a result.
__device__ __forceinline__ void publish_group_best(unsigned long long* gth,
                                                   unsigned long long* gm, int K,
                                                   uint64_t best, uint64_t others_min) {
  atomicMax(gm + blockIdx.x % K, best);
  const uint64_t v = others_min < best ? others_min : best;
  if (v > 0ull) atomicMax(gth, v);
}

// The least of the other K - 1 groups' maxima of a row (all ones for K = 1).
__device__ __forceinline__ uint64_t others_min(const unsigned long long* gm, int K) {
  const int mine = blockIdx.x % K;
  uint64_t v = ~0ull;
#pragma unroll 8
  for (int g = 0; g < K; ++g) {
    const uint64_t x = g == mine ? ~0ull : __ldcg(gm + g);
    v = x < v ? x : v;
  }
  return v;
}

// Shared-memory footprint of the epilogue (bytes) for N rows, top-K and NG
// warpgroups.
__host__ __device__ constexpr size_t epi_smem_bytes(int N, int K, int NG = 1) {
  return static_cast<size_t>(N) * K * 8                    // lists
         + static_cast<size_t>(NG) * 2 * 16 * 132 * 4       // transposed chunks, 2 per group
         + static_cast<size_t>(N) * 8                       // running (max, sum) per row
         + static_cast<size_t>(N) * 8                       // per-tile copy of the row bounds
         + static_cast<size_t>(N) * 8                       // best keys as last published
         + static_cast<size_t>(N) * 8                       // other groups' least maximum
         + static_cast<size_t>(NG) * 4 * 32 * 8;            // entrant staging, 32 keys per warp
}

// NG warpgroups (1 or 2) share the epilogue.  The head rows come in chunks of
// 16 (one 16-column TMEM load); chunk CH belongs to group CH % NG, which hands
// it over (one vocabulary entry per thread) and processes it alone, each of
// its four warps owning 4 of the 16 rows (row c to warp c % 4).  The groups
// synchronise only within themselves (named barrier 1 + group).
template <int N, int NG = 1>
struct LogitsEpilogue {
  static_assert(NG == 1 || NG == 2, "epilogue warpgroups");
  static constexpr bool kLaneLocal = N <= 64;
  static constexpr int kChunks = N / 16;
  static constexpr int kSlots = kLaneLocal ? 4 * ((kChunks + NG - 1) / NG) : 1;
  static constexpr int kTPitch = 132;  // floats per transposed row
  static constexpr int kThreads = NG * 128;
  float lm[kSlots], ls[kSlots];
  uint64_t* lists;          // [N][K], one sorted list per row
  unsigned long long* gth;  // [N] global per-row lower bound of the K-th key (or null)
  unsigned long long* gmx;  // [N][32] per-row best key of each CTA group (or null)
  uint64_t* gcache;         // [N] this tile's copy of gth
  uint64_t* gpub;           // [N] this CTA's best key per row as last published
  uint64_t* gomin;          // [N] the other CTA groups' least best key, per tile
  uint64_t* stg;            // [32] entrant staging of this warp
  float* T;                 // [2][16][kTPitch] of this group
  float2* run;              // [N] (N > 64)
  int K, M, lane, w4, g, t;
  int nchunk;               // chunks handed over so far (selects the T buffer)
  bool bad;

  __device__ __forceinline__ void bar() {
    asm volatile("bar.sync %0, 128;" ::"r"(1 + g) : "memory");
  }

  // Row of this warp's slot s (lane-local path): local chunk s / 4, row s % 4.
  __device__ __forceinline__ int slot_row(int s) const {
    return ((s >> 2) * NG + g) * 16 + w4 + 4 * (s & 3);
  }

  __device__ __forceinline__ void init(uint8_t* smem, int K_, int M_,
                                       unsigned long long* gth_ = nullptr,
                                       unsigned long long* gmx_ = nullptr) {
    gth = gth_;
    gmx = gth_ ? gmx_ : nullptr;
    lists = reinterpret_cast<uint64_t*>(smem);
    float* T0 = reinterpret_cast<float*>(lists + static_cast<size_t>(N) * K_);
    run = reinterpret_cast<float2*>(T0 + NG * 2 * 16 * kTPitch);
    gcache = reinterpret_cast<uint64_t*>(run + N);
    K = K_;
    M = M_;
    const int tt = threadIdx.x % kThreads;
    g = tt >> 7;
    t = tt & 127;
    lane = threadIdx.x & 31;
    w4 = t >> 5;
    T = T0 + g * 2 * 16 * kTPitch;
    gpub = gcache + N;
    gomin = gpub + N;
    stg = gomin + N + (tt >> 5) * 32;
    nchunk = 0;
    bad = false;
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
      lm[i] = -INFINITY;
      ls[i] = 0.f;
    }
    for (int i = tt; i < N * K_; i += kThreads) lists[i] = 0ull;
    for (int c = tt; c < N; c += kThreads) {
      run[c] = make_float2(-INFINITY, 0.f);
      gcache[c] = 0ull;
      gpub[c] = 0ull;
      gomin[c] = 0ull;
    }
    asm volatile("bar.sync 3, %0;" ::"r"(kThreads) : "memory");
  }

  // At the start of a tile: this warp's rows' global bounds and the other
  // CTA groups' least best key, all loads in flight together (the list
  // update and the bound publishing then read shared memory only).
  __device__ __forceinline__ void tile_begin() {
    if (!gth) return;
    for (int i = lane;; i += 32) {
      const int c = ((i >> 2) * NG + g) * 16 + w4 + 4 * (i & 3);
      if (c >= M) break;
      gcache[c] = __ldcg(gth + c);
      if (gmx) gomin[c] = others_min(gmx + static_cast<size_t>(c) * 32, K);
    }
    __syncwarp();
  }

  // Stage x (rows c0..c0+15 of vocabulary entry t of the tile) transposed.
  __device__ __forceinline__ float* stage(const float (&x)[16]) {
    float* Tb = T + (nchunk & 1) * 16 * kTPitch;
#pragma unroll
    for (int j = 0; j < 16; ++j) Tb[j * kTPitch + t] = x[j];
    ++nchunk;
    bar();
    return Tb;
  }

  // Top-K update of row c with this lane's 4 values (vocabulary v0 + lane + 32 i).
  __device__ __forceinline__ void topk4(int c, const float (&xv)[4], uint32_t v0, int V) {
    uint64_t* L = lists + static_cast<size_t>(c) * K;
    const uint64_t gb = gcache[c];
    const uint64_t k_before = L[K - 1];
    const uint64_t th = k_before > gb ? k_before : gb;
    uint64_t key[4];
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t v = v0 + lane + 32 * i;
      key[i] = (static_cast<int>(v) < V && xv[i] == xv[i]) ? make_key(xv[i], v) : 0ull;
      cnt += key[i] > th ? 1 : 0;
    }
    const int total = static_cast<int>(__reduce_add_sync(kFull, static_cast<unsigned>(cnt)));
    if (total == 0) return;  // the common case once the bounds have filled
    list_update(L, K, stg, th, key[0], key[1], key[2], key[3], cnt, total);
    // publish improved bounds: the list's K-th key (once the list is full)
    // and this CTA's best key for its group (gpub: as last published)
    const uint64_t k_after = L[K - 1], best = L[0];
    if (gth && lane == 0 && k_after > th) atomicMax(gth + c, k_after);
    if (gmx && best > gpub[c]) {
      if (lane == 0) {
        publish_group_best(gth + c, gmx + static_cast<size_t>(c) * 32, K, best, gomin[c]);
        gpub[c] = best;
      }
      __syncwarp();
    }
  }

  __device__ __forceinline__ void load4(const float* Tb, int j, uint32_t v0, int V, float (&xv)[4],
                                        bool (&fin)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      xv[i] = Tb[j * kTPitch + lane + 32 * i];
      const bool valid = static_cast<int>(v0 + lane + 32 * i) < V;
      if (valid && (xv[i] != xv[i] || xv[i] == INFINITY)) bad = true;
      fin[i] = valid && xv[i] > -INFINITY && xv[i] < INFINITY;
    }
  }

  // <= 64 rows: chunk CH (rows 16 CH .. 16 CH + 15, a chunk of this group)
  // with compile-time slots.
  template <int CH>
  __device__ __forceinline__ void chunk_static(const float (&x)[16], uint32_t v0, int V) {
    const float* Tb = stage(x);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = w4 + 4 * jj;
      const int c = CH * 16 + j;
      if (c >= M) continue;  // uniform across the warp
      float xv[4];
      bool fin[4];
      load4(Tb, j, v0, V, xv, fin);
      constexpr int kBase = (CH / NG) * 4;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (!fin[i]) continue;
        const float d = xv[i] - lm[kBase + jj];
        const float e = fast_exp(-fabsf(d));
        const bool up = d > 0.f;
        ls[kBase + jj] = up ? fmaf(ls[kBase + jj], e, 1.f) : ls[kBase + jj] + e;
        lm[kBase + jj] = up ? xv[i] : lm[kBase + jj];
      }
      topk4(c, xv, v0, V);
    }
  }

  // > 64 rows: chunk starting at row c0 (a chunk of this group, runtime).
  __device__ __forceinline__ void chunk_dyn(const float (&x)[16], int c0, uint32_t v0, int V) {
    const float* Tb = stage(x);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int j = w4 + 4 * jj;
      const int c = c0 + j;
      if (c >= M) continue;
      float xv[4];
      bool fin[4];
      load4(Tb, j, v0, V, xv, fin);
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) mx = fin[i] ? fmaxf(mx, xv[i]) : mx;
      mx = warp_max_f(mx);
      if (mx != -INFINITY) {
        float se = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) se += fin[i] ? fast_exp(xv[i] - mx) : 0.f;
        se = warp_sum_f(se);
        if (lane == 0) {
          float2 r = run[c];
          lse_merge(r.x, r.y, mx, se);
          run[c] = r;
        }
      }
      topk4(c, xv, v0, V);
    }
  }

  // Write this CTA's partials: one (max, sum-exp) pair and one list per row,
  // each by the row's owner warp.
  __device__ __forceinline__ void finish(int cta, float* pm, float* ps, int cta_stride,
                                         uint64_t* ptop, int list_stride, int* err) {
    __syncwarp();
    if constexpr (kLaneLocal) {
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const int c = slot_row(s);
        float m = lm[s], sm = ls[s];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(kFull, m, o);
          const float s2 = __shfl_xor_sync(kFull, sm, o);
          lse_merge(m, sm, m2, s2);
        }
        if (lane == 0 && c < M) {
          pm[(size_t)c * cta_stride + cta] = m;
          ps[(size_t)c * cta_stride + cta] = sm;
        }
      }
    }
    for (int c0 = g * 16; c0 < M; c0 += 16 * NG) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int c = c0 + w4 + 4 * jj;
        if (c >= M) break;
        if constexpr (!kLaneLocal) {
          if (lane == 0) {
            pm[(size_t)c * cta_stride + cta] = run[c].x;
            ps[(size_t)c * cta_stride + cta] = run[c].y;
          }
        }
        if (lane < K) ptop[((size_t)c * list_stride + cta) * K + lane] = lists[(size_t)c * K + lane];
      }
    }
    if (bad) atomicOr(err, DT_ERR_NONFINITE);
  }
};

}  // namespace dt
