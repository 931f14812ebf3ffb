// Head call for many head rows (64 and more): the corrected logits
//   ell[m, v] = z_d[v] + sum_h S[m, h] Wout[v, h]
// with the online log-sum-exp and the per-row top-K fused into the epilogue
// ("DARTree: Teaching a Chain-Trained Corrector to Think in Trees", Core
// Mechanism: a single batched head call per depth for every branch;
// "Technische Samenvatting:
// DARTree", Methodologie 1: the top-k children of every branch, scored from
// the normalised corrected distribution).
//
// Orientation.  Here the head rows are the MMA M (one or two M = 128
// halves, padded) and a vocabulary tile of NV = 128 or 256 entries is the
// MMA N.  The accumulator then holds one head row per TMEM lane: an
// epilogue thread reads its own row's logits of the tile with tcgen05.ld
// and keeps the row's running (max, sum-exp), its top-K list and threshold
// -- no transposition, no cross-lane reduction, a compare per value.  (The
// kernel for fewer than 64 rows, k_head_tc, puts the vocabulary on M
// instead.)  The states are re-read from L2 for every tile; the wider tile
// halves that stream per weight byte (one CTA with MH = 2 and NV = 256 has a
// single accumulator: the MMAs of a tile wait for the previous tile's
// epilogue).
//
// Warp roles: warps 0..4MH-1 epilogue (warp w reads TMEM lane quarter w % 4
// of half w / 4), warp 4MH TMA producer (per 64-wide K step: MH boxes of
// 128 state rows and NV / 128 boxes of 128 Wout rows, 128-byte swizzle),
// warp 4MH+1 TMEM allocator + single-thread MMA issuer.  Two accumulators
// where 2 x MH x NV columns fit in TMEM, else one.  Persistent: each CTA
// owns a contiguous range of vocabulary tiles.
//
// Pair mode (129..256 rows).  With 256 rows one CTA's shared memory is the
// bottleneck: per K step its MMAs read both row halves' states and the Wout
// tile twice.  A cluster of two CTAs instead computes M = 256 x N = 256
// with the two-CTA MMA: each CTA holds 128 state rows and 128 of the tile's
// Wout rows, the leader issues the MMAs for both, both CTAs' copies complete
// on the leader's stage barrier, the MMA commits arrive in both CTAs, and
// each CTA's TMEM receives its 128 rows x 256 columns.  Each CTA runs two
// epilogue warpgroups, one per half of the tile's columns (warps 0-3 and
// 4-7), each a separate partial slot for the row merge.
//
// Per CTA and row the result is one (max, sum-exp) pair and one sorted list
// of K keys, the same partials as k_head_tc, merged across CTAs by the row
// merge kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dt {
namespace {

// MH halves of 128 head rows (MMA M) x NV vocabulary entries (MMA N) per
// tile.  kPair: a CTA pair computes one M = 256 x N = NV tile with the
// two-CTA MMA; each CTA holds 128 of the rows (MH = 1) and NV / 2 of the
// tile's Wout rows, and its TMEM holds its 128 rows x NV columns.
//
// kHalfS (one CTA, at most 64 live rows): the stage holds a 64-row state box
// ([states 8 KB][Wout]); the MMA's A rows 64..127 then read the first Wout
// rows of the same stage, which only the never-read TMEM lanes 64..127 see.
// The smaller stage leaves room for one more in flight.
template <int MH, int NV, bool kPair = false, bool kHalfS = false>
struct RowsCfg {
  static constexpr int kRows = 128 * MH;             // head rows of this CTA (padded)
  static constexpr int kABytes = (kHalfS ? 64 : kRows) * kTileH * 2;  // states, 128 B rows
  static constexpr int kBRows = kPair ? NV / 2 : NV; // Wout rows of the tile in this CTA
  static constexpr int kBBytes = kBRows * kTileH * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kAccCols = MH * NV;           // TMEM columns of one accumulator
  static constexpr int kBufs = 2 * kAccCols <= 512 ? 2 : 1;
  static constexpr uint32_t kTmemCols = kBufs * kAccCols < 32 ? 32 : kBufs * kAccCols;
  // epilogue warpgroups: one per 128-row half (one CTA), or two per CTA of
  // a pair, each taking half of every tile's columns
  static constexpr int kColGroups = kPair ? 2 : 1;
  static constexpr int kEpiWarps = 4 * MH * kColGroups;
  static constexpr int kProducer = kEpiWarps;
  static constexpr int kMma = kEpiWarps + 1;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static_assert(NV == 128 || NV == 256, "vocabulary tile");
  static_assert(!kPair || (MH == 1 && NV == 256), "pair tile");
  static_assert(!kHalfS || (MH == 1 && !kPair), "64-row state box");
  static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "TMEM columns");
  // instruction descriptor: bf16 x bf16 -> fp32, K-major A and B, N = NV,
  // M = 128 (one CTA) or 256 (the pair)
  static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                     (static_cast<uint32_t>(NV >> 3) << 17) |
                                     (static_cast<uint32_t>((kPair ? 256 : 128) >> 4) << 24);
};

// ----------------------------------------------------- two-CTA (pair) PTX
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Cluster address of the variable at `p` in the CTA of the given rank.
__device__ __forceinline__ uint32_t map_to_rank(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// 2-D tiled load into this CTA's shared memory whose bytes complete on an
// mbarrier of either CTA of the pair (bar: cluster address).  x a multiple
// of 64 bf16 elements.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
// Arrive on an mbarrier of either CTA of the cluster (cluster address).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Once the pair's MMAs issued so far complete, arrive on the mbarrier at
// `bar`'s offset in the CTAs of `mask` (bit = rank in the pair).
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_u32(bar)), "h"(mask)
      : "memory");
}
template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)), "r"(NCOLS)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(NCOLS)
               : "memory");
}
// Bounded wait with cluster-scope acquire (the barrier receives arrivals
// from the other CTA of the pair); gives up like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* err,
                                                  long long limit) {
  const uint32_t a = smem_u32(bar);
  auto try_wait = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
  };
  if (try_wait()) return true;
  const long long lim = limit > 0 ? limit : kWaitLimitCycles;
  const long long t0 = clock64();
  while (!try_wait()) {
    if (clock64() - t0 > lim) {
      atomicOr(err, DT_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

constexpr int kRowsMaxStages = 8;

// Each thread of the warp reads 32 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Threshold value of a key bound: values below it cannot beat the key (0,
// the empty bound, lets every value through).
__device__ __forceinline__ float bound_value(uint64_t th) {
  return th == 0ull ? -INFINITY : key_value(th);
}

// Sorted insert (best first) of `key`, which beats the K-th key, into the
// list whose slot i is Lr[i * stride]; returns the new K-th key.
__device__ __noinline__ uint64_t list_insert_row(uint64_t* Lr, int stride, int K, uint64_t key) {
  int pos = K - 1;
  while (pos > 0) {
    const uint64_t prev = Lr[(pos - 1) * stride];
    if (prev >= key) break;
    Lr[pos * stride] = prev;
    --pos;
  }
  Lr[pos * stride] = key;
  return Lr[(K - 1) * stride];
}

// This CTA's best key of a row improved: raise its group's maximum (group =
// unit % K, unit = the CTA or CTA pair owning a vocabulary range), then the row's bound gth to the least of the K group maxima (K
// distinct keys at or above it; the new value stands in for this CTA's
// group).  One thread.
__device__ __noinline__ void publish_group_best(unsigned long long* gth, unsigned long long* gm,
                                                int K, int unit, uint64_t best) {
  const int mine = unit % K;
  atomicMax(gm + mine, best);
  uint64_t mn = ~0ull;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i < K) {
      uint64_t v = __ldcg(gm + i);
      if (i == mine) v = v > best ? v : best;
      mn = v < mn ? v : mn;
    }
  }
  if (mn != ~0ull && mn > 0ull) atomicMax(gth, mn);
}

constexpr float kLog2e = 1.4426950408889634f;

// A thread's top-K list of its head row, best first.  KR > 0: in KR
// registers (K <= KR), the list in the last K slots and slots before it
// holding ~0 (above every key, so never displaced) -- the K-th key is then
// always the last slot; KR == 0: K keys in shared memory, slot i at
// L[i * stride].  Empty slots hold key 0.
template <int KR>
struct RowList {
  uint64_t L[KR];
  int K;
  __device__ __forceinline__ void init(uint64_t*, int, int K_) {
    K = K_;
#pragma unroll
    for (int i = 0; i < KR; ++i) L[i] = i < KR - K ? ~0ull : 0ull;
  }
  __device__ __forceinline__ uint64_t best() const {
    uint64_t b = 0ull;
#pragma unroll
    for (int i = 0; i < KR; ++i) b = (L[i] != ~0ull && L[i] > b) ? L[i] : b;
    return b;
  }
  // insert a key that beats the K-th; returns the new K-th key
  __device__ __forceinline__ uint64_t insert(uint64_t key) {
#pragma unroll
    for (int i = KR - 1; i > 0; --i) {
      const uint64_t up = L[i - 1];
      L[i] = key > up ? up : (key > L[i] ? key : L[i]);
    }
    L[0] = key > L[0] ? key : L[0];
    return L[KR - 1];
  }
  __device__ __forceinline__ void store(uint64_t* dst) const {
#pragma unroll
    for (int i = 0; i < KR; ++i)
      if (i >= KR - K) dst[i - (KR - K)] = L[i];
  }
};

template <>
struct RowList<0> {
  uint64_t* L;
  int stride, K;
  __device__ __forceinline__ void init(uint64_t* l, int st, int K_) {
    L = l;
    stride = st;
    K = K_;
  }
  __device__ __forceinline__ uint64_t best() const { return L[0]; }
  __device__ __forceinline__ uint64_t insert(uint64_t key) {
    return list_insert_row(L, stride, K, key);
  }
  __device__ __forceinline__ void store(uint64_t* dst) const {
    for (int i = 0; i < K; ++i) dst[i] = L[i * stride];
  }
};

template <int MH, int NV, int KR, bool kPair, bool kHalfS>
__global__ void __launch_bounds__(RowsCfg<MH, NV, kPair, kHalfS>::kThreads, 1)
    k_head_rows(const __grid_constant__ CUtensorMap tmap_w,
                const __grid_constant__ CUtensorMap tmap_s, const TcParams p) {
  using C = RowsCfg<MH, NV, kPair, kHalfS>;
  static_assert(KR == 0 || KR == 8 || KR == 32, "register list capacity");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  uint8_t* stage_base = smem;  // stage: [states kABytes][Wout kBBytes]
  // top-K lists (K > 8 only), slot-major: slot i of list r at lists[i * kListRows + r]
  uint64_t* lists = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(S) * C::kStageBytes);
  constexpr int kListRows = C::kRows * C::kColGroups;  // lists per CTA: (column group, row)
  uint64_t* bars = lists + (KR > 0 ? 0 : static_cast<size_t>(p.K) * kListRows);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // unit = the CTA, or the CTA pair (cluster ranks 0 = leader, 1 = peer)
  const uint32_t rank = kPair ? cluster_rank() : 0u;
  const int unit = kPair ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int n_units = kPair ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  const int n_tiles = (p.rows + NV - 1) / NV;
  const int t_begin = static_cast<int>((static_cast<long long>(unit) * n_tiles) / n_units);
  const int t_end = static_cast<int>((static_cast<long long>(unit + 1) * n_tiles) / n_units);
  const int nk = p.H / kTileH;
  // each tile starts its contraction at a tile-dependent K step (spreads the
  // concurrent CTAs' reads over DRAM channels)
  auto kb_at = [&](int t, int i) {
    int j = i + (t * 5) % nk;
    if (j >= nk) j -= nk;
    return j;
  };

  if (warp == C::kMma) {
    if constexpr (kPair)
      tmem_alloc_pair<C::kTmemCols>(tmem_slot);  // the same columns in both CTAs
    else
      tmem_alloc<C::kTmemCols>(tmem_slot);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kPair ? 2 * C::kEpiWarps : C::kEpiWarps);  // pair: both CTAs' warps
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::kProducer && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_s);
  }
  if (KR == 0 && warp < C::kEpiWarps)
    for (int i = threadIdx.x; i < p.K * kListRows; i += 32 * C::kEpiWarps) lists[i] = 0ull;
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // both CTAs' barriers exist before either signals
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the states, z and the bounds come from earlier kernels
  pdl_trigger();

  if (warp == C::kProducer) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_s = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int t = t_begin; t < t_end && !*abort_flag; ++t) {
        for (int i = 0; i < nk; ++i) {
          const int kb = kb_at(t, i);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, p.wait_limit)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* dst = stage_base + static_cast<size_t>(stage) * C::kStageBytes;
          if constexpr (kPair) {
            // this CTA's 128 state rows and 128 Wout rows; both CTAs' bytes
            // complete on the leader's barrier, which the leader arms
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
            const uint32_t fb = map_to_rank(&full[stage], 0);
            tma_load_2d_pair(dst, &tmap_s, fb, kb * kTileH, static_cast<int>(rank) * 128, pol_s);
            const int wr = t * NV + static_cast<int>(rank) * 128;  // first weight row
            if (p.w_tiled)
              tma_load_2d_pair(dst + C::kABytes, &tmap_w, fb, 0, (wr / 128 * p.w_nk + kb) * 128,
                               pol_w);
            else
              tma_load_2d_pair(dst + C::kABytes, &tmap_w, fb, kb * kTileH, wr, pol_w);
          } else {
            mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
#pragma unroll
            for (int h = 0; h < MH; ++h)
              tma_load_2d(dst + h * (128 * 128), &tmap_s, &full[stage], kb * kTileH, h * 128,
                          pol_s);
#pragma unroll
            for (int j = 0; j < NV / 128; ++j) {
              const int wr = t * NV + j * 128;  // first weight row of the box
              if (p.w_tiled)
                tma_load_2d(dst + C::kABytes + j * (128 * 128), &tmap_w, &full[stage], 0,
                            (wr / 128 * p.w_nk + kb) * 128, pol_w);
              else
                tma_load_2d(dst + C::kABytes + j * (128 * 128), &tmap_w, &full[stage],
                            kb * kTileH, wr, pol_w);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every issued copy must have landed before the CTA may exit
      // (pair: the peer's copies complete on the leader's barriers, so the
      // leader drains both, and the final cluster barrier holds the peer)
      const long long first = issued > S ? issued - S : 0;
      for (long long n = first; n < issued && rank == 0; ++n) {
        const int s = static_cast<int>(n % S);
        if (!mbar_wait(&full[s], static_cast<uint32_t>((n / S) & 1), p.err)) break;
      }
      if (kPair && rank != 0 && *abort_flag) {
        // after a timeout the peer may have issued a stage the leader never
        // consumed (whose completion it cannot observe): hold the CTA for
        // ~50 us, far longer than a copy takes to land
        const long long t0 = clock64();
        while (clock64() - t0 < 100000) {
        }
      }
    }
  } else if (warp == C::kMma) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0 && rank == 0) {  // pair: the leader issues for both CTAs
      constexpr uint32_t idesc = C::kIdesc;
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int t = t_begin; t < t_end && !*abort_flag; ++t, ++it) {
        const int a = C::kBufs == 2 ? (it & 1) : 0;
        const uint32_t par = static_cast<uint32_t>(C::kBufs == 2 ? (it >> 1) : it) & 1u;
        const bool free_acc = kPair ? mbar_wait_cluster(&tempty[a], par ^ 1u, p.err, p.wait_limit)
                                    : mbar_wait(&tempty[a], par ^ 1u, p.err, p.wait_limit);
        if (!free_acc) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(a * C::kAccCols);
        bool ok = true;
        for (int i = 0; i < nk; ++i) {
          if (!mbar_wait(&full[stage], phase, p.err, p.wait_limit)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stage_base + static_cast<size_t>(stage) * C::kStageBytes);
          const uint32_t b_addr = a_addr + C::kABytes;
          if constexpr (kPair) {
#pragma unroll
            for (int k = 0; k < kTileH / 16; ++k)
              tc_mma_bf16_pair(d0, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32),
                               idesc, (i != 0 || k != 0) ? 1u : 0u);
            tc_commit_pair(&empty[stage], 3);  // the stage is free in both CTAs
          } else {
#pragma unroll
            for (int h = 0; h < MH; ++h) {
#pragma unroll
              for (int k = 0; k < kTileH / 16; ++k)
                tc_mma_bf16(d0 + static_cast<uint32_t>(h * NV),
                            smem_desc_sw128(a_addr + h * (128 * 128) + k * 32),
                            smem_desc_sw128(b_addr + k * 32), idesc, (i != 0 || k != 0) ? 1u : 0u);
            }
            tc_commit(&empty[stage]);
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kPair)
          tc_commit_pair(&tfull[a], 3);
        else
          tc_commit(&tfull[a]);
      }
      // all issued MMAs complete before TMEM is released
      if constexpr (kPair)
        tc_commit_pair(done, 1);
      else
        tc_commit(done);
      mbar_wait(done, 0, p.err);
    }
  } else {
    // --------------------------------------------------------- epilogue
    // thread = head row; its running (max, sum-exp), its top-K list (in
    // registers for K <= KR, else in shared memory) and K-th key
    const int gi = warp >> 2, wq = warp & 3;
    const int h = kPair ? 0 : gi;   // this thread's 128-row half (one CTA)
    const int cg = kPair ? gi : 0;  // this thread's half of the tile's columns (pair)
    constexpr int kChunks = NV / 32 / C::kColGroups;  // 32-column chunks per tile and thread
    const int slot = unit * C::kColGroups + cg;       // the partial slot of this (row, columns)
    const int row = static_cast<int>(rank) * 128 + h * 128 + wq * 32 + lane;
    const bool live = row < p.M;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int req = live ? row / p.rows_per_req : 0;
    const float* zrow = p.z + static_cast<long long>(req) * p.z_req_stride;
    const bool z_vec = (p.z_req_stride & 3) == 0 && (reinterpret_cast<uintptr_t>(p.z) & 15) == 0;
    const int K = p.K, V = p.rows;
    RowList<KR> list;
    list.init(lists + cg * C::kRows + h * 128 + wq * 32 + lane, kListRows, K);
    float m = -INFINITY, s = 0.f;
    uint64_t kth = 0ull;       // the list's K-th key (0 until it holds K keys)
    uint64_t best_pub = 0ull;  // this row's best key as last published
    bool bad = false;
    // the base logits of one 32-entry chunk (loaded one chunk ahead)
    auto load_z = [&](int vb, float (&zv)[32]) {
      const int nv = V - vb < 32 ? V - vb : 32;
      if (live && z_vec && nv == 32) {
        const float4* z4 = reinterpret_cast<const float4*>(zrow + vb);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 u = __ldg(z4 + j);
          zv[4 * j] = u.x;
          zv[4 * j + 1] = u.y;
          zv[4 * j + 2] = u.z;
          zv[4 * j + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) zv[j] = (live && j < nv) ? __ldg(zrow + vb + j) : 0.f;
      }
    };
    float zn[32];
    if (t_begin < t_end) load_z(t_begin * NV + cg * kChunks * 32, zn);
    int it = 0;
    for (int t = t_begin; t < t_end; ++t, ++it) {
      const int a = C::kBufs == 2 ? (it & 1) : 0;
      const uint32_t par = static_cast<uint32_t>(C::kBufs == 2 ? (it >> 1) : it) & 1u;
      // the row's global bound, read before the wait
      uint64_t gb = 0ull;
      if (p.gth && live) gb = __ldcg(p.gth + row);
      int okl = 0;
      if (lane == 0)
        okl = (!*abort_flag && (kPair ? mbar_wait_cluster(&tfull[a], par, p.err, p.wait_limit)
                                      : mbar_wait(&tfull[a], par, p.err, p.wait_limit)))
                  ? 1
                  : 0;
      if (__shfl_sync(kFullMask, okl, 0) == 0) {  // the warp leaves together
        if (lane == 0) *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + lane_base + static_cast<uint32_t>(a * C::kAccCols + h * NV);
      const uint64_t th0 = kth > gb ? kth : gb;
      uint64_t th = th0;
      float thv = bound_value(th);
#pragma unroll 1
      for (int q = 0; q < kChunks; ++q) {
        const int qq = cg * kChunks + q;  // chunk within the tile
        const int vb = t * NV + qq * 32;
        int nv = V - vb < 32 ? V - vb : 32;  // valid entries of this chunk
        nv = nv < 0 ? 0 : nv;
        float x[32];
        __syncwarp();
        tmem_ld32(tb + static_cast<uint32_t>(qq * 32), x);  // the whole warp, live or not
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] += zn[j];
        {  // next chunk's base logits, in flight while this one is processed
          const int vn = q + 1 < kChunks ? vb + 32 : (t + 1) * NV + cg * kChunks * 32;
          if (q + 1 < kChunks || t + 1 < t_end) load_z(vn, zn);
        }
        if (!live) continue;
        // x * 0 is NaN exactly for NaN and +-inf: one probe per value
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) pr[j & 3] = fmaf(x[j], 0.f, pr[j & 3]);
        if (nv == 32 && (pr[0] + pr[1]) + (pr[2] + pr[3]) == 0.f) {
          // all 32 finite: four independent chains for the maximum and sum
          float c4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
          for (int j = 4; j < 32; ++j) c4[j & 3] = fmaxf(c4[j & 3], x[j]);
          const float cm = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
          if (cm > m) {
            s *= fast_exp(m - cm);  // 0 while m is -inf (s is 0 then too)
            m = cm;
          }
          const float ml = m * kLog2e;
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 32; ++j) s4[j & 3] += exp2f(fmaf(x[j], kLog2e, -ml));
          s += (s4[0] + s4[1]) + (s4[2] + s4[3]);
        } else {
          // a tail chunk or a non-finite value: per-value checks
          float cm = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (j < nv) {
              if (x[j] != x[j] || x[j] == INFINITY) bad = true;
              if (x[j] > -INFINITY && x[j] < INFINITY) cm = fmaxf(cm, x[j]);
            }
          }
          if (cm > m) {
            s *= fast_exp(m - cm);
            m = cm;
          }
          if (m != -INFINITY) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nv && x[j] > -INFINITY && x[j] < INFINITY) s += fast_exp(x[j] - m);
          }
        }
        // top-K: a value below the bound's value cannot enter.  While the
        // list is short the chunk bounds itself: the least of G >= K group
        // maxima (groups of 32 / G values) has G values at or above it.
        float cb = -INFINITY;
        if (kth == 0ull && K <= 16) {
          float pm[16];  // maxima of the pairs of valid, non-NaN values
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            pm[i] = -INFINITY;
            if (2 * i < nv && x[2 * i] == x[2 * i]) pm[i] = x[2 * i];
            if (2 * i + 1 < nv && x[2 * i + 1] == x[2 * i + 1]) pm[i] = fmaxf(pm[i], x[2 * i + 1]);
          }
          cb = INFINITY;
          if (K <= 8) {  // 8 groups of 4
#pragma unroll
            for (int i = 0; i < 8; ++i) cb = fminf(cb, fmaxf(pm[2 * i], pm[2 * i + 1]));
          } else {  // 16 groups of 2
#pragma unroll
            for (int i = 0; i < 16; ++i) cb = fminf(cb, pm[i]);
          }
        }
        const float thv_e = fmaxf(thv, cb);
        uint32_t cand = 0u;  // the chunk's candidates, one bit per entry
#pragma unroll
        for (int j = 0; j < 32; ++j) cand |= (j < nv && x[j] >= thv_e) ? 1u << j : 0u;
        while (cand) {  // rare: one insertion site, the value picked by index
          const int j = __ffs(cand) - 1;
          cand &= cand - 1u;
          float xj = x[0];
#pragma unroll
          for (int i = 1; i < 32; ++i) xj = j == i ? x[i] : xj;
          const uint64_t key = make_key(xj, static_cast<uint32_t>(vb + j));
          if (key > th) {  // exact test against the bound as it stands now
            kth = list.insert(key);
            th = kth > gb ? kth : gb;
          }
        }
        thv = bound_value(th);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair && rank != 0)
          mbar_arrive_cluster(map_to_rank(&tempty[a], 0));  // the leader's accumulator barrier
        else
          mbar_arrive(&tempty[a]);
      }
      // publish improved bounds: the list's K-th key (once the list is
      // full) and this CTA's best key for its group
      if (p.gth && live && kth > th0) atomicMax(p.gth + row, kth);
      if (p.gth && p.gmx && live) {
        const uint64_t best = list.best();
        if (best > best_pub) {
          publish_group_best(p.gth + row, p.gmx + static_cast<size_t>(row) * 32, K, slot, best);
          best_pub = best;
        }
      }
    }
    if (live) {
      const int cta = slot;
      p.pm[static_cast<size_t>(row) * p.cta_stride + cta] = m;
      p.ps[static_cast<size_t>(row) * p.cta_stride + cta] = s;
      list.store(p.ptop + (static_cast<size_t>(row) * p.list_stride + cta) * K);
    }
    if (bad) atomicOr(p.err, DT_ERR_NONFINITE);
  }

  tc_fence_before();
  __syncthreads();
  // pair: neither CTA leaves (or frees its TMEM) while the other may still
  // signal it or the leader's MMAs may still use its memory
  if constexpr (kPair) cluster_sync_all();
  if (warp == C::kMma) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair<C::kTmemCols>(tmem_base);
    else
      tmem_dealloc<C::kTmemCols>(tmem_base);
  }
}

template <int MH, int NV, int KR, bool kPair, bool kHalfS>
cudaError_t launch_rows(const CUtensorMap& tw, const CUtensorMap& ts, const TcParams& p, int units,
                        cudaStream_t st) {
  using C = RowsCfg<MH, NV, kPair, kHalfS>;
  const size_t lists = KR > 0 ? 0 : static_cast<size_t>(p.K) * C::kRows * C::kColGroups * 8;
  const size_t fixed = 1024 + lists + 64 * 8 + 64;
  const size_t budget = 227 * 1024 - 512;  // no static shared memory in this kernel
  int stages = budget > fixed ? static_cast<int>((budget - fixed) / C::kStageBytes) : 0;
  const int cap = p.max_stages > 0 ? p.max_stages : kRowsMaxStages;
  if (stages > cap) stages = cap;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  TcParams q = p;
  q.stages = stages;
  const size_t smem = fixed + static_cast<size_t>(stages) * C::kStageBytes;
  if constexpr (kPair)
    return launch_kernel_cluster(k_head_rows<MH, NV, KR, kPair, kHalfS>, dim3(2 * units),
                                 dim3(C::kThreads), smem, st, q.pdl != 0, 2, tw, ts, q);
  else
    return launch_kernel(k_head_rows<MH, NV, KR, kPair, kHalfS>, dim3(units), dim3(C::kThreads),
                         smem, st, q.pdl != 0, tw, ts, q);
}

// The top-K lists: in registers for K <= 8; for K <= 32 as well where one
// warpgroup of epilogue threads leaves the registers (one 128-row CTA);
// else in shared memory.
template <int MH, int NV, bool kPair, bool kHalfS = false>
cudaError_t launch_rows_k(const CUtensorMap& tw, const CUtensorMap& ts, const TcParams& p,
                          int units, cudaStream_t st) {
  if (p.K <= 8) return launch_rows<MH, NV, 8, kPair, kHalfS>(tw, ts, p, units, st);
  if constexpr (MH == 1 && !kPair)
    if (p.K <= 32) return launch_rows<MH, NV, 32, kPair, kHalfS>(tw, ts, p, units, st);
  return launch_rows<MH, NV, 0, kPair, kHalfS>(tw, ts, p, units, st);
}

template <int MH, int NV, bool kPair, bool kHalfS = false>
cudaError_t set_rows_attrs() {
  cudaError_t e = set_max_dynamic_smem(k_head_rows<MH, NV, 8, kPair, kHalfS>);
  if constexpr (MH == 1 && !kPair)
    if (e == cudaSuccess) e = set_max_dynamic_smem(k_head_rows<MH, NV, 32, kPair, kHalfS>);
  return e != cudaSuccess ? e : set_max_dynamic_smem(k_head_rows<MH, NV, 0, kPair, kHalfS>);
}

int g_max_pairs = 0;  // CTA pairs of the pair kernel that can be resident together

}  // namespace

cudaError_t init_head_rows_attrs() {
  cudaError_t e;
  if ((e = set_rows_attrs<1, 128, false>()) != cudaSuccess) return e;
  if ((e = set_rows_attrs<2, 128, false>()) != cudaSuccess) return e;
  if ((e = set_rows_attrs<1, 256, false>()) != cudaSuccess) return e;
  if ((e = set_rows_attrs<2, 256, false>()) != cudaSuccess) return e;
  if ((e = set_rows_attrs<1, 256, true>()) != cudaSuccess) return e;
  if ((e = set_rows_attrs<1, 256, false, true>()) != cudaSuccess) return e;
  // resident clusters of two at the largest shared-memory footprint
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(RowsCfg<1, 256, true>::kThreads);
  cfg.dynamicSmemBytes = 227 * 1024 - 2048;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, k_head_rows<1, 256, 0, true, false>, &cfg);
  if (e != cudaSuccess) return e;
  g_max_pairs = n;
  return cudaSuccess;
}

cudaError_t launch_head_rows(int M, int nv, bool pair, const CUtensorMap& tw, const CUtensorMap& ts,
                             const TcParams& p, int units, cudaStream_t st, int* units_used) {
  if (M < 1 || M > kMaxRows || (nv != 128 && nv != 256)) return cudaErrorInvalidValue;
  if (pair) {  // 129..256 rows over a CTA pair, 256-entry vocabulary tiles
    if (M <= 128 || nv != 256) return cudaErrorInvalidValue;
    if (units > g_max_pairs) units = g_max_pairs;
    if (units < 1) return cudaErrorInvalidConfiguration;
    *units_used = 2 * units;  // partial slots: two column halves per pair
    return launch_rows_k<1, 256, true>(tw, ts, p, units, st);
  }
  *units_used = units;
  if (p.s_rows == 64) {  // 64-row state boxes (the map's box), 256-entry tiles
    if (M > 64 || nv != 256) return cudaErrorInvalidValue;
    return launch_rows_k<1, 256, false, true>(tw, ts, p, units, st);
  }
  if (M <= 128)
    return nv == 128 ? launch_rows_k<1, 128, false>(tw, ts, p, units, st)
                     : launch_rows_k<1, 256, false>(tw, ts, p, units, st);
  return nv == 128 ? launch_rows_k<2, 128, false>(tw, ts, p, units, st)
                   : launch_rows_k<2, 256, false>(tw, ts, p, units, st);
}

}  // namespace dt
