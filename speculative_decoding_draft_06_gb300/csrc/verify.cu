// The verification consumer of a built tree: one attention layer of the
// target over the prefix and the draft tree with the emitted ancestor mask,
// and the longest accepted prefix under the target's predictions
// ("DARTree: Teaching a Chain-Trained Corrector to Think in Trees", Core
// Mechanism: with the tree and its mask a single target forward verifies
// all branches, and the longest prefix the target agrees with is kept; "Technische Samenvatting: DARTree", Methodologie 2, Verificatie).
//
// Tree attention on the 5th-generation tensor cores.  A CTA owns 128 query
// rows (one TMEM lane each) of one request and one key/value head, and a
// share of the key range (the keys are split over CTAs until one wave fills
// the GPU; the splits of a query tile are one thread-block cluster, which
// exchanges the partial rows in distributed shared memory, each split
// combining the rows it owns).
// Query row q of a key/value head is (node q / g, query head hk * g + q % g),
// g = Hq / Hkv.  Row 0 (the root) sees the prefix; node i >= 1 sees the
// prefix and the tree nodes of mask row i - 1.
//
// Warp roles (320 threads): warps 0-7 softmax (two warpgroups; a thread
// owns a query row = TMEM lane, its group half of each key tile and half of
// the head dimensions of O), warp 8 TMA producer (the query tile, and
// 128-key tiles of K and of the blocked, transposed value cache, 128-byte
// swizzle, two stages whose keys and values have separate barriers), warp 9
// TMEM allocator + single-thread MMA issuer.
// One pass over the CTA's keys with an online softmax: S = Q K^T (M = 128
// rows, N = 128 keys, K = 128 head dims) into double-buffered TMEM, P =
// 2^(s - m) rounded to bf16 and stored to tensor memory (double-buffered;
// each lane holds its row's weights, two keys per 32-bit column), O += P V
// (M = 128, N = 128 head dims, K = 128 keys; A = P read from tensor memory,
// B = the value tile in shared memory) in TMEM.  The reference maximum m is raised only
// when a tile beats it by more than 8 (base 2), which rescales O in TMEM.
// The rounded weights also form the normaliser, so O is an exact convex
// combination of the visible values with weights within 2^-8 of the exact
// softmax.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "../../include/dartree.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dt {
namespace {

constexpr int kDh = 128;           // head dimension (fixed)
constexpr int kQRows = 128;        // query rows per CTA (TMEM lanes)
constexpr int kKeys = 128;         // keys per tile
constexpr int kVBlock = 64;        // keys per value-cache block (one swizzle atom)
constexpr int kPBufs = 2;          // P buffers in tensor memory
constexpr int kAttnThreads = 320;
constexpr int kSoftmaxThreads = 256;   // two warpgroups, one per half of each key tile
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kHalf = kKeys / 2;       // keys of a tile per warpgroup
constexpr int kStages = 2;
constexpr int kMaxSplit = 8;  // key splits of a query tile: one (portable) cluster
constexpr int kQBytes = kQRows * kDh * 2;        // 32 KB: 2 swizzle atoms of 64 head dims
constexpr int kKBytes = kKeys * kDh * 2;         // 32 KB: 2 atoms of 64 head dims
constexpr int kVBytes = kDh * kKeys * 2;         // 32 KB: 2 blocks of 128 head dims x 64 keys
constexpr int kStageBytes = kKBytes + kVBytes;
constexpr uint32_t kTmemCols = 512;  // S0 [0,128) S1 [128,256) O [256,384) P0 [384,448) P1 [448,512)
constexpr uint32_t kColO = 256;
constexpr uint32_t kColP = 384;      // P buffer b: 64 columns of bf16 pairs (128 keys) per lane

struct AttnParams {
  int Lp, B, L, Hq, Hkv, g, words, rows;  // L = Lp + B keys; rows = (B + 1) * g
  float scale_log2;                       // scale * log2(e)
  const uint16_t* Q;                      // [R][B+1][Hq][dh]
  const uint32_t* mask;                   // [R][B][words]
  float* O;                               // [R][B+1][Hq][dh]
  uint16_t* O16;                          // same, bf16 bits, or null
  int* err;
  long long wait_limit;
  int n_split, q_tiles;                   // n_split > 1: a cluster of n_split CTAs per query tile
  int q_tma;                              // the query tile by TMA (128 % g == 0), else by the threads
  unsigned long long g_magic;             // ceil(2^32 / g): q / g = (q g_magic) >> 32 for every row q
};

// Thread-block cluster access (the key splits of a query tile).
__device__ __forceinline__ uint32_t cl_addr(const void* p, int rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(a)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(rank));
  return a;
}
__device__ __forceinline__ void cl_st_f4(uint32_t a, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void cl_st_f2(uint32_t a, float2 v) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y)
               : "memory");
}
__device__ __forceinline__ void cl_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 2^x (approximate hardware exp2; -inf -> +0).
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> packed bf16 pair, round to nearest even: lo in the low half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// 4-D tiled load (x, y, z, w) into shared memory, bytes completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Byte offset of 16-byte granule gr (of 8 in a 128-byte row) of row r in a
// 128-byte swizzled atom.
__device__ __forceinline__ uint32_t sw128(int r, int gr) {
  return static_cast<uint32_t>(r * 128 + ((gr ^ (r & 7)) << 4));
}

constexpr int kOPitch = kDh + 4;  // floats per staged O row (16-byte rows spread over the banks)

// Output row q of a query tile (node q / g, query head hk g + q % g; the
// quotient by a multiply with the rounded-up reciprocal, exact for the
// row counts the host admits).
__device__ __forceinline__ size_t out_row(const AttnParams& p, int r, int hk, int q) {
  const int node = static_cast<int>((static_cast<unsigned long long>(q) * p.g_magic) >> 32);
  const int h = hk * p.g + (q - node * p.g);
  return ((static_cast<size_t>(r) * (p.B + 1) + node) * p.Hq + h) * kDh;
}

// One row of 128 head dims by one warp: lane i writes dims 4i .. 4i + 3
// (512 contiguous bytes of fp32, 256 of bf16).
__device__ __forceinline__ void store_row(const AttnParams& p, size_t base, float4 v) {
  const int lane = threadIdx.x & 31;
  *reinterpret_cast<float4*>(p.O + base + 4 * lane) = v;
  if (p.O16)
    *reinterpret_cast<uint2*>(p.O16 + base + 4 * lane) =
        make_uint2(cvt_bf16x2(v.x, v.y), cvt_bf16x2(v.z, v.w));
}

// Each query row's base-2 (max, sum) of this CTA's keys, as finish_tile
// staged it.
__shared__ float2 sh_ml[kQRows];

// The end of a query tile's keys in this CTA (the 256 softmax threads;
// thread = (row, half of the head dims), holding its unnormalised O half
// and the row's max m and sum l in base 2).  The rows are staged in shared
// memory (sO, the pipeline's stage buffers, free once the last product has
// landed) so that each warp then moves whole rows with 512-byte accesses.
// One split: O = O_row / l, stored here.  Several: the cluster's exchange
// and combine follow (split_exchange, split_combine).
__device__ __forceinline__ void finish_tile(const AttnParams& p, int r, int hk, int qt, int row,
                                            int half, const float (&o)[kDh / 2], float m, float l,
                                            float* sO) {
  constexpr int kOH = kDh / 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* dst = sO + row * kOPitch + half * kOH;
#pragma unroll
  for (int i = 0; i < kOH; i += 4)
    *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
  if (half == 0) sh_ml[row] = make_float2(m, l);
  asm volatile("bar.sync 1, 256;" ::: "memory");
  if (p.n_split > 1) return;
  const int q0 = qt * kQRows;
  for (int rr = warp; rr < kQRows; rr += 8) {
    if (q0 + rr >= p.rows) break;
    const float lr = sh_ml[rr].y;
    const float inv = lr > 0.f ? 1.f / lr : 0.f;
    float4 v = *reinterpret_cast<const float4*>(sO + rr * kOPitch + 4 * lane);
    v.x *= inv;
    v.y *= inv;
    v.z *= inv;
    v.w *= inv;
    store_row(p, out_row(p, r, hk, q0 + rr), v);
  }
}

// Several splits: split s owns rows [s RS, (s + 1) RS) of the query tile
// (RS = ceil(128 / n)).  Every split sends the rows the others own -- its
// unnormalised O row and (m, l) -- into the owner's receive buffer in
// shared memory (distributed shared memory; slot s of the owner's n - 1
// slots, the owner's own split skipped).  The 256 softmax threads, after
// the cluster has started.
__device__ __forceinline__ void split_exchange(const AttnParams& p, int qt, int split,
                                               const float* sO, float* recv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n_split, rs = (kQRows + n - 1) / n;
  const int q0 = qt * kQRows;
  const int live = p.rows - q0 < kQRows ? p.rows - q0 : kQRows;  // rows of the tile that exist
  float2* recv_ml = reinterpret_cast<float2*>(recv + static_cast<size_t>(n - 1) * rs * kDh);
  for (int d = 0; d < n; ++d) {
    if (d == split) continue;
    const int slot = split < d ? split : split - 1;
    const int b = d * rs;
    const int cnt = (b + rs < live ? b + rs : live) - b;
    // the slot's rows in rank d's receive buffer (one address map per rank)
    const uint32_t dst = cl_addr(recv + static_cast<size_t>(slot) * rs * kDh + 4 * lane, d);
    const uint32_t dst_ml = cl_addr(recv_ml + slot * rs, d);
    for (int i = warp; i < cnt; i += 8) {
      const float4 v = *reinterpret_cast<const float4*>(sO + (b + i) * kOPitch + 4 * lane);
      cl_st_f4(dst + static_cast<uint32_t>(i * kDh * 4), v);
      if (lane == 0) cl_st_f2(dst_ml + static_cast<uint32_t>(i * 8), sh_ml[b + i]);
    }
  }
}

// The rows this split owns, from every split's (m, l, O) in split order
// (deterministic):
//   M = max_s m_s, L = sum_s l_s 2^(m_s - M), O = sum_s O_s 2^(m_s - M) / L.
// After the cluster barrier that follows every split's exchange.  N = the
// split count, so that the per-row work is straight-line code: every
// split's rows are a base and a row stride (the own split's in sO and
// sh_ml, the others' in the receive buffer).
template <int N>
__device__ __forceinline__ void combine_rows(const AttnParams& p, int r, int hk, int qt, int split,
                                             const float* sO, const float* recv) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int rs = (kQRows + N - 1) / N;
  const int q0 = qt * kQRows;
  const int live = p.rows - q0 < kQRows ? p.rows - q0 : kQRows;
  const int b = split * rs;
  const int cnt = (b + rs < live ? b + rs : live) - b;
  const float2* recv_ml = reinterpret_cast<const float2*>(recv + static_cast<size_t>(N - 1) * rs * kDh);
  const float* vb[N];
  int vs[N];
  const float2* mb[N];
#pragma unroll
  for (int s2 = 0; s2 < N; ++s2) {
    const bool own = s2 == split;
    const int slot = s2 < split ? s2 : s2 - 1;
    vb[s2] = own ? sO + b * kOPitch + 4 * lane : recv + static_cast<size_t>(slot) * rs * kDh + 4 * lane;
    vs[s2] = own ? kOPitch : kDh;
    mb[s2] = own ? sh_ml + b : recv_ml + slot * rs;
  }
  for (int i = warp; i < cnt; i += 8) {
    float2 ml[N];
    float4 v[N];
#pragma unroll
    for (int s2 = 0; s2 < N; ++s2) {
      ml[s2] = mb[s2][i];
      v[s2] = *reinterpret_cast<const float4*>(vb[s2] + i * vs[s2]);
    }
    float M = ml[0].x;
#pragma unroll
    for (int s2 = 1; s2 < N; ++s2) M = fmaxf(M, ml[s2].x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s2 = 0; s2 < N; ++s2) {
      const float f = ml[s2].x == -INFINITY ? 0.f : fast_ex2(ml[s2].x - M);
      L += ml[s2].y * f;
      acc.x += v[s2].x * f;
      acc.y += v[s2].y * f;
      acc.z += v[s2].z * f;
      acc.w += v[s2].w * f;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    store_row(p, out_row(p, r, hk, q0 + b + i),
              make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
  }
}

__device__ __forceinline__ void split_combine(const AttnParams& p, int r, int hk, int qt,
                                              int split, const float* sO, const float* recv) {
  switch (p.n_split) {
    case 2: combine_rows<2>(p, r, hk, qt, split, sO, recv); break;
    case 3: combine_rows<3>(p, r, hk, qt, split, sO, recv); break;
    case 4: combine_rows<4>(p, r, hk, qt, split, sO, recv); break;
    case 5: combine_rows<5>(p, r, hk, qt, split, sO, recv); break;
    case 6: combine_rows<6>(p, r, hk, qt, split, sO, recv); break;
    case 7: combine_rows<7>(p, r, hk, qt, split, sO, recv); break;
    default: combine_rows<8>(p, r, hk, qt, split, sO, recv); break;
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    k_tree_attention(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_vt, const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sStage = sQ + kQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStage + kStages * kStageBytes);
  // keys and values of a stage have their own barriers: the keys are free
  // once QK^T has read them, two tiles before the values
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + kStages;
  uint64_t* v_full = k_empty + kStages;
  uint64_t* v_empty = v_full + kStages;
  uint64_t* s_full = v_empty + kStages;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;   // [2]
  uint64_t* p_empty = p_full + 2;   // [2]
  uint64_t* o_done = p_empty + 2;
  uint64_t* q_full = o_done + 1;    // the query tile's copies (q_tma)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_full + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // several key splits: the rows this split owns, as the others send them
  float* recv = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.n_split > 1) cl_arrive_relaxed();  // (waited on before the first remote store)
  const int r = blockIdx.z, hk = blockIdx.y;
  const int qt = blockIdx.x / p.n_split, split = blockIdx.x % p.n_split;
  const int q0 = qt * kQRows;
  // key tiles of this CTA: the query tile's largest node bounds the tree
  // keys any of its rows can see
  const int last_node = min(p.B, (q0 + kQRows - 1) / p.g);
  const int t_all = (p.Lp + last_node + kKeys - 1) / kKeys;
  const int t_beg = split * t_all / p.n_split, t_end = (split + 1) * t_all / p.n_split;
  const int nt = t_end - t_beg;

  // the keys, and the values, of the CTA's key tile f into its stage
  auto issue_k = [&](int f) {
    const int t = t_beg + f;
    const int stage = f % kStages;
    uint8_t* k_dst = sStage + stage * kStageBytes;
    mbar_arrive_expect_tx(&k_full[stage], kKBytes);
    tma_load_4d(k_dst, &tm_k, &k_full[stage], 0, t * kKeys, hk, r);
    tma_load_4d(k_dst + kKBytes / 2, &tm_k, &k_full[stage], 64, t * kKeys, hk, r);
  };
  auto issue_v = [&](int f) {
    const int t = t_beg + f;
    const int stage = f % kStages;
    uint8_t* v_dst = sStage + stage * kStageBytes + kKBytes;
    mbar_arrive_expect_tx(&v_full[stage], kVBytes);
    tma_load_4d(v_dst, &tm_vt, &v_full[stage], 0, 0, 2 * t, hk + p.Hkv * r);
    tma_load_4d(v_dst + kVBytes / 2, &tm_vt, &v_full[stage], 0, 0, 2 * t + 1, hk + p.Hkv * r);
  };
  const int n_pre = nt < kStages ? nt : kStages;  // tiles loaded during the setup

  if (warp == kMmaWarp) tmem_alloc<kTmemCols>(tmem_slot);
  if (warp == kProducerWarp && lane == 0) {
    // the producer's own barriers, and the first stages' copies while the
    // query tile is staged (the stages start empty)
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(q_full, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
    if (p.q_tma) {
      // rows (node, query head) of the tile: a box of 128 / g nodes by the
      // g query heads of this key/value head, per 64 head dims
      const int nodes = kQRows / p.g;
      mbar_arrive_expect_tx(q_full, kQBytes);
      tma_load_4d(sQ, &tm_q, q_full, 0, hk * p.g, qt * nodes, r);
      tma_load_4d(sQ + kQRows * 128, &tm_q, q_full, 64, hk * p.g, qt * nodes, r);
    }
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_vt);
    for (int f = 0; f < n_pre; ++f) {
      issue_k(f);
      issue_v(f);
    }
  }
  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], 8);  // one arrival per softmax warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&p_full[b], 8);
      mbar_init(&p_empty[b], 1);
    }
    mbar_init(o_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // otherwise the query tile, written by the softmax threads in the
  // swizzled layout
  if (!p.q_tma && threadIdx.x < kQRows) {
    const int row = threadIdx.x, q = q0 + row;
    const bool valid = q < p.rows;
    const uint4* src = nullptr;
    if (valid) {
      const int node = q / p.g, h = hk * p.g + q % p.g;
      src = reinterpret_cast<const uint4*>(
          p.Q + ((static_cast<size_t>(r) * (p.B + 1) + node) * p.Hq + h) * kDh);
    }
#pragma unroll
    for (int gi = 0; gi < 16; ++gi) {
      const uint4 v = valid ? __ldg(src + gi) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(sQ + (gi >> 3) * (kQRows * 128) + sw128(row, gi & 7)) = v;
    }
    fence_proxy_async_smem();  // visible to the tensor cores
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      long long k_issued = n_pre, v_issued = n_pre;
      for (int f = n_pre; f < nt && !*abort_flag; ++f) {
        const int stage = f % kStages;
        const uint32_t ph = static_cast<uint32_t>((f / kStages) & 1);
        // the keys once QK^T of tile f - 2 has read its stage's, then the
        // values once the product of tile f - 2 has
        if (!mbar_wait(&k_empty[stage], ph ^ 1u, p.err, p.wait_limit)) {
          *abort_flag = 1;
          break;
        }
        issue_k(f);
        ++k_issued;
        if (!mbar_wait(&v_empty[stage], ph ^ 1u, p.err, p.wait_limit)) {
          *abort_flag = 1;
          break;
        }
        issue_v(f);
        ++v_issued;
      }
      // drain: every issued copy must have landed before the CTA may exit
      for (int kv = 0; kv < 2; ++kv) {
        const long long issued = kv == 0 ? k_issued : v_issued;
        uint64_t* full = kv == 0 ? k_full : v_full;
        const long long first = issued > kStages ? issued - kStages : 0;
        for (long long n = first; n < issued; ++n) {
          const int s = static_cast<int>(n % kStages);
          if (!mbar_wait(&full[s], static_cast<uint32_t>((n / kStages) & 1), p.err)) break;
        }
      }
      if (p.q_tma) mbar_wait(q_full, 0, p.err);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_m128<kKeys>();
      constexpr uint32_t idesc_o = idesc_bf16_m128<kDh>();
      const uint32_t q_addr = smem_u32(sQ);
      bool ok = true;
      auto wait = [&](uint64_t* bar, uint32_t par) {
        if (ok && !*abort_flag && mbar_wait(bar, par, p.err, p.wait_limit)) return true;
        ok = false;
        *abort_flag = 1;
        return false;
      };
      // S[b] = Q K^T for the tile in stage `stage`
      auto issue_s = [&](int u, int stage) {
        const int b = u & 1;
        if (!wait(&s_empty[b], (static_cast<uint32_t>(u >> 1) & 1u) ^ 1u)) return false;
        if (!wait(&k_full[stage], static_cast<uint32_t>((u / kStages) & 1))) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(sStage + stage * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < kDh / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32u;  // 16 head dims within the 128-byte row
          tc_mma_bf16(tmem_base + static_cast<uint32_t>(b * kKeys),
                      smem_desc_sw128(q_addr + (kk >> 2) * (kQRows * 128) + off),
                      smem_desc_sw128(k_addr + (kk >> 2) * (kKeys * 128) + off), idesc_s,
                      kk != 0 ? 1u : 0u);
        }
        tc_commit(&s_full[b]);
        tc_commit(&k_empty[stage]);  // the keys are read once the scores are done
        return true;
      };
      // O += P V for tile j (its stage), then release P and the stage
      auto issue_o = [&](int j) {
        const int stage = j % kStages, pb = j % kPBufs;
        if (!wait(&p_full[pb], static_cast<uint32_t>(j / kPBufs) & 1u)) return false;
        if (!wait(&v_full[stage], static_cast<uint32_t>((j / kStages) & 1))) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(sStage + stage * kStageBytes + kKBytes);
        const uint32_t pa = tmem_base + kColP + static_cast<uint32_t>(pb * (kKeys / 2));
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32u;  // 16 keys within the 128-byte row
          // A = P from tensor memory: keys 16 kk .. 16 kk + 15 are 8 columns
          tc_mma_bf16_ta(tmem_base + kColO, pa + static_cast<uint32_t>(kk * 8),
                         smem_desc_sw128(v_addr + (kk >> 2) * (kDh * 128) + off), idesc_o,
                         (j != 0 || kk != 0) ? 1u : 0u);
        }
        tc_commit(&p_empty[pb]);
        tc_commit(&v_empty[stage]);
        return true;
      };
      if (p.q_tma && nt > 0) wait(q_full, 0);
      // scores of tile j, then the product of tile j - 1
      for (int j = 0; j < nt && ok; ++j) {
        if (!issue_s(j, j % kStages)) break;
        if (j > 0 && !issue_o(j - 1)) break;
      }
      if (ok && nt > 0) issue_o(nt - 1);
      tc_commit(o_done);
      mbar_wait(o_done, 0, p.err);
    }
  } else {
    // -------------------------------------------------------- softmax
    __shared__ float red[2][kQRows];      // per-row exchange between the two groups
    __shared__ float red2[2][2][kQRows];  // per-tile row maxima (double-buffered)
    __shared__ int stop_slot[2][8];       // per-tile stop marks of the 8 warps
    const int wg = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane, q = q0 + row;
    const int node = q < p.rows ? q / p.g : 0;
    const uint32_t* mrow =
        (q < p.rows && node >= 1) ? p.mask + (static_cast<size_t>(r) * p.B + node - 1) * p.words
                                  : nullptr;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const int col0 = wg * kHalf;  // this group's keys within a tile
    // the row's mask words covering this group's half of tile t (three
    // words from the one holding the half's first tree key; zero for the
    // root row and beyond the row)
    auto mask_words = [&](int t, uint32_t (&w)[3]) {
      w[0] = w[1] = w[2] = 0u;
      const int j0 = t * kKeys + col0;
      if (mrow && j0 + kHalf > p.Lp) {
        const int wb = (j0 > p.Lp ? j0 - p.Lp : 0) >> 5;
#pragma unroll
        for (int k = 0; k < 3; ++k)
          if (wb + k < p.words) w[k] = __ldg(mrow + wb + k);
      }
    };
    // scaled scores of this group's half of tile t, -inf where not visible
    auto load_s = [&](int u, int t, const uint32_t (&w)[3], float (&s)[kHalf]) {
      const int b = u & 1;
      const uint32_t taddr = tmem_base + lane_base + static_cast<uint32_t>(b * kKeys + col0);
#pragma unroll
      for (int c = 0; c < kHalf; c += 16) {
        float x[16];
        tmem_ld16(taddr + c, x);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[c + i] = x[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[b]);  // S[b] may be overwritten
      const int j0 = t * kKeys + col0;
      if (j0 + kHalf <= p.Lp) {
#pragma unroll
        for (int c = 0; c < kHalf; ++c) s[c] *= p.scale_log2;
      } else {
        // visibility of keys j0 .. j0 + 63 as one 64-bit word: the np prefix
        // keys, then the mask bits from tree index tf on, cut at L
        const int np = p.Lp > j0 ? p.Lp - j0 : 0;  // < 64 here
        const int tf = j0 > p.Lp ? j0 - p.Lp : 0;
        const uint32_t lo = __funnelshift_r(w[0], w[1], tf & 31);
        const uint32_t hi = __funnelshift_r(w[1], w[2], tf & 31);
        uint64_t vis = ((static_cast<uint64_t>(hi) << 32) | lo) << np;
        if (np > 0) vis |= (1ull << np) - 1;
        const int nv = p.L - j0;  // keys of the window below L
        if (nv < kHalf) vis &= nv > 0 ? (1ull << nv) - 1 : 0ull;
        const uint32_t v0 = static_cast<uint32_t>(vis), v1 = static_cast<uint32_t>(vis >> 32);
#pragma unroll
        for (int c = 0; c < kHalf; ++c) {
          const bool seen = (((c < 32 ? v0 : v1) >> (c & 31)) & 1u) != 0u;
          s[c] = seen ? s[c] * p.scale_log2 : -INFINITY;
        }
      }
    };
    // One pass with an online maximum.  P uses a reference maximum m that
    // is raised only when a tile's row maximum exceeds it by more than 8
    // (base 2), so weights stay <= 2^8; raising it rescales l and the O
    // accumulated so far (after the products issued so far have landed).
    // The two groups meet at a named barrier every tile, so every decision
    // to stop is taken by all 256 threads together at that barrier: a warp
    // whose wait ran out marks its stop slot and goes on to the barrier.
    bool go = true;
    float m = -INFINITY, l = 0.f;
    constexpr int kOH = kDh / 2;
    // a warp-uniform bounded wait (lane 0 polls, the warp takes its answer)
    auto wait_w = [&](uint64_t* bar, uint32_t par) {
      int okl = 0;
      if (lane == 0) okl = mbar_wait(bar, par, p.err, p.wait_limit) ? 1 : 0;
      return __shfl_sync(kFullMask, okl, 0) != 0;
    };
    for (int j = 0; j < nt; ++j) {
      uint32_t mw[3];
      mask_words(t_beg + j, mw);  // (in flight during the wait)
      const bool okw = go && !*abort_flag && wait_w(&s_full[j & 1], static_cast<uint32_t>(j >> 1) & 1u);
      float s[kHalf];
      float mh = -INFINITY;
      if (okw) {
        tc_fence_after();
        load_s(j, t_beg + j, mw, s);
#pragma unroll
        for (int c = 0; c < kHalf; ++c) mh = fmaxf(mh, s[c]);
      }
      red2[j & 1][wg][row] = mh;  // the row maximum of the tile, both halves
      if (lane == 0) stop_slot[j & 1][warp] = okw ? 0 : 1;
      asm volatile("bar.sync 1, 256;" ::: "memory");
      int stop = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) stop |= stop_slot[j & 1][w];
      if (stop) {  // the same for all 256 threads
        go = false;
        *abort_flag = 1;
        break;
      }
      const float mx = fmaxf(red2[j & 1][0][row], red2[j & 1][1][row]);
      const bool raise = mx > m + 8.f;  // the same in both groups
      bool failed = false;
      if (__any_sync(kFullMask, raise)) {
        const float m_new = raise ? mx : m;
        const float alpha = raise ? fast_ex2(m - m_new) : 1.f;  // 0 when m was -inf
        l *= alpha;
        m = m_new;
        if (j > 0) {  // O holds the products of tiles 0..j-1: wait for the last
          failed = !wait_w(&p_empty[(j - 1) % kPBufs],
                           static_cast<uint32_t>((j - 1) / kPBufs) & 1u);
          if (!failed) {
            tc_fence_after();
            const uint32_t oaddr = tmem_base + lane_base + kColO + wg * kOH;
#pragma unroll
            for (int c = 0; c < kOH; c += 16) {
              float x[16];
              tmem_ld16(oaddr + c, x);
#pragma unroll
              for (int i = 0; i < 16; ++i) x[i] *= alpha;
              tmem_st16(oaddr + c, x);
            }
            tmem_wait_st();
          }
        }
      }
      const float sub = m == -INFINITY ? 0.f : m;
      uint32_t pk[kHalf / 2];
#pragma unroll
      for (int c = 0; c < kHalf; c += 2) {
        const uint32_t v = cvt_bf16x2(fast_ex2(s[c] - sub), fast_ex2(s[c + 1] - sub));
        l += __uint_as_float(v << 16) + __uint_as_float(v & 0xFFFF0000u);
        pk[c / 2] = v;
      }
      // the product that last read this P buffer has finished
      const int pb = j % kPBufs;
      if (!failed)
        failed = !wait_w(&p_empty[pb], (static_cast<uint32_t>(j / kPBufs) & 1u) ^ 1u);
      if (failed) {  // stop at the next tile's barrier, with the other group
        go = false;
        *abort_flag = 1;
        continue;
      }
      // this group's 64 keys of the tile: 32 columns of its lane's P row
      tmem_st32(tmem_base + lane_base + kColP + static_cast<uint32_t>(pb * (kKeys / 2) + wg * 32),
                pk);
      tmem_wait_st();
      tc_fence_before();  // P and the rescaled O are ordered before the next product
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    // (a group that stopped early still meets the other at every barrier
    // below; the barriers inside the loop are met by both while neither
    // has stopped, and a stop sets the abort flag both then see)
    red[wg][row] = l;  // the two halves' sums -> the row's
    asm volatile("bar.sync 1, 256;" ::: "memory");
    l = red[0][row] + red[1][row];
    // this group's half of the head dimensions of O
    float o[kOH];
    if (go && nt > 0 && wait_w(o_done, 0)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kOH; c += 16) {
        float x[16];
        tmem_ld16(tmem_base + lane_base + kColO + wg * kOH + c, x);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[c + i] = x[i];
      }
    } else {
#pragma unroll
      for (int c = 0; c < kOH; ++c) o[c] = 0.f;
      if (nt > 0) l = 0.f;
    }
    // the stage buffers are free: every product (the last reader) has landed
    finish_tile(p, r, hk, qt, row, wg, o, m, l, reinterpret_cast<float*>(sStage));
  }

  // several splits: every CTA of the query tile's cluster sends the rows the
  // others own and combines its own (every thread of every CTA meets both
  // cluster barriers, whatever path it took above)
  if (p.n_split > 1) {
    cl_wait();  // every CTA of the cluster runs: its receive buffer exists
    if (warp < kSoftmaxThreads / 32)
      split_exchange(p, qt, split, reinterpret_cast<const float*>(sStage), recv);
    cl_sync();  // every row delivered
    if (warp < kSoftmaxThreads / 32)
      split_combine(p, r, hk, qt, split, reinterpret_cast<const float*>(sStage), recv);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc<kTmemCols>(tmem_base);
  }
}

// ---------------------------------------------------------------- accept

struct AcceptParams {
  int B, max_len;
  const int32_t* parent;  // [R][B]
  const int32_t* token;
  const int32_t* n_out;   // [R]
  const int32_t* pred;    // [R][B+1]
  int32_t* len;           // [R]
  int32_t* nodes;         // [R][max_len]
  int32_t* bonus;         // [R]
};

// One warp per request: at each step the lanes scan the tree for the child
// of the current node carrying the predicted token (siblings have distinct
// tokens: at most one matches).
__global__ void __launch_bounds__(32) k_accept(const AcceptParams p) {
  const int r = blockIdx.x, lane = threadIdx.x;
  const int32_t* par = p.parent + static_cast<size_t>(r) * p.B;
  const int32_t* tok = p.token + static_cast<size_t>(r) * p.B;
  const int32_t* pred = p.pred + static_cast<size_t>(r) * (p.B + 1);
  const int n = min(max(p.n_out[r], 0), p.B);
  int cur = -1, len = 0;
  for (int step = 0; step <= p.B; ++step) {  // bounded by the tree size
    const int32_t want = pred[cur + 1];
    int found = -1;
    for (int base = 0; base < n && found < 0; base += 32) {
      const int m = base + lane;
      const bool hit = m < n && par[m] == cur && tok[m] == want;
      const unsigned b = __ballot_sync(kFullMask, hit);
      if (b) found = base + __ffs(b) - 1;
    }
    if (found < 0) break;
    if (lane == 0 && len < p.max_len) p.nodes[static_cast<size_t>(r) * p.max_len + len] = found;
    ++len;
    cur = found;
  }
  if (lane == 0) {
    p.len[r] = len;
    p.bonus[r] = pred[cur + 1];
    for (int i = len; i < p.max_len; ++i) p.nodes[static_cast<size_t>(r) * p.max_len + i] = -1;
  }
}

dartree_status fail(dartree_status s, const char* why) {
  set_context_free_error(why);
  return s;
}


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

bool encode_4d(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[4],
               const cuuint64_t (&strides)[3], const cuuint32_t (&box)[4]) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}


__device__ int g_attn_err;  // error word when the caller passes none

}  // namespace
}  // namespace dt

extern "C" size_t dartree_tree_attention_workspace(int32_t R, int32_t Lp, int32_t B, int32_t Hq,
                                                   int32_t Hkv) {
  // the key splits exchange their rows in distributed shared memory: no
  // device scratch is needed
  (void)R;
  (void)Lp;
  (void)B;
  (void)Hq;
  (void)Hkv;
  return 0;
}

extern "C" dartree_status dartree_tree_attention(const void* Q, const void* K, const void* Vt,
                                                 const uint32_t* mask, int32_t R,
                                                 int32_t Lp, int32_t B, int32_t Hq, int32_t Hkv,
                                                 int32_t dh, float scale, float* O, void* O_bf16,
                                                 void* work, size_t work_bytes, int32_t* err,
                                                 void* stream) {
  using namespace dt;
  (void)work;  // (the key splits need no scratch: kept for the interface)
  (void)work_bytes;
  if (!Q || !K || !Vt || !O || (B > 0 && !mask))
    return fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (R < 1 || Lp < 0 || B < 0 || B > DARTREE_MAX_B || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
      Lp + B < 1 || !(scale > 0.f))
    return fail(DARTREE_ERR_INVALID_ARG, "bad R, Lp, B, Hq, Hkv or scale");
  if (dh != kDh) return fail(DARTREE_ERR_UNSUPPORTED, "head dimension must be 128");
  const uintptr_t al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                       reinterpret_cast<uintptr_t>(Vt) | reinterpret_cast<uintptr_t>(O) |
                       reinterpret_cast<uintptr_t>(O_bf16);
  if (al & 15) return fail(DARTREE_ERR_INVALID_ARG, "Q, K, Vt and O must be 16-byte aligned");
  const int L = Lp + B;
  const int g = Hq / Hkv;
  CUtensorMap tm_q, tm_k, tm_vt;
  const int nblk = (L + kVBlock - 1) / kVBlock;
  {  // keys [R][Hkv][L][dh]: a tile is 64 consecutive rows of one head
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kDh), static_cast<cuuint64_t>(L),
                                static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(R)};
    const cuuint64_t str[3] = {static_cast<cuuint64_t>(kDh) * 2,
                               static_cast<cuuint64_t>(L) * kDh * 2,
                               static_cast<cuuint64_t>(Hkv) * L * kDh * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kKeys), 1, 1};
    if (!encode_4d(&tm_k, K, dims, str, box)) return fail(DARTREE_ERR_CUDA, "key tensor map");
  }
  {  // values [R][Hkv][nblk][dh][64]: a tile is one contiguous transposed block
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kVBlock), static_cast<cuuint64_t>(kDh),
                                static_cast<cuuint64_t>(nblk),
                                static_cast<cuuint64_t>(Hkv) * R};
    const cuuint64_t str[3] = {static_cast<cuuint64_t>(kVBlock) * 2,
                               static_cast<cuuint64_t>(kVBlock) * kDh * 2,
                               static_cast<cuuint64_t>(nblk) * kVBlock * kDh * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(kVBlock), static_cast<cuuint32_t>(kDh), 1,
                               1};
    if (!encode_4d(&tm_vt, Vt, dims, str, box)) return fail(DARTREE_ERR_CUDA, "value tensor map");
  }
  const bool q_tma = kQRows % g == 0;
  if (q_tma) {  // queries [R][B+1][Hq][dh]: a tile is 128 / g nodes x g heads
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kDh), static_cast<cuuint64_t>(Hq),
                                static_cast<cuuint64_t>(B) + 1, static_cast<cuuint64_t>(R)};
    const cuuint64_t str[3] = {static_cast<cuuint64_t>(kDh) * 2,
                               static_cast<cuuint64_t>(Hq) * kDh * 2,
                               static_cast<cuuint64_t>(B + 1) * Hq * kDh * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(g),
                               static_cast<cuuint32_t>(kQRows / g), 1};
    if (!encode_4d(&tm_q, Q, dims, str, box)) return fail(DARTREE_ERR_CUDA, "query tensor map");
  } else {
    tm_q = tm_k;  // (not read: the threads stage the query tile)
  }
  AttnParams p{};
  p.Lp = Lp;
  p.B = B;
  p.L = L;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = g;
  p.q_tma = q_tma ? 1 : 0;
  // q / g by a multiply: with m = ceil(2^32 / g) = (2^32 + e) / g, e < g,
  // (q m) >> 32 = floor(q / g + q e / (g 2^32)) = q / g while q e < 2^32;
  // here q < (B + 1) g <= 1025 g and e < g
  p.g_magic = ((1ull << 32) + static_cast<unsigned long long>(g) - 1) / static_cast<unsigned long long>(g);
  if (static_cast<unsigned long long>(B + 1) * g * g >= (1ull << 32))
    return fail(DARTREE_ERR_UNSUPPORTED, "too many query heads per key/value head");
  p.words = (B + 31) / 32;
  p.rows = (B + 1) * p.g;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.Q = static_cast<const uint16_t*>(Q);
  p.mask = mask;
  p.O = O;
  p.O16 = static_cast<uint16_t*>(O_bf16);
  p.err = err;
  cudaError_t e;
  if (!p.err) {
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p.err), g_attn_err);
    if (e != cudaSuccess) return fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  }
  const size_t smem0 =
      1024 + kQBytes + static_cast<size_t>(kStages) * kStageBytes + 256;
  // split the keys so that one wave of CTAs fills the GPU: the splits of a
  // query tile are one cluster (at most kMaxSplit CTAs)
  p.q_tiles = (p.rows + kQRows - 1) / kQRows;
  const int tiles = R * Hkv * p.q_tiles;
  const int key_tiles = (L + kKeys - 1) / kKeys;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int n_split = sms / tiles;  // one CTA per SM
  n_split = n_split < kMaxSplit ? n_split : kMaxSplit;
  // a split keeps at least 3 key tiles (tuning: DARTREE_ATTN_SPLIT_MIN): with
  // fewer, the exchange and the combine cost more than the tiles they save
  int min_tiles = 3;
  if (const char* v = getenv("DARTREE_ATTN_SPLIT_MIN")) min_tiles = atoi(v) > 0 ? atoi(v) : 1;
  const int by_keys = key_tiles / min_tiles;
  n_split = n_split < by_keys ? n_split : by_keys;
  if (const char* v = getenv("DARTREE_ATTN_MAX_SPLIT"))  // (test knob)
    if (atoi(v) >= 1 && atoi(v) < n_split) n_split = atoi(v);
  if (n_split < 1) n_split = 1;
  p.n_split = n_split;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rs = (kQRows + n_split - 1) / n_split;
  const size_t recv_bytes =
      n_split > 1 ? static_cast<size_t>(n_split - 1) * rs * (kDh * 4 + 8) : 0;
  const size_t smem = smem0 + recv_bytes;
  // the receive buffer is largest for the split count that maximises
  // (n - 1) ceil(128 / n) (7: 114 rows), not for the largest count
  int recv_rows_max = 0;
  for (int n = 2; n <= kMaxSplit; ++n) {
    const int rows_n = (n - 1) * ((kQRows + n - 1) / n);
    recv_rows_max = rows_n > recv_rows_max ? rows_n : recv_rows_max;
  }
  e = cudaFuncSetAttribute(k_tree_attention, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem0 + static_cast<size_t>(recv_rows_max) *
                                                        (kDh * 4 + 8)));
  if (e != cudaSuccess) return fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  const dim3 grid(p.q_tiles * n_split, Hkv, R);
  e = n_split > 1 ? launch_kernel_cluster(k_tree_attention, grid, dim3(kAttnThreads), smem, st,
                                          false, n_split, tm_q, tm_k, tm_vt, p)
                  : launch_kernel(k_tree_attention, grid, dim3(kAttnThreads), smem, st, false,
                                  tm_q, tm_k, tm_vt, p);
  if (e != cudaSuccess) return fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  return DARTREE_OK;
}

extern "C" dartree_status dartree_accept(const int32_t* parent, const int32_t* token,
                                         const int32_t* n_out, const int32_t* pred, int32_t R,
                                         int32_t B, int32_t max_len, int32_t* accept_len,
                                         int32_t* accept_nodes, int32_t* bonus, void* stream) {
  using namespace dt;
  if (!parent || !token || !n_out || !pred || !accept_len || !bonus ||
      (max_len > 0 && !accept_nodes))
    return fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (R < 1 || B < 1 || B > DARTREE_MAX_B || max_len < 0)
    return fail(DARTREE_ERR_INVALID_ARG, "bad R, B or max_len");
  AcceptParams p{B, max_len, parent, token, n_out, pred, accept_len, accept_nodes, bonus};
  cudaError_t e = launch_kernel(k_accept, dim3(R), dim3(32), 0, static_cast<cudaStream_t>(stream),
                                false, p);
  if (e != cudaSuccess) return fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  return DARTREE_OK;
}
