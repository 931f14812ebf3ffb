// The verification consumer of a built tree: one attention layer of the
// target over the prefix and the draft tree with the emitted ancestor mask,
// and the longest accepted prefix under the target's predictions
// ("DARTree: Teaching a Chain-Trained Corrector to Think in Trees", Core
// Mechanism: the verification tree and sparse attention mask let the target
// check every branch in ONE forward, then the longest matching prefix is
// accepted; "Technische Samenvatting: DARTree", Methodologie 2, Verificatie).
//
// Tree attention, flash-style, one pass with an online softmax: a CTA owns
// 64 query rows (4 warps x 16) of one request and one key/value head; key
// and value tiles of 64 positions stream through double-buffered shared
// memory (16-byte async copies, XOR-swizzled rows); scores and P.V run on
// bf16 warp-level MMAs (m16n8k16, fp32 accumulation), P staying in
// registers between the two products.  Query row q of a key/value head is
// (node q / g, query head hk * g + q % g), g = Hq / Hkv.  Row 0 (the root)
// sees the prefix; node i >= 1 sees the prefix and the tree nodes of mask
// row i - 1.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/dartree.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dt {
namespace {

constexpr int kDh = 128;          // head dimension (fixed)
constexpr int kQRows = 64;        // query rows per CTA
constexpr int kKeys = 64;         // keys per tile
constexpr int kAttnThreads = 128;
constexpr int kRowBytes = kDh * 2;  // 256 B per bf16 row
constexpr int kTileBytes = kKeys * kRowBytes;

struct AttnParams {
  int Lp, B, Hq, Hkv, g, words, rows;  // rows = (B + 1) * g query rows per key/value head
  float scale_log2;                     // scale * log2(e)
  const uint16_t* Q;                    // [R][B+1][Hq][dh]
  const uint16_t* Kp;                   // [R][Lp][Hkv][dh]
  const uint16_t* Vp;
  const uint16_t* Kt;                   // [R][B][Hkv][dh]
  const uint16_t* Vt;
  const uint32_t* mask;                 // [R][B][words]
  float* O;                             // [R][B+1][Hq][dh]
  uint16_t* O16;                        // same, bf16 bits, or null
  // key split (flash-decoding): CTA (tile, split) covers a share of the key
  // tiles; the last split to finish a query tile combines the partials
  int n_split, q_tiles;
  float* part_O;                        // [tiles][n_split][64][dh] unnormalised
  float2* part_ml;                      // [tiles][n_split][64] (max, sum) in base 2
  int* cnt;                             // [tiles] arrivals, zero before the launch
};

// Byte offset of 16-byte chunk c of row r in a swizzled [rows][256 B] tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;  // 0: fill with zeros, read nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += a (16x16, row) * b (16x8, col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

// Two fp32 -> packed bf16 pair (round to nearest even), lower column first.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return static_cast<uint32_t>(float_to_bf16_bits(lo)) |
         (static_cast<uint32_t>(float_to_bf16_bits(hi)) << 16);
}

// Stage key/value tile `t` (keys t*64 .. t*64+63 of prefix + tree) of head hk.
__device__ __forceinline__ void load_kv(const AttnParams& p, int r, int hk, int t, uint32_t sK,
                                        uint32_t sV) {
  for (int e = threadIdx.x; e < kKeys * 16; e += kAttnThreads) {
    const int row = e >> 4, c = e & 15;
    const int j = t * kKeys + row;
    const uint16_t *k, *v;
    bool valid = true;
    if (j < p.Lp) {
      const size_t o = ((static_cast<size_t>(r) * p.Lp + j) * p.Hkv + hk) * kDh + c * 8;
      k = p.Kp + o;
      v = p.Vp + o;
    } else if (j < p.Lp + p.B) {
      const size_t o = ((static_cast<size_t>(r) * p.B + (j - p.Lp)) * p.Hkv + hk) * kDh + c * 8;
      k = p.Kt + o;
      v = p.Vt + o;
    } else {
      k = p.Kp;  // any mapped address; nothing is read
      v = p.Kp;
      valid = false;
    }
    cp_async16(sK + swz(row, c), k, valid);
    cp_async16(sV + swz(row, c), v, valid);
  }
}

// Publish this CTA's partial (unnormalised O, row max and sum in base 2);
// the last split of the query tile to arrive combines all of them:
//   M = max_s m_s, L = sum_s l_s 2^(m_s - M), O = sum_s O_s 2^(m_s - M) / L.
__device__ __forceinline__ void combine_splits(const AttnParams& p, int r, int hk, int qt, int split,
                                            const float (&o)[16][4], float m_a, float m_b,
                                            float l_a, float l_b) {
  __shared__ int last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t tile = (static_cast<size_t>(r) * p.Hkv + hk) * p.q_tiles + qt;
  float* po = p.part_O + (tile * p.n_split + split) * kQRows * kDh;
  float2* pml = p.part_ml + (tile * p.n_split + split) * kQRows;
  const int ra = warp * 16 + (lane >> 2), rb = ra + 8;  // rows within the tile
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int col = i * 8 + (lane & 3) * 2;
    *reinterpret_cast<float2*>(po + ra * kDh + col) = make_float2(o[i][0], o[i][1]);
    *reinterpret_cast<float2*>(po + rb * kDh + col) = make_float2(o[i][2], o[i][3]);
  }
  if ((lane & 3) == 0) {
    pml[ra] = make_float2(m_a, l_a);
    pml[rb] = make_float2(m_b, l_b);
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last = (atomicAdd(p.cnt + tile, 1) == p.n_split - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float* all_o = p.part_O + tile * p.n_split * kQRows * kDh;
  const float2* all_ml = p.part_ml + tile * p.n_split * kQRows;
  for (int e = threadIdx.x; e < kQRows * (kDh / 4); e += kAttnThreads) {
    const int row = e / (kDh / 4), c4 = (e % (kDh / 4)) * 4;
    const int q = qt * kQRows + row;
    if (q >= p.rows) continue;
    float M = -INFINITY;
    for (int s = 0; s < p.n_split; ++s) M = fmaxf(M, __ldcg(&all_ml[s * kQRows + row]).x);
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < p.n_split; ++s) {  // fixed order: deterministic
      const float2 ml = __ldcg(&all_ml[s * kQRows + row]);
      if (ml.x == -INFINITY) continue;
      const float f = exp2f(ml.x - M);
      L += ml.y * f;
      const float4 v =
          __ldcg(reinterpret_cast<const float4*>(all_o + (s * kQRows + row) * kDh + c4));
      acc.x += v.x * f;
      acc.y += v.y * f;
      acc.z += v.z * f;
      acc.w += v.w * f;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float4 out = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    const int node = q / p.g, h = hk * p.g + q % p.g;
    const size_t base = ((static_cast<size_t>(r) * (p.B + 1) + node) * p.Hq + h) * kDh + c4;
    *reinterpret_cast<float4*>(p.O + base) = out;
    if (p.O16)
      *reinterpret_cast<uint2*>(p.O16 + base) =
          make_uint2(pack_bf16(out.x, out.y), pack_bf16(out.z, out.w));
  }
  if (threadIdx.x == 0) p.cnt[tile] = 0;
}

__global__ void __launch_bounds__(kAttnThreads) k_tree_attention(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sKV = sQ + kQRows * kRowBytes;  // [2 stages][K tile, V tile]
  const int r = blockIdx.z, hk = blockIdx.y;
  const int qt = blockIdx.x / p.n_split, split = blockIdx.x % p.n_split;
  const int q0 = qt * kQRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- query tile: 64 rows of (node, head) gathered into shared memory
  for (int e = threadIdx.x; e < kQRows * 16; e += kAttnThreads) {
    const int row = e >> 4, c = e & 15;
    const int q = q0 + row;
    const bool valid = q < p.rows;
    const int node = q / p.g, h = hk * p.g + q % p.g;
    const uint16_t* src =
        valid ? p.Q + ((static_cast<size_t>(r) * (p.B + 1) + node) * p.Hq + h) * kDh + c * 8 : p.Q;
    cp_async16(sQ + swz(row, c), src, valid);
  }
  const int n_keys = p.Lp + p.B;
  const int n_tiles = (n_keys + kKeys - 1) / kKeys;
  // the largest node of this tile bounds the tree keys any row can see
  const int last_node = min(p.B, (q0 + kQRows - 1) / p.g);
  const int t_all = min(n_tiles, (p.Lp + last_node + kKeys - 1) / kKeys);
  const int t_beg = split * t_all / p.n_split, t_end = (split + 1) * t_all / p.n_split;
  if (t_beg < t_end) load_kv(p, r, hk, t_beg, sKV, sKV + kTileBytes);
  cp_async_commit();

  // this thread's two query rows (within the warp's 16) and their nodes
  const int qa = q0 + warp * 16 + (lane >> 2), qb = qa + 8;
  const int node_a = qa / p.g, node_b = qb / p.g;
  const uint32_t* mrow_a =
      (node_a >= 1 && qa < p.rows) ? p.mask + (static_cast<size_t>(r) * p.B + node_a - 1) * p.words
                                   : nullptr;
  const uint32_t* mrow_b =
      (node_b >= 1 && qb < p.rows) ? p.mask + (static_cast<size_t>(r) * p.B + node_b - 1) * p.words
                                   : nullptr;

  float o[16][4];  // 16 x 128 output of the warp: 16 column tiles of 8
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
  uint32_t qf[8][4];  // A fragments of the warp's 16 query rows, 8 k-steps

  for (int t = t_beg; t < t_end; ++t) {
    const int st = t - t_beg;
    const uint32_t sK = sKV + (st & 1) * 2 * kTileBytes, sV = sK + kTileBytes;
    if (t + 1 < t_end) {
      const uint32_t nK = sKV + ((st + 1) & 1) * 2 * kTileBytes;
      load_kv(p, r, hk, t + 1, nK, nK + kTileBytes);
    }
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (t == t_beg) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4(sQ + swz(row, ks * 2 + (lane >> 4)), qf[ks]);
      }
    }
    // ---- S = Q K^T for 64 keys: 8 column tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
      for (int n2 = 0; n2 < 4; ++n2) {  // two key tiles per ldmatrix
        uint32_t b[4];
        const int krow = n2 * 16 + (lane & 7) + (lane >> 4) * 8;
        ldsm_x4(sK + swz(krow, ks * 2 + ((lane >> 3) & 1)), b);
        mma_bf16(s[2 * n2], qf[ks], b[0], b[1]);
        mma_bf16(s[2 * n2 + 1], qf[ks], b[2], b[3]);
      }
    }
    // ---- visibility, online softmax (base 2), P in registers
    const int j0 = t * kKeys;
    float mx_a = m_a, mx_b = m_b;
    if (j0 + kKeys <= p.Lp) {  // prefix keys only: every row sees all of them
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] *= p.scale_log2;
        mx_a = fmaxf(mx_a, fmaxf(s[n][0], s[n][1]));
        mx_b = fmaxf(mx_b, fmaxf(s[n][2], s[n][3]));
      }
    } else {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = j0 + n * 8 + (lane & 3) * 2 + (e & 1);
          const bool row_b = e >= 2;
          const uint32_t* mr = row_b ? mrow_b : mrow_a;
          bool vis = j < p.Lp;
          if (!vis && j < n_keys && mr != nullptr) {
            const int tt = j - p.Lp;
            vis = (__ldg(mr + (tt >> 5)) >> (tt & 31)) & 1u;
          }
          const float v = vis ? s[n][e] * p.scale_log2 : -INFINITY;
          s[n][e] = v;
          if (row_b) mx_b = fmaxf(mx_b, v); else mx_a = fmaxf(mx_a, v);
        }
      }
    }
#pragma unroll
    for (int o2 = 1; o2 <= 2; o2 <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(kFullMask, mx_a, o2));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(kFullMask, mx_b, o2));
    }
    // (ex2 of -inf is +0: invisible keys get weight 0 without a test)
    const float al_a = (mx_a == -INFINITY) ? 1.f : fast_ex2(m_a - mx_a);
    const float al_b = (mx_b == -INFINITY) ? 1.f : fast_ex2(m_b - mx_b);
    m_a = mx_a;
    m_b = mx_b;
    const float sub_a = (m_a == -INFINITY) ? 0.f : m_a, sub_b = (m_b == -INFINITY) ? 0.f : m_b;
    uint32_t pf[4][4];  // A fragments of P: 4 k-steps of 16 keys
    float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      // the bf16-rounded weights are used for both P.V and the normaliser
      const uint32_t pa = cvt_bf16x2(fast_ex2(s[n][0] - sub_a), fast_ex2(s[n][1] - sub_a));
      const uint32_t pb = cvt_bf16x2(fast_ex2(s[n][2] - sub_b), fast_ex2(s[n][3] - sub_b));
      ps_a += __uint_as_float(pa << 16) + __uint_as_float(pa & 0xFFFF0000u);
      ps_b += __uint_as_float(pb << 16) + __uint_as_float(pb & 0xFFFF0000u);
      const int ks = n >> 1, hi = n & 1;
      pf[ks][hi * 2 + 0] = pa;
      pf[ks][hi * 2 + 1] = pb;
    }
    l_a = l_a * al_a + ps_a;
    l_b = l_b * al_b + ps_b;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      o[i][0] *= al_a;
      o[i][1] *= al_a;
      o[i][2] *= al_b;
      o[i][3] *= al_b;
    }
    // ---- O += P V: 16 column tiles of 8 (head dim), 4 k-steps of 16 keys
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int d2 = 0; d2 < 8; ++d2) {  // two head-dim tiles per ldmatrix
        uint32_t b[4];
        const int vrow = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(sV + swz(vrow, d2 * 2 + (lane >> 4)), b);
        mma_bf16(o[2 * d2], pf[ks], b[0], b[1]);
        mma_bf16(o[2 * d2 + 1], pf[ks], b[2], b[3]);
      }
    }
    __syncthreads();  // the stage is refilled by the next iteration
  }
  cp_async_wait<0>();

  // ---- normalise and write the two rows of this thread
#pragma unroll
  for (int o2 = 1; o2 <= 2; o2 <<= 1) {
    l_a += __shfl_xor_sync(kFullMask, l_a, o2);
    l_b += __shfl_xor_sync(kFullMask, l_b, o2);
  }
  if (p.n_split > 1) {
    combine_splits(p, r, hk, qt, split, o, m_a, m_b, l_a, l_b);
    return;
  }
  const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f, inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int q = half ? qb : qa;
    if (q >= p.rows) continue;
    const int node = q / p.g, h = hk * p.g + q % p.g;
    const size_t base = ((static_cast<size_t>(r) * (p.B + 1) + node) * p.Hq + h) * kDh;
    const float inv = half ? inv_b : inv_a;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int col = i * 8 + (lane & 3) * 2;
      const float x0 = o[i][half * 2] * inv, x1 = o[i][half * 2 + 1] * inv;
      *reinterpret_cast<float2*>(p.O + base + col) = make_float2(x0, x1);
      if (p.O16) *reinterpret_cast<uint32_t*>(p.O16 + base + col) = pack_bf16(x0, x1);
    }
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

}  // namespace
}  // namespace dt

namespace dt {
namespace {
constexpr int kMaxSplit = 16;

size_t split_bytes(int R, int B, int Hq, int Hkv, int n_split) {
  const size_t q_tiles = (static_cast<size_t>(B + 1) * (Hq / Hkv) + kQRows - 1) / kQRows;
  const size_t tiles = static_cast<size_t>(R) * Hkv * q_tiles;
  const size_t o = tiles * n_split * kQRows * kDh * 4, ml = tiles * n_split * kQRows * 8;
  return o + ml + tiles * 4 + 64;
}
}  // namespace
}  // namespace dt

extern "C" size_t dartree_tree_attention_workspace(int32_t R, int32_t Lp, int32_t B, int32_t Hq,
                                                   int32_t Hkv) {
  (void)Lp;
  if (R < 1 || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return 0;
  return dt::split_bytes(R, B, Hq, Hkv, dt::kMaxSplit);
}

extern "C" dartree_status dartree_tree_attention(const void* Q, const void* Kp, const void* Vp,
                                                 const void* Kt, const void* Vt,
                                                 const uint32_t* mask, int32_t R, int32_t Lp,
                                                 int32_t B, int32_t Hq, int32_t Hkv, int32_t dh,
                                                 float scale, float* O, void* O_bf16, void* work,
                                                 size_t work_bytes, void* stream) {
  using namespace dt;
  if (!Q || !Kt || !Vt || !O || (Lp > 0 && (!Kp || !Vp)) || (B > 0 && !mask))
    return fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (R < 1 || Lp < 0 || B < 0 || B > DARTREE_MAX_B || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 ||
      Lp + B < 1 || !(scale > 0.f))
    return fail(DARTREE_ERR_INVALID_ARG, "bad R, Lp, B, Hq, Hkv or scale");
  if (dh != kDh) return fail(DARTREE_ERR_UNSUPPORTED, "head dimension must be 128");
  const uintptr_t al = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(Kt) |
                       reinterpret_cast<uintptr_t>(Vt) | reinterpret_cast<uintptr_t>(Kp) |
                       reinterpret_cast<uintptr_t>(Vp) | reinterpret_cast<uintptr_t>(O) |
                       reinterpret_cast<uintptr_t>(O_bf16);
  if (al & 15) return fail(DARTREE_ERR_INVALID_ARG, "Q, K, V and O must be 16-byte aligned");
  AttnParams p{};
  p.Lp = Lp;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.g = Hq / Hkv;
  p.words = (B + 31) / 32;
  p.rows = (B + 1) * p.g;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.Q = static_cast<const uint16_t*>(Q);
  p.Kp = static_cast<const uint16_t*>(Lp > 0 ? Kp : Kt);
  p.Vp = static_cast<const uint16_t*>(Lp > 0 ? Vp : Vt);
  p.Kt = static_cast<const uint16_t*>(Kt);
  p.Vt = static_cast<const uint16_t*>(Vt);
  p.mask = mask;
  p.O = O;
  p.O16 = static_cast<uint16_t*>(O_bf16);
  const size_t smem = static_cast<size_t>(kQRows) * kRowBytes + 4 * static_cast<size_t>(kTileBytes);
  cudaError_t e = cudaFuncSetAttribute(k_tree_attention,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  // split the keys so that one wave of CTAs fills the GPU, as the workspace allows
  p.q_tiles = (p.rows + kQRows - 1) / kQRows;
  const int tiles = R * Hkv * p.q_tiles;
  const int key_tiles = (Lp + B + kKeys - 1) / kKeys;
  int dev = 0, sms = 148, per_sm = 1;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_tree_attention, kAttnThreads, smem);
  if (per_sm < 1) per_sm = 1;
  int n_split = (per_sm * sms) / tiles;  // one full wave of CTAs
  n_split = n_split < kMaxSplit ? n_split : kMaxSplit;
  n_split = n_split < key_tiles ? n_split : key_tiles;
  if (n_split < 1) n_split = 1;
  if ((reinterpret_cast<uintptr_t>(work) & 15) != 0) work = nullptr;
  while (n_split > 1 && (work == nullptr || split_bytes(R, B, Hq, Hkv, n_split) > work_bytes))
    --n_split;
  p.n_split = n_split;
  if (n_split > 1) {
    const size_t ot = static_cast<size_t>(tiles) * n_split * kQRows * kDh * 4;
    const size_t mt = static_cast<size_t>(tiles) * n_split * kQRows * 8;
    uint8_t* wb = static_cast<uint8_t*>(work);
    p.part_O = reinterpret_cast<float*>(wb);
    p.part_ml = reinterpret_cast<float2*>(wb + ot);
    p.cnt = reinterpret_cast<int*>(wb + ot + mt);
    e = cudaMemsetAsync(p.cnt, 0, sizeof(int) * tiles, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(DARTREE_ERR_CUDA, cudaGetErrorString(e));
  }
  const dim3 grid(p.q_tiles * n_split, Hkv, R);
  e = launch_kernel(k_tree_attention, grid, dim3(kAttnThreads), smem,
                                static_cast<cudaStream_t>(stream), false, p);
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
