// Kernels of the build variants.
//
//  * Markov correction head: the state after a token depends on that token
//    alone, s' = q(tanh(E[tok])) -- the recurrent head with A = 0, so a state
//    step reads M rows of E instead of streaming A ("Technische Samenvatting:
//    DARTree", Experimentele Resultaten, Ablatie: DARTree on the DSpark
//    drafter, whose correction head is Markov).
//  * Base-logit candidates: at every depth the K candidate tokens are the
//    top-K of the base logits z_d, shared by all branches, and the head
//    scores only those K tokens per branch, normalised over the K
//    ("Technische Samenvatting: DARTree", Methodologie 1: Kandidaat Selectie
//    from the base logits; Gebatchte Correctie of those candidates for all
//    branches in one batch).  The head call then reads K rows of Wout per
//    request instead of all V.
//  * Sequential best-first growth, the baseline DARTree replaces: one head
//    call per expanded node, with the heap logic on the device between the
//    calls ("Technische Samenvatting: DARTree", Probleemstelling, Causale
//    Correctie: pop one node, correct it, push its children, then the next;
//    Experimentele Resultaten, Ablatie: latency of the sequential build).
#include <cuda_runtime.h>

#include "block.cuh"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dt {

// ------------------------------------------------------------ Markov state

__global__ void __launch_bounds__(256) k_state_markov(const MarkovParams p) {
  pdl_wait();
  pdl_trigger();
  const int q = blockIdx.y;
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= p.H) return;
  float out = 0.f;
  if (q < p.M_out) {
    int tok = __ldg(p.tok + q);
    if (tok < 0 || tok >= p.V) {  // only after an upstream failure
      atomicOr(p.err, DT_ERR_BAD_INDEX);
      tok = 0;
    }
    const size_t e = static_cast<size_t>(tok) * p.H + h;
    const float u = p.bf16 ? bf16_bits_to_float(__ldg(static_cast<const uint16_t*>(p.E) + e))
                           : __ldg(static_cast<const float*>(p.E) + e);
    out = tanhf(u);
  }
  const size_t o = static_cast<size_t>(q) * p.H + h;
  if (p.bf16)
    static_cast<uint16_t*>(p.S_out)[o] = float_to_bf16_bits(out);
  else
    static_cast<float*>(p.S_out)[o] = out;
}

cudaError_t launch_state_markov(const MarkovParams& p, cudaStream_t st) {
  return launch_kernel(k_state_markov, dim3((p.H + 255) / 256, p.n_out), dim3(256), 0, st,
                       p.pdl != 0, p);
}

// ------------------------------------------------------ base-logit top-K

constexpr int kBaseThreads = 256;
constexpr int kBaseWarps = kBaseThreads / 32;
constexpr int kBaseBatch = 8;  // loads in flight per thread

// Block (chunk, row): top-K of z[row][chunk*8192 ...) by (z desc, token
// asc) -- a sorted list per warp (one key per lane per step, inserted only
// when it beats the list's K-th key), folded across the warps.  The last
// chunk block of the row merges the chunk lists into the row's candidates.
__global__ void __launch_bounds__(kBaseThreads) k_base_topk(const BaseTopkParams p) {
  __shared__ uint64_t lists[kBaseWarps][kMaxK];
  __shared__ uint64_t wl[kBaseWarps][32];
  __shared__ int last_flag;
  pdl_wait();
  pdl_trigger();
  const int chunk = blockIdx.x, row = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K;
  const int p2 = pow2_ceil32(K);
  uint64_t* L = lists[warp];
  if (lane < K) L[lane] = 0ull;
  __syncwarp();
  const float* z = p.z + static_cast<size_t>(row) * p.V;
  const int v_end = min(p.V, (chunk + 1) * kBaseChunk);
  bool bad = false;
  for (int base = chunk * kBaseChunk; base < v_end; base += kBaseThreads * kBaseBatch) {
    float x[kBaseBatch];
#pragma unroll
    for (int i = 0; i < kBaseBatch; ++i) {
      const int v = base + i * kBaseThreads + threadIdx.x;
      x[i] = v < v_end ? __ldg(z + v) : -INFINITY;
    }
#pragma unroll
    for (int i = 0; i < kBaseBatch; ++i) {
      const int v = base + i * kBaseThreads + threadIdx.x;
      const bool valid = v < v_end;
      if (valid && (x[i] != x[i] || x[i] == INFINITY)) bad = true;
      const uint64_t key = (valid && x[i] == x[i]) ? make_key(x[i], static_cast<uint32_t>(v)) : 0ull;
      const unsigned bal = __ballot_sync(kFullMask, key > L[K - 1]);
      if (bal == 0u) continue;
      if (__popc(bal) <= 2)
        list_insert_lanes(L, K, key, bal);
      else
        list_merge_batch(L, K, key > L[K - 1] ? key : 0ull);
    }
  }
  if (bad) atomicOr(p.err, DT_ERR_NONFINITE);
  uint64_t v = lane < K ? L[lane] : 0ull;
  v = block_tree_merge(v, wl, p2);
  uint64_t* part = p.part + static_cast<size_t>(row) * p.n_chunks * K;
  if (warp == 0 && lane < K) part[static_cast<size_t>(chunk) * K + lane] = v;
  // ---- the last chunk block of the row merges the chunk lists
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) last_flag = (atomicAdd(p.cnt + row, 1) == p.n_chunks - 1);
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  if (threadIdx.x == 0) p.cnt[row] = 0;
  v = 0ull;
  for (int l = warp; l < p.n_chunks; l += kBaseWarps) {
    uint64_t y;
    merge_operands(part + static_cast<size_t>(l) * K, K, p2, v, y);
    v = warp_merge_desc(v, y, p2);
  }
  v = block_tree_merge(v, wl, p2);
  if (warp == 0 && lane < K) {
    if (v == 0ull) atomicOr(p.err, DT_ERR_BAD_INDEX);  // fewer than K real entries
    p.cand[static_cast<size_t>(row) * K + lane] = v ? static_cast<int32_t>(key_index(v)) : 0;
  }
}

cudaError_t launch_base_topk(const BaseTopkParams& p, cudaStream_t st) {
  return launch_kernel(k_base_topk, dim3(p.n_chunks, p.rows), dim3(kBaseThreads), 0, st,
                       p.pdl != 0, p);
}

// ------------------------------------------- corrected candidate logits

constexpr int kCandThreads = 256;
constexpr int kCandWarps = kCandThreads / 32;

// Dot product of a state row and a weight row (H a multiple of 8 for bf16),
// lanes striding over 16-byte pieces; fp32 accumulation, warp-reduced.  A
// blocked bf16 row (blocks of 128 rows x 64 columns) has its 16-byte piece i
// at piece (i / 8) * 1024 + i % 8 from the row's start in its first block.
__device__ __forceinline__ float warp_dot(const void* s, const void* w, int H, bool bf16,
                                          bool blocked = false) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f;
  if (bf16) {
    const uint4* a = static_cast<const uint4*>(s);
    const uint4* b = static_cast<const uint4*>(w);
    for (int i = lane; i < H / 8; i += 32) {
      const uint4 x = __ldg(a + i), y = __ldg(b + (blocked ? (i >> 3) * 1024 + (i & 7) : i));
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        acc = fmaf(__uint_as_float(xs[k] << 16), __uint_as_float(ys[k] << 16), acc);
        acc = fmaf(__uint_as_float(xs[k] & 0xFFFF0000u), __uint_as_float(ys[k] & 0xFFFF0000u), acc);
      }
    }
  } else {
    const float* a = static_cast<const float*>(s);
    const float* b = static_cast<const float*>(w);
    for (int i = lane; i < H; i += 32) acc = fmaf(__ldg(a + i), __ldg(b + i), acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFullMask, acc, o);
  return acc;
}

// Block m = head row m: e_j = fp32(z_d[c_j] + S[m] . Wout[c_j]) for the K
// candidates c_j of the row's request; writes the row's (max, sum-exp) over
// the K values and the K keys (e desc, token asc) as its one partial.
__global__ void __launch_bounds__(kCandThreads) k_cand_logits(const CandParams p) {
  __shared__ uint64_t keys[kMaxK];
  pdl_wait();
  pdl_trigger();
  const int m = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int req = m / p.rows_per_req;
  const int32_t* cand = p.cand + static_cast<size_t>(req) * p.cand_req_stride;
  const float* z = p.z + static_cast<size_t>(req) * p.z_req_stride;
  const size_t eb = p.bf16 ? 2 : 4;
  const uint8_t* srow = static_cast<const uint8_t*>(p.S) + static_cast<size_t>(m) * p.H * eb;
  for (int j = warp; j < p.K; j += kCandWarps) {
    const int c = __ldg(cand + j);
    const bool blocked = p.bf16 && p.w_tiled;
    // row c: row-major, or row c % 128 of its first 128 x 64 block
    const size_t w_off = blocked ? (static_cast<size_t>(c >> 7) * p.w_nk * 8192 +
                                    static_cast<size_t>(c & 127) * 64) * 2
                                 : static_cast<size_t>(c) * p.H * eb;
    const uint8_t* wrow = static_cast<const uint8_t*>(p.Wout) + w_off;
    const float dot = warp_dot(srow, wrow, p.H, p.bf16 != 0, blocked);
    if (lane == 0) {
      const float e = dot + __ldg(z + c);
      if (e != e || e == INFINITY) atomicOr(p.err, DT_ERR_NONFINITE);
      keys[j] = (e == e) ? make_key(e, static_cast<uint32_t>(c)) : 0ull;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  const uint64_t k = lane < p.K ? keys[lane] : 0ull;
  const float e = lane < p.K && k ? key_value(k) : -INFINITY;
  const float mx = warp_max_f(e);
  const float s = warp_sum_f(mx == -INFINITY || e == -INFINITY ? 0.f : expf(e - mx));
  const uint64_t srt = warp_sort_desc(k);
  if (lane < p.K) p.ptop[static_cast<size_t>(m) * p.list_stride * p.K + lane] = srt;
  if (lane == 0) {
    p.pm[static_cast<size_t>(m) * p.cta_stride] = mx;
    p.ps[static_cast<size_t>(m) * p.cta_stride] = s;
  }
}

cudaError_t launch_cand_logits(const CandParams& p, cudaStream_t st) {
  return launch_kernel(k_cand_logits, dim3(p.M), dim3(kCandThreads), 0, st, p.pdl != 0, p);
}

// The blocked layout of a row-major bf16 matrix: output 16-byte piece o is
// piece o % 8 of row o / 8 % 128 of block o / 1024 = (b, k) = (block / nk,
// block % nk), i.e. columns 64 k + 8 (o % 8) .. of row 128 b + o / 8 % 128
// (zero past V).  Grid-stride; one 16-byte load and store per piece.
__global__ void k_block_weights(const uint4* __restrict__ W, int V, int H, uint4* __restrict__ out,
                                long long n_pieces) {
  const int nk = H / 64;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long o = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; o < n_pieces;
       o += step) {
    const long long block = o >> 10;
    const int within = static_cast<int>(o & 1023);
    const long long row = (block / nk) * 128 + (within >> 3);
    const int k = static_cast<int>(block % nk);
    out[o] = row < V ? __ldg(W + row * (H / 8) + k * 8 + (within & 7)) : make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_block_weights(const uint16_t* W, int V, int H, uint16_t* out,
                                 cudaStream_t st) {
  const long long n_pieces = (static_cast<long long>(V) + 127) / 128 * 128 * (H / 8);
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long want = (n_pieces + 255) / 256;
  const int grid = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
  k_block_weights<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(W), V, H,
                                        reinterpret_cast<uint4*>(out), n_pieces);
  return cudaGetLastError();
}

// ------------------------------------------------ best-first baseline

constexpr int kBfThreads = 1024;

__global__ void __launch_bounds__(256) k_bestfirst_init(const BestFirstParams p) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  if (threadIdx.x == 0) {
    p.st[r * 4 + 0] = 0;
    p.st[r * 4 + 1] = 0;
    p.st[r * 4 + 2] = -1;  // the first call expands the root
    p.st[r * 4 + 3] = 1;
    p.z_row[r] = 0;
    p.n_out[r] = 0;
  }
  const size_t ob = static_cast<size_t>(r) * p.B;
  for (int q = threadIdx.x; q < p.B; q += blockDim.x) {
    p.parent[ob + q] = -1;
    p.token[ob + q] = -1;
    p.depth[ob + q] = 0;
    p.score[ob + q] = 0.f;
  }
  for (int e = threadIdx.x; e < p.B * p.words; e += blockDim.x)
    p.mask[static_cast<size_t>(r) * p.B * p.words + e] = 0u;
}

cudaError_t launch_bestfirst_init(const BestFirstParams& p, cudaStream_t st) {
  return launch_kernel(k_bestfirst_init, dim3(p.R), dim3(256), 0, st, p.pdl != 0, p);
}

__device__ __forceinline__ void copy_state(void* dst, const void* src, int H, bool bf16) {
  const size_t n = static_cast<size_t>(H) * (bf16 ? 2 : 4) / 16;  // H % 8 == 0
  const uint4* s = static_cast<const uint4*>(src);
  uint4* d = static_cast<uint4*>(dst);
  for (size_t i = threadIdx.x; i < n; i += blockDim.x) d[i] = s[i];
}

// One block per request, after head call `c`: the expanded node's state is
// archived under its rank and its K children join the node table (ids in
// rank order, score = node score + logp, one fp32 add); then the best
// unpopped node under (key desc, id asc), key = score + beta * depth, is
// popped -- an argmax over the table, which is what a max-heap pop returns
// -- and written as output rank n_pop with its ancestor-mask row.  If the
// budget allows and its depth is below D, the next call expands it: its
// parent's state is staged and its token and depth recorded.
__global__ void __launch_bounds__(kBfThreads) k_bestfirst_step(const BestFirstParams p) {
  __shared__ unsigned long long best;
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const bool bf16 = p.bf16 != 0;
  const size_t rowb = static_cast<size_t>(p.H) * (bf16 ? 2 : 4);
  int* st = p.st + r * 4;
  int n_nodes = st[0];
  const int n_pop = st[1], cur = st[2], expand = st[3];
  const size_t nb = static_cast<size_t>(r) * p.max_nodes;
  if (threadIdx.x == 0) best = 0ull;
  if (expand) {
    const int dep = cur < 0 ? 0 : p.node_dep[nb + cur];
    const float sc = cur < 0 ? 0.f : p.node_score[nb + cur];
    if (cur >= 0) {
      const int rk = p.node_rank[nb + cur];
      copy_state(static_cast<uint8_t*>(p.S_pop) + (static_cast<size_t>(r) * p.B + rk) * rowb,
                 static_cast<const uint8_t*>(p.S_call) + r * rowb, p.H, bf16);
    }
    for (int j = threadIdx.x; j < p.K; j += blockDim.x) {
      const size_t id = nb + n_nodes + j;
      int tok = p.row_tok[r * p.K + j];
      if (tok < 0) {  // only after an upstream failure
        atomicOr(p.err, DT_ERR_BAD_INDEX);
        tok = 0;
      }
      p.node_par[id] = cur;
      p.node_tok[id] = tok;
      p.node_dep[id] = dep + 1;
      p.node_score[id] = __fadd_rn(sc, p.row_logp[r * p.K + j]);
      p.node_rank[id] = -1;
    }
    n_nodes += p.K;
  }
  __syncthreads();
  // ---- pop: the best node still in the heap
  unsigned long long mine = 0ull;
  if (n_pop < p.B) {
    for (int id = threadIdx.x; id < n_nodes; id += blockDim.x) {
      if (p.node_rank[nb + id] >= 0) continue;
      const float key = __fadd_rn(p.node_score[nb + id],
                                  __fmul_rn(p.beta, static_cast<float>(p.node_dep[nb + id])));
      const unsigned long long k = make_key(key, static_cast<uint32_t>(id));
      mine = k > mine ? k : mine;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long x = shfl_xor_u64(mine, o);
    mine = x > mine ? x : mine;
  }
  if ((threadIdx.x & 31) == 0 && mine) atomicMax(&best, mine);
  __syncthreads();
  int next = 0, m = -1;
  if (best) {
    m = static_cast<int>(key_index(best));
    const int q = n_pop;
    const int par = p.node_par[nb + m];
    const int pr = par < 0 ? -1 : p.node_rank[nb + par];
    const int dep = p.node_dep[nb + m];
    const size_t ob = static_cast<size_t>(r) * p.B;
    const size_t mb = static_cast<size_t>(r) * p.B * p.words;
    for (int w = threadIdx.x; w < p.words; w += blockDim.x) {
      uint32_t bits = pr >= 0 ? p.mask[mb + static_cast<size_t>(pr) * p.words + w] : 0u;
      if (w == (q >> 5)) bits |= 1u << (q & 31);
      p.mask[mb + static_cast<size_t>(q) * p.words + w] = bits;
    }
    next = (q + 1 < p.B && dep < p.D) ? 1 : 0;
    if (next) {  // stage the parent's state for the state step of the next call
      const void* src = pr < 0
          ? static_cast<const void*>(static_cast<const uint8_t*>(p.S_root) + r * rowb)
          : static_cast<const void*>(static_cast<const uint8_t*>(p.S_pop) +
                                     (static_cast<size_t>(r) * p.B + pr) * rowb);
      copy_state(static_cast<uint8_t*>(p.S_stage) + r * rowb, src, p.H, bf16);
    }
    if (threadIdx.x == 0) {
      p.node_rank[nb + m] = q;
      p.parent[ob + q] = pr;
      p.token[ob + q] = p.node_tok[nb + m];
      p.depth[ob + q] = dep;
      p.score[ob + q] = p.node_score[nb + m];
      p.n_out[r] = q + 1;
      if (next) {
        p.tok_next[r] = p.node_tok[nb + m];
        p.z_row[r] = dep;  // the children of a depth-d node use z_{d+1}
      }
    }
  }
  if (threadIdx.x == 0) {
    st[0] = n_nodes;
    st[1] = n_pop + (best ? 1 : 0);
    st[2] = next ? m : cur;
    st[3] = next;
  }
}

cudaError_t launch_bestfirst_step(const BestFirstParams& p, cudaStream_t st) {
  return launch_kernel(k_bestfirst_step, dim3(p.R), dim3(kBfThreads), 0, st, p.pdl != 0, p);
}

// Stage the base logits the next call scores with: z_stage[r] = z[r][z_row[r]]
// (the depth of the children of the node that call expands).
__global__ void __launch_bounds__(256) k_bestfirst_z(const BestFirstParams p) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.y;
  const int d = p.z_row[r];
  const float* src = p.z + (static_cast<size_t>(r) * p.D + d) * p.V;
  float* dst = p.z_stage + static_cast<size_t>(r) * p.V;
  const int v0 = blockIdx.x * 1024 + threadIdx.x;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = v0 + i * 256;
    if (v < p.V) dst[v] = __ldg(src + v);
  }
}

cudaError_t launch_bestfirst_z(const BestFirstParams& p, cudaStream_t st) {
  return launch_kernel(k_bestfirst_z, dim3((p.V + 1023) / 1024, p.R), dim3(256), 0, st,
                       p.pdl != 0, p);
}

}  // namespace dt
