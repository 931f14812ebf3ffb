// Head call with fp32 weights and at most 16 head rows.
//
// Corrected logits ell[m, v] = z_d[v] + sum_h S[m, h] Wout[v, h] for every
// head row at once ("DARTree: Teaching a Chain-Trained Corrector to Think in
// Trees", Core Mechanism: one batched head call per depth), fused with the
// online log-sum-exp and the per-row top-K (LogitsEpilogue), as in the
// tensor-core kernel.  fp32 weights keep fp32 products (TF32 would round the
// operands far outside a 1e-5 score tolerance), so the products are FFMA.
//
// With fp32 weights the output projection is small (33 MB at V = 32000,
// H = 256) and the call is bound by latency, not by a pipe.  A CTA of 640
// threads owns 128-row tiles.  Warps 4-19 compute the dot products: four
// threads share a weight row (dot_tiles: the row's four threads read 64
// contiguous bytes per load, the loads software-pipelined over the CTA's
// tiles) and multiply them with the head rows (staged in shared memory);
// the four partial sums meet by two shuffles.  Warps 0-3 run the epilogue only (thread t = vocabulary entry t
// of the tile): the tile sums pass through a double buffer in shared memory
// with named barriers (full: the dot warps arrive, the epilogue warps wait;
// empty: the reverse), so the epilogue of tile i, which is longest on a
// CTA's first tile while its lists fill, runs under the loads of tile i + 1
// instead of delaying a quarter of them.  The epilogue warps load a tile's
// base logits and row bounds before they wait for its sums.
//
// With A given, the next depth's state contraction U = A S_in rides along:
// A's H rows are ceil(H / 128) more tiles after the vocabulary's, whose sums
// the epilogue warps store as U[m][h] (the selection then finishes the step
// as tanh(U[parent] + E[token])).  The call is latency-bound, so the extra
// tiles cost little, and the state step needs no launch of its own.
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dt {
namespace {

constexpr int kF32Threads = 640;  // 4 epilogue warps + 16 dot-product warps
constexpr int kF32Epi = 128;      // epilogue threads (warps 0-3)
constexpr int kF32Chunk = 256;    // columns per load round (16 float4 per thread)

// named barriers (0 is __syncthreads; the epilogue uses 1 and 3)
__device__ __forceinline__ void nb_sync(int id) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kF32Threads) : "memory");
}
__device__ __forceinline__ void nb_arrive(int id) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(kF32Threads) : "memory");
}
constexpr int kBarStage = 2;  // the head rows are staged
constexpr int kBarFull = 4;   // + buffer: the tile sums are written
constexpr int kBarEmpty = 6;  // + buffer: the epilogue has read them

// The head rows (written by the previous kernel) into shared memory, every
// thread's share, after the wait for that kernel; then all 640 threads meet
// (a named barrier: the two warp groups reach it from different code).
__device__ __forceinline__ void stage_head_rows(const TcParams& p, float* sS, int ldS) {
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e < 16 * ldS; e += kF32Threads) {
    const int j = e / ldS, c = e % ldS;
    sS[e] = (j < p.M && c < p.H) ? __ldcg(p.S_f32 + static_cast<size_t>(j) * p.H + c) : 0.f;
  }
  nb_sync(kBarStage);
}

// The dot-product warps' loop over this CTA's tiles for J live head rows.
// Thread (row r_in, quarter part) reads the row's float4 granules part,
// part + 4, ... of each 256-column chunk, in batches of NB (8 for up to 4
// head rows, else 4: two batches' registers beside J accumulators).
// The batches of all the CTA's tiles form one stream, software-pipelined:
// the loads of batch b + 2 are issued once batch b is multiplied (also
// across a tile's end, so the next tile's loads are in flight during the
// tile's reduction and hand-over), and the memory system does not wait for
// the FFMAs.  A tile's four partial sums per row meet by two shuffles and
// go to the tile-sum buffer (double-buffered with the epilogue warps).
template <int J, int NB>
__device__ __forceinline__ void dot_tiles(const TcParams& p, float* sS, int ldS, float* sX,
                                          int t_begin, int n_t, int r_in, int part) {
  constexpr int kPer = 16 / NB;  // batches per chunk
  const int per_tile = kPer * ((p.H + kF32Chunk - 1) / kF32Chunk);  // batches per tile (even)
  const int total = n_t * per_tile;
  auto load = [&](int bt, float4 (&w)[NB]) {
    const int i = bt / per_tile, rem = bt - i * per_tile;
    const int c0 = (rem / kPer) * kF32Chunk, k0 = (rem % kPer) * NB;
    const int t = t_begin + i;
    const bool st = t >= p.n_tiles;  // a tile of A's rows
    const int row = (st ? t - p.n_tiles : t) * kTileV + r_in;
    const bool valid = row < (st ? p.H : p.rows);
    const float4* wrow = reinterpret_cast<const float4*>(
        (st ? p.A_f32 : p.W_f32) + static_cast<size_t>(valid ? row : 0) * p.H + c0);
    const int hn = p.H - c0 < kF32Chunk ? p.H - c0 : kF32Chunk;
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int g = part + 4 * (k0 + k);
      w[k] = (valid && 4 * g < hn) ? __ldg(wrow + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto fma = [&](int bt, const float4 (&w)[NB], float (&acc)[J]) {
    const int rem = bt % per_tile;
    const int c0 = (rem / kPer) * kF32Chunk, k0 = (rem % kPer) * NB;
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int col = c0 + 4 * (part + 4 * (k0 + k));
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const float4 s = *reinterpret_cast<const float4*>(sS + j * ldS + col);
        acc[j] = fmaf(w[k].x, s.x, acc[j]);
        acc[j] = fmaf(w[k].y, s.y, acc[j]);
        acc[j] = fmaf(w[k].z, s.z, acc[j]);
        acc[j] = fmaf(w[k].w, s.w, acc[j]);
      }
    }
  };
  float acc[J];
#pragma unroll
  for (int j = 0; j < J; ++j) acc[j] = 0.f;
  float4 wa[NB], wb[NB];
  // the weights are constant: the first two batches go out before the wait
  // for the previous kernel, and land while the head rows are staged
  if (total > 0) {
    load(0, wa);
    load(1, wb);
  }
  stage_head_rows(p, sS, ldS);
  for (int bt = 0; bt < total; bt += 2) {  // a pair of batches of one tile
    fma(bt, wa, acc);
    if (bt + 2 < total) load(bt + 2, wa);
    fma(bt + 1, wb, acc);
    if (bt + 3 < total) load(bt + 3, wb);
    if ((bt + 2) % per_tile == 0) {  // the tile's end
      const int i = bt / per_tile, b = i & 1;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        acc[j] += __shfl_xor_sync(kFullMask, acc[j], 1);
        acc[j] += __shfl_xor_sync(kFullMask, acc[j], 2);
      }
      if (i >= 2) nb_sync(kBarEmpty + b);  // the epilogue has read tile i - 2
      if (part == 0) {
        float* X = sX + b * kTileV * 17;
#pragma unroll
        for (int j = 0; j < 16; ++j) X[r_in * 17 + j] = j < J ? acc[j] : 0.f;
      }
      nb_arrive(kBarFull + b);
#pragma unroll
      for (int j = 0; j < J; ++j) acc[j] = 0.f;
    }
  }
}

// J: at least the live head rows (4, 8 or 16), NB: the dot-product batch;
// one instantiation per row count keeps each kernel's code to its own loop.
template <int J, int NB>
__global__ void __launch_bounds__(kF32Threads, 1) k_head_f32(const TcParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int ldS = (p.H + kF32Chunk - 1) / kF32Chunk * kF32Chunk;  // padded row pitch
  float* sS = reinterpret_cast<float*>(smem_raw);                   // [16][ldS] head rows
  float* sX = sS + 16 * ldS;                                        // [2][128][17] tile sums
  uint8_t* epi_smem = reinterpret_cast<uint8_t*>(sX + 2 * kTileV * 17);

  const int tid = threadIdx.x, warp = tid >> 5;
  // vocabulary tiles, then (with A) the state tiles
  const int n_all = p.n_tiles + (p.A_f32 ? (p.H + kTileV - 1) / kTileV : 0);
  const int t_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * n_all) / gridDim.x);
  const int t_end = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * n_all) / gridDim.x);
  const int n_t = t_end - t_begin;  // this CTA's tiles

  LogitsEpilogue<16> epi;
  if (warp < 4) epi.init(epi_smem, p.K, p.M, p.gth, p.gmx);

  if (warp >= 4) {
    // ---- dot-product warps: 128 weight rows x 4 quarters
    const int dt = tid - kF32Epi;
    const int r_in = dt >> 2, part = dt & 3;
    dot_tiles<J, NB>(p, sS, ldS, sX, t_begin, n_t, r_in, part);
    return;
  }

  // ---- epilogue warps: thread tid = vocabulary entry tid of the tile
  stage_head_rows(p, sS, ldS);
  const bool one_req = p.rows_per_req >= p.M;
  for (int i = 0; i < n_t; ++i) {
    const int b = i & 1, t = t_begin + i;
    const bool st_tile = t >= p.n_tiles;
    // the row bounds and the base logits, loaded before the sums are ready
    if (!st_tile) epi.tile_begin();
    const int v = t * kTileV + tid;
    const bool vv = !st_tile && v < p.rows;
    const float z1 = (one_req && vv) ? __ldg(p.z + v) : 0.f;
    nb_sync(kBarFull + b);
    const float* X = sX + b * kTileV * 17;
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = X[tid * 17 + j];
    if (i + 2 < n_t) nb_arrive(kBarEmpty + b);  // the dot warps may refill buffer b
    if (st_tile) {  // U[m][h] = (A S_in)[h, m], coalesced over h
      const int hh = (t - p.n_tiles) * kTileV + tid;
      if (hh < p.H) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < p.M) p.U_f32[static_cast<size_t>(j) * p.H + hh] = x[j];
      }
      continue;
    }
    if (one_req) {
#pragma unroll
      for (int j = 0; j < 16; ++j) x[j] += z1;
    } else {
      int req_prev = -1;
      float zv = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int req = j / p.rows_per_req;
        if (req != req_prev) {
          req_prev = req;
          zv = (vv && j < p.M) ? __ldg(p.z + static_cast<size_t>(req) * p.z_req_stride + v) : 0.f;
        }
        x[j] += zv;
      }
    }
    epi.template chunk_static<0>(x, static_cast<uint32_t>(t * kTileV), p.rows);
  }
  epi.finish(blockIdx.x, p.pm, p.ps, p.cta_stride, p.ptop, p.list_stride, p.err);
}

size_t f32_smem(int H, int K) {
  const int ldS = (H + kF32Chunk - 1) / kF32Chunk * kF32Chunk;
  return static_cast<size_t>(16) * ldS * 4 + static_cast<size_t>(2) * kTileV * 17 * 4 +
         epi_smem_bytes(16, K);
}

}  // namespace

bool head_f32_fits(int M, int H, int K) {
  return M >= 1 && M <= 16 && H % 4 == 0 && f32_smem(H, K) <= 200 * 1024;
}

cudaError_t init_head_f32_attrs() {
  cudaError_t e = set_max_dynamic_smem(k_head_f32<4, 8>);
  if (e == cudaSuccess) e = set_max_dynamic_smem(k_head_f32<8, 4>);
  return e != cudaSuccess ? e : set_max_dynamic_smem(k_head_f32<16, 4>);
}

cudaError_t launch_head_f32(const TcParams& p, int grid, cudaStream_t st) {
  if (!head_f32_fits(p.M, p.H, p.K) || (reinterpret_cast<uintptr_t>(p.W_f32) & 15) ||
      (p.A_f32 && ((reinterpret_cast<uintptr_t>(p.A_f32) & 15) || !p.U_f32)))
    return cudaErrorInvalidValue;
  auto k = p.M <= 4 ? k_head_f32<4, 8> : p.M <= 8 ? k_head_f32<8, 4> : k_head_f32<16, 4>;
  return launch_kernel(k, dim3(grid), dim3(kF32Threads), f32_smem(p.H, p.K), st,
                       p.pdl != 0, p);
}

}  // namespace dt
