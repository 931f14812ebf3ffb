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
// H = 256) and the call is bound by latency, not by a pipe: with one thread
// per weight row and four warps per SM, each thread waited through rounds of
// dependent loads.  Here a CTA of 512 threads owns 128-row tiles and four
// threads share a weight row: thread (row, part) reads the row's float4
// granules part, part + 4, part + 8, ... of each 256-column chunk -- its 16
// loads issued before any is used, and the four threads of a row together
// read 64 contiguous bytes per load -- multiplies them with the head rows
// (staged in shared memory), and the four partial sums meet by two shuffles.
// Sixteen warps per SM keep enough loads in flight.  The sums of a tile then
// go through shared memory to warps 0-3 (thread t = vocabulary entry t, the
// epilogue's layout), which run the epilogue while the other warps start the
// next tile's loads.
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dt {
namespace {

constexpr int kF32Threads = 512;
constexpr int kF32Chunk = 256;  // columns per load round (16 float4 per thread)

// granules g = part + 4 k of a 256-column chunk (columns c0 + 4 g .. + 3),
// in batches of NB loads issued together (16 for up to 8 head rows; two
// batches of 8 for 16 rows, to stay within the registers of 512 threads)
template <int J, int NB>
__device__ __forceinline__ void chunk_dot(const float* wrow, bool valid, int part, int hn,
                                          const float* sS, int ldS, int c0, float (&acc)[16]) {
#pragma unroll
  for (int k0 = 0; k0 < 16; k0 += NB) {
    float4 w[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      const int g = part + 4 * (k0 + k);
      w[k] = (valid && 4 * g < hn) ? __ldg(reinterpret_cast<const float4*>(wrow + c0) + g)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
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
  }
}

__global__ void __launch_bounds__(kF32Threads, 1) k_head_f32(const TcParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int ldS = (p.H + kF32Chunk - 1) / kF32Chunk * kF32Chunk;  // padded row pitch
  float* sS = reinterpret_cast<float*>(smem_raw);                   // [16][ldS] head rows
  float* sX = sS + 16 * ldS;                                        // [2][128][17] tile sums
  uint8_t* epi_smem = reinterpret_cast<uint8_t*>(sX + 2 * kTileV * 17);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int r_in = tid >> 2, part = tid & 3;  // weight row of the tile, its quarter
  const int t_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * p.n_tiles) / gridDim.x);
  const int t_end =
      static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.n_tiles) / gridDim.x);

  LogitsEpilogue<16> epi;
  if (warp < 4) epi.init(epi_smem, p.K, p.M, p.gth, p.gmx);
  pdl_wait();  // the head rows come from the previous kernel
  pdl_trigger();
  for (int e = tid; e < 16 * ldS; e += kF32Threads) {
    const int j = e / ldS, c = e % ldS;
    sS[e] = (j < p.M && c < p.H) ? __ldcg(p.S_f32 + static_cast<size_t>(j) * p.H + c) : 0.f;
  }
  __syncthreads();
  const int J = p.M;  // live head rows (1..16)
  const bool one_req = p.rows_per_req >= p.M;
  int buf = 0;
  for (int t = t_begin; t < t_end; ++t, buf ^= 1) {
    // the epilogue warps' row bounds, read while the tile's loads are in flight
    if (warp < 4) epi.tile_begin();
    // ---- all 512 threads: the tile's dot products
    const int row = t * kTileV + r_in;
    const bool valid = row < p.rows;
    const float* wrow = p.W_f32 + static_cast<size_t>(valid ? row : 0) * p.H;
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int c0 = 0; c0 < p.H; c0 += kF32Chunk) {
      const int hn = p.H - c0 < kF32Chunk ? p.H - c0 : kF32Chunk;
      if (J <= 4)
        chunk_dot<4, 16>(wrow, valid, part, hn, sS, ldS, c0, acc);
      else if (J <= 8)
        chunk_dot<8, 16>(wrow, valid, part, hn, sS, ldS, c0, acc);
      else
        chunk_dot<16, 8>(wrow, valid, part, hn, sS, ldS, c0, acc);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      acc[j] += __shfl_xor_sync(kFullMask, acc[j], 1);
      acc[j] += __shfl_xor_sync(kFullMask, acc[j], 2);
    }
    float* X = sX + buf * kTileV * 17;
    if (part == 0) {
#pragma unroll
      for (int j = 0; j < 16; ++j) X[r_in * 17 + j] = acc[j];
    }
    // the tile's sums are complete, and (double buffer) the epilogue of the
    // tile before last has read its buffer
    __syncthreads();
    if (warp >= 4) continue;
    // ---- warps 0-3: thread tid = vocabulary entry tid of the tile
    const int v = t * kTileV + tid;
    const bool vv = v < p.rows;
    float x[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = X[tid * 17 + j];
    if (one_req) {
      const float z1 = vv ? __ldg(p.z + v) : 0.f;
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
  if (warp < 4) epi.finish(blockIdx.x, p.pm, p.ps, p.cta_stride, p.ptop, p.list_stride, p.err);
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

cudaError_t init_head_f32_attrs() { return set_max_dynamic_smem(k_head_f32); }

cudaError_t launch_head_f32(const TcParams& p, int grid, cudaStream_t st) {
  if (!head_f32_fits(p.M, p.H, p.K) || (reinterpret_cast<uintptr_t>(p.W_f32) & 15))
    return cudaErrorInvalidValue;
  return launch_kernel(k_head_f32, dim3(grid), dim3(kF32Threads), f32_smem(p.H, p.K), st,
                       p.pdl != 0, p);
}

}  // namespace dt
