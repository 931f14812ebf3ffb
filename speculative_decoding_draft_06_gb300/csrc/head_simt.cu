// Head call (fused corrected logits + log-sum-exp + top-K) for fp32 weights
// on the CUDA cores, for calls that the TMA-fed fp32 kernel (head_f32.cu)
// does not take: more than 16 head rows, or weight rows that are not
// 16-byte multiples.
//
// fp32 weights keep fp32 products: TF32 tensor cores round the operands to
// 10 mantissa bits, which is far outside a 1e-5 score tolerance, so this
// path uses FFMA.  Same epilogue as the tensor-core kernel ("DARTree:
// Teaching a Chain-Trained Corrector to Think in Trees", Core Mechanism: one
// batched head call per depth yields every branch's corrected distribution).
//
// A CTA of 128 threads owns contiguous 128-row weight tiles; thread t owns
// weight row tile*128 + t and reads it straight from global memory with
// 16-byte loads, eight in flight (the row's cache lines stay in L1 between
// its loads).  The 16 head rows of a chunk are staged in shared memory in
// slices of 256 columns and read as broadcasts; each thread keeps 16
// head-row accumulators in registers, of which only the first 4 or 8 are
// computed when no more rows of the chunk carry data.
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace dt {

constexpr int kSimtH = 256;  // state columns staged per slice

template <int N>
__global__ void __launch_bounds__(128) k_head_simt(const TcParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float* sS = reinterpret_cast<float*>(smem_raw);                // [16][256] state slice
  uint8_t* tail = reinterpret_cast<uint8_t*>(sS + 16 * kSimtH);  // epilogue

  const int tid = threadIdx.x;
  const int t_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * p.n_tiles) / gridDim.x);
  const int t_end =
      static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.n_tiles) / gridDim.x);

  LogitsEpilogue<N> epi;
  epi.init(tail, p.K, p.M, p.gth);
  pdl_wait();
  pdl_trigger();
  const int mcols = p.M < N ? p.M : N;  // columns that carry data

  for (int t = t_begin; t < t_end; ++t) {
    const int row = t * kTileV + tid;
    const bool valid = row < p.rows;
    // contraction of 16 head rows c0..c0+15 against this thread's weight row
    const float* wrow = p.W_f32 + static_cast<size_t>(valid ? row : 0) * p.H;
    const bool w_vec = (p.H & 3) == 0 && (reinterpret_cast<uintptr_t>(p.W_f32) & 15) == 0;
    // the first J of the chunk's 16 head rows (the others are zero): J = 4 or
    // 8 when only that many rows of the chunk carry data
    auto dot_j = [&](auto jc, float (&acc)[16], int c0) {
      constexpr int J = decltype(jc)::value;
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.f;
      for (int h0 = 0; h0 < p.H; h0 += kSimtH) {
        const int hn = p.H - h0 < kSimtH ? p.H - h0 : kSimtH;  // columns of this slice
        __syncthreads();
        for (int e = tid; e < J * kSimtH; e += kTileV) {
          const int r = e / kSimtH, c = e % kSimtH;
          const int m = c0 + r;
          sS[e] = (m < p.M && c < hn) ? __ldg(p.S_f32 + static_cast<size_t>(m) * p.H + h0 + c)
                                      : 0.f;
        }
        __syncthreads();
        if (w_vec && (hn & 31) == 0) {
          for (int hb = 0; hb < hn; hb += 32) {  // 32 columns: eight 16-byte loads
            float4 w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
              w[q] = valid ? __ldg(reinterpret_cast<const float4*>(wrow + h0 + hb) + q)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float* sc = sS + hb + 4 * q;
#pragma unroll
              for (int j = 0; j < J; ++j) {
                const float4 sv = *reinterpret_cast<const float4*>(sc + j * kSimtH);
                acc[j] = fmaf(w[q].x, sv.x, acc[j]);
                acc[j] = fmaf(w[q].y, sv.y, acc[j]);
                acc[j] = fmaf(w[q].z, sv.z, acc[j]);
                acc[j] = fmaf(w[q].w, sv.w, acc[j]);
              }
            }
          }
        } else {
          for (int hh = 0; hh < hn; ++hh) {
            const float w = valid ? __ldg(wrow + h0 + hh) : 0.f;
#pragma unroll
            for (int j = 0; j < J; ++j) acc[j] = fmaf(w, sS[j * kSimtH + hh], acc[j]);
          }
        }
      }
    };
    auto dot16 = [&](float (&acc)[16], int c0) {
      const int live = mcols - c0;  // the same for the whole block
      if (live <= 4)
        dot_j(IntC<4>{}, acc, c0);
      else if (live <= 8)
        dot_j(IntC<8>{}, acc, c0);
      else
        dot_j(IntC<16>{}, acc, c0);
    };
    auto add_z = [&](float (&acc)[16], int c0) {
      int req_prev = -1;
      float zv = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c = c0 + j;
        const int req = c / p.rows_per_req;
        if (req != req_prev) {
          req_prev = req;
          zv = (valid && c < p.M) ? __ldg(p.z + static_cast<size_t>(req) * p.z_req_stride + row)
                                  : 0.f;
        }
        acc[j] += zv;
      }
    };
    epi.tile_begin();
    const uint32_t v0 = static_cast<uint32_t>(t * kTileV);
    if constexpr (N <= 64) {
      static_for<0, N / 16>([&](auto i) {
        constexpr int CH = decltype(i)::value;
        if (CH * 16 < mcols) {
          float acc[16];
          dot16(acc, CH * 16);
          add_z(acc, CH * 16);
          epi.template chunk_static<CH>(acc, v0, p.rows);
        }
      });
    } else {
      for (int c0 = 0; c0 < mcols; c0 += 16) {
        float acc[16];
        dot16(acc, c0);
        add_z(acc, c0);
        epi.chunk_dyn(acc, c0, v0, p.rows);
      }
    }
  }
  epi.finish(blockIdx.x, p.pm, p.ps, p.cta_stride, p.ptop, p.list_stride, p.err);
}

template <int N>
static cudaError_t launch_simt_n(const TcParams& p, int grid, cudaStream_t st) {
  const size_t smem = 16 * kSimtH * 4 + epi_smem_bytes(N, p.K);
  return launch_kernel(k_head_simt<N>, dim3(grid), dim3(128), smem, st, p.pdl != 0, p);
}

#ifndef DT_N
#error "compile head_simt.cu with -DDT_N=<16|32|64|128|256>"
#endif

#define DT_CAT2(a, b) a##b
#define DT_CAT(a, b) DT_CAT2(a, b)

cudaError_t DT_CAT(init_head_simt_attrs_, DT_N)() { return set_max_dynamic_smem(k_head_simt<DT_N>); }

cudaError_t DT_CAT(launch_head_simt_, DT_N)(const TcParams& p, int grid, cudaStream_t st) {
  return launch_simt_n<DT_N>(p, grid, st);
}

}  // namespace dt
