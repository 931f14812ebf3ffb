// Batched head contraction on the 5th-generation tensor cores (bf16 weights).
//
// One kernel shape serves both dense steps of a DARTree head call:
//   * corrected logits  ell[m, v] = z_d[v] + sum_h S[m, h] Wout[v, h]
//     ("DARTree: Teaching a Chain-Trained Corrector to Think in Trees", Core
//     Mechanism: a single batched head call per depth yields a corrected
//     distribution for every branch), fused with the online log-sum-exp and the
//     per-row top-K (LogitsEpilogue) -- the logits never reach HBM;
//   * state step        S'[m, h] = bf16(tanh(sum_j A[h, j] S[m, j] + E[tok_m, h]))
//     ("Technische Samenvatting: DARTree", Methodologie 1: the kept branches
//     carry their correction states forward).
//
// Swap-AB: the weight matrix supplies the 128-row MMA "M" side (vocabulary or
// hidden rows) and the head rows are the MMA N (16..256), so tiny head
// batches still fill the tensor core's M dimension.  Both operands are
// K-major bf16 tiles of 128 B rows loaded by TMA with the 128-byte swizzle;
// the fp32 accumulator lives in TMEM (two buffers, so the epilogue of tile i
// overlaps the MMAs of tile i+1).
//
// Warp roles: warps 0..4G-1 epilogue (G warpgroups; TMEM lane quarter =
// warp % 4), warp 4G TMA producer, warp 4G+1 TMEM allocator + single-thread
// MMA issuer.  The logits kernel for more than 16 head rows runs two epilogue
// warpgroups, which take alternate 16-row chunks of each accumulator tile, so
// every SM sub-partition has two epilogue warps to overlap the latency of the
// top-K updates.  Each CTA owns a contiguous range of 128-row weight tiles
// (persistent, one CTA per SM).
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dt {

constexpr int kDefaultMaxStages = 8;

template <int N>
struct TcLayout {
  static constexpr int kABytes = kTileV * kTileH * 2;  // 16 KB
  static constexpr int kBBytes = N * kTileH * 2;       // N rows of 128 B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * N < 32 ? 32 : 2 * N;
};

// Epilogue warpgroups of a kernel variant.
template <int N, bool kLogits>
struct TcRoles {
  static constexpr int kGroups = (kLogits && N > 16) ? 2 : 1;
  static constexpr int kEpiWarps = 4 * kGroups;
  static constexpr int kProducer = kEpiWarps;
  static constexpr int kMma = kEpiWarps + 1;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
};

// State step epilogue (all 128 epilogue threads; thread = hidden unit `row`).
// Unsplit: output row q takes column slot[q] of U = A S_in (its parent's
// row), adds E[tok[q]], tanh, rounds to bf16 (zeros past M_out); the rows'
// slots and tokens are staged in shared memory, and each batch of 16 rows
// issues its embedding loads together.  Split-K: this CTA's partial U for
// every input row goes to part[split][c][hidden]; k_state_finish sums the
// splits and finishes the rows.
template <int N>
__device__ __forceinline__ void state_epilogue(const TcParams& p, uint32_t tbase, int tile,
                                               int split, int warp, int lane, int row,
                                               bool valid) {
  const int lr = warp * 32 + lane;
  if (p.n_split > 1) {
    float* mine = p.part + static_cast<size_t>(split) * kMaxRows * p.H + row;
    for (int c0 = 0; c0 < p.M; c0 += 16) {
      float x[16];
      tmem_ld16(tbase + c0, x);
      if (valid) {
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (c0 + j < p.M) mine[static_cast<size_t>(c0 + j) * p.H] = x[j];
      }
    }
    return;
  }
  constexpr int kB = 16;  // output rows per batch
  __shared__ int s_col[kMaxRows], s_tok[kMaxRows];
  const int n_out = pad_rows(p.M_out);
  bool bad = false;
  for (int q = lr; q < n_out; q += 128) {
    int col = q < p.M_out ? __ldg(p.slot + q) : 0;
    int tok = q < p.M_out ? __ldg(p.tok + q) : 0;
    if (col < 0 || col >= p.M) col = 0;  // (never, unless upstream failed)
    if (tok < 0 || tok >= p.V_tok) {     // only after an upstream failure
      bad = true;
      tok = 0;
    }
    s_col[q] = col;
    s_tok[q] = tok;
  }
  if (bad) atomicOr(p.err, DT_ERR_BAD_INDEX);
  asm volatile("bar.sync 1, 128;" ::: "memory");
  for (int q0 = 0; q0 < n_out; q0 += kB) {
    float u[kB], e[kB];
    if (valid) {
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int q = q0 + j < n_out ? q0 + j : 0;
        e[j] = bf16_bits_to_float(__ldg(p.E_bf16 + static_cast<size_t>(s_tok[q]) * p.H + row));
      }
    }
#pragma unroll
    for (int j = 0; j < kB; ++j) {
      const int q = q0 + j < n_out ? q0 + j : 0;
      uint32_t r;
      asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];"
                   : "=r"(r)
                   : "r"(tbase + static_cast<uint32_t>(s_col[q])));
      u[j] = __uint_as_float(r);
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    if (valid) {
#pragma unroll
      for (int j = 0; j < kB; ++j) {
        const int q = q0 + j;
        if (q < n_out) {
          const float out = q < p.M_out ? tanhf(u[j] + e[j]) : 0.f;
          p.S_out_bf16[static_cast<size_t>(q) * p.H + row] = float_to_bf16_bits(out);
        }
      }
    }
  }
}

template <int N, bool kLogits>
__global__ void __launch_bounds__(TcRoles<N, kLogits>::kThreads, 1)
    k_head_tc(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_s,
              const TcParams p) {
  using L = TcLayout<N>;
  using R = TcRoles<N, kLogits>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int S = p.stages;
  uint8_t* stage_base = smem;
  uint8_t* after = smem + static_cast<size_t>(S) * L::kStageBytes;
  uint8_t* epi_smem = after;  // logits epilogue: lists, transposed chunks, row state
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(after + (kLogits ? epi_smem_bytes(N, p.K, R::kGroups) : 0));
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // work of this CTA: logits -- tiles blockIdx.x, blockIdx.x + gridDim.x,
  // ... over the whole contraction (the CTAs stream neighbouring tiles at
  // the same time); state -- one tile and one slice of the contraction
  // (split-K, reduced through global scratch).  tile_of maps the CTA's
  // i-th tile to its index.
  const int nk_all = p.H / kTileH;
  int t_begin, t_end, kb_begin = 0, kb_end = nk_all, split = 0;
  if constexpr (kLogits) {
    t_begin = 0;
    t_end = (p.n_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
            static_cast<int>(gridDim.x);
  } else {
    t_begin = blockIdx.x / p.n_split;
    t_end = t_begin + 1;
    split = blockIdx.x % p.n_split;
    kb_begin = split * nk_all / p.n_split;
    kb_end = (split + 1) * nk_all / p.n_split;
  }
  // The contraction of each tile starts at a tile-dependent k-block and
  // wraps around.  Tiles are 128 consecutive weight rows, so at a common
  // k-block every CTA would read 128-byte pieces at the same offset of
  // power-of-two-strided rows -- the same low address bits everywhere, which
  // concentrates the stream on a few DRAM channels.  Rotating the start
  // spreads concurrent CTAs over different offsets.
  const int kb_span = kb_end - kb_begin;
  auto tile_of = [&](int ti) {
    return kLogits ? static_cast<int>(blockIdx.x) + ti * static_cast<int>(gridDim.x) : ti;
  };
  auto kb_at = [&](int t, int i) {
    int j = i + (t * 5) % kb_span;
    if (j >= kb_span) j -= kb_span;
    return kb_begin + j;
  };

  if (warp == R::kMma) tmem_alloc<L::kTmemCols>(tmem_slot);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], R::kEpiWarps);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == R::kProducer && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_s);
  }
  LogitsEpilogue<N, R::kGroups> epi;
  if (kLogits && warp < R::kEpiWarps) epi.init(epi_smem, p.K, p.M, p.gth, p.gmx);
  __shared__ int epi_go[2];  // per-tile decision of each epilogue warpgroup
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // prologue done; from here on the kernel reads and writes shared buffers.
  // A state step whose operands were complete before the previous kernel
  // began streams them at once and waits only in its epilogue (the unsplit
  // epilogue reads the previous kernel's selection (slot, tok); the split
  // one waits after storing its partials) -- the contraction then overlaps
  // the previous kernel.
  const bool early = !kLogits && p.early_operands;
  if (!early) pdl_wait();
  pdl_trigger();

  if (warp == R::kProducer) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_s = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      for (int ti = t_begin; ti < t_end && !*abort_flag; ++ti) {
        const int t = tile_of(ti);
        for (int i = 0; i < kb_span; ++i) {
          const int kb = kb_at(t, i);
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.err, p.wait_limit)) {
            *abort_flag = 1;
            break;
          }
          uint8_t* a_dst = stage_base + static_cast<size_t>(stage) * L::kStageBytes;
          uint8_t* b_dst = a_dst + L::kABytes;
          mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
          if (kLogits && p.w_tiled)
            tma_load_2d(a_dst, &tmap_w, &full[stage], 0, (t * p.w_nk + kb) * kTileV, pol_w);
          else
            tma_load_2d(a_dst, &tmap_w, &full[stage], kb * kTileH, t * kTileV, pol_w);
          tma_load_2d(b_dst, &tmap_s, &full[stage], kb * kTileH, 0, pol_s);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // drain: every issued copy must have landed before the CTA may exit
      const long long first = issued > S ? issued - S : 0;
      for (long long n = first; n < issued; ++n) {
        const int s = static_cast<int>(n % S);
        const uint32_t par = static_cast<uint32_t>((n / S) & 1);
        if (!mbar_wait(&full[s], par, p.err)) break;
      }
    }
  } else if (warp == R::kMma) {
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_m128<N>();
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int ti = t_begin; ti < t_end && !*abort_flag; ++ti, ++it) {
        const int t = tile_of(ti);
        const int a = it & 1;
        if (!mbar_wait(&tempty[a], (static_cast<uint32_t>(it >> 1) & 1u) ^ 1u, p.err,
                       p.wait_limit)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * N);
        bool ok = true;
        for (int i = 0; i < kb_span; ++i) {
          if (!mbar_wait(&full[stage], phase, p.err, p.wait_limit)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr =
              smem_u32(stage_base + static_cast<size_t>(stage) * L::kStageBytes);
          const uint32_t b_addr = a_addr + L::kABytes;
#pragma unroll
          for (int k = 0; k < kTileH / 16; ++k) {
            tc_mma_bf16(d_tmem, smem_desc_sw128(a_addr + k * 32), smem_desc_sw128(b_addr + k * 32),
                        idesc, (i != 0 || k != 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[a]);
      }
      // all issued MMAs complete before TMEM is released
      tc_commit(done);
      mbar_wait(done, 0, p.err);
    }
  } else {
    // --------------------------------------------------------- epilogue
    // The warps of a group synchronise with a named barrier, so they must
    // take every decision together: one thread per group waits for the
    // accumulator and broadcasts whether to go on (a timed-out wait ends all
    // four warps' loops at once).  Every group waits for every tile, so each
    // arrival on tempty belongs to the tile it was meant for.
    // Split-K partials need nothing from the previous kernel and go to a
    // scratch that only the finish kernel after this one reads: they are
    // stored first, and the wait (which keeps the kernels' completion order)
    // comes after them.
    const bool wait_last = early && p.n_split > 1;
    if (early && !wait_last) pdl_wait();
    int it = 0;
    const int grp = warp >> 2;
    const int wq = warp & 3;  // TMEM lane quarter
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    // all rows of one request (the usual case): one base logit per thread
    // and tile, loaded before the accumulator wait
    const bool one_req = kLogits && p.rows_per_req >= p.M;
    for (int ti = t_begin; ti < t_end; ++ti, ++it) {
      const int t = tile_of(ti);
      const int a = it & 1;
      const int row = t * kTileV + wq * 32 + lane;  // vocabulary (or hidden) index
      const bool valid = row < p.rows;
      float z1 = 0.f;
      if constexpr (kLogits) {
        if (one_req && valid) z1 = __ldg(p.z + row);
        epi.tile_begin();  // the rows' global bounds, also ahead of the wait
      }
      if ((threadIdx.x & 127) == 0) {
        const bool ok = !*abort_flag &&
                        mbar_wait(&tfull[a], static_cast<uint32_t>(it >> 1) & 1u, p.err,
                                  p.wait_limit);
        if (!ok) *abort_flag = 1;
        epi_go[grp] = ok;
      }
      asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory");
      if (!epi_go[grp]) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + lane_base + static_cast<uint32_t>(a * N);
      if constexpr (kLogits) {
        int req_prev = -1;
        float zv = 0.f;
        auto add_z = [&](float (&x)[16], int c0) {
          if (one_req) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] += z1;
            return;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c = c0 + j;
            const int req = c / p.rows_per_req;
            if (req != req_prev) {
              req_prev = req;
              zv = (valid && c < p.M) ? __ldg(p.z + static_cast<size_t>(req) * p.z_req_stride + row)
                                      : 0.f;
            }
            x[j] += zv;
          }
        };
        const uint32_t v0 = static_cast<uint32_t>(t * kTileV);
        if constexpr (N <= 64) {
          static_for<0, N / 16>([&](auto i) {
            constexpr int CH = decltype(i)::value;
            if (CH % R::kGroups == grp && CH * 16 < p.M) {  // same for the group's warps
              float x[16];
              tmem_ld16(tbase + CH * 16, x);
              add_z(x, CH * 16);
              epi.template chunk_static<CH>(x, v0, p.rows);
            }
          });
        } else {
          const int c_end = (p.M + 15) & ~15;
          for (int c0 = 16 * grp; c0 < c_end; c0 += 16 * R::kGroups) {
            float x[16];
            tmem_ld16(tbase + c0, x);
            add_z(x, c0);
            epi.chunk_dyn(x, c0, v0, p.rows);
          }
        }
      } else {
        state_epilogue<N>(p, tbase, t, split, warp, lane, row, valid);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
    }
    if constexpr (kLogits) {
      epi.finish(blockIdx.x, p.pm, p.ps, p.cta_stride, p.ptop, p.list_stride, p.err);
    }
    if (wait_last) pdl_wait();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == R::kMma) {
    tc_fence_after();
    tmem_dealloc<L::kTmemCols>(tmem_base);
  }
}

template <int N, bool kLogits>
static cudaError_t launch_tc_n(const CUtensorMap& tw, const CUtensorMap& ts, const TcParams& p,
                               int grid, cudaStream_t st) {
  using L = TcLayout<N>;
  using R = TcRoles<N, kLogits>;
  size_t fixed = 1024 + (kLogits ? epi_smem_bytes(N, p.K, R::kGroups) : 0) + 64 * 8 + 64;
  // per-SM shared memory is 228 KB, 1 KB of it reserved per resident CTA,
  // less the kernel's own static shared memory (at most 4 KB)
  auto stages_for = [&](int cps) -> int {
    const size_t budget = (cps == 1 ? 227 * 1024 : 228 * 1024 / cps - 1024) - 4096;
    return budget > fixed ? static_cast<int>((budget - fixed) / L::kStageBytes) : 0;
  };
  // two CTAs per SM only where both fit with a real pipeline, else one
  int cps = p.ctas_per_sm > 1 ? p.ctas_per_sm : 1;
  if (cps > 1 && stages_for(cps) < 3) cps = 1;
  int stages = stages_for(cps);
  const int cap = p.max_stages > 0 ? p.max_stages : kDefaultMaxStages;
  if (stages > cap) stages = cap;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  TcParams q = p;
  q.stages = stages;
  const size_t smem = fixed + static_cast<size_t>(stages) * L::kStageBytes;
  return launch_kernel(k_head_tc<N, kLogits>, dim3(grid), dim3(R::kThreads), smem, st, q.pdl != 0, tw, ts,
                       q);
}

#ifndef DT_N
#error "compile head_tc.cu with -DDT_N=<16|32|64|128|256>"
#endif

#define DT_CAT2(a, b) a##b
#define DT_CAT(a, b) DT_CAT2(a, b)

cudaError_t DT_CAT(init_head_tc_attrs_, DT_N)() {
  cudaError_t e = set_max_dynamic_smem(k_head_tc<DT_N, true>);
  if (e != cudaSuccess) return e;
  return set_max_dynamic_smem(k_head_tc<DT_N, false>);
}

cudaError_t DT_CAT(launch_head_tc_, DT_N)(bool logits, const CUtensorMap& tw, const CUtensorMap& ts,
                                           const TcParams& p, int grid, cudaStream_t st) {
  return logits ? launch_tc_n<DT_N, true>(tw, ts, p, grid, st)
                : launch_tc_n<DT_N, false>(tw, ts, p, grid, st);
}

}  // namespace dt
