// Block-wide selection helpers shared by the selection kernels: a bitonic
// sort of 64-bit keys in shared memory and a tree fold of per-warp sorted
// lists (keys as in common.cuh: value desc, index asc).
#pragma once
#include <cstdint>

#include "common.cuh"

namespace dt {

// Sort keys[0..n) descending; n is a power of two.
inline __device__ void block_sort_desc(uint64_t* keys, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint64_t a = keys[i], b = keys[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// Fold the per-warp lists wl[w] (descending, p2 keys) into warp 0's `v` by
// a pairwise tree: log2(warps) levels of one merge each.  All threads of the
// block call it; on return warp 0's lanes 0..p2-1 hold the best p2 keys.
inline __device__ uint64_t block_tree_merge(uint64_t v, uint64_t (*wl)[32], int p2) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  wl[warp][lane] = lane < p2 ? v : 0ull;
  __syncthreads();
  for (int stride = 1; stride < nw; stride <<= 1) {
    if ((warp & (2 * stride - 1)) == 0 && warp + stride < nw) {
      uint64_t y;
      merge_operands(wl[warp + stride], p2, p2, v, y);
      v = warp_merge_desc(v, y, p2);
      __syncwarp();
      wl[warp][lane] = lane < p2 ? v : 0ull;
    }
    __syncthreads();
  }
  return v;
}

// The k largest of n distinct keys keys[0..n) (shared memory) into
// out[0..k) in descending order: key i belongs at out[r], r = the number of
// keys above it, whenever r < k (each count stops once it reaches k, so
// most keys are dropped after a short scan).  Slots of out beyond n keep
// their contents.  All threads of the block call it; the caller
// synchronises before reading out.
inline __device__ void block_rank_select(const uint64_t* keys, int n, int k, uint64_t* out) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint64_t x = keys[i];
    int above = 0, j = 0;
    for (; j + 8 <= n && above < k; j += 8) {
#pragma unroll
      for (int u = 0; u < 8; ++u) above += keys[j + u] > x ? 1 : 0;
    }
    for (; j < n && above < k; ++j) above += keys[j] > x ? 1 : 0;
    if (above < k) out[above] = x;
  }
}

// Radix select of the k largest of n distinct 64-bit keys (k <= n).
// Most significant digit first, 8 bits per pass: each pass histograms the
// digit of the keys that share the prefix found so far, and one warp picks
// the digit whose class holds the k-th largest (scanning the 256 bins from
// the top).  When that class is taken whole, its prefix is the threshold and
// the passes stop early; otherwise the next pass refines within the class.
// Then the keys at or above the threshold (exactly k) are gathered into
// out[0..k) in any order.  keys may be in shared or global memory; out,
// hist (256 counters) and sh (4 ints) in shared memory.  All threads of the
// block call it; returns the threshold.
inline __device__ uint64_t block_radix_select(const uint64_t* keys, int n, int k, uint64_t* out,
                                              unsigned* hist, int* sh) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint64_t prefix = 0ull, mask = 0ull;
  int kr = k;  // rank of the k-th largest within the current class
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const uint64_t key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 255 - 8l .. 248 - 8l (highest digits first)
      unsigned c[8], tot = 0u;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        tot += c[j];
      }
      unsigned inc = tot;  // inclusive prefix over lanes
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += y;
      }
      const unsigned exc = inc - tot;
      const bool here = exc < static_cast<unsigned>(kr) && static_cast<unsigned>(kr) <= inc;
      if (here) {
        unsigned above = exc;
        int j = 0;
        while (above + c[j] < static_cast<unsigned>(kr)) above += c[j++];
        sh[0] = 255 - 8 * lane - j;                        // the digit
        sh[1] = static_cast<int>(above);                   // keys of the class above it
        sh[2] = static_cast<int>(c[j]);                    // keys with this digit
      }
    }
    __syncthreads();
    const int digit = sh[0], above = sh[1], cnt = sh[2];
    prefix |= static_cast<uint64_t>(digit) << shift;
    mask |= 255ull << shift;
    kr -= above;
    __syncthreads();
    if (kr == cnt) break;  // the whole class is selected: prefix is the threshold
  }
  if (threadIdx.x == 0) sh[3] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint64_t key = keys[i];
    if (key >= prefix) out[atomicAdd(&sh[3], 1)] = key;
  }
  __syncthreads();
  return prefix;
}

}  // namespace dt
