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

}  // namespace dt
