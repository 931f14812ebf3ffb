// Device-side definitions shared by the DARTree kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace dt {

// Bits of the device error word (folded into a status by dartree_sync_status).
enum : int {
  DT_ERR_NONFINITE = 1,   // NaN or +inf base logit / corrected logit
  DT_ERR_TIMEOUT = 2,     // a bounded pipeline wait gave up
  DT_ERR_CLOSURE = 4,     // Top-B selected a node whose parent is unselected
  DT_ERR_EMPTY_ROW = 8,   // a corrected row has no finite logit
  DT_ERR_BAD_INDEX = 16,  // a token / row index out of range was clamped
};

constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at GB300 clocks
// (pipeline waits may be given a shorter limit to test the timeout path;
// waits for copies or MMAs already in flight always use the full limit)

constexpr int kMaxK = 32;      // children per node
constexpr int kMaxRows = 256;  // head rows per call (R * W), one MMA N
constexpr int kTileV = 128;    // vocabulary rows per MMA tile (MMA M)
constexpr int kTileH = 64;     // bf16 elements per 128-byte swizzle row (K step)
constexpr int kEpiWarps = 4;   // epilogue warps (one per TMEM lane quarter)

// --------------------------------------------------------- ordered keys
// Selections use a total order: value descending, then index ascending.
// A 64-bit key encodes both so that "better" == "larger key":
//   high 32 bits: the float's bits mapped to an unsigned order (-0 -> +0),
//   low 32 bits : 0xFFFFFFFF - index.
// The key 0 is below every real key and marks an empty slot.
__device__ __forceinline__ uint32_t float_order(float x) {
  if (x == 0.0f) x = 0.0f;  // one zero
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float order_float(uint32_t o) {
  const uint32_t b = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
  return __uint_as_float(b);
}

__device__ __forceinline__ uint64_t make_key(float x, uint32_t idx) {
  return (static_cast<uint64_t>(float_order(x)) << 32) | (0xFFFFFFFFu - idx);
}
__device__ __forceinline__ float key_value(uint64_t k) {
  return order_float(static_cast<uint32_t>(k >> 32));
}
__device__ __forceinline__ uint32_t key_index(uint64_t k) {
  return 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFu);
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float fast_exp(float x) {  // e^x, x <= 0 in practice
  return exp2f(x * 1.4426950408889634f);
}

constexpr unsigned kFullMask = 0xFFFFFFFFu;

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(kFullMask, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(kFullMask, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int mask) {
  const uint32_t lo = __shfl_xor_sync(kFullMask, static_cast<uint32_t>(v), mask);
  const uint32_t hi = __shfl_xor_sync(kFullMask, static_cast<uint32_t>(v >> 32), mask);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// (m, s) <- (m, s) (+) (m2, s2): log-sum-exp pairs, s = sum exp(x - m).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mx = fmaxf(m, m2);
  if (mx == -INFINITY) {
    m = -INFINITY;
    s = 0.f;
    return;
  }
  s = s * expf(m - mx) + s2 * expf(m2 - mx);
  m = mx;
}

// Smallest power of two >= k (k <= 32).
__host__ __device__ __forceinline__ int pow2_ceil32(int k) {
  return k <= 1 ? 1 : k <= 2 ? 2 : k <= 4 ? 4 : k <= 8 ? 8 : k <= 16 ? 16 : 32;
}

// Warp-wide merge of two descending key lists of length p2 (a power of two
// <= 32); the result is the best p2 keys, descending, in lanes 0..p2-1.
//   p2 == 32: v = a[lane], y = b[31 - lane].
//   p2 <= 16: v = a[lane] in lanes < p2 and b[2*p2 - 1 - lane] in lanes
//             p2 .. 2*p2-1 (a bitonic sequence); y is unused.
// One half-cleaner keeps the larger of each mirrored pair, then a bitonic
// merge sorts the surviving half.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t v, uint64_t y, int p2) {
  const int lane = threadIdx.x & 31;
  int s;
  if (p2 == 32) {
    v = v > y ? v : y;
    s = 16;
  } else {
    const uint64_t o = shfl_xor_u64(v, p2);
    v = (lane & p2) ? (v < o ? v : o) : (v > o ? v : o);
    s = p2 >> 1;
  }
  for (; s > 0; s >>= 1) {
    const uint64_t o = shfl_xor_u64(v, s);
    v = (lane & s) ? (v < o ? v : o) : (v > o ? v : o);
  }
  return v;
}

// Operands for folding the descending list L (K valid keys, zero-padded to
// p2) into a running list held in lanes 0..p2-1 (v): on return (v, y) are
// the arguments of warp_merge_desc.
__device__ __forceinline__ void merge_operands(const uint64_t* L, int K, int p2, uint64_t& v,
                                               uint64_t& y) {
  const int lane = threadIdx.x & 31;
  if (p2 == 32) {
    const int j = 31 - lane;
    y = j < K ? L[j] : 0ull;
  } else {
    const int j = 2 * p2 - 1 - lane;
    const uint64_t b = (lane >= p2 && lane < 2 * p2 && j < K) ? L[j] : 0ull;
    v = lane < p2 ? v : b;
    y = 0ull;
  }
}

// Programmatic dependent launch.  A kernel launched with it may start while
// the previous kernel on the stream is still running; everything before
// pdl_wait() must touch no memory that another kernel writes or still reads.
// pdl_wait() returns once every earlier kernel has completed and its writes
// are visible; pdl_trigger() lets the next kernel begin its own prologue.
// Both are no-ops for an ordinary launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `k` on `st`, with programmatic dependent launch when `pdl`.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Launch `k` as clusters of `cl` CTAs along x (grid.x a multiple of cl),
// with programmatic dependent launch when `pdl`.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_cluster(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t st, bool pdl, int cl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = cl;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// Opt a kernel into the largest dynamic shared memory it can use: the
// per-block limit minus its static shared memory.
template <typename Kern>
inline cudaError_t set_max_dynamic_smem(Kern* k) {
  cudaFuncAttributes a{};
  cudaError_t e = cudaFuncGetAttributes(&a, k);
  if (e != cudaSuccess) return e;
  const int limit = 227 * 1024 - static_cast<int>(a.sharedSizeBytes);
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
}

// Padded column count for r valid head rows (an MMA N: 16, 32, 64, 128, 256).
__host__ __device__ __forceinline__ int pad_rows(int r) {
  return r <= 16 ? 16 : r <= 32 ? 32 : r <= 64 ? 64 : r <= 128 ? 128 : 256;
}

// Compile-time loop helpers (for register arrays indexed by constants).
template <int V>
struct IntC {
  static constexpr int value = V;
};

template <int B, int E, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  if constexpr (B < E) {
    f(IntC<B>{});
    static_for<B + 1, E>(f);
  }
}

}  // namespace dt
