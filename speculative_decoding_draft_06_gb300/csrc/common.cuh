// Device-side definitions shared by the DARTree kernels.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace dt {

// Bits of the device error word (folded into a status by dartree_sync_status).
enum : int {
  DT_ERR_NONFINITE = 1,   // NaN or +inf base logit / corrected logit
  DT_ERR_TIMEOUT = 2,     // a bounded pipeline wait gave up
  DT_ERR_CLOSURE = 4,     // Top-B selected a node whose parent is unselected
  DT_ERR_EMPTY_ROW = 8,   // a corrected row has no finite logit
};

constexpr long long kWaitLimitCycles = 4000000000LL;  // ~2 s at GB300 clocks

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
