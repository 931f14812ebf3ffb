// Head state step that allocates nothing: dartree_state_step_noalloc.
//
// Who needs it: code that runs under a memory manager which owns the device
// heap -- an inference server or framework whose caching allocator has
// already reserved the GPU's memory, a plugin that is handed buffers but may
// not add allocations of its own -- and latency-critical paths that cannot
// afford cudaMalloc/cudaFree (they synchronise the device).  Such callers
// cannot create a dartree context, whose workspace is allocated by
// dartree_create.
//
// The computation is the tensor-core state step of a build (split-K
// contraction of A with the parent states, reduced through scratch memory,
// tanh, bf16 rounding).  Its scratch lives in the file-scope device arrays
// below instead of a context: a fixed ~12 MiB that every GPU which loads
// this library keeps until the process exits.
//
// Set-up: the first call on each device (that device current) looks up the
// arrays' device addresses with cudaGetSymbolAddress, fills the identity
// row map and sets the kernels' shared-memory attributes.  That first call
// synchronises with the device, so make it before any stream capture.  Later
// calls on the device only enqueue work.
//
// All calls share the arrays and the arrays keep the previous call's
// contents.  Each call copies its parent states into the staging array and
// zeroes the staging rows between M and the MMA's padded row count; the
// split-K partials and the output rows are fully written before they are
// read, so nothing else needs clearing.  Calls whose work overlaps on the GPU
// (different streams, or different host threads without ordering) race on
// the arrays and give wrong results.
//
// Device checks: the kernels OR a timeout (a bounded pipeline wait ran out)
// or a bad index into a per-device check word that also lives here.  The word
// gathers the flags of every call until dartree_sync_status(NULL, stream)
// reads it: that call synchronises the stream, returns TIMEOUT or
// DEVICE_CHECK when a flag is set (so a failed step is never reported as OK)
// and clears the word for the calls that follow.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/dartree.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kNaMaxH = 4096;                  // largest head width
constexpr int kNaSlots = 64;                   // partial tiles (tile x split) held

// Scratch of the context-free state step.  The host-side names below are
// stand-ins, not device addresses: host code must use the addresses that
// cudaGetSymbolAddress returns.
// split-K partials [n_split][256][H]: n_split * H <= kNaSlots * 128
static __device__ __align__(256) float g_na_part[kNaSlots * dt::kMaxRows * dt::kTileV];  // 8 MiB
static __device__ __align__(256) uint16_t g_na_in[dt::kMaxRows * kNaMaxH];               // 2 MiB
static __device__ __align__(256) uint16_t g_na_out[dt::kMaxRows * kNaMaxH];              // 2 MiB
static __device__ __align__(256) int32_t g_na_iota[dt::kMaxRows];
static __device__ __align__(256) int g_na_err;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceScratch {
  bool ready = false;
  int num_sms = 0;
  float* part = nullptr;
  uint16_t* in = nullptr;
  uint16_t* out = nullptr;
  int32_t* iota = nullptr;
  int* err = nullptr;
};

constexpr int kMaxDevices = 64;
DeviceScratch g_dev[kMaxDevices];
std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;

dartree_status na_fail(dartree_status s, const std::string& why) {
  dt::set_context_free_error(why);
  return s;
}

dartree_status na_cuda_fail(const char* what, cudaError_t e) {
  return na_fail(DARTREE_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

// 2-D bf16 tensor map: rows x cols, box of 64 columns x box_rows rows.
bool encode(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(dt::kTileH), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Once per device, with that device current.
dartree_status setup(int dev, DeviceScratch** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceScratch& d = g_dev[dev];
  if (d.ready) {
    *out = &d;
    return DARTREE_OK;
  }
  cudaDeviceProp prop{};
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return na_cuda_fail("device query", e);
  if (prop.major != 10 || prop.minor != 3)
    return na_fail(DARTREE_ERR_UNSUPPORTED, "needs a compute capability 10.3 device");
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
      return na_fail(DARTREE_ERR_CUDA, "cuTensorMapEncodeTiled entry point");
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  if ((e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.part), g_na_part)) != cudaSuccess ||
      (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.in), g_na_in)) != cudaSuccess ||
      (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.out), g_na_out)) != cudaSuccess ||
      (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.iota), g_na_iota)) != cudaSuccess ||
      (e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_na_err)) != cudaSuccess)
    return na_cuda_fail("cudaGetSymbolAddress", e);
  int32_t h_iota[dt::kMaxRows];
  for (int i = 0; i < dt::kMaxRows; ++i) h_iota[i] = i;
  if ((e = cudaMemcpy(d.iota, h_iota, sizeof h_iota, cudaMemcpyHostToDevice)) != cudaSuccess)
    return na_cuda_fail("identity row map", e);
  if ((e = dt::init_head_attrs()) != cudaSuccess) return na_cuda_fail("kernel attributes", e);
  d.num_sms = prop.multiProcessorCount;
  d.ready = true;
  *out = &d;
  return DARTREE_OK;
}

}  // namespace

extern "C" dartree_status dartree_state_step_noalloc(const void* S_par, const int32_t* tok,
                                                     const void* A, const void* E, int32_t H,
                                                     int32_t M, void* S_out, void* stream) {
  if (!S_par || !tok || !A || !E || !S_out)
    return na_fail(DARTREE_ERR_INVALID_ARG, "null pointer argument");
  if (M < 1 || H < dt::kTileH || H % dt::kTileH != 0)
    return na_fail(DARTREE_ERR_INVALID_ARG, "need M >= 1 and H a positive multiple of 64");
  if (M > dt::kMaxRows || H > kNaMaxH)
    return na_fail(DARTREE_ERR_UNSUPPORTED,
                   "dartree_state_step_noalloc handles M <= 256 rows and H <= 4096 (got M=" +
                       std::to_string(M) + ", H=" + std::to_string(H) + ")");
  // A is read by TMA (16-byte aligned base); E by 8-byte loads of four bf16
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(E)) & 15)
    return na_fail(DARTREE_ERR_INVALID_ARG, "A and E must be 16-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return na_cuda_fail("cudaGetDevice", e);
  if (dev < 0 || dev >= kMaxDevices) return na_fail(DARTREE_ERR_UNSUPPORTED, "device index");
  DeviceScratch* d = nullptr;
  dartree_status s = setup(dev, &d);
  if (s != DARTREE_OK) return s;

  const int N = dt::pad_rows(M);
  const int tiles = (H + dt::kTileV - 1) / dt::kTileV;
  const int nk = H / dt::kTileH;
  int n_split = kNaSlots / tiles;
  if (n_split > d->num_sms / tiles) n_split = d->num_sms / tiles;
  if (n_split > nk) n_split = nk;
  if (n_split < 1) n_split = 1;

  CUtensorMap tm_a, tm_s;
  if (!encode(&tm_a, A, H, H, dt::kTileV) || !encode(&tm_s, d->in, dt::kMaxRows, H, N))
    return na_fail(DARTREE_ERR_CUDA, "cuTensorMapEncodeTiled failed");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rb = static_cast<size_t>(H) * 2;
  e = cudaMemcpyAsync(d->in, S_par, M * rb, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess && N > M) e = cudaMemsetAsync(d->in + static_cast<size_t>(M) * H, 0, (N - M) * rb, st);
  if (e != cudaSuccess) return na_cuda_fail("staging", e);

  dt::TcParams p{};
  p.rows = H;
  p.H = H;
  p.M = M;
  p.M_out = M;
  p.slot = d->iota;
  p.tok = tok;
  p.n_tiles = tiles;
  p.err = d->err;
  p.E_bf16 = static_cast<const uint16_t*>(E);
  p.S_out_bf16 = d->out;
  p.n_split = n_split;
  p.part = d->part;
  p.V_tok = 0x7FFFFFFF;  // tokens are the caller's to keep in [0, V)
  // test knob (as for contexts): shorten the pipeline waits to provoke TIMEOUT
  if (const char* v = getenv("DARTREE_WAIT_LIMIT_CYCLES")) p.wait_limit = atoll(v);
  e = dt::launch_head_tc(N, false, tm_a, tm_s, p, tiles * n_split, st);
  if (e == cudaSuccess && n_split > 1) {
    dt::StateFinishParams f{};
    f.H = H;
    f.M_in = M;
    f.M_out = M;
    f.n_out = N;
    f.n_split = n_split;
    f.V_tok = p.V_tok;
    f.part = d->part;
    f.slot = d->iota;
    f.tok = tok;
    f.E = p.E_bf16;
    f.S_out = d->out;
    f.err = d->err;
    e = dt::launch_state_finish(f, st);
  }
  if (e != cudaSuccess) return na_cuda_fail("state step launch", e);
  e = cudaMemcpyAsync(S_out, d->out, M * rb, cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return na_cuda_fail("output copy", e);
  return DARTREE_OK;
}

// The device checks of the calls above on the current device: synchronise
// `st`, read the check word, clear it.  Returns the flags (0: none), or -1
// when the device was never set up by a call (nothing to report).
int dt::noalloc_take_status(cudaStream_t st, cudaError_t* err) {
  *err = cudaSuccess;
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return 0;
  if (dev < 0 || dev >= kMaxDevices) return -1;
  int* word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_dev[dev].ready) return -1;
    word = g_dev[dev].err;
  }
  if ((*err = cudaStreamSynchronize(st)) != cudaSuccess) return 0;
  int h = 0;
  if ((*err = cudaMemcpy(&h, word, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return 0;
  if (h != 0 && (*err = cudaMemset(word, 0, sizeof(int))) != cudaSuccess) return 0;
  return h;
}
