// moe_route_static_scratch: moe_route without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they route: a plugin that a
// host framework hands only its input and output buffers, a runtime whose device memory is
// a fixed budget reserved up front, or code that runs inside an allocator's own callback.
// For them this entry point keeps the routing scan's scratch (the per-block expert counts)
// in a fixed array that lives in the library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds
// kStaticScratchInts int32 (1 MiB) of it until the process exits. Host code cannot use the
// variable's name as a device address, so a call looks the address up with
// cudaGetSymbolAddress (with the device current) whenever the current context differs from
// the one the cached address belongs to: the first call on each device, and the first call
// after that device's context was destroyed and recreated (cudaDeviceReset), when the module
// may be loaded at another address. Such a first call should come before any stream
// capture. Every call on a device shares the one array, so calls whose kernels overlap on
// the GPU (other streams, other threads) race and must be serialised by the caller. Nothing
// in the array has to start at zero: the counting pass writes every entry it later reads.
#include <cuda.h>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kStaticScratchInts = 1 << 18;  // 1 MiB: ceil(T / 128) * E entries at most
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int32_t g_scan_scratch[kStaticScratchInts];
static __device__ __align__(256) DeviceStatus g_status_sink;

struct StaticScratch {
  int32_t* scratch;
  DeviceStatus* sink;
};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no link against libcuda).
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    tried = true;
  }
  return fn;
}

std::mutex g_mu;
StaticScratch g_addr[kMaxDevices];
CUcontext g_ctx[kMaxDevices];  // context the cached addresses belong to (null: none yet)

cudaError_t current_ctx(CUcontext* out) {
  CtxGetCurrentFn get = ctx_get_current();
  if (!get) return cudaErrorNotSupported;
  return get(out) == CUDA_SUCCESS ? cudaSuccess : cudaErrorContextIsDestroyed;
}

// Device addresses of the two arrays in the current context (looked up again whenever the
// context is not the one they were looked up in).
cudaError_t static_scratch(StaticScratch* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  CUcontext ctx = nullptr;
  e = current_ctx(&ctx);
  if (e != cudaSuccess) return e;
  if (ctx == nullptr || ctx != g_ctx[dev]) {
    StaticScratch a{};
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&a.scratch), g_scan_scratch);  // makes the context current
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(&a.sink), g_status_sink);
    if (e != cudaSuccess) return e;
    e = current_ctx(&ctx);
    if (e != cudaSuccess) return e;
    g_addr[dev] = a;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool ok16(const void* p) { return p != nullptr && ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_static_scratch(const moe_config_t* cfg, const float* logits,
                                                 int32_t* topk_idx, float* topk_w, int32_t* counts,
                                                 int32_t* offsets, int32_t* row_token,
                                                 int32_t* tok_row, int32_t* device_status,
                                                 moe_stream_t stream) {
  size_t need = 0;
  moe_status_t v = moe_workspace_size(cfg, &need);  // validates the configuration
  if (v != MOE_OK) return v;
  if ((int64_t)scan_blocks(*cfg) * cfg->E > kStaticScratchInts) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) {
    cudaError_t e = cudaSuccess;
    if (ok16(counts)) e = cudaMemsetAsync(counts, 0, (size_t)cfg->E * 4, (cudaStream_t)stream);
    if (e == cudaSuccess && ok16(offsets))
      e = cudaMemsetAsync(offsets, 0, (size_t)(cfg->E + 1) * 4, (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (!ok16(logits) || !ok16(topk_idx) || !ok16(topk_w) || !ok16(counts) || !ok16(offsets) ||
      !ok16(row_token) || !ok16(tok_row))
    return MOE_ERR_INVALID_ARG;
  if (device_status && ((uintptr_t)device_status & 7u)) return MOE_ERR_INVALID_ARG;
  StaticScratch s{};
  if (static_scratch(&s) != cudaSuccess) return MOE_ERR_CUDA;
  DeviceStatus* st = device_status ? reinterpret_cast<DeviceStatus*>(device_status) : s.sink;
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = launch_route_topk(*cfg, logits, topk_idx, topk_w, st, cs);
  if (e == cudaSuccess)
    e = launch_route_scan(*cfg, topk_idx, counts, offsets, row_token, tok_row, s.scratch, st, cs);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
