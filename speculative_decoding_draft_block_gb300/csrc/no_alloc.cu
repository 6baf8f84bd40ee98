// ds_verify_static: ds_verify with its scratch in a file-scope device array.
//
// Some callers cannot hand the library a workspace:
//   * plain C hosts that embed the library without any device allocator of
//     their own;
//   * serving loops that must not allocate between steps, because
//     cudaMalloc / cudaFree synchronise the device and stall the other
//     streams.
// For them this entry point takes the same arguments as ds_verify, ignores
// `workspace` / `workspace_bytes`, and uses a statically allocated scratch
// array of kScratchBytes bytes that lives as long as the loaded module. It
// allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
//
// Set-up: the first call on each device (with that device current) takes the
// array's device address with cudaGetSymbolAddress and caches it per device,
// together with the id of the context it belongs to; a call in a later
// context (after cudaDeviceReset) looks the address up again. Make one call
// on every device before capturing work into a CUDA graph, so that the
// capture does not include the set-up query.
//
// Zero-initialisation: none is needed. ds_verify writes every scratch word it
// reads within the same call (per-row results for rows 0..L_b, the final-draw
// descriptors, the chunk and group records).
//
// Concurrency: there is one scratch array per device. Two calls on the same
// device whose executions overlap (different streams, or different host
// threads) race on it; the caller must order them (one stream, or events).
//
// Limit: calls whose ds_verify_workspace_bytes(B, K, V, r) exceeds
// kScratchBytes return DS_ERR_WORKSPACE without launching anything.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "internal.h"

namespace ds {
namespace {

constexpr size_t kScratchBytes = size_t(DS_VERIFY_STATIC_SCRATCH_BYTES);
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

// The driver's id of the current context (unique for the life of the
// process), or 0 if it cannot be read; taken through the runtime's
// entry-point query so the library needs no link to the driver library.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx[kMaxDevices] = {};

// Device address of the scratch array on the current device. It is looked up
// once per device and context: after cudaDeviceReset the device gets a new
// primary context, where the module (and the array) may sit elsewhere, so a
// changed context id triggers a new lookup.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // 0 when no context is current yet (the lookup below creates it) or the id
  // cannot be read: then the address is looked up again
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr || ctx == 0 || ctx != g_ctx[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace ds

extern "C" ds_status ds_verify_static(const ds_verify_args* a, ds_stream_t stream) {
  if (a == nullptr) return DS_ERR_INVALID_ARG;
  const size_t need = ds_verify_workspace_bytes(a->B, a->K, a->V, a->r);
  if (need == 0) return DS_ERR_INVALID_ARG;
  if (need > ds::kScratchBytes) return DS_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (ds::scratch_address(&scratch) != cudaSuccess) return DS_ERR_CUDA;
  ds_verify_args b = *a;
  b.workspace = scratch;
  b.workspace_bytes = ds::kScratchBytes;
  return ds_verify(&b, stream);
}
