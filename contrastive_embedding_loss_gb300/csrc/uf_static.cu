// uf_static.cu -- uf_contrastive_fwd_bwd_static: the loss for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand this library a workspace: code that runs where the
// allocator is off limits (a real-time or safety-certified host that allocates
// everything up front and forbids cudaMalloc afterwards, a plugin whose host
// application owns all device memory, or a process whose CUDA allocator is a pool it
// must not grow).  For them this file holds the scratch itself, in one fixed-size
// device array that exists from the moment the library's module is loaded on a GPU
// until the process exits.  The entry point allocates nothing: it looks up the array's
// device address, checks that the call fits, and runs the ordinary entry point with the
// array as its workspace.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/uf_contrastive.h"

namespace {

// The scratch shared by every call on a device.  In host code this name is only a
// stand-in for the symbol; its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_workspace[UF_STATIC_WORKSPACE_BYTES];

std::mutex g_static_mu;
void* g_static_ptr[64] = {};              // per-device address of g_static_workspace
unsigned long long g_static_ctx[64] = {};  // id of the context that address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current context (the driver never reuses one within a process), or 0.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array on `device` (which must be current); nullptr on failure.
// The address is looked up at a device's first call and again whenever the device's
// context has changed since (after cudaDeviceReset the module, and the array with it, is
// loaded afresh at another address).
void* static_workspace(int device) {
  if (device < 0 || device >= 64) return nullptr;
  unsigned long long ctx = current_context_id();  // 0 while no context is current on this thread
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[device] || ctx == 0 || g_static_ctx[device] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
    if (ctx == 0) ctx = current_context_id();  // the lookup made the primary context current
    g_static_ptr[device] = p;
    g_static_ctx[device] = ctx;
  }
  return g_static_ptr[device];
}

}  // namespace

extern "C" uf_status_t uf_contrastive_fwd_bwd_static(const void* A, const void* B, int64_t Na, int64_t Nb, int D,
                                                      const int* prefixes, int n_prefix, int kind,
                                                      float logit_scale, float bias, const float* prefix_weights,
                                                      float* loss_per_prefix, float* row_terms, float* col_terms,
                                                      float* dA, float* dB, int* device_status, void* stream) {
  const size_t need = uf_contrastive_workspace_min(Na, Nb, D, prefixes, n_prefix, kind, dA != nullptr);
  if (need == 0) return UF_INVALID_ARGUMENT;
  if (need > static_cast<size_t>(UF_STATIC_WORKSPACE_BYTES)) return UF_WORKSPACE_TOO_SMALL;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return UF_CUDA_ERROR;
  void* ws = static_workspace(device);
  if (!ws) return UF_CUDA_ERROR;
  // Every element of the workspace is written before it is read, so nothing in the
  // array needs clearing between calls.
  return uf_contrastive_fwd_bwd(A, B, Na, Nb, D, prefixes, n_prefix, kind, logit_scale, bias, prefix_weights,
                                loss_per_prefix, row_terms, col_terms, dA, dB, ws, UF_STATIC_WORKSPACE_BYTES,
                                device_status, stream);
}
