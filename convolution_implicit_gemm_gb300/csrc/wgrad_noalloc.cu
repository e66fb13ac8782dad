// wgrad_noalloc.cu -- the weight gradient for callers that cannot allocate.
//
// conv2d_wgrad needs a device workspace for its split-K partial sums, and it
// expects the caller to provide it.  Some callers cannot: code that runs
// under a memory manager which owns all device memory and only hands it input
// and output buffers (a plugin inside a host framework, for example), and
// code that must not call cudaMalloc on its hot path because the call can
// synchronise the device and can fail under memory pressure.  For them,
// conv2d_wgrad_noalloc keeps the partial sums in one fixed array that lives in
// this library's device image, so the call itself allocates nothing.
//
// The array is IGCONV_WGRAD_NOALLOC_SCRATCH_BYTES (32 MiB).  Every GPU that
// loads the library holds it until the process exits.  All calls on a device
// share it: calls whose kernels overlap on the GPU (different streams, or
// different host threads) race on it and must be serialised by the caller.
// Each call overwrites every partial it later reads, so the array never needs
// clearing.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "igconv.h"

namespace {

static __device__ __align__(256) unsigned char g_wgrad_scratch[IGCONV_WGRAD_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);

constexpr int kMaxScratchDevices = 64;
struct ScratchSlot {
  unsigned long long ctx_id;  // unique ID of the context the address belongs to
  void* ptr;
};
std::mutex g_scratch_mu;
ScratchSlot g_scratch[kMaxScratchDevices] = {};
PFN_ctxGetCurrent g_ctx_current = nullptr;
PFN_ctxGetId g_ctx_id = nullptr;

// Unique ID of the calling thread's current context (0 when none is current
// yet).  cudaDeviceReset destroys a device's primary context and the next
// runtime call creates a new one with a new ID, in which the array has a new
// address.
bool current_context_id(unsigned long long* id) {
  *id = 0;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return false;
  return ctx == nullptr || g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current device's context.  In
// host code the array's name only stands in for the symbol, so the address is
// looked up with cudaGetSymbolAddress the first time a context of a device
// calls, and cached with that context's ID; a call from a new context (after
// cudaDeviceReset) looks it up again.
igconv_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices)
    return IGCONV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_ctx_current || !g_ctx_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                         &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess)
      return IGCONV_ERR_CUDA;
    g_ctx_current = reinterpret_cast<PFN_ctxGetCurrent>(f1);
    g_ctx_id = reinterpret_cast<PFN_ctxGetId>(f2);
  }
  unsigned long long id = 0;
  if (!current_context_id(&id)) return IGCONV_ERR_CUDA;
  ScratchSlot& slot = g_scratch[dev];
  if (slot.ptr == nullptr || id == 0 || slot.ctx_id != id) {
    // the lookup also makes the device's primary context current if no
    // runtime call has done so yet
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_wgrad_scratch) != cudaSuccess || p == nullptr)
      return IGCONV_ERR_CUDA;
    if (!current_context_id(&id) || id == 0) return IGCONV_ERR_CUDA;
    slot.ctx_id = id;
    slot.ptr = p;
  }
  *out = slot.ptr;
  return IGCONV_OK;
}

}  // namespace

extern "C" igconv_status_t conv2d_wgrad_noalloc(const igconv_problem_t* prob,
                                                igconv_dtype_t dtype, igconv_dtype_t dw_dtype,
                                                const void* X, const void* dY, const void* Cin,
                                                void* dW, float alpha, float beta, void* stream) {
  const size_t need = conv2d_wgrad_workspace_size(prob, dtype, dw_dtype);
  if (need == 0) {
    // an invalid problem: let the regular entry point name the error
    return conv2d_wgrad(prob, dtype, dw_dtype, X, dY, Cin, dW, alpha, beta, nullptr, 0, stream);
  }
  // (a problem whose fastest plan needs more than the scratch array may still
  // fit its split-K plan; conv2d_wgrad picks the plan the size allows and
  // returns WORKSPACE when none fits)
  void* scratch = nullptr;
  const igconv_status_t st = scratch_address(&scratch);
  if (st != IGCONV_OK) return st;
  return conv2d_wgrad(prob, dtype, dw_dtype, X, dY, Cin, dW, alpha, beta, scratch,
                      static_cast<size_t>(IGCONV_WGRAD_NOALLOC_SCRATCH_BYTES), stream);
}
