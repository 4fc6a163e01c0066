// qmv_noalloc.cu -- qmv_moe_layer for callers that cannot allocate device memory.
//
// Some hosts of this library may not allocate GPU memory at all while they
// decode: an inference server that hands every byte of the device to its own
// pool before serving starts, a plugin running inside another application's
// CUDA context with a fixed budget, or code that runs while a stream is being
// captured and must not call the allocator. qmv_moe_layer needs scratch space
// for the layer's intermediate activations, which such callers cannot
// provide. qmv_moe_layer_noalloc runs the same layer with that scratch in the
// fixed array below, which is part of the library's device image: every GPU
// that loads the library holds it until the process exits.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qmv.h"
#include "qmv_internal.h"

namespace {

constexpr size_t kScratchBytes = QMV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The layer's scratch: h between the two launches (bf16 for the MX formats,
// fp16 with QMV_FLAG_X_F16, fp32 for the codebook formats). In host code this
// name is only a host-side stand-in for the device array: passing it to a
// kernel would be wrong, so the host side uses the device address that
// cudaGetSymbolAddress returns in the current context.
static __device__ __align__(256) unsigned char g_layer_scratch[kScratchBytes];

// The array's address belongs to the context it was looked up in. The cache
// keys it by the context's process-unique id (cuCtxGetId), so a call made in
// another context on the same device -- a host application's own context, or
// the primary context created again after cudaDeviceReset -- looks it up anew.
// The driver functions are reached through the runtime's entry-point query,
// so the library links no driver library.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct Cached {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};

std::mutex g_mu;
Cached g_cache[kMaxDevices];
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

bool resolve_driver_functions() {
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult st;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &st) == cudaSuccess &&
        st == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &st) == cudaSuccess &&
        st == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
  });
  return g_ctx_get_current != nullptr && g_ctx_get_id != nullptr;
}

// Id of the context current on this thread, or 0.
unsigned long long current_context_id() {
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int lookup_symbol(void** p) {
  *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(p, g_layer_scratch);
  if (e != cudaSuccess || *p == nullptr) {
    cudaGetLastError();
    return qmv::record_error(QMV_ECUDA, "qmv_moe_layer_noalloc: cudaGetSymbolAddress of the scratch array failed");
  }
  return QMV_OK;
}

// Device address of g_layer_scratch in the current context of the current
// device: looked up on the first call in each context (which also loads the
// library's device code into it, if the runtime has not yet) and cached.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return qmv::record_error(QMV_ECUDA, "qmv_moe_layer_noalloc: cudaGetDevice failed");
  }
  if (dev < 0 || dev >= kMaxDevices) return qmv::record_error(QMV_EINVAL, "qmv_moe_layer_noalloc: device index out of range");
  if (!resolve_driver_functions()) {
    return qmv::record_error(QMV_ECUDA, "qmv_moe_layer_noalloc: cuCtxGetCurrent / cuCtxGetId not available");
  }
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = current_context_id();
  void* p = nullptr;
  if (id == 0) {
    // no context bound yet: the lookup makes the runtime bind the device's
    // primary context
    const int rc = lookup_symbol(&p);
    if (rc != QMV_OK) return rc;
    id = current_context_id();
    if (id == 0) return qmv::record_error(QMV_ECUDA, "qmv_moe_layer_noalloc: no current CUDA context");
  }
  Cached& c = g_cache[dev];
  if (c.ptr == nullptr || c.ctx_id != id) {
    if (p == nullptr) {
      const int rc = lookup_symbol(&p);
      if (rc != QMV_OK) return rc;
    }
    c.ctx_id = id;
    c.ptr = p;
  }
  *out = c.ptr;
  return QMV_OK;
}

}  // namespace

extern "C" int qmv_moe_layer_noalloc(const qmv_wdesc* gate_up_desc, const void* w_gate_up_dev,
                                     const qmv_wdesc* down_desc, const void* w_down_dev, const void* x_dev,
                                     const int32_t* ids_dev, int32_t ntok, int32_t top_k, void* y_dev,
                                     uint32_t flags, void* stream) {
  const size_t need = qmv_moe_layer_workspace_bytes(gate_up_desc, ntok, top_k);
  if (need == 0) {
    return qmv::record_error(QMV_EINVAL, "qmv_moe_layer_noalloc: invalid gate/up descriptor, ntok or top_k");
  }
  if (need > kScratchBytes) {
    return qmv::record_error(QMV_ESIZE,
                             "qmv_moe_layer_noalloc: this layer needs %zu bytes of scratch, more than the %zu-byte "
                             "static scratch array (use qmv_moe_layer with a workspace instead)",
                             need, kScratchBytes);
  }
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != QMV_OK) return rc;
  return qmv_moe_layer(gate_up_desc, w_gate_up_dev, down_desc, w_down_dev, x_dev, ids_dev, ntok, top_k, scratch,
                       kScratchBytes, y_dev, flags, stream);
}
