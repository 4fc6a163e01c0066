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

#include <cuda_runtime.h>

#include "../../include/qmv.h"
#include "qmv_internal.h"

namespace {

constexpr size_t kScratchBytes = QMV_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The layer's scratch (h, and for codebook layers its q8_1 copy). In host
// code this name is only a host-side stand-in for the device array: passing it
// to a kernel would be wrong, so the host side uses the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_layer_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_layer_scratch on the current device, looked up on the
// first call per device (with that device current) and cached.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return qmv::record_error(QMV_ECUDA, "qmv_moe_layer_noalloc: cudaGetDevice failed");
  }
  if (dev < 0 || dev >= kMaxDevices) return qmv::record_error(QMV_EINVAL, "qmv_moe_layer_noalloc: device index out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_layer_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return qmv::record_error(QMV_ECUDA, "qmv_moe_layer_noalloc: cudaGetSymbolAddress of the scratch array failed");
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
