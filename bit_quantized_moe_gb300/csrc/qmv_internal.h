// qmv_internal.h -- host-side interface between the C ABI and the kernel launchers.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qmv_layout.h"

namespace qmv {

// Everything a matvec launch needs; filled and validated by the C ABI layer.
struct MatvecArgs {
  int fmt = 0;
  int N = 0, K = 0, n_experts = 1;
  const void* w = nullptr;        // GPU weight layout, expert 0
  uint64_t expert_stride = 0;     // bytes between experts
  const void* x = nullptr;        // bf16 vectors (MXFP4) or q8_1 vectors
  int nvec = 0;                   // activation vectors in x
  int per_slot = 0;
  const int32_t* ids = nullptr;   // null: dense
  int ntok = 1, top_k = 1;
  void* y = nullptr;
  int32_t* dbg = nullptr;         // integer block sums (CB formats) or null
  uint32_t lut[4] = {0, 0, 0, 0}; // 16 int8 codebook bytes
  bool prefetch = false;          // QMV_FLAG_PREFETCH_INPUTS
  bool x_f32 = false;             // QMV_FLAG_X_F32: fp32 x, quantized to q8_1 in the kernel
  bool x_f16 = false;             // QMV_FLAG_X_F16: MX formats, fp16 x and y
  bool glu = false;               // gate/up-interleaved matrix, store silu(gate) * up
  int out_n = 0;                  // output rows per slot (0: N)
  int path = 0;                   // 0: cost model, 1: tensor cores where possible, 2: CUDA cores
  cudaStream_t stream = nullptr;
};

// Name of the CUDA call a launcher made last on this thread (for error messages).
extern thread_local const char* g_launch_stage;

// Dynamic shared memory a launch of `a` needs (0 if it exceeds the device limit).
size_t matvec_smem_bytes(const MatvecArgs& a);

// Launch plan of `a` for an explicit device shape (qmv_debug_plan).
void debug_plan(const MatvecArgs& a, int sm_count, int ctas_per_sm, size_t smem_per_sm, int64_t out[12]);

cudaError_t launch_matvec_mxfp4(const MatvecArgs& a);
cudaError_t launch_matvec_cb2(const MatvecArgs& a);
cudaError_t launch_matvec_cb3(const MatvecArgs& a);
cudaError_t launch_matvec_cb4(const MatvecArgs& a);
cudaError_t launch_matvec_mxfp8(const MatvecArgs& a);

// Compute-rate probe of the chunk routine (qmv_debug_chunk_rate).
cudaError_t launch_chunk_rate_mxfp4(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                    int64_t* threads, cudaStream_t s);
cudaError_t launch_chunk_rate_mxfp8(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                    int64_t* threads, cudaStream_t s);
cudaError_t launch_chunk_rate_cb2(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s);
cudaError_t launch_chunk_rate_cb3(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s);
cudaError_t launch_chunk_rate_cb4(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights,
                                  int64_t* threads, cudaStream_t s);

// Dense verify batches of the MX formats (5..16 bf16 tokens) on the tensor
// cores: whether a call takes that path, and its launcher.
bool verify_supported(const MatvecArgs& a);
cudaError_t launch_verify(const MatvecArgs& a);

cudaError_t launch_quantize_q8(const float* x, int nvec, int K, void* xq, cudaStream_t s);
cudaError_t launch_swiglu_bf16(const void* g, const void* u, void* h, int64_t n, cudaStream_t s);
// Output types of the combine.
enum : int { kOutBF16 = 0, kOutF16 = 1, kOutF32 = 2 };
cudaError_t launch_combine(int dtype, const void* ys, const float* w, const int32_t* ids, int ntok, int top_k,
                           int n_experts, int N, void* y, cudaStream_t s);
cudaError_t launch_dequant(int fmt, int N, int K, const void* w, const uint32_t lut[4], float* out,
                           cudaStream_t s);

cudaError_t launch_wait_probe(unsigned long long limit_ns, cudaStream_t s);

// Phase probe (build variant -DQMV_PHASE_PROBE, never the product build):
// lane 0 of every warp records %globaltimer at the phases of a launch into
// g_phase[launch slot][CTA][warp][phase], for the launches made while the
// probe is enabled (qmv_debug_phase_probe), slots dealt in launch order. The
// phases (kPh*) run from kernel start to the warp's end.
enum : int {
  kPhStart = 0,        // kernel entry
  kPhWorkList = 1,     // work list built (first CTA barrier passed)
  kPhEarlyTiles = 2,   // tile copies before griddepcontrol.wait issued
  kPhDepWait = 3,      // griddepcontrol.wait returned
  kPhActLoads = 4,     // first round of activation loads issued
  kPhRingIssued = 5,   // every ring stage's first tile copy issued
  kPhActStaged = 6,    // activations staged (CTA barrier passed)
  kPhTile0Ready = 7,   // first tile landed
  kPhTile0Done = 8,    // first tile computed
  kPhTile1Ready = 9,
  kPhTile2Ready = 10,
  kPhLastDone = 11,    // last tile computed
  kPhEnd = 12,         // warp done (after its stores)
  kPhases = 16
};
constexpr int kProbeSlots = 8, kProbeCtas = 512, kProbeWarps = 16;

// Phase probe (probe build only): launches made while on record their phases.
extern bool g_phase_probe_on;
int phase_mxfp4(unsigned long long* out, size_t n, int clear);
int phase_mxfp8(unsigned long long* out, size_t n, int clear);
int phase_cb2(unsigned long long* out, size_t n, int clear);
int phase_cb3(unsigned long long* out, size_t n, int clear);
int phase_cb4(unsigned long long* out, size_t n, int clear);

uint32_t status_act(int clear);
uint32_t status_mxfp4(int clear);
uint32_t status_cb2(int clear);
uint32_t status_cb3(int clear);
uint32_t status_cb4(int clear);
uint32_t status_mxfp8(int clear);
uint32_t status_verify(int clear);

// Sets the calling thread's qmv_last_error() message and returns `code`.
int record_error(int code, const char* fmt, ...);

// Per-device cached properties.
int device_sm_count();
size_t device_max_smem_optin();
size_t device_smem_per_sm();

}  // namespace qmv
