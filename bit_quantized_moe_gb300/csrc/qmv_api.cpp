// qmv_api.cpp -- the C ABI (include/qmv.h): argument checks, error reporting,
// dispatch to the launchers. Nothing here reads device memory or synchronizes,
// except qmv_device_status.
#include "../../include/qmv.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "qmv_internal.h"
#include "qmv_layout.h"

namespace qmv {
thread_local const char* g_launch_stage = "";
bool g_phase_probe_on = false;

void pack_expert(const Geometry& g, const uint8_t* codes, const uint8_t* scales, uint8_t* out);
void pack_gate_up_expert(const Geometry& g, int N, const uint8_t* gate_codes, const uint8_t* gate_scales,
                         const uint8_t* up_codes, const uint8_t* up_scales, uint8_t* out);
void unpack_expert(const Geometry& g, const uint8_t* in, uint8_t* codes, uint8_t* scales);

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int ok() {
  g_last_error.clear();
  return QMV_OK;
}

int cuda_fail(cudaError_t e, const char* where) {
  cudaGetLastError();  // clear a non-sticky error so later calls start clean
  return fail(QMV_ECUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_desc(const qmv_wdesc* d) {
  if (d == nullptr) return fail(QMV_EINVAL, "descriptor is NULL");
  if (d->fmt < QMV_MXFP4 || d->fmt > QMV_MXFP8) return fail(QMV_EINVAL, "unknown format %d", d->fmt);
  if (d->N < 1 || d->N > QMV_MAX_N) return fail(QMV_ESHAPE, "N=%d outside [1, %d]", d->N, QMV_MAX_N);
  if (d->K < 32 || d->K > QMV_MAX_K || d->K % 32 != 0)
    return fail(QMV_ESHAPE, "K=%d must be a multiple of 32 in [32, %d]", d->K, QMV_MAX_K);
  if (d->n_experts < 1) return fail(QMV_EINVAL, "n_experts=%d must be >= 1", d->n_experts);
  return QMV_OK;
}

void lut_words(const qmv_wdesc* d, uint32_t out[4]) {
  for (int w = 0; w < 4; ++w) {
    uint32_t v = 0;
    for (int b = 0; b < 4; ++b) v |= (uint32_t)(uint8_t)d->lut[4 * w + b] << (8 * b);
    out[w] = v;
  }
}

struct DevInfo {
  int sm_count = 0;
  size_t smem_optin = 0;
  size_t smem_per_sm = 0;
};

std::mutex g_dev_mu;
DevInfo g_dev[64];

const DevInfo* dev_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (di.sm_count == 0) {
    int sms = 0, smem = 0, smem_sm = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return nullptr;
    if (cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
      return nullptr;
    di.sm_count = sms;
    di.smem_optin = (size_t)smem;
    di.smem_per_sm = (size_t)smem_sm;
  }
  return &di;
}

cudaError_t launch_for(const MatvecArgs& a) {
  switch (a.fmt) {
    case MXFP4: return launch_matvec_mxfp4(a);
    case CB2: return launch_matvec_cb2(a);
    case CB3: return launch_matvec_cb3(a);
    case MXFP8: return launch_matvec_mxfp8(a);
    default: return launch_matvec_cb4(a);
  }
}

// Launch flags valid for a call of format fmt (dbg: the block-sum export).
int check_flags(int fmt, uint32_t flags, bool dbg, const char* name) {
  if (flags & ~(uint32_t)(QMV_FLAG_PREFETCH_INPUTS | QMV_FLAG_X_F32 | QMV_FLAG_X_F16 | QMV_FLAG_PATH_TENSOR |
                          QMV_FLAG_PATH_CUDA_CORES))
    return fail(QMV_EINVAL, "%s: unknown flags 0x%x", name, flags);
  if ((flags & QMV_FLAG_PATH_TENSOR) && (flags & QMV_FLAG_PATH_CUDA_CORES))
    return fail(QMV_EINVAL, "%s: QMV_FLAG_PATH_TENSOR and QMV_FLAG_PATH_CUDA_CORES together", name);
  if ((flags & QMV_FLAG_X_F32) && (fmt_is_mx(fmt) || dbg))
    return fail(QMV_EINVAL, "%s: QMV_FLAG_X_F32 applies to the codebook formats only (not block sums)", name);
  if ((flags & QMV_FLAG_X_F16) && !fmt_is_mx(fmt))
    return fail(QMV_EINVAL, "%s: QMV_FLAG_X_F16 applies to the MX formats only", name);
  return QMV_OK;
}

// Rows of the gate/up-interleaved matrix of a projection with N rows.
int gate_up_rows(int N) { return 2 * ((N + kRows / 2 - 1) / (kRows / 2) * (kRows / 2)); }

// A gather of more than QMV_MAX_LAYER_SLOTS routed slots takes the sorted
// tensor-core gather when its slots share experts: the tensor-core work item
// decodes an expert's weights once for up to 16 of its slots, so it pays
// when experts carry several slots each. With few slots per expert (many
// experts, a uniform router) the CUDA-core gather streams the same weights
// and decodes them more cheaply, so the call runs as CUDA-core gathers of
// whole tokens, QMV_MAX_LAYER_SLOTS slots at a time (an expert shared by two
// of them is streamed by each). Measured on GB300 (2880^2 MXFP4 and
// 7168 x 2048 / 2048 x 7168 codebook experts, 64-128 slots): the MX tensor
// path breaks even at 4 slots per expert; CB4's (one accumulator per block,
// drained on the CUDA cores) at about 7 (8 per expert: 150 against 195 us,
// 6.4: 186 against 191, 4: 283 against 208); CB2 / CB3's (two accumulators
// per 32-group) at about 12.
constexpr int kSortedMinSlotsPerExpertMx = 4;
constexpr int kSortedMinSlotsPerExpertCb4 = 8;
constexpr int kSortedMinSlotsPerExpertCb = 12;

bool sorted_gather_pays(const MatvecArgs& a) {
  const int nslots = a.ntok * a.top_k;
  const int experts = a.n_experts < nslots ? a.n_experts : nslots;
  const int need = fmt_is_mx(a.fmt) ? kSortedMinSlotsPerExpertMx
                   : (a.fmt == CB4 ? kSortedMinSlotsPerExpertCb4 : kSortedMinSlotsPerExpertCb);
  return nslots >= need * experts;
}

// Codebook dense verify batches take the tensor cores only when the
// CUDA-core path's weight streams (one per 4 tokens, side by side) would
// overflow the L2 cache: below that the repeated streams hit L2 and the
// CUDA cores are faster (measured on GB300: 7168 x 2048 CB3 and 2048 x 7168
// CB2 at 16 tokens 10.4 / 11.3 us on the CUDA cores against 13.4 / 17.9 us
// on the tensor cores; 7168^2 CB4 47.0 against 29.2 us).
constexpr uint64_t kCbDenseTensorBytes = 64ull << 20;

bool dense_tensor_pays(const MatvecArgs& a) {
  if (fmt_is_mx(a.fmt)) return true;
  const uint64_t streams = (uint64_t)(a.ntok + 3) / 4;
  return streams * make_geometry(a.fmt, a.N, a.K).expert > kCbDenseTensorBytes;
}

// Whether the call runs on the tensor cores (dense verify batch or sorted
// gather), else on the CUDA-core matvec (one launch, or one per token range
// for a gather of more than QMV_MAX_LAYER_SLOTS slots).
bool use_tensor_cores(const MatvecArgs& a) {
  if (a.path == 2 || !verify_supported(a)) return false;
  return a.path == 1 || (a.ids == nullptr ? dense_tensor_pays(a) : sorted_gather_pays(a));
}

// Tokens per CUDA-core launch of a gather (all of them up to
// QMV_MAX_LAYER_SLOTS routed slots).
int gather_launch_tokens(const MatvecArgs& a) {
  return (a.ids != nullptr && a.ntok * a.top_k > QMV_MAX_LAYER_SLOTS) ? QMV_MAX_LAYER_SLOTS / a.top_k : a.ntok;
}

// The CUDA-core gather of tokens [t0, t0 + n): ids, activations, outputs and
// block sums offset to the range's first slot.
MatvecArgs token_range(const MatvecArgs& a, int t0, int n) {
  MatvecArgs b = a;
  const int s0 = t0 * a.top_k;
  const size_t xvec = fmt_is_mx(a.fmt) ? (size_t)a.K * 2
                                       : (a.x_f32 ? (size_t)a.K * 4 : (size_t)q8_vec_bytes(a.K));
  const size_t ysz = fmt_is_mx(a.fmt) ? 2 : 4;
  b.ntok = n;
  b.ids = a.ids + s0;
  b.x = static_cast<const uint8_t*>(a.x) + (size_t)(a.per_slot ? s0 : t0) * xvec;
  b.nvec = a.per_slot ? n * a.top_k : n;
  b.y = static_cast<uint8_t*>(a.y) + (size_t)s0 * a.out_n * ysz;
  if (a.dbg != nullptr) b.dbg = a.dbg + (size_t)s0 * a.N * (a.K / fmt_group(a.fmt));
  return b;
}

// Validates one matvec call and fills `a` (no launch).
int prepare_matvec(const qmv_wdesc* desc_in, const void* w, const void* x, int per_slot, const int32_t* ids,
                   int ntok, int top_k, void* y, int32_t* dbg, size_t dbg_bytes, cudaStream_t stream,
                   const char* name, uint32_t flags, bool glu, MatvecArgs& a) {
  int rc = check_desc(desc_in);
  if (rc) return rc;
  qmv_wdesc glu_desc;
  const qmv_wdesc* desc = desc_in;
  if (glu) {
    if (desc_in->N > QMV_MAX_N / 2) return fail(QMV_ESHAPE, "%s: N=%d too large for gate/up fusion", name, desc_in->N);
    glu_desc = *desc_in;
    glu_desc.N = gate_up_rows(desc_in->N);
    desc = &glu_desc;
  }
  rc = check_flags(desc->fmt, flags, dbg != nullptr, name);
  if (rc) return rc;
  if (w == nullptr || x == nullptr || y == nullptr)
    return fail(QMV_EINVAL, "%s: weight, activation and output pointers must be non-NULL", name);
  if (ntok < 1 || ntok > QMV_MAX_NTOK) return fail(QMV_EINVAL, "%s: ntok=%d outside [1, %d]", name, ntok, QMV_MAX_NTOK);
  const bool gather = ids != nullptr;
  if (gather) {
    if (top_k < 1 || top_k > QMV_MAX_TOPK)
      return fail(QMV_EINVAL, "%s: top_k=%d outside [1, %d]", name, top_k, QMV_MAX_TOPK);
    if (ntok * top_k > QMV_MAX_SLOTS)
      return fail(QMV_EINVAL, "%s: ntok * top_k = %d routed slots > %d", name, ntok * top_k, QMV_MAX_SLOTS);
  } else if (desc->n_experts != 1) {
    return fail(QMV_EINVAL, "%s: a dense matvec needs n_experts == 1 (got %d)", name, desc->n_experts);
  }
  if (!aligned16(w) || !aligned16(x) || !aligned16(y) || (gather && !aligned16(ids)))
    return fail(QMV_EALIGN, "%s: device pointers must be 16-byte aligned", name);
  if (dbg != nullptr) {
    if (fmt_is_mx(desc->fmt)) return fail(QMV_EINVAL, "%s: block sums exist only for codebook formats", name);
    if (!aligned16(dbg)) return fail(QMV_EALIGN, "%s: sums pointer must be 16-byte aligned", name);
    const int span = fmt_group(desc->fmt);
    const size_t slots = gather ? (size_t)ntok * top_k : (size_t)ntok;
    const size_t need = slots * desc->N * (desc->K / span) * sizeof(int32_t);
    if (dbg_bytes < need) return fail(QMV_ESIZE, "%s: sums buffer %zu bytes < %zu", name, dbg_bytes, need);
  }
  const Geometry g = make_geometry(desc->fmt, desc->N, desc->K);
  a = MatvecArgs();
  a.fmt = desc->fmt;
  a.N = desc->N;
  a.K = desc->K;
  a.n_experts = desc->n_experts;
  a.w = w;
  a.expert_stride = g.expert;
  a.x = x;
  a.per_slot = gather ? (per_slot != 0) : 0;
  a.nvec = (gather && a.per_slot) ? ntok * top_k : ntok;
  a.ids = ids;
  a.ntok = ntok;
  a.top_k = gather ? top_k : 1;
  a.y = y;
  a.dbg = dbg;
  lut_words(desc, a.lut);
  a.prefetch = (flags & QMV_FLAG_PREFETCH_INPUTS) != 0;
  a.x_f32 = (flags & QMV_FLAG_X_F32) != 0;
  a.x_f16 = (flags & QMV_FLAG_X_F16) != 0;
  a.glu = glu;
  a.out_n = desc_in->N;
  a.path = (flags & QMV_FLAG_PATH_TENSOR) ? 1 : ((flags & QMV_FLAG_PATH_CUDA_CORES) ? 2 : 0);
  a.stream = stream;
  const DevInfo* di = dev_info();
  if (di == nullptr) return cuda_fail(cudaGetLastError(), name);
  if (use_tensor_cores(a)) return QMV_OK;   // tensor-core path, fixed shared memory
  const size_t smem = matvec_smem_bytes(token_range(a, 0, gather_launch_tokens(a)));
  if (smem == 0 || smem > di->smem_optin)
    return fail(QMV_ESHAPE, "%s: %d activation vectors of K=%d do not fit in shared memory", name, a.nvec,
                desc->K);
  return QMV_OK;
}

int run_matvec(const qmv_wdesc* desc_in, const void* w, const void* x, int per_slot, const int32_t* ids,
               int ntok, int top_k, void* y, int32_t* dbg, size_t dbg_bytes, cudaStream_t stream,
               const char* name, uint32_t flags = 0, bool glu = false) {
  MatvecArgs a;
  const int rc = prepare_matvec(desc_in, w, x, per_slot, ids, ntok, top_k, y, dbg, dbg_bytes, stream, name, flags,
                                glu, a);
  if (rc) return rc;
  g_launch_stage = "";
  cudaError_t e = cudaSuccess;
  if (use_tensor_cores(a)) {
    e = launch_verify(a);
  } else {
    const int per = gather_launch_tokens(a);
    for (int t0 = 0; t0 < a.ntok && e == cudaSuccess; t0 += per) {
      e = launch_for(per < a.ntok ? token_range(a, t0, a.ntok - t0 < per ? a.ntok - t0 : per) : a);
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(QMV_ECUDA, "%s: %s failed: %s (%s)", name, g_launch_stage, cudaGetErrorName(e),
                cudaGetErrorString(e));
  }
  return ok();
}

}  // namespace

int record_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int device_sm_count() {
  const DevInfo* di = dev_info();
  return di ? di->sm_count : 1;
}

size_t device_max_smem_optin() {
  const DevInfo* di = dev_info();
  return di ? di->smem_optin : 0;
}

size_t device_smem_per_sm() {
  const DevInfo* di = dev_info();
  return di ? di->smem_per_sm : 0;
}

}  // namespace qmv

using namespace qmv;

extern "C" {

int32_t qmv_scale_group(int32_t fmt) { return (fmt >= 0 && fmt < kNumFmts) ? fmt_group(fmt) : 0; }

int32_t qmv_code_bits(int32_t fmt) { return (fmt >= 0 && fmt < kNumFmts) ? fmt_bits(fmt) : 0; }

size_t qmv_canonical_code_bytes(const qmv_wdesc* d) {
  if (check_desc(d)) return 0;
  return (size_t)d->N * d->K * fmt_bits(d->fmt) / 8;
}

size_t qmv_canonical_scale_bytes(const qmv_wdesc* d) {
  if (check_desc(d)) return 0;
  return (size_t)d->N * (d->K / fmt_group(d->fmt));
}

size_t qmv_packed_expert_bytes(const qmv_wdesc* d) {
  if (check_desc(d)) return 0;
  return (size_t)make_geometry(d->fmt, d->N, d->K).expert;
}

size_t qmv_packed_bytes(const qmv_wdesc* d) {
  if (check_desc(d)) return 0;
  return (size_t)make_geometry(d->fmt, d->N, d->K).expert * d->n_experts;
}

int qmv_pack_weights(const qmv_wdesc* d, const uint8_t* codes, const uint8_t* scales, void* out,
                     size_t out_bytes) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!codes || !scales || !out) return fail(QMV_EINVAL, "qmv_pack_weights: NULL buffer");
  const Geometry g = make_geometry(d->fmt, d->N, d->K);
  const size_t need = (size_t)g.expert * d->n_experts;
  if (out_bytes < need) return fail(QMV_ESIZE, "qmv_pack_weights: output %zu bytes < %zu", out_bytes, need);
  const size_t cb = (size_t)d->N * d->K * fmt_bits(d->fmt) / 8;
  const size_t sb = (size_t)d->N * (d->K / fmt_group(d->fmt));
  for (int e = 0; e < d->n_experts; ++e) {
    pack_expert(g, codes + e * cb, scales + e * sb, static_cast<uint8_t*>(out) + (size_t)e * g.expert);
  }
  return ok();
}

int qmv_unpack_weights(const qmv_wdesc* d, const void* packed, size_t packed_bytes, uint8_t* codes,
                       uint8_t* scales) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!codes || !scales || !packed) return fail(QMV_EINVAL, "qmv_unpack_weights: NULL buffer");
  const Geometry g = make_geometry(d->fmt, d->N, d->K);
  const size_t need = (size_t)g.expert * d->n_experts;
  if (packed_bytes < need)
    return fail(QMV_ESIZE, "qmv_unpack_weights: input %zu bytes < %zu", packed_bytes, need);
  const size_t cb = (size_t)d->N * d->K * fmt_bits(d->fmt) / 8;
  const size_t sb = (size_t)d->N * (d->K / fmt_group(d->fmt));
  for (int e = 0; e < d->n_experts; ++e) {
    unpack_expert(g, static_cast<const uint8_t*>(packed) + (size_t)e * g.expert, codes + e * cb, scales + e * sb);
  }
  return ok();
}

size_t qmv_act_q8_vec_bytes(int32_t K) {
  if (K < 32 || K > QMV_MAX_K || K % 32) return 0;
  return (size_t)q8_vec_bytes(K);
}

size_t qmv_act_q8_bytes(int32_t nvec, int32_t K) {
  if (nvec < 1) return 0;
  return (size_t)nvec * qmv_act_q8_vec_bytes(K);
}

int qmv_quantize_act_q8(const float* x, int32_t nvec, int32_t K, void* xq, size_t xq_bytes, void* stream) {
  if (!x || !xq) return fail(QMV_EINVAL, "qmv_quantize_act_q8: NULL pointer");
  if (nvec < 1 || nvec > QMV_MAX_SLOTS)
    return fail(QMV_EINVAL, "qmv_quantize_act_q8: nvec=%d outside [1, %d]", nvec, QMV_MAX_SLOTS);
  if (K < 32 || K > QMV_MAX_K || K % 32)
    return fail(QMV_ESHAPE, "qmv_quantize_act_q8: K=%d must be a multiple of 32 in [32, %d]", K, QMV_MAX_K);
  if (!aligned16(x) || !aligned16(xq)) return fail(QMV_EALIGN, "qmv_quantize_act_q8: pointers must be 16-byte aligned");
  const size_t need = qmv_act_q8_bytes(nvec, K);
  if (xq_bytes < need) return fail(QMV_ESIZE, "qmv_quantize_act_q8: output %zu bytes < %zu", xq_bytes, need);
  cudaError_t e = launch_quantize_q8(x, nvec, K, xq, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmv_quantize_act_q8");
  return ok();
}

int qmv_act_q8_unpack(const void* xq, int32_t nvec, int32_t K, int8_t* q, uint16_t* d) {
  if (!xq || !q || !d) return fail(QMV_EINVAL, "qmv_act_q8_unpack: NULL pointer");
  if (nvec < 1 || K < 32 || K > QMV_MAX_K || K % 32) return fail(QMV_ESHAPE, "qmv_act_q8_unpack: bad shape");
  const size_t vb = (size_t)q8_vec_bytes(K);
  for (int v = 0; v < nvec; ++v) {
    const uint8_t* src = static_cast<const uint8_t*>(xq) + v * vb;
    std::memcpy(q + (size_t)v * K, src, K);
    std::memcpy(d + (size_t)v * (K / 32), src + K, (size_t)(K / 32) * 2);
  }
  return ok();
}

int qmv_dense(const qmv_wdesc* desc, const void* w, const void* x, int32_t ntok, void* y, void* stream) {
  return run_matvec(desc, w, x, 0, nullptr, ntok, 1, y, nullptr, 0, static_cast<cudaStream_t>(stream),
                    "qmv_dense");
}

int qmv_moe_gather(const qmv_wdesc* desc, const void* w, const void* x, int32_t per_slot_x, const int32_t* ids,
                   int32_t ntok, int32_t top_k, void* y, void* stream) {
  if (ids == nullptr) return fail(QMV_EINVAL, "qmv_moe_gather: ids must be non-NULL");
  return run_matvec(desc, w, x, per_slot_x, ids, ntok, top_k, y, nullptr, 0, static_cast<cudaStream_t>(stream),
                    "qmv_moe_gather");
}

int qmv_dense_ex(const qmv_wdesc* desc, const void* w, const void* x, int32_t ntok, void* y, uint32_t flags,
                 void* stream) {
  return run_matvec(desc, w, x, 0, nullptr, ntok, 1, y, nullptr, 0, static_cast<cudaStream_t>(stream),
                    "qmv_dense_ex", flags);
}

int qmv_moe_gather_ex(const qmv_wdesc* desc, const void* w, const void* x, int32_t per_slot_x, const int32_t* ids,
                      int32_t ntok, int32_t top_k, void* y, uint32_t flags, void* stream) {
  if (ids == nullptr) return fail(QMV_EINVAL, "qmv_moe_gather_ex: ids must be non-NULL");
  return run_matvec(desc, w, x, per_slot_x, ids, ntok, top_k, y, nullptr, 0, static_cast<cudaStream_t>(stream),
                    "qmv_moe_gather_ex", flags);
}

size_t qmv_packed_gate_up_expert_bytes(const qmv_wdesc* d) {
  if (check_desc(d)) return 0;
  if (d->N > QMV_MAX_N / 2) return 0;
  return (size_t)make_geometry(d->fmt, gate_up_rows(d->N), d->K).expert;
}

int qmv_pack_gate_up(const qmv_wdesc* d, const uint8_t* gate_codes, const uint8_t* gate_scales,
                     const uint8_t* up_codes, const uint8_t* up_scales, void* out, size_t out_bytes) {
  int rc = check_desc(d);
  if (rc) return rc;
  if (!gate_codes || !gate_scales || !up_codes || !up_scales || !out)
    return fail(QMV_EINVAL, "qmv_pack_gate_up: NULL buffer");
  if (d->N > QMV_MAX_N / 2) return fail(QMV_ESHAPE, "qmv_pack_gate_up: N=%d too large", d->N);
  const Geometry g = make_geometry(d->fmt, gate_up_rows(d->N), d->K);
  const size_t need = (size_t)g.expert * d->n_experts;
  if (out_bytes < need) return fail(QMV_ESIZE, "qmv_pack_gate_up: output %zu bytes < %zu", out_bytes, need);
  const size_t cb = (size_t)d->N * d->K * fmt_bits(d->fmt) / 8;
  const size_t sb = (size_t)d->N * (d->K / fmt_group(d->fmt));
  for (int e = 0; e < d->n_experts; ++e) {
    pack_gate_up_expert(g, d->N, gate_codes + e * cb, gate_scales + e * sb, up_codes + e * cb, up_scales + e * sb,
                        static_cast<uint8_t*>(out) + (size_t)e * g.expert);
  }
  return ok();
}

int qmv_moe_gate_up_swiglu(const qmv_wdesc* desc, const void* w, const void* x, const int32_t* ids, int32_t ntok,
                           int32_t top_k, void* h, uint32_t flags, void* stream) {
  if (ids == nullptr) return fail(QMV_EINVAL, "qmv_moe_gate_up_swiglu: ids must be non-NULL");
  return run_matvec(desc, w, x, 0, ids, ntok, top_k, h, nullptr, 0, static_cast<cudaStream_t>(stream),
                    "qmv_moe_gate_up_swiglu", flags, true);
}

// Workspace of qmv_moe_layer: h (MXFP4: bf16; codebooks: fp32).
size_t qmv_moe_layer_workspace_bytes(const qmv_wdesc* gu, int32_t ntok, int32_t top_k) {
  if (check_desc(gu) || ntok < 1 || ntok > QMV_MAX_NTOK || top_k < 1 || top_k > QMV_MAX_TOPK ||
      ntok * top_k > QMV_MAX_SLOTS)
    return 0;
  const size_t slots = (size_t)ntok * top_k;
  if (fmt_is_mx(gu->fmt)) return (slots * gu->N * 2 + 255) / 256 * 256;
  if (gu->N % 32) return 0;
  return (slots * gu->N * 4 + 255) / 256 * 256;
}

int qmv_moe_layer(const qmv_wdesc* gu, const void* w_gu, const qmv_wdesc* down, const void* w_down, const void* x,
                  const int32_t* ids, int32_t ntok, int32_t top_k, void* ws, size_t ws_bytes, void* y,
                  uint32_t flags, void* stream) {
  const char* name = "qmv_moe_layer";
  int rc = check_desc(gu);
  if (rc) return rc;
  rc = check_desc(down);
  if (rc) return rc;
  if (!ids || !ws) return fail(QMV_EINVAL, "%s: ids and workspace must be non-NULL", name);
  if (fmt_is_mx(gu->fmt) != fmt_is_mx(down->fmt))
    return fail(QMV_EINVAL, "%s: gate/up and down must both be MX formats or both codebook formats", name);
  if (down->K != gu->N) return fail(QMV_ESHAPE, "%s: down K=%d must equal gate/up N=%d", name, down->K, gu->N);
  if (down->n_experts != gu->n_experts)
    return fail(QMV_EINVAL, "%s: gate/up and down expert counts differ (%d, %d)", name, gu->n_experts, down->n_experts);
  if (ntok < 1 || ntok > QMV_MAX_NTOK || top_k < 1 || top_k > QMV_MAX_TOPK || ntok * top_k > QMV_MAX_SLOTS)
    return fail(QMV_EINVAL, "%s: ntok=%d / top_k=%d out of range", name, ntok, top_k);
  const size_t need = qmv_moe_layer_workspace_bytes(gu, ntok, top_k);
  if (ws_bytes < need) return fail(QMV_ESIZE, "%s: workspace %zu bytes < %zu", name, ws_bytes, need);
  if (!aligned16(ws)) return fail(QMV_EALIGN, "%s: workspace must be 16-byte aligned", name);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // gate/up with SwiGLU into h, then down on the per-slot h. The down gather
  // prefetches its weights and ids (they were complete before the layer's
  // first launch). Codebooks: the down launch quantizes the fp32 h to q8_1 as
  // it stages it.
  rc = run_matvec(gu, w_gu, x, 0, ids, ntok, top_k, ws, nullptr, 0, s, name, flags, true);
  if (rc) return rc;
  const uint32_t down_flags = QMV_FLAG_PREFETCH_INPUTS | (flags & (QMV_FLAG_X_F16 | QMV_FLAG_PATH_TENSOR |
                                                                    QMV_FLAG_PATH_CUDA_CORES)) |
                              (fmt_is_mx(gu->fmt) ? 0u : (uint32_t)QMV_FLAG_X_F32);
  return run_matvec(down, w_down, ws, 1, ids, ntok, top_k, y, nullptr, 0, s, name, down_flags);
}

int qmv_moe_combine_ex(const qmv_wdesc* down, const void* ys, const float* weights, const int32_t* ids,
                       int32_t ntok, int32_t top_k, void* y, uint32_t flags, void* stream) {
  const char* name = "qmv_moe_combine";
  int rc = check_desc(down);
  if (rc) return rc;
  if (flags & ~(uint32_t)QMV_FLAG_X_F16) return fail(QMV_EINVAL, "%s: unknown flags 0x%x", name, flags);
  if ((flags & QMV_FLAG_X_F16) && !fmt_is_mx(down->fmt))
    return fail(QMV_EINVAL, "%s: QMV_FLAG_X_F16 applies to the MX formats only", name);
  if (!ys || !weights || !ids || !y) return fail(QMV_EINVAL, "%s: NULL pointer", name);
  if (ntok < 1 || ntok > QMV_MAX_NTOK || top_k < 1 || top_k > QMV_MAX_TOPK || ntok * top_k > QMV_MAX_SLOTS)
    return fail(QMV_EINVAL, "%s: ntok=%d / top_k=%d out of range", name, ntok, top_k);
  if (!aligned16(ys) || !aligned16(weights) || !aligned16(ids) || !aligned16(y))
    return fail(QMV_EALIGN, "%s: pointers must be 16-byte aligned", name);
  const int dtype = !fmt_is_mx(down->fmt) ? kOutF32 : ((flags & QMV_FLAG_X_F16) ? kOutF16 : kOutBF16);
  cudaError_t e = launch_combine(dtype, ys, weights, ids, ntok, top_k, down->n_experts, down->N, y,
                                 static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

int qmv_moe_combine(const qmv_wdesc* down, const void* ys, const float* weights, const int32_t* ids, int32_t ntok,
                    int32_t top_k, void* y, void* stream) {
  return qmv_moe_combine_ex(down, ys, weights, ids, ntok, top_k, y, 0u, stream);
}

size_t qmv_moe_layer_combine_workspace_bytes(const qmv_wdesc* gu, const qmv_wdesc* down, int32_t ntok, int32_t top_k) {
  const size_t layer = qmv_moe_layer_workspace_bytes(gu, ntok, top_k);
  if (layer == 0 || check_desc(down)) return 0;
  const size_t elem = fmt_is_mx(down->fmt) ? 2 : 4;
  return layer + ((size_t)ntok * top_k * down->N * elem + 255) / 256 * 256;
}

int qmv_moe_layer_combine(const qmv_wdesc* gu, const void* w_gu, const qmv_wdesc* down, const void* w_down,
                          const void* x, const int32_t* ids, const float* weights, int32_t ntok, int32_t top_k,
                          void* ws, size_t ws_bytes, void* y, uint32_t flags, void* stream) {
  const char* name = "qmv_moe_layer_combine";
  const size_t need = qmv_moe_layer_combine_workspace_bytes(gu, down, ntok, top_k);
  if (need == 0) return fail(QMV_EINVAL, "%s: invalid descriptors, ntok or top_k", name);
  if (ws == nullptr || ws_bytes < need) return fail(QMV_ESIZE, "%s: workspace %zu bytes < %zu", name, ws_bytes, need);
  if (!weights || !y) return fail(QMV_EINVAL, "%s: NULL pointer", name);
  const size_t layer = qmv_moe_layer_workspace_bytes(gu, ntok, top_k);
  void* ys = static_cast<uint8_t*>(ws) + layer;
  int rc = qmv_moe_layer(gu, w_gu, down, w_down, x, ids, ntok, top_k, ws, layer, ys, flags, stream);
  if (rc) return rc;
  return qmv_moe_combine_ex(down, ys, weights, ids, ntok, top_k, y, flags & QMV_FLAG_X_F16, stream);
}

int qmv_debug_plan(const qmv_wdesc* desc, int32_t ntok, int32_t top_k, int32_t gather, int32_t per_slot_x,
                   uint32_t flags, int32_t sm_count, int32_t ctas_per_sm, int64_t smem_per_sm, int64_t* out,
                   int32_t n_out) {
  const char* name = "qmv_debug_plan";
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!out || n_out < 12) return fail(QMV_ESIZE, "%s: out needs 12 entries", name);
  if (ntok < 1 || ntok > QMV_MAX_NTOK || top_k < 1 || top_k > QMV_MAX_TOPK ||
      (gather && ntok * top_k > QMV_MAX_LAYER_SLOTS))
    return fail(QMV_EINVAL, "%s: ntok=%d / top_k=%d out of range for the CUDA-core matvec", name, ntok, top_k);
  if (sm_count < 1 || ctas_per_sm < 1 || smem_per_sm < 1) return fail(QMV_EINVAL, "%s: bad device shape", name);
  rc = check_flags(desc->fmt, flags, false, name);
  if (rc) return rc;
  MatvecArgs a;
  a.fmt = desc->fmt;
  a.N = desc->N;
  a.K = desc->K;
  a.n_experts = desc->n_experts;
  static const int32_t dummy = 0;
  a.ids = gather ? &dummy : nullptr;
  a.per_slot = (gather && per_slot_x) ? 1 : 0;
  a.ntok = ntok;
  a.top_k = gather ? top_k : 1;
  a.nvec = a.per_slot ? ntok * top_k : ntok;
  a.prefetch = (flags & QMV_FLAG_PREFETCH_INPUTS) != 0;
  a.x_f32 = (flags & QMV_FLAG_X_F32) != 0;
  a.x_f16 = (flags & QMV_FLAG_X_F16) != 0;
  debug_plan(a, sm_count, ctas_per_sm, (size_t)smem_per_sm, out);
  return ok();
}

int qmv_debug_path(const qmv_wdesc* desc, int32_t ntok, int32_t top_k, int32_t gather, int32_t glu,
                   uint32_t flags, int64_t* out, int32_t n_out) {
  const char* name = "qmv_debug_path";
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!out || n_out < 2) return fail(QMV_ESIZE, "%s: out needs 2 entries", name);
  if (ntok < 1 || ntok > QMV_MAX_NTOK || top_k < 1 || top_k > QMV_MAX_TOPK ||
      (gather && ntok * top_k > QMV_MAX_SLOTS) || (glu && !gather))
    return fail(QMV_EINVAL, "%s: ntok=%d / top_k=%d / gather=%d / glu=%d out of range", name, ntok, top_k, gather,
                glu);
  rc = check_flags(desc->fmt, flags, false, name);
  if (rc) return rc;
  MatvecArgs a;
  a.fmt = desc->fmt;
  a.N = glu ? gate_up_rows(desc->N) : desc->N;
  a.K = desc->K;
  a.n_experts = desc->n_experts;
  static const int32_t dummy = 0;
  a.ids = gather ? &dummy : nullptr;
  a.ntok = ntok;
  a.top_k = gather ? top_k : 1;
  a.x_f32 = (flags & QMV_FLAG_X_F32) != 0;
  a.x_f16 = (flags & QMV_FLAG_X_F16) != 0;
  a.glu = glu != 0;
  a.out_n = desc->N;
  a.path = (flags & QMV_FLAG_PATH_TENSOR) ? 1 : ((flags & QMV_FLAG_PATH_CUDA_CORES) ? 2 : 0);
  out[0] = use_tensor_cores(a) ? 1 : 0;
  out[1] = gather_launch_tokens(a);
  return ok();
}

int qmv_debug_block_sums(const qmv_wdesc* desc, const void* w, const void* x, int32_t per_slot_x,
                         const int32_t* ids, int32_t ntok, int32_t top_k, void* y, int32_t* sums,
                         size_t sums_bytes, void* stream) {
  return qmv_debug_block_sums_ex(desc, w, x, per_slot_x, ids, ntok, top_k, y, sums, sums_bytes, 0u, stream);
}

int qmv_debug_block_sums_ex(const qmv_wdesc* desc, const void* w, const void* x, int32_t per_slot_x,
                            const int32_t* ids, int32_t ntok, int32_t top_k, void* y, int32_t* sums,
                            size_t sums_bytes, uint32_t flags, void* stream) {
  if (sums == nullptr) return fail(QMV_EINVAL, "qmv_debug_block_sums: sums must be non-NULL");
  if (flags & ~(uint32_t)(QMV_FLAG_PREFETCH_INPUTS | QMV_FLAG_PATH_TENSOR | QMV_FLAG_PATH_CUDA_CORES))
    return fail(QMV_EINVAL, "qmv_debug_block_sums: flags 0x%x (prefetch and path flags only)", flags);
  return run_matvec(desc, w, x, per_slot_x, ids, ntok, top_k, y, sums, sums_bytes,
                    static_cast<cudaStream_t>(stream), "qmv_debug_block_sums", flags);
}

int qmv_swiglu_bf16(const void* g, const void* u, void* h, int64_t n, void* stream) {
  if (!g || !u || !h) return fail(QMV_EINVAL, "qmv_swiglu_bf16: NULL pointer");
  if (n < 0) return fail(QMV_EINVAL, "qmv_swiglu_bf16: n=%lld < 0", (long long)n);
  if (!aligned16(g) || !aligned16(u) || !aligned16(h))
    return fail(QMV_EALIGN, "qmv_swiglu_bf16: pointers must be 16-byte aligned");
  if (n == 0) return ok();
  cudaError_t e = launch_swiglu_bf16(g, u, h, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmv_swiglu_bf16");
  return ok();
}

int qmv_debug_dequant(const qmv_wdesc* desc, const void* w, int32_t expert, float* out, size_t out_bytes,
                      void* stream) {
  int rc = check_desc(desc);
  if (rc) return rc;
  if (!w || !out) return fail(QMV_EINVAL, "qmv_debug_dequant: NULL pointer");
  if (expert < 0 || expert >= desc->n_experts) return fail(QMV_EINVAL, "qmv_debug_dequant: expert %d out of range", expert);
  if (!aligned16(w) || !aligned16(out)) return fail(QMV_EALIGN, "qmv_debug_dequant: pointers must be 16-byte aligned");
  const size_t need = (size_t)desc->N * desc->K * sizeof(float);
  if (out_bytes < need) return fail(QMV_ESIZE, "qmv_debug_dequant: output %zu bytes < %zu", out_bytes, need);
  const Geometry g = make_geometry(desc->fmt, desc->N, desc->K);
  uint32_t lut[4];
  lut_words(desc, lut);
  cudaError_t e = launch_dequant(desc->fmt, desc->N, desc->K, static_cast<const uint8_t*>(w) + (size_t)expert * g.expert,
                                 lut, out, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmv_debug_dequant");
  return ok();
}

int qmv_device_status(uint32_t* flags, int32_t clear) {
  if (!flags) return fail(QMV_EINVAL, "qmv_device_status: NULL pointer");
  uint32_t v = 0;
  const uint32_t parts[7] = {status_mxfp4(clear), status_cb2(clear),   status_cb3(clear),   status_cb4(clear),
                             status_mxfp8(clear), status_verify(clear), status_act(clear)};
  for (uint32_t p : parts) {
    if (p == 0xffffffffu) return cuda_fail(cudaGetLastError(), "qmv_device_status");
    v |= p;
  }
  *flags = v;
  return ok();
}

int qmv_debug_chunk_rate(int32_t fmt, int32_t nv, int32_t ctas_per_sm, int32_t iters, float* sink,
                         size_t sink_bytes, int64_t* weights, int64_t* threads, void* stream) {
  const char* name = "qmv_debug_chunk_rate";
  if (fmt < 0 || fmt >= kNumFmts) return fail(QMV_EINVAL, "%s: unknown format %d", name, fmt);
  if (nv < 1 || nv > 4) return fail(QMV_EINVAL, "%s: nv=%d outside [1, 4]", name, nv);
  if (ctas_per_sm < 1 || ctas_per_sm > 2) return fail(QMV_EINVAL, "%s: ctas_per_sm=%d outside [1, 2]", name, ctas_per_sm);
  if (iters < 1 || iters > (1 << 20)) return fail(QMV_EINVAL, "%s: iters=%d outside [1, 2^20]", name, iters);
  if (!weights || !threads) return fail(QMV_EINVAL, "%s: NULL output pointer", name);
  if (sink != nullptr && !aligned16(sink)) return fail(QMV_EALIGN, "%s: sink must be 16-byte aligned", name);
  if (dev_info() == nullptr) return cuda_fail(cudaGetLastError(), name);
  int64_t w = 0, t = 0;
  cudaError_t (*fn)(int, int, int, float*, int64_t*, int64_t*, cudaStream_t) = nullptr;
  switch (fmt) {
    case MXFP4: fn = launch_chunk_rate_mxfp4; break;
    case MXFP8: fn = launch_chunk_rate_mxfp8; break;
    case CB2: fn = launch_chunk_rate_cb2; break;
    case CB3: fn = launch_chunk_rate_cb3; break;
    default: fn = launch_chunk_rate_cb4; break;
  }
  cudaError_t e = fn(nv, ctas_per_sm, iters, nullptr, &w, &t, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, name);
  *weights = w;
  *threads = t;
  if (sink == nullptr) return ok();
  if (sink_bytes < (size_t)t * sizeof(float)) return fail(QMV_ESIZE, "%s: sink %zu bytes < %zu", name, sink_bytes,
                                                          (size_t)t * sizeof(float));
  e = fn(nv, ctas_per_sm, iters, sink, &w, &t, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, name);
  return ok();
}

size_t qmv_debug_phase_entries(void) { return (size_t)kProbeSlots * kProbeCtas * kProbeWarps * kPhases; }

int qmv_debug_phase_probe(int32_t enable) {
#ifdef QMV_PHASE_PROBE
  g_phase_probe_on = enable != 0;
  return ok();
#else
  (void)enable;
  return fail(QMV_EINVAL, "qmv_debug_phase_probe: this library was built without the phase probe "
              "(build.py --phase-probe builds the variant that has it)");
#endif
}

int qmv_debug_phase_read(int32_t fmt, uint64_t* out, size_t n, int32_t clear) {
  if (!out) return fail(QMV_EINVAL, "qmv_debug_phase_read: NULL pointer");
  if (n < qmv_debug_phase_entries()) return fail(QMV_ESIZE, "qmv_debug_phase_read: %zu entries < %zu", n,
                                                 qmv_debug_phase_entries());
#ifdef QMV_PHASE_PROBE
  unsigned long long* o = reinterpret_cast<unsigned long long*>(out);
  int rc = -1;
  switch (fmt) {
    case QMV_MXFP4: rc = phase_mxfp4(o, n, clear); break;
    case QMV_MXFP8: rc = phase_mxfp8(o, n, clear); break;
    case QMV_CB2: rc = phase_cb2(o, n, clear); break;
    case QMV_CB3: rc = phase_cb3(o, n, clear); break;
    case QMV_CB4: rc = phase_cb4(o, n, clear); break;
    default: return fail(QMV_EINVAL, "qmv_debug_phase_read: unknown format %d", fmt);
  }
  if (rc != 0) return cuda_fail(cudaGetLastError(), "qmv_debug_phase_read");
  return ok();
#else
  (void)fmt;
  (void)clear;
  return fail(QMV_EINVAL, "qmv_debug_phase_read: this library was built without the phase probe");
#endif
}

int qmv_debug_wait_probe(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull)
    return fail(QMV_EINVAL, "qmv_debug_wait_probe: limit %llu ns outside (0, 1 s]", (unsigned long long)limit_ns);
  cudaError_t e = launch_wait_probe(limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "qmv_debug_wait_probe");
  return ok();
}

const char* qmv_last_error(void) { return g_last_error.c_str(); }

const char* qmv_version(void) { return "qmv 0.1 (sm_103a)"; }

}  // extern "C"
