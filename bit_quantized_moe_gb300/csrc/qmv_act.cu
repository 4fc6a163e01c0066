// qmv_act.cu -- activation-side kernels: the q8_1 quantizer, SwiGLU, and the
// weight-layout decoder used by the tests.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "qmv_device.cuh"
#include "qmv_internal.h"
#include "qmv_layout.h"
#include "qmv_matvec.cuh"

namespace qmv {

// ---------------------------------------------------------------------------
// q8_1: one warp per block of 32 activations, lane i owns element i.
// amax = max|x|, d = amax / 127, q = round_half_away(x * (1/d)) clamped to
// +-127, d stored as fp16 (RNE). Divisions and the product are IEEE-rounded
// fp32 operations (no contraction, no approximate reciprocal).
// ---------------------------------------------------------------------------
__global__ void quantize_q8_kernel(const float* __restrict__ x, int nvec, int K, uint8_t* __restrict__ xq,
                                   uint32_t vec_bytes) {
  const int lane = threadIdx.x & 31;
  const int blocks_per_vec = K / 32;
  const long total = (long)nvec * blocks_per_vec;
  pdl_wait();
  for (long b = (long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); b < total;
       b += (long)gridDim.x * (blockDim.x / 32)) {
    const int v = (int)(b / blocks_per_vec);
    const int blk = (int)(b % blocks_per_vec);
    const float xi = x[(size_t)v * K + (size_t)blk * 32 + lane];
    float amax = fabsf(xi);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    float r = roundf(__fmul_rn(xi, id));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    uint8_t* out = xq + (size_t)v * vec_bytes;
    out[(size_t)blk * 32 + lane] = (uint8_t)(int8_t)(int)r;
    if (lane == 0) reinterpret_cast<__half*>(out + K)[blk] = __float2half_rn(d);
  }
  pdl_launch_dependents();
}

cudaError_t launch_quantize_q8(const float* x, int nvec, int K, void* xq, cudaStream_t s) {
  const long warps = (long)nvec * (K / 32);
  const int threads = 256;
  long grid = (warps + 7) / 8;
  const long cap = (long)device_sm_count() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  quantize_q8_kernel<<<(unsigned)grid, threads, 0, s>>>(x, nvec, K, static_cast<uint8_t*>(xq),
                                                         (uint32_t)q8_vec_bytes(K));
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// SwiGLU: h = silu(g) * u, silu(z) = z / (1 + exp(-z)), fp32 arithmetic (swiglu_f32).
// ---------------------------------------------------------------------------
__global__ void swiglu_kernel(const __nv_bfloat16* __restrict__ g, const __nv_bfloat16* __restrict__ u,
                              __nv_bfloat16* __restrict__ h, int64_t n) {
  pdl_wait();
  const int64_t n8 = n / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 gv = reinterpret_cast<const uint4*>(g)[i];
    const uint4 uv = reinterpret_cast<const uint4*>(u)[i];
    const __nv_bfloat16* ge = reinterpret_cast<const __nv_bfloat16*>(&gv);
    const __nv_bfloat16* ue = reinterpret_cast<const __nv_bfloat16*>(&uv);
    uint4 hv;
    __nv_bfloat16* he = reinterpret_cast<__nv_bfloat16*>(&hv);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      he[k] = __float2bfloat16_rn(swiglu_f32(__bfloat162float(ge[k]), __bfloat162float(ue[k])));
    }
    reinterpret_cast<uint4*>(h)[i] = hv;
  }
  for (int64_t i = n8 * 8 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    h[i] = __float2bfloat16_rn(swiglu_f32(__bfloat162float(g[i]), __bfloat162float(u[i])));
  }
  pdl_launch_dependents();
}

cudaError_t launch_swiglu_bf16(const void* g, const void* u, void* h, int64_t n, cudaStream_t s) {
  const int threads = 256;
  long grid = (long)((n / 8 + threads - 1) / threads);
  const long cap = (long)device_sm_count() * 4;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  swiglu_kernel<<<(unsigned)grid, threads, 0, s>>>(static_cast<const __nv_bfloat16*>(g),
                                                   static_cast<const __nv_bfloat16*>(u),
                                                   static_cast<__nv_bfloat16*>(h), n);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Router-weighted combine of per-slot outputs: y[t][n] = sum over valid slots
// j (ids[t][j] in [0, E)) of w[t][j] * ys[t][j][n], fp32 fma in slot order
// (the same order every run), stored as T. Thread per output element.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_out(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float load_out(const __half* p, int64_t i) { return __half2float(p[i]); }
__device__ __forceinline__ float load_out(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ void store_val(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_val(__half* p, int64_t i, float v) { p[i] = __float2half_rn(v); }
__device__ __forceinline__ void store_val(float* p, int64_t i, float v) { p[i] = v; }

template <typename T>
__global__ void combine_kernel(const T* __restrict__ ys, const float* __restrict__ w, const int32_t* __restrict__ ids,
                               int ntok, int top_k, int n_experts, int N, T* __restrict__ y) {
  pdl_wait();
  const int64_t total = (int64_t)ntok * N;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / N);
    const int n = (int)(i % N);
    float acc = 0.0f;
    for (int j = 0; j < top_k; ++j) {
      const int s = t * top_k + j;
      const int e = ids[s];
      if (e < 0 || e >= n_experts) continue;
      acc = fmaf(w[s], load_out(ys, (int64_t)s * N + n), acc);
    }
    store_val(y, i, acc);
  }
  pdl_launch_dependents();
}

cudaError_t launch_combine(int dtype, const void* ys, const float* w, const int32_t* ids, int ntok, int top_k,
                           int n_experts, int N, void* y, cudaStream_t s) {
  const int threads = 256;
  const long total = (long)ntok * N;
  long grid = (total + threads - 1) / threads;
  const long cap = (long)device_sm_count() * 4;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  // Programmatic dependent launch after the down gather that produced ys.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (s != nullptr) ? 1 : 0;
  if (dtype == kOutBF16) {
    return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16>, static_cast<const __nv_bfloat16*>(ys), w, ids,
                              ntok, top_k, n_experts, N, static_cast<__nv_bfloat16*>(y));
  }
  if (dtype == kOutF16) {
    return cudaLaunchKernelEx(&cfg, combine_kernel<__half>, static_cast<const __half*>(ys), w, ids, ntok, top_k,
                              n_experts, N, static_cast<__half*>(y));
  }
  return cudaLaunchKernelEx(&cfg, combine_kernel<float>, static_cast<const float*>(ys), w, ids, ntok, top_k,
                            n_experts, N, static_cast<float*>(y));
}

// ---------------------------------------------------------------------------
// Weight-layout decoder: one warp per tile, the matvec kernels' decode
// routines, out[n][k] = value(code) * 2^(e-127).
// ---------------------------------------------------------------------------
template <int FMT>
__global__ void dequant_kernel(const uint8_t* __restrict__ w, int N, int K, uint32_t l0, uint32_t l1,
                               uint32_t l2, uint32_t l3, float* __restrict__ out) {
  const Geometry g = make_geometry(FMT, N, K);
  const int rt = blockIdx.x / g.chunks;
  const int c = blockIdx.x % g.chunks;
  const int lane = threadIdx.x;
  const int L = (c == g.chunks - 1) ? g.last_lanes : 32;
  if (lane >= L) return;
  const uint8_t* st = w + tile_offset(g, rt, c);
  const uint8_t* scl = st + tile_code_bytes(FMT, L) + lane * kRows * lane_scale_bytes(FMT);
  const uint32_t t[4] = {l0, l1, l2, l3};
  for (int r = 0; r < kRows; ++r) {
    const int row = rt * kRows + r;
    if (row >= N) break;
    float val[32];
    if constexpr (FMT == MXFP8) {
      const uint4* cp = reinterpret_cast<const uint4*>(st + (size_t)(r * L + lane) * 32);
      const uint4 a = cp[0], b = cp[1];
      const uint32_t w8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      for (int q = 0; q < 8; ++q) {
        uint32_t h[2];
        e4m3x4_to_f16x2(w8[q], h);
        for (int hb = 0; hb < 2; ++hb) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[hb]));
          val[4 * q + 2 * hb] = f.x;
          val[4 * q + 2 * hb + 1] = f.y;
        }
      }
    } else if constexpr (FMT == MXFP4) {
      const uint4 cw = *reinterpret_cast<const uint4*>(st + (size_t)(r * L + lane) * 16);
      const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
      for (int q = 0; q < 4; ++q) {
        uint32_t h[4];
        e2m1x8_to_f16x2(w4[q], h);
        for (int b = 0; b < 4; ++b) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[b]));
          val[8 * q + 2 * b] = f.x;
          val[8 * q + 2 * b + 1] = f.y;
        }
      }
    } else {
      uint32_t wv[8];
      if constexpr (FMT == CB2) {
        const uint2 u = *reinterpret_cast<const uint2*>(st + (size_t)(r * L + lane) * 8);
        decode_cb2(u.x, u.y, t[0], wv);
      } else if constexpr (FMT == CB3) {
        const uint2 u = *reinterpret_cast<const uint2*>(st + (size_t)(r * L + lane) * 8);
        const uint32_t hc =
            *reinterpret_cast<const uint32_t*>(st + (size_t)kRows * L * 8 + (size_t)(r * L + lane) * 4);
        decode_cb3(u.x, u.y, hc, t[0], t[1], wv);
      } else {
        const uint4 u = *reinterpret_cast<const uint4*>(st + (size_t)(r * L + lane) * 16);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
        decode_cb4(w4, t, wv);
      }
      for (int i = 0; i < 32; ++i) val[i] = (float)(int8_t)((wv[i >> 2] >> (8 * (i & 3))) & 0xffu);
    }
    for (int i = 0; i < 32; ++i) {
      const int gi = i / fmt_group(FMT);
      const float s = e8m0_to_f32(scl[r * lane_scale_bytes(FMT) + gi]);
      out[(size_t)row * K + (size_t)c * kChunkK + lane * kLaneK + i] = val[i] * s;
    }
  }
}

cudaError_t launch_dequant(int fmt, int N, int K, const void* w, const uint32_t lut[4], float* out,
                           cudaStream_t s) {
  const Geometry g = make_geometry(fmt, N, K);
  const unsigned grid = (unsigned)(g.row_tiles * g.chunks);
  const uint8_t* wp = static_cast<const uint8_t*>(w);
  switch (fmt) {
    case MXFP4: dequant_kernel<MXFP4><<<grid, 32, 0, s>>>(wp, N, K, lut[0], lut[1], lut[2], lut[3], out); break;
    case CB2: dequant_kernel<CB2><<<grid, 32, 0, s>>>(wp, N, K, lut[0], lut[1], lut[2], lut[3], out); break;
    case CB3: dequant_kernel<CB3><<<grid, 32, 0, s>>>(wp, N, K, lut[0], lut[1], lut[2], lut[3], out); break;
    case MXFP8: dequant_kernel<MXFP8><<<grid, 32, 0, s>>>(wp, N, K, lut[0], lut[1], lut[2], lut[3], out); break;
    default: dequant_kernel<CB4><<<grid, 32, 0, s>>>(wp, N, K, lut[0], lut[1], lut[2], lut[3], out); break;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Wait probe: one CTA waits on an mbarrier phase that nothing completes, with
// the same bounded wait the matvec kernels use, and records the timeout in the
// status word. Exercises the timeout path without a fault or a hang.
// ---------------------------------------------------------------------------
__global__ void wait_probe_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(smem_addr(&bar), 0, limit_ns);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) set_status(kStatusWaitProbe);
}

cudaError_t launch_wait_probe(unsigned long long limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

QMV_DEFINE_STATUS_ACCESSOR(status_act)

size_t matvec_smem_bytes(const MatvecArgs& a) {
  const LaunchPlan plan = plan_launch(a, device_sm_count(), kCtasPerSm, device_smem_per_sm());
  // room for the kernel's static shared variables (128 bytes with alignment)
  return (size_t)plan.smem.total + 256;
}

// The CUDA-core matvec's launch plan for an explicit device shape (no device
// is queried): see qmv_debug_plan.
void debug_plan(const MatvecArgs& a, int sm_count, int ctas_per_sm, size_t smem_per_sm, int64_t out[12]) {
  const LaunchPlan L = plan_launch(a, sm_count, ctas_per_sm, smem_per_sm);
  const Geometry g = make_geometry(a.fmt, a.N, a.K);
  const int64_t v[12] = {L.nv, L.warps, L.stages, L.items, L.grid, L.splits, L.split_chunks, L.items_per_cta,
                         L.x_slots, L.contig, (int64_t)L.smem.total, g.row_tiles};
  for (int i = 0; i < 12; ++i) out[i] = v[i];
}

}  // namespace qmv
