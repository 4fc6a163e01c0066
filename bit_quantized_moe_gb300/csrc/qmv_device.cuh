// qmv_device.cuh -- sm_103a device primitives: bulk asynchronous copies into
// shared memory completed on mbarriers, bounded waits, status flags.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmv {

// A wait on an mbarrier gives up after this long, sets a status flag and lets
// the kernel return instead of hanging the GPU.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;   // 2 s
constexpr unsigned long long kDrainLimitNs = 200000000ull;   // 0.2 s

// Status bits (qmv_device_status).
enum : uint32_t {
  kStatusWaitX = 1u,      // activation staging copy did not complete
  kStatusWaitTile = 2u,   // weight tile copy did not complete
  kStatusDrain = 4u,      // a copy was still in flight when giving up
  kStatusWaitProbe = 8u,  // the wait probe's barrier (which nothing completes) timed out
  kStatusPlan = 16u,      // a CTA needed more staged activation vectors than planned
};

// One status word per translation unit; read back by that unit's accessor.
static __device__ uint32_t g_status;

__device__ __forceinline__ void set_status(uint32_t bits) { atomicOr(&g_status, bits); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One wait attempt. The thread is suspended (not spinning) until the phase
// completes or about kSuspendHintNs elapse, so waiting warps take no issue
// slots from warps that compute.
constexpr uint32_t kSuspendHintNs = 1000000;   // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of an mbarrier for at most `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// L2 policy for data read exactly once per call (streamed weights).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy global -> this CTA's shared memory; completes `bytes` of
// transaction count on the mbarrier. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void* src, uint32_t bytes,
                                                   uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
      "[%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Programmatic dependent launch: wait for the preceding kernel's memory to be
// visible / allow the next kernel to start launching. Both are no-ops when the
// launch did not opt in.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// E8M0 byte -> fp32 2^(e-127); e = 0 -> 2^-127 (subnormal), e = 255 -> NaN.
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  uint32_t bits = e << 23;
  bits = (e == 0u) ? 0x00400000u : bits;
  bits = (e == 255u) ? 0x7fc00000u : bits;
  return __uint_as_float(bits);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
  return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Four E2M1 codes (two bytes, low nibble first) -> two f16x2 (exact).
__device__ __forceinline__ void e2m1x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n .reg .b8 a, b, c, d;\n mov.b32 {a, b, c, d}, %2;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Eight E2M1 codes (one 32-bit word, nibble i = code i) -> four f16x2.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n .reg .b8 a, b, c, d;\n mov.b32 {a, b, c, d}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, a;\n cvt.rn.f16x2.e2m1x2 %1, b;\n"
      " cvt.rn.f16x2.e2m1x2 %2, c;\n cvt.rn.f16x2.e2m1x2 %3, d;\n}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Four E4M3 codes (one 32-bit word, byte i = code i) -> two f16x2: h[0]
// holds codes 0 (low half) and 1, h[1] codes 2 and 3. Every E4M3 value,
// subnormals included, is exact in f16; the NaN codes give f16 NaN.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t (&h)[2]) {
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n"
      " cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
      : "=r"(h[0]), "=r"(h[1])
      : "r"(w));
}

}  // namespace qmv

// Defines `uint32_t NAME(int clear)` that returns (and optionally clears) this
// translation unit's status word. Synchronizes the device.
#define QMV_DEFINE_STATUS_ACCESSOR(NAME)                                        \
  uint32_t NAME(int clear) {                                                    \
    uint32_t v = 0;                                                             \
    if (cudaMemcpyFromSymbol(&v, qmv::g_status, sizeof(v)) != cudaSuccess) {    \
      return 0xffffffffu;                                                       \
    }                                                                           \
    if (clear) {                                                                \
      const uint32_t z = 0;                                                     \
      if (cudaMemcpyToSymbol(qmv::g_status, &z, sizeof(z)) != cudaSuccess) {    \
        return 0xffffffffu;                                                     \
      }                                                                         \
    }                                                                           \
    return v;                                                                   \
  }
