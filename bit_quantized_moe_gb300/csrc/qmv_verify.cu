// qmv_verify.cu -- batched products on the fifth-generation tensor cores
// (tcgen05) for every weight format: dense calls of 5..16 tokens (a
// speculative-decoding verify batch) and sorted expert gathers of 33..128
// routed slots.
//
// A verify batch applies one weight matrix to several tokens at once
// ("perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on RDNA ...", "Depends on":
// the batched ROCmFPX MMQ that runs the verify batch). With more than a few
// tokens the product is a skinny GEMM, D[n][t] = sum_k W[n][k] x[t][k], and
// the CUDA-core matvec becomes ALU-bound (one FMA or dp4a lane per weight and
// token). Here the CUDA cores only decode and one thread issues tcgen05.mma
// (kind::f16, M = 128 rows, N = 16 tokens, K = 16) into tensor memory.
//
// MX formats (verify_mx_kernel) -- bf16 operands, one accumulator per row:
//   A (weights, in tensor memory: lane = row, bf16 pairs along the columns):
//      code x 2^(e - e_ref) as bf16, where e_ref is the row's
//      first E8M0 byte in the CTA's K range plus kRefMargin (at most 254).
//      The factor 2^(e - e_ref) (e - e_ref in [-24, 0]) is an exact f16, so
//      one mixed-precision FMA
//      (fma.rn.f32.f16, f16 inputs, fp32 result) makes each product exactly
//      and cvt.rn.bf16x2.f32 packs it without rounding (E2M1: two
//      significant bits, E4M3: four, far above bf16's smallest subnormal).
//   B (activations): the bf16 vectors as they are.
//   Products of bf16 values are exact in fp32, so the accumulator holds
//      sum_k code x 2^(e - e_ref) x x in fp32, and the epilogue multiplies it
//      by 2^(e_ref - 127) ("perf(rocm): add an mxfp4 arm ...", "Current
//      Behavior": E8M0 scale 2^(e-127)): a power of two, exact unless the
//      product leaves fp32's normal range. The result differs from the
//      CUDA-core path only in the order of the fp32 additions. A row holding
//      a scale byte outside [e_ref - 24, e_ref] (its bytes spread wider than
//      the margin allows, or the NaN byte 255) is flagged while it is decoded
//      and recomputed exactly on the CUDA cores after the MMAs (sum over
//      groups of 2^(e-127) x sum(code x x) in fp32).
//
// Codebook formats (verify_kernel) -- exact integer block sums:
//   A (weights): codebook values through the byte permute table of the
//      CUDA-core kernel into int8 and from there to f16 (exact).
//   B (activations): the q8_1 codes as f16 (exact), their fp16 scale d kept
//      aside.
//   One tensor-memory accumulator per E8M0 group (16 columns per half-block
//      scale of CB2 / CB3): every product and partial sum is an integer below
//      2^24, so each accumulator is the exact integer block sum
//      sum_{i in h} lut[c_i] * q_i. The decoding warps drain each finished
//      accumulator (tcgen05.ld) and apply d_b * 2^(e-127) in fp32 (two
//      half-blocks: d_b * (2^(e0-127) * isum0 + 2^(e1-127) * isum1)), the dot
//      structure of the review reply in "perf(ggml/hip): optimize ROCMFPX
//      fp3/fp2 MMVQ on RDNA ...".
//
// Work decomposition: a CTA owns 128 rows (16 row tiles of the packed
// layout) and one of `split` K ranges; the `split` CTAs of a row block form a
// thread-block cluster and add their partial sums through distributed shared
// memory in rank order (deterministic), each rank storing a share of the
// outputs. Per CTA: 8 decoding warps, their weight loads issued a window of
// steps ahead, and one warp that issues the MMAs. A stages of 64 columns,
// each with a "full" barrier (one arrival per decoding warp that writes it)
// and an "empty" one (tcgen05.commit). MX: three stages in tensor memory; warp
// w writes rows 32 (w % 4) .. + 31 (its quadrant of lanes) of the steps of
// parity w / 4, both 32-groups of the step for its row (one tcgen05.st of 16
// columns each). Codebooks: stages in tensor memory after the accumulators
// (four for CB4, two for CB2 / CB3); warp w decodes rows 32 (w % 4) .. + 31
// (the tensor-memory lanes it may read and write) and group w / 4 of every
// step, one tcgen05.st of 16 columns per block; the accumulators of a few
// steps (four, or three when a step has four blocks) live in tensor memory,
// each step's with an "accumulated" barrier (tcgen05.commit) and a
// "drained" one, and a warp drains step st - kLag after decoding step st. A
// sorted gather adds a second grid dimension of work items, one (expert, up
// to 16 of its slots) pair each.
//
// Operand layouts: A in tensor memory, lane = row, column j of a stage =
// elements 2j and 2j + 1 of the step (low half first); B (activations,
// tokens padded to 16 with zeros) in shared memory as no-swizzle K-major
// "canonical" core matrices of 8 rows x 16 bytes, core matrix (token group
// g, k group kk) at kk * 256 + g * 128.
// Descriptor leading byte offset = the K-direction stride, stride byte
// offset = the row-direction stride.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "qmv_device.cuh"
#include "qmv_internal.h"
#include "qmv_layout.h"
#include "qmv_matvec.cuh"

namespace qmv {
namespace cg = cooperative_groups;

namespace {

constexpr int kVRows = 128;      // rows per CTA (MMA M)
constexpr int kVTok = 16;        // MMA N: tokens, padded
constexpr int kDecoders = 256;   // decoding threads: two per row
constexpr int kVThreads = kDecoders + 32;   // plus one warp that issues the MMAs
constexpr int kVStepK = 64;      // columns per step (one A stage): 2 groups of 32
constexpr int kLag = 2;          // codebooks: a decoding warp drains step st - kLag after decoding step st
constexpr int kScaleRing = 8;    // codebooks: steps of E8M0 bytes kept for the drains
constexpr int kVMaxSplit = 8;    // cluster size limit (portable)
constexpr int kVMaxSlots = 128;  // routed slots of a sorted gather
constexpr int kVMaxSteps = 24;   // activation operand <= 48 KB (two CTAs per SM)
constexpr int kMaxSpread = 24;   // MX: e - e_ref down to -24 (2^-24: f16's smallest subnormal)
constexpr int kRefMargin = 12;   // MX: e_ref = first scale byte + 12: bytes within -12 .. +12 of the first

// Codebooks: accumulators per step and tensor-memory columns.
template <int FMT>
struct CbAcc {
  static constexpr int span = fmt_group(FMT);                  // columns per accumulator (one scale)
  static constexpr int blocks = kVStepK / span;                // accumulators per step: 2 or 4
  // Tensor memory (256 columns): the accumulators of acc_steps steps, then
  // a_bufs stages of the A operand (32 columns each): CB4 4 steps (128
  // columns) and 4 stages; CB2 / CB3 3 steps (192 columns) and 2 stages.
  static constexpr int acc_steps = blocks == 4 ? 3 : 4;
  static constexpr int acc_cols = acc_steps * blocks * kVTok;
  static constexpr int a_bufs = (256 - acc_cols) / 32;
  static constexpr uint32_t tm_cols = 256u;
  // A stage b of step st is rewritten at step st + a_bufs once MMA(st) is
  // done; the drain of st runs after decoding st + kLag: with a_bufs >= kLag
  // neither waits on the other in a cycle. (A lag of 3 for CB4 measured the
  // same as 2 on GB300.)
  static_assert(a_bufs >= 2 && a_bufs <= 4 && kLag <= a_bufs && kLag < acc_steps, "A and accumulator rings");
};

template <int FMT>
struct VFmt {
  static constexpr int spl = lane_scale_bytes(FMT);            // E8M0 bytes per lane block: 1 or 2
  // Weight loads in flight per thread: MX formats, 4 lane blocks (the two
  // 32-groups of 2 steps; measured on GB300: 2 steps beat 1, 3 and 4 steps
  // for MXFP4 and equal 4 for MXFP8). The codebook kernels are bound by
  // issue rather than load latency, and fewer blocks leave registers to the
  // drains: CB4 1 (7168^2 x 16 tokens: 29.2 us against 30.9 with 2, 33.2
  // with 4, 39.7 with 6), CB2 / CB3 2 (128-slot gathers 78.7 / 89.0 us
  // against 94.6 / 99.6 with 4 and 100.7 / 101.6 with 8 / 6).
  static constexpr int window = fmt_is_mx(FMT) ? 4 : (FMT == CB4 ? 1 : 2);
  static constexpr int words = (FMT == CB3) ? 3 : lane_code_bytes(FMT) / 4;
};

struct VParams {
  const uint8_t* w;
  const uint8_t* x;        // bf16 vectors (MX), q8_1 vectors, or fp32 vectors (codebooks with x_f32)
  void* y;                 // [slot][N]: bf16 (MX) or fp32 (codebooks)
  int32_t* dbg;            // integer block sums (codebooks) or null
  int N, K, T;
  int row_tiles, chunks, last_lanes;
  uint32_t full_tile;
  uint64_t rowtile;
  uint32_t x_vec_bytes;
  int x_f32;               // codebooks: x is fp32, quantized to q8_1 while staged
  uint32_t lut[4];         // codebook values + 128, one byte per code
  int groups;   // K / 32
  int split;    // CTAs (cluster ranks) per row block
  int steps;    // steps of the longest K range
  int prefetch; // weights were not written by the preceding kernel: load them before griddepcontrol.wait
  // sorted gather (ids != null): slots grouped by expert, <= 16 slots per work item
  const int32_t* ids;
  int top_k, nslots, per_slot, n_experts;
  uint64_t expert_stride;
};

__device__ __forceinline__ uint64_t mma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;   // tcgen05 descriptor version; base offset 0, no swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulator (bits 4-5 = 1), A and B
// both f16 (bits 7-9 and 10-12 = 0), both K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kVTok >> 3) << 17) | ((uint32_t)(kVRows >> 4) << 24);
// The same with A and B both bf16 (bits 7-9 and 10-12 = 1): MX formats.
constexpr uint32_t kIdescBf16 = kIdesc | (1u << 7) | (1u << 10);

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Eight fp32 accumulator columns of this warp's 32 tensor-memory lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// MX: scale of a lane block outside the matrix (its codes are zero).
constexpr uint32_t kNoScale = 0x100u;

// Lane block of one row and one 32-group: codes and E8M0 byte(s) (two, the
// half-blocks, for CB2 / CB3).
template <int FMT>
struct Block {
  uint32_t c[VFmt<FMT>::words];
  uint32_t e;
};

template <int FMT>
__device__ __forceinline__ void load_block(const VParams& p, const uint8_t* w, int rt, int r8, int g, bool valid,
                                           Block<FMT>& b) {
  if (!valid) {
#pragma unroll
    for (int i = 0; i < VFmt<FMT>::words; ++i) b.c[i] = 0;
    b.e = (VFmt<FMT>::spl == 2) ? 0x7f7fu : (fmt_is_mx(FMT) ? kNoScale : 0x7fu);
    return;
  }
  const int c = g >> 5, l = g & 31;
  const int L = (c == p.chunks - 1) ? p.last_lanes : 32;
  const uint8_t* tile = w + (uint64_t)rt * p.rowtile + (uint64_t)c * p.full_tile;
  const size_t li = (size_t)(r8 * L + l);
  if constexpr (FMT == MXFP4 || FMT == CB4) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(tile + li * 16));
    b.c[0] = v.x; b.c[1] = v.y; b.c[2] = v.z; b.c[3] = v.w;
  } else if constexpr (FMT == MXFP8) {
    const uint4* src = reinterpret_cast<const uint4*>(tile + li * 32);
    const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
    b.c[0] = v0.x; b.c[1] = v0.y; b.c[2] = v0.z; b.c[3] = v0.w;
    b.c[4] = v1.x; b.c[5] = v1.y; b.c[6] = v1.z; b.c[7] = v1.w;
  } else {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(tile + li * 8));
    b.c[0] = v.x; b.c[1] = v.y;
    if constexpr (FMT == CB3) b.c[2] = __ldg(reinterpret_cast<const uint32_t*>(tile + (size_t)kRows * L * 8 + li * 4));
  }
  const uint8_t* sp = tile + tile_code_bytes(FMT, L) + (size_t)(l * kRows + r8) * VFmt<FMT>::spl;
  if constexpr (VFmt<FMT>::spl == 2) {
    b.e = __ldg(reinterpret_cast<const unsigned short*>(sp));
  } else {
    b.e = __ldg(sp);
  }
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Four int8 values stored with a bias of 128 (v + 128 in each byte) -> two
// f16x2 holding exactly v: the byte under the f16 exponent of 1024 gives
// 1024 + v + 128, and subtracting 1152 is exact.
__device__ __forceinline__ void biased_i8x4_to_f16x2(uint32_t v, uint32_t& lo, uint32_t& hi) {
  lo = sub_f16x2(prmt(v, 0x64646464u, 0x4140u), 0x64806480u);
  hi = sub_f16x2(prmt(v, 0x64646464u, 0x4342u), 0x64806480u);
}


// Codebooks: 32 codes of a lane block -> 32 exact f16 element values
// (unscaled integers) as 16 f16x2 words in K order (low half first).
template <int FMT>
__device__ __forceinline__ void decode_words(const Block<FMT>& b, const uint32_t (&lut)[4], uint32_t (&out)[16]) {
  static_assert(!fmt_is_mx(FMT), "codebook decode");
  uint32_t v[8];
  if constexpr (FMT == CB2) {
    decode_cb2(b.c[0], b.c[1], lut[0], v);
  } else if constexpr (FMT == CB3) {
    decode_cb3(b.c[0], b.c[1], b.c[2], lut[0], lut[1], v);
  } else {
    const uint32_t w4[4] = {b.c[0], b.c[1], b.c[2], b.c[3]};
    decode_cb4(w4, lut, v);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) biased_i8x4_to_f16x2(v[i], out[2 * i], out[2 * i + 1]);
}

// f16 bits of 2^d for -24 <= d <= 0 (normal down to 2^-14, subnormal below;
// the fp32 power of two converts exactly).
__device__ __forceinline__ uint16_t pow2_f16(int d) {
  return __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)(d + 127) << 23)));
}

// Two f16 element values times the f16 power of two m -> bf16x2: each
// product made exactly in fp32 by the mixed-precision FMA (f16 inputs, fp32
// sum with +0), then packed (low half = first element). Exact whenever the
// product is a bf16 value, which holds for every E2M1 / E4M3 code times
// 2^-24 .. 1.
__device__ __forceinline__ uint32_t scaled_pair_bf16(uint32_t h2, uint16_t m) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n .reg .f32 a, b;\n mov.b32 {lo, hi}, %1;\n"
      " fma.rn.f32.f16 a, lo, %2, %3;\n fma.rn.f32.f16 b, hi, %2, %3;\n"
      " cvt.rn.bf16x2.f32 %0, b, a;\n}"
      : "=r"(r)
      : "r"(h2), "h"(m), "f"(0.0f));
  return r;
}

// Codebooks, activation operand B: one (token t, local 32-group gl) unit --
// the 32 q8_1 codes as f16 into four core-matrix rows -- and its fp16 scale
// d (as fp32) for the drain.
template <int FMT>
__device__ __forceinline__ void stage_unit_q8(const VParams& p, int vec, int g, bool valid, uint8_t* bbuf, int gl,
                                              int t, float* aux) {
  uint32_t w[16];
  float f = 0.0f;
  if (!valid) {
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = 0;
  } else {
    uint32_t qw[8];
    if (p.x_f32) {
      float xf[32];
      const float4* src = reinterpret_cast<const float4*>(p.x + (size_t)vec * p.x_vec_bytes + (size_t)g * 128);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 v = src[i];
        xf[4 * i] = v.x; xf[4 * i + 1] = v.y; xf[4 * i + 2] = v.z; xf[4 * i + 3] = v.w;
      }
      f = __half2float(__float2half_rn(q8_block(xf, qw)));
    } else {
      const uint8_t* xv = p.x + (size_t)vec * p.x_vec_bytes;
      const uint4* src = reinterpret_cast<const uint4*>(xv + (size_t)g * 32);
      const uint4 a = src[0], b = src[1];
      qw[0] = a.x; qw[1] = a.y; qw[2] = a.z; qw[3] = a.w;
      qw[4] = b.x; qw[5] = b.y; qw[6] = b.z; qw[7] = b.w;
      f = __half2float(reinterpret_cast<const __half*>(xv + p.K)[g]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) biased_i8x4_to_f16x2(qw[i] ^ 0x80808080u, w[2 * i], w[2 * i + 1]);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int kk = gl * 4 + q;
    *reinterpret_cast<uint4*>(bbuf + (size_t)kk * 256 + (t >> 3) * 128 + (t & 7) * 16) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
  aux[gl * kVTok + t] = f;
}

// 16 bytes global -> shared without a register round trip (cp.async, L2
// only); src_bytes = 0 writes zeros (and reads nothing).
__device__ __forceinline__ void cp_async16(uint8_t* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// MX, activation operand B: the bf16 columns [32 g0, 32 g0 + 64 steps) of
// tokens t < T, zero beyond the CTA's range and for padding tokens. Units of
// 8 columns (16 bytes), every one of a thread's copies in flight at once
// (cp.async); the caller waits for them (cp_async_wait_all) before the
// barrier that publishes the operand.
__device__ __forceinline__ void stage_x_bf16_async(const VParams& p, int T, int g0, int g1, int steps, int tid,
                                                   const int* slot, uint8_t* bbuf) {
  const int n_units = steps * (kVStepK / 8) * kVTok;
  const int k_end = g1 * 32;
  for (int u = tid; u < n_units; u += kDecoders) {
    const int t = u % kVTok, kk = u / kVTok;
    const int k = g0 * 32 + kk * 8;
    const bool valid = t < T && k < k_end;
    const int vec = (p.ids == nullptr) ? t : (p.per_slot ? slot[t < T ? t : 0] : slot[t < T ? t : 0] / p.top_k);
    const uint8_t* src = valid ? p.x + (size_t)vec * p.x_vec_bytes + (size_t)k * 2 : p.x;
    cp_async16(bbuf + (size_t)kk * 256 + (t >> 3) * 128 + (t & 7) * 16, src, valid ? 16u : 0u);
  }
}

// Shared-memory state of a sorted gather's work item.
struct GatherSmem {
  int ids[kVMaxSlots];
  int cnt[kVMaxSlots];
  int slot[kVTok];   // slot of each of the item's tokens
  int item[3];       // expert, first rank, tokens
};

// Sorted gather: work item blockIdx.y is the (expert, group of <= 16 of its
// slots) pair of that index, experts in order of their first slot and slots
// in slot order. Each CTA derives it from the ids in shared memory: thread s
// finds its expert's slot count and its rank among them; the first slot of
// each expert counts the work items of the experts before it. Slots with an
// invalid id get zero rows (written by the CTAs of work item 0). Returns the
// item's token count, or -1 for an index past the last item (every CTA of a
// cluster shares blockIdx.y, so a cluster exits as a whole, before it
// allocates tensor memory). Called by every thread of the CTA.
template <int FMT>
__device__ int gather_work_item(const VParams& p, int tid, int rank, int rb, GatherSmem& gs) {
  if (!p.prefetch) pdl_wait();
  if (tid == 0) gs.item[0] = -1;
  int e = -1;
  if (tid < p.nslots) {
    e = p.ids[tid];
    if (e < 0 || e >= p.n_experts) e = -1;
    gs.ids[tid] = e;
  }
  __syncthreads();
  int cnt = 0, rk = 0;
  bool first = false;
  if (tid < p.nslots && e >= 0) {
    for (int q = 0; q < p.nslots; ++q) {
      const int eq = gs.ids[q];
      cnt += (eq == e);
      rk += (eq == e && q < tid);
    }
    first = (rk == 0);
  }
  if (tid < p.nslots) gs.cnt[tid] = first ? cnt : 0;
  __syncthreads();
  if (first) {
    int before = 0;
    for (int q = 0; q < tid; ++q) before += (gs.cnt[q] + kVTok - 1) / kVTok;
    const int mine = (cnt + kVTok - 1) / kVTok;
    const int y = (int)blockIdx.y;
    if (y >= before && y < before + mine) {
      gs.item[0] = e;
      gs.item[1] = (y - before) * kVTok;
      gs.item[2] = min(kVTok, cnt - (y - before) * kVTok);
    }
  }
  __syncthreads();
  if (gs.item[0] >= 0 && e == gs.item[0] && rk >= gs.item[1] && rk < gs.item[1] + gs.item[2]) {
    gs.slot[rk - gs.item[1]] = tid;
  }
  if (blockIdx.y == 0) {
    if (p.prefetch) pdl_wait();   // outputs are written only after the preceding kernel completed
    for (int i = rank * kVThreads + tid; i < p.nslots * kVRows; i += p.split * kVThreads) {
      const int sl = i / kVRows, orow = rb * kVRows + i % kVRows;
      if (gs.ids[sl] < 0 && orow < p.N) {
        if constexpr (fmt_is_mx(FMT)) {
          static_cast<__nv_bfloat16*>(p.y)[(size_t)sl * p.N + orow] = __float2bfloat16_rn(0.f);
        } else {
          static_cast<float*>(p.y)[(size_t)sl * p.N + orow] = 0.f;
        }
      }
    }
  }
  __syncthreads();
  return gs.item[0] < 0 ? -1 : gs.item[2];
}

// The partial sums part[t][row] of the `split` CTAs of a row block meet in
// rank order through distributed shared memory; rank q stores outputs q,
// q + split, ... (bf16 for MX, fp32 for the codebooks). Called by every
// thread of every CTA of the cluster.
template <int FMT>
__device__ void cluster_store(const VParams& p, const float* part, int rank, int rb, int T, const int* slot,
                              int tid) {
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  for (int i = rank * kVThreads + tid; i < kVRows * T; i += p.split * kVThreads) {  // all 9 warps
    const int t = i / kVRows, rw = i % kVRows;
    const int orow = rb * kVRows + rw;
    if (orow >= p.N) continue;
    float v[kVMaxSplit];
#pragma unroll
    for (int q = 0; q < kVMaxSplit; ++q) {
      v[q] = (q < p.split) ? cluster.map_shared_rank(const_cast<float*>(part), q)[t * kVRows + rw] : 0.f;
    }
    float a = 0.f;
#pragma unroll
    for (int q = 0; q < kVMaxSplit; ++q) a += v[q];   // rank order; absent ranks add +0
    const int oslot = (p.ids == nullptr) ? t : slot[t];
    if constexpr (fmt_is_mx(FMT)) {
      static_cast<__nv_bfloat16*>(p.y)[(size_t)oslot * p.N + orow] = __float2bfloat16_rn(a);
    } else {
      static_cast<float*>(p.y)[(size_t)oslot * p.N + orow] = a;
    }
  }
  cluster.sync();
}

// MX: the rows whose reference byte is -1 (scale bytes spanning more than
// kMaxSpread octaves, or the NaN byte 255), recomputed on the CUDA cores: sum
// over groups of 2^(e-127) * (sum of code x x) in fp32 (the CUDA-core path's
// formula), one warp per row, the lanes taking groups and adding their sums
// in a fixed shuffle order; the result replaces part[.][row]. The activations
// are read from the staged operand B.
template <int FMT>
__device__ void recompute_rows(const VParams& p, const uint8_t* w, int rb, int g0, int g1, int T,
                               const uint8_t* bbuf, const int* s_eref, float* part, int warp, int lane) {
  for (int rr = warp; rr < kVRows; rr += kVThreads / 32) {
    if (s_eref[rr] >= 0) continue;
    const int orow = rb * kVRows + rr;
    if (orow >= p.N) continue;
    float sum[kVTok];
#pragma unroll
    for (int t = 0; t < kVTok; ++t) sum[t] = 0.f;
    for (int g = g0 + lane; g < g1; g += 32) {
      Block<FMT> bk;
      load_block<FMT>(p, w, orow >> 3, orow & 7, g, true, bk);
      const float sc = e8m0_to_f32(bk.e);
      uint32_t hw[16];
      if constexpr (FMT == MXFP4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t hq[4];
          e2m1x8_to_f16x2(bk.c[q], hq);
#pragma unroll
          for (int i = 0; i < 4; ++i) hw[4 * q + i] = hq[i];
        }
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint32_t hq[2];
          e4m3x4_to_f16x2(bk.c[q], hq);
          hw[2 * q] = hq[0];
          hw[2 * q + 1] = hq[1];
        }
      }
      const int kl0 = (g - g0) * 32;
#pragma unroll 1
      for (int t = 0; t < kVTok; ++t) {
        if (t < T) {
          const uint8_t* xt = bbuf + (t >> 3) * 128 + (t & 7) * 16;
          float d = 0.f;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(&hw[i]));
            const int k = kl0 + 2 * i;
            const uint32_t xb = *reinterpret_cast<const uint32_t*>(xt + (size_t)(k >> 3) * 256 + (k & 7) * 2);
            d = fmaf(wf.x, __uint_as_float(xb << 16), d);
            d = fmaf(wf.y, __uint_as_float(xb & 0xffff0000u), d);
          }
          sum[t] = fmaf(sc, d, sum[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kVTok; ++t) {
      float v = sum[t];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) part[t * kVRows + rr] = v;
    }
  }
}

// MX: 16 fp32 tensor-memory columns x 32 lanes of this warp's quadrant from
// 16 registers per thread (thread l -> lane base + l).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                  "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
               : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// MMA with A read from tensor memory (M = 128 lanes, K = 16 bf16 or f16
// in 8 columns), B from shared memory.
template <bool BF16>
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t accumulate) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
               :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(BF16 ? kIdescBf16 : kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t accumulate) {
  mma_ts<true>(d_tmem, a_tmem, b, accumulate);
}

// MX: 32 codes of a lane block -> 16 bf16x2 words code x 2^(e - e_ref) in K
// order. e - e_ref is clamped to [-24, 0]; returns whether that changed it
// (or the byte is 255), in which case the row is recomputed on the CUDA
// cores and its accumulator is not used. A block outside the matrix (scale
// kNoScale, zero codes) is never flagged.
template <int FMT>
__device__ __forceinline__ bool decode_ref(const Block<FMT>& b, int eref, uint32_t (&out)[16]) {
  int d = (int)b.e - eref;
  const bool bad = (d < -kMaxSpread || d > 0) && b.e != kNoScale;
  d = d < -kMaxSpread ? -kMaxSpread : (d > 0 ? 0 : d);
  const uint16_t m = pow2_f16(d);
  if constexpr (FMT == MXFP4) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t h[4];
      e2m1x8_to_f16x2(b.c[q], h);
#pragma unroll
      for (int i = 0; i < 4; ++i) out[4 * q + i] = scaled_pair_bf16(h[i], m);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t h[2];
      e4m3x4_to_f16x2(b.c[q], h);
      out[2 * q] = scaled_pair_bf16(h[0], m);
      out[2 * q + 1] = scaled_pair_bf16(h[1], m);
    }
  }
  return bad;
}

constexpr int kShortKSteps = 8;         // MX: steps per CTA up to which the 3-CTA build runs
constexpr int kTmAStages = 3;          // MX: A operand stages in tensor memory (32 columns each)
constexpr uint32_t kTmACol0 = 32;      // MX: first A column (the accumulator takes columns 0..15)
constexpr uint32_t kTmCols = 128;      // MX: tensor-memory columns per CTA (accumulator + 3 stages)

// MX formats: bf16 operands code x 2^(e - e_ref), one accumulator per row
// for the CTA's whole K range, 2^(e_ref - 127) applied in the epilogue. The
// A operand lives in tensor memory: lane = row, a step's 64 columns in 32
// columns of bf16 pairs; warp w decodes rows 32 (w % 4) .. + 31 (its
// quadrant of lanes) and the steps of parity w / 4, both lane blocks of the
// step for its row, and writes them with one tcgen05.st each. CTAS: the CTAs
// per SM the registers are sized for (3 for short K ranges, where it measured
// faster; 2 otherwise).
template <int FMT, int CTAS>
__global__ void __launch_bounds__(kVThreads, CTAS) verify_mx_kernel(const __grid_constant__ VParams p) {
  using F = VFmt<FMT>;
  static_assert(fmt_is_mx(FMT), "MX formats");
  constexpr int kWin = F::window / 2;   // steps of loads in flight per thread (two lane blocks each)
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t empty[kTmAStages];   // A stage read by the MMAs (tcgen05.commit)
  __shared__ __align__(8) uint64_t full[kTmAStages];    // A stage written by the 4 warps of its parity
  __shared__ __align__(8) uint64_t done;                // every MMA complete (tcgen05.commit)
  __shared__ uint32_t tmem_slot;
  __shared__ int s_eref[kVRows];                        // row reference byte e_ref; -1: recomputed
  __shared__ uint8_t s_bad[2][kVRows];                  // per parity: a block outside the window
  __shared__ GatherSmem gs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)(blockIdx.x % (unsigned)p.split);
  const int rb = (int)(blockIdx.x / (unsigned)p.split);
  const int g0 = (int)((long)rank * p.groups / p.split);
  const int g1 = (int)((long)(rank + 1) * p.groups / p.split);
  const int steps = (g1 - g0 + 1) / 2;

  int T = p.T;
  const uint8_t* w = p.w;
  if (p.ids != nullptr) {
    T = gather_work_item<FMT>(p, tid, rank, rb, gs);
    if (T < 0) return;
    w = p.w + (uint64_t)gs.item[0] * p.expert_stride;
  }
  uint8_t* bbuf = smem;                                  // steps x 64 columns x 16 tokens
  float* part = reinterpret_cast<float*>(smem + (size_t)p.steps * (kVStepK / 8) * 256);  // 16 x 128 fp32

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&tmem_slot)), "r"(kTmCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int i = 0; i < kTmAStages; ++i) {
      mbar_init(smem_addr(&empty[i]), 1);
      mbar_init(smem_addr(&full[i]), 4);
    }
    mbar_init(smem_addr(&done), 1);
    fence_mbar_init();
  }
  const bool decoder = tid < kDecoders;
  const int quad = warp & 3, par = (warp >> 2) & 1;
  const int r = quad * 32 + lane;                       // row of the block (= tensor-memory lane)
  const int row = rb * kVRows + r;
  const int rt = row >> 3, r8 = row & 7;
  const bool row_ok = decoder && rt < p.row_tiles;
  // this thread's steps: st = par, par + 2, ...; step k of them loads groups
  // g0 + 2 st and g0 + 2 st + 1 of its row
  Block<FMT> win[kWin][2];
  if (!p.prefetch) {
    pdl_wait();
    if (decoder) stage_x_bf16_async(p, T, g0, g1, steps, tid, gs.slot, bbuf);
  }
  Block<FMT> first;
  load_block<FMT>(p, w, rt, r8, g0, row_ok, first);   // the row's reference scale byte
#pragma unroll
  for (int u = 0; u < kWin; ++u) {
    const int st = par + 2 * u, g = g0 + 2 * st;
    load_block<FMT>(p, w, rt, r8, g, row_ok && st < steps && g < g1, win[u][0]);
    load_block<FMT>(p, w, rt, r8, g + 1, row_ok && st < steps && g + 1 < g1, win[u][1]);
  }
  if (p.prefetch) {
    pdl_wait();
    if (decoder) stage_x_bf16_async(p, T, g0, g1, steps, tid, gs.slot, bbuf);
  }
  pdl_launch_dependents();
  cp_async_wait_all();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  bool any_bad = false;

  if (decoder) {
    const int e_first = (int)first.e;
    const int eref = min((e_first == (int)kNoScale ? 127 : e_first) + kRefMargin, 254);
    bool bad = false;
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);   // this warp's lane quadrant
    for (int k0 = 0; par + 2 * k0 < steps; k0 += kWin) {
#pragma unroll
      for (int u = 0; u < kWin; ++u) {
        const int k = k0 + u, st = par + 2 * k;
        if (st < steps) {
          const int sa = st % kTmAStages;
          if (st >= kTmAStages) {
            // the MMAs that read this stage kTmAStages steps ago are done
            ok &= mbar_wait_bounded(smem_addr(&empty[sa]), (uint32_t)((st / kTmAStages) - 1) & 1u, kWaitLimitNs);
          }
          tc_fence_after();
          const uint32_t col = tq + kTmACol0 + (uint32_t)sa * 32;
          uint32_t v[16];
          bad |= decode_ref<FMT>(win[u][0], eref, v);
          tmem_st16(col, v);
          bad |= decode_ref<FMT>(win[u][1], eref, v);
          tmem_st16(col + 16, v);
          const int stn = st + 2 * kWin, gn = g0 + 2 * stn;
          load_block<FMT>(p, w, rt, r8, gn, row_ok && stn < steps && gn < g1, win[u][0]);
          load_block<FMT>(p, w, rt, r8, gn + 1, row_ok && stn < steps && gn + 1 < g1, win[u][1]);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&full[sa]));
        }
      }
    }
    s_bad[par][r] = bad ? 1 : 0;
    if (par == 0) s_eref[r] = eref;
    any_bad = bad;
  } else if (lane == 0) {
    // MMA issue: step st once the 4 warps of its parity have written its A
    // stage; one accumulator for the whole K range.
    for (int st = 0; st < steps; ++st) {
      const int sa = st % kTmAStages;
      ok &= mbar_wait_bounded(smem_addr(&full[sa]), (uint32_t)(st / kTmAStages) & 1u, kWaitLimitNs);
      tc_fence_after();
      const uint32_t a0 = tmem + kTmACol0 + (uint32_t)sa * 32;
      const uint32_t b0 = smem_addr(bbuf + (size_t)st * (kVStepK / 8) * 256);
#pragma unroll
      for (int j = 0; j < kVStepK / 16; ++j) {
        mma_bf16_ts(tmem, a0 + (uint32_t)j * 8, mma_desc(b0 + j * 2 * 256, 256, 128), (st > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit(smem_addr(&empty[sa]));
    }
    mma_commit(smem_addr(&done));
  }
  __syncwarp();
  ok &= mbar_wait_bounded(smem_addr(&done), 0u, kWaitLimitNs);
  if (!__all_sync(0xffffffffu, ok) && lane == 0) set_status(kStatusWaitTile);
  tc_fence_before();
  any_bad = __syncthreads_or(any_bad) != 0;   // every row's e_ref and flags are in shared memory
  tc_fence_after();

  // Accumulator rows 32 w .. 32 w + 31 (tensor-memory lanes of warp w) ->
  // partial sums part[t][row] = D x 2^(e_ref - 127); a flagged row gets
  // e_ref = -1 here (this thread's own row) and is recomputed below.
  if (warp < 4) {
    float v0[8], v1[8];
    const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
    tmem_ld8(ta, v0);
    tmem_ld8(ta + 8u, v1);
    tmem_wait_ld();
    const int rr = warp * 32 + lane;
    int er = s_eref[rr];
    if (s_bad[0][rr] | s_bad[1][rr]) {
      er = -1;
      s_eref[rr] = -1;
    }
    const float f = e8m0_to_f32(er < 0 ? 127u : (uint32_t)er);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      part[t * kVRows + rr] = v0[t] * f;
      part[(t + 8) * kVRows + rr] = v1[t] * f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (any_bad) {
    recompute_rows<FMT>(p, w, rb, g0, g1, T, bbuf, s_eref, part, warp, lane);
    __syncthreads();
  }
  cluster_store<FMT>(p, part, rank, rb, T, gs.slot, tid);
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(kTmCols));
  }
}

// Codebook formats: f16 integer operands, one tensor-memory accumulator per
// (half-)block scale, drained by the decoding warps into fp32 row sums. The
// A operand is a ring of steps in tensor memory after the accumulators (lane
// = row, a step's 64 columns in 32 columns of f16 pairs, each decoding warp
// writing its quadrant of lanes and its 32-group with one tcgen05.st).
template <int FMT>
__global__ void __launch_bounds__(kVThreads, 2) verify_kernel(const __grid_constant__ VParams p) {
  using F = VFmt<FMT>;
  using C = CbAcc<FMT>;
  static_assert(!fmt_is_mx(FMT), "codebook formats");
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int kBufs = C::a_bufs;
  __shared__ __align__(8) uint64_t empty[kBufs];       // A stage read by the MMAs (tcgen05.commit)
  __shared__ __align__(8) uint64_t full[kBufs];        // A stage written by all decoding warps
  constexpr int kAcc = C::acc_steps;
  __shared__ __align__(8) uint64_t accd[kAcc];         // a step's accumulators complete (tcgen05.commit)
  __shared__ __align__(8) uint64_t accf[kAcc];         // a step's accumulators drained (one arrival per decoding warp)
  __shared__ __align__(8) uint64_t done;               // every MMA complete (tcgen05.commit)
  __shared__ uint32_t tmem_slot;
  __shared__ GatherSmem gs;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)(blockIdx.x % (unsigned)p.split);
  const int rb = (int)(blockIdx.x / (unsigned)p.split);
  const int g0 = (int)((long)rank * p.groups / p.split);
  const int g1 = (int)((long)(rank + 1) * p.groups / p.split);
  const int steps = (g1 - g0 + 1) / 2;

  int T = p.T;
  const uint8_t* w = p.w;
  if (p.ids != nullptr) {
    T = gather_work_item<FMT>(p, tid, rank, rb, gs);
    if (T < 0) return;
    w = p.w + (uint64_t)gs.item[0] * p.expert_stride;
  }
  uint8_t* bbuf = smem;                                               // steps x 64 columns x 16 tokens
  uint16_t* sc = reinterpret_cast<uint16_t*>(bbuf + (size_t)p.steps * (kVStepK / 8) * 256);  // [ring][2][128]
  float* aux = reinterpret_cast<float*>(sc + kScaleRing * 2 * kVRows);  // [2 steps][16]: 2^-s or d
  float* part = aux + (size_t)p.steps * 2 * kVTok;                    // 16 x 128 fp32 partial sums

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&tmem_slot)), "r"(C::tm_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(smem_addr(&empty[i]), 1);
      mbar_init(smem_addr(&full[i]), kDecoders / 32);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(smem_addr(&accd[i]), 1);
      mbar_init(smem_addr(&accf[i]), kDecoders / 32);
    }
    mbar_init(smem_addr(&done), 1);
    fence_mbar_init();
  }
  // Decoding warp w takes rows 32 (w % 4) .. + 31 of the block
  // -- the tensor-memory lanes its drains may read -- and group 2 * step +
  // w / 4 of every step: lane l decodes row 32 (w % 4) + l, and later drains
  // that row's accumulator of the same group for all 16 tokens, with the
  // E8M0 byte it decoded itself. The first window of loads goes out first
  // (before griddepcontrol.wait when the caller guarantees the weights are
  // not the preceding kernel's output), then the activations.
  const bool decoder = tid < kDecoders;
  const int h = (warp >> 2) & 1;                 // group of the step
  const int r = (warp & 3) * 32 + lane;          // row of the block
  const int row = rb * kVRows + r;
  const int rt = row >> 3, r8 = row & 7;
  const bool row_ok = decoder && rt < p.row_tiles;
  uint32_t lut[4] = {p.lut[0], p.lut[1], p.lut[2], p.lut[3]};
  constexpr int kWindow = F::window;
  Block<FMT> win[kWindow];
  if (!p.prefetch) pdl_wait();
#pragma unroll
  for (int u = 0; u < kWindow; ++u) {
    const int g = g0 + 2 * u + h;
    load_block<FMT>(p, w, rt, r8, g, row_ok && u < steps && g < g1, win[u]);
  }
  if (p.prefetch) pdl_wait();
  pdl_launch_dependents();

  // Activation operand: tokens t < T of groups [g0, g0 + 2 steps), zero
  // beyond the CTA's range and for padding tokens.
  if (decoder) {
    const int n_units = 2 * steps * kVTok;
    for (int u = tid; u < n_units; u += kDecoders) {
      const int t = u % kVTok, gl = u / kVTok;
      const int g = g0 + gl;
      const bool valid = t < T && g < g1;
      const int vec = (p.ids == nullptr) ? t : (p.per_slot ? gs.slot[t < T ? t : 0] : gs.slot[t < T ? t : 0] / p.top_k);
      stage_unit_q8<FMT>(p, vec, g, valid, bbuf, gl, t, aux);
    }
  }

  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  // Drain of step sd: this thread's row, its group 2 sd + h, 16 tokens in
  // two halves of 8 columns; the scale byte is the one this thread stored
  // when it decoded the block (its own earlier write, no barrier needed).
  const uint32_t tlane = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  float acc[kVTok];
#pragma unroll
  for (int i = 0; i < kVTok; ++i) acc[i] = 0.f;
  uint16_t* my_sc = sc + warp * 32 + lane;       // [kScaleRing][256 decoding threads]
  auto drain = [&](int sd) {
    ok = ok && mbar_wait_bounded(smem_addr(&accd[sd % kAcc]), (uint32_t)(sd / kAcc) & 1u, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return;
    tc_fence_after();
    constexpr int per = C::blocks / 2;   // accumulators per 32-group: 1, or 2 half-blocks
    const uint32_t col0 = (uint32_t)(((sd % kAcc) * C::blocks + h * per) * kVTok);
    const int gl = 2 * sd + h;
    const float* f = aux + gl * kVTok;
    const uint32_t eb = my_sc[(sd % kScaleRing) * kDecoders];
    const float s0 = e8m0_to_f32(eb & 0xffu), s1 = e8m0_to_f32(eb >> 8);
#pragma unroll
    for (int th = 0; th < 2; ++th) {
      float v[per][8];
#pragma unroll
      for (int j = 0; j < per; ++j) tmem_ld8(tlane + col0 + (uint32_t)(j * kVTok + th * 8), v[j]);
      tmem_wait_ld();
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int tt = th * 8 + t;
        if constexpr (per == 2) {
          acc[tt] = fmaf(f[tt], fmaf(s0, v[0][t], s1 * v[1][t]), acc[tt]);
        } else {
          acc[tt] = fmaf(f[tt], s0 * v[0][t], acc[tt]);
        }
      }
      const int g = g0 + gl;
      if (p.dbg != nullptr && row < p.N && g < g1) {
        const int nb = p.K / C::span;
#pragma unroll
        for (int j = 0; j < per; ++j) {
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int tt = th * 8 + t;
            if (tt < T) {
              const int slot = (p.ids == nullptr) ? tt : gs.slot[tt];
              p.dbg[((size_t)slot * p.N + row) * nb + g * per + j] = (int32_t)v[j][t];
            }
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&accf[sd % kAcc]));
  };

  if (decoder) {
    for (int s0 = 0; s0 < steps && ok; s0 += kWindow) {
#pragma unroll
      for (int u = 0; u < kWindow; ++u) {
        const int st = s0 + u;
        if (st < steps && ok) {
          const int b = st % kBufs;
          if (st >= kBufs) {
            // the MMAs that read this stage kBufs steps ago are done
            ok = ok && mbar_wait_bounded(smem_addr(&empty[b]), (uint32_t)((st / kBufs) - 1) & 1u, kWaitLimitNs);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
          tc_fence_after();   // after the MMAs that read the stage
          uint32_t v[16];
          decode_words<FMT>(win[u], lut, v);
          tmem_st16(tlane + (uint32_t)C::acc_cols + (uint32_t)b * 32u + (uint32_t)h * 16u, v);
          my_sc[(st % kScaleRing) * kDecoders] = (uint16_t)win[u].e;
          const int gn = g0 + 2 * (st + kWindow) + h;
          load_block<FMT>(p, w, rt, r8, gn, row_ok && st + kWindow < steps && gn < g1, win[u]);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&full[b]));
          if (st >= kLag) drain(st - kLag);
        }
      }
    }
    for (int sd = steps - kLag > 0 ? steps - kLag : 0; sd < steps && ok; ++sd) drain(sd);
  } else if (lane == 0) {
    // MMA issue: step st once every decoding warp has written its A stage
    // and the accumulators it reuses have been drained.
    for (int st = 0; st < steps && ok; ++st) {
      const int b = st % kBufs;
      ok = mbar_wait_bounded(smem_addr(&full[b]), (uint32_t)(st / kBufs) & 1u, kWaitLimitNs);
      if (ok && st >= kAcc) {
        ok = mbar_wait_bounded(smem_addr(&accf[st % kAcc]), (uint32_t)((st / kAcc) - 1) & 1u, kWaitLimitNs);
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t a0 = tmem + (uint32_t)C::acc_cols + (uint32_t)b * 32u;
      const uint32_t b0 = smem_addr(bbuf + (size_t)st * (kVStepK / 8) * 256);
#pragma unroll
      for (int j = 0; j < kVStepK / 16; ++j) {
        const int blk = j * 16 / C::span;
        const uint32_t col = (uint32_t)(((st % kAcc) * C::blocks + blk) * kVTok);
        mma_ts<false>(tmem + col, a0 + (uint32_t)j * 8u, mma_desc(b0 + j * 2 * 256, 256, 128),
                      (j * 16 % C::span) != 0 ? 1u : 0u);
      }
      mma_commit(smem_addr(&empty[b]));
      mma_commit(smem_addr(&accd[st % kAcc]));
    }
    mma_commit(smem_addr(&done));
    if (!mbar_wait_bounded(smem_addr(&done), 0u, kWaitLimitNs)) ok = false;
  }
  if (!ok && lane == 0) set_status(kStatusWaitTile);

  // Partial sums part[t][row].
  __syncthreads();
  if (decoder && h == 0) {
#pragma unroll
    for (int t = 0; t < kVTok; ++t) part[t * kVRows + r] = acc[t];
  }
  __syncthreads();
  if (decoder && h == 1) {
#pragma unroll
    for (int t = 0; t < kVTok; ++t) part[t * kVRows + r] += acc[t];
  }
  tc_fence_before();

  cluster_store<FMT>(p, part, rank, rb, T, gs.slot, tid);
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(C::tm_cols));
  }
}

}  // namespace

// Tensor-core plan: rows in blocks of 128, K cut into `split` ranges (one
// cluster rank each) so that the grid covers about two CTAs per SM. Taken by
// dense calls of 5..16 tokens and gathers of 33..128 routed slots, with bf16
// (MX) or q8_1 / fp32 (codebook) activations, not the gate/up fusion.
bool verify_supported(const MatvecArgs& a) {
  if (a.x_f16 || a.glu) return false;
  if (fmt_is_mx(a.fmt) && a.dbg != nullptr) return false;
  if (a.ids != nullptr) {
    // sorted gather: beyond the decode gather's 32 routed slots
    const int nslots = a.ntok * a.top_k;
    if (nslots <= 32 || nslots > kVMaxSlots) return false;
  } else if (a.ntok <= 4 || a.ntok > kVTok) {
    return false;
  }
  const int groups = a.K / 32;
  return (groups + kVMaxSplit - 1) / kVMaxSplit <= 2 * kVMaxSteps;
}

// Dynamic shared memory: the activation operand and the partial sums; for
// the codebooks also the ring of scale bytes and the per-group activation
// scales.
static size_t verify_smem_bytes(bool mx, int steps) {
  const size_t b = (size_t)steps * (kVStepK / 8) * 256, part = (size_t)kVTok * kVRows * 4;
  if (mx) return b + part;
  return b + (size_t)kScaleRing * 2 * kVRows * 2 + (size_t)steps * 2 * kVTok * 4 + part;
}

template <int FMT>
static cudaError_t launch_verify_fmt(const MatvecArgs& a) {
  const Geometry g = make_geometry(a.fmt, a.N, a.K);
  VParams p;
  p.w = static_cast<const uint8_t*>(a.w);
  p.x = static_cast<const uint8_t*>(a.x);
  p.y = a.y;
  p.dbg = a.dbg;
  p.N = a.N;
  p.K = a.K;
  p.T = a.ntok;
  p.row_tiles = g.row_tiles;
  p.chunks = g.chunks;
  p.last_lanes = g.last_lanes;
  p.full_tile = g.full_tile;
  p.rowtile = g.rowtile;
  p.x_f32 = a.x_f32 ? 1 : 0;
  p.x_vec_bytes = fmt_is_mx(a.fmt) ? (uint32_t)a.K * 2u : (a.x_f32 ? (uint32_t)a.K * 4u : (uint32_t)q8_vec_bytes(a.K));
  for (int i = 0; i < 4; ++i) p.lut[i] = a.lut[i] ^ 0x80808080u;
  p.groups = a.K / 32;
  const int row_blocks = (a.N + kVRows - 1) / kVRows;
  // About one wave of two CTAs per SM: a sorted gather's grid.y is an upper
  // bound of its work items (ceil(slots / 16) + distinct experts, known only
  // on the device); K is split for about one item per expert that can occur.
  const int nslots = a.ids ? a.ntok * a.top_k : 0;
  const int experts = a.ids ? (a.n_experts < nslots ? a.n_experts : nslots) : 1;
  const int items = a.ids ? (nslots + kVTok - 1) / kVTok + experts : 1;
  int split = (2 * device_sm_count()) / (row_blocks * experts);
  if (split > kVMaxSplit) split = kVMaxSplit;
  if (split > p.groups / 2) split = p.groups / 2;
  if (split < 1) split = 1;
  while ((p.groups + split - 1) / split > 2 * kVMaxSteps && split < kVMaxSplit) ++split;
  p.split = split;
  p.steps = ((p.groups + split - 1) / split + 1) / 2;
  p.prefetch = a.prefetch ? 1 : 0;
  p.ids = a.ids;
  p.top_k = a.top_k;
  p.nslots = nslots;
  p.per_slot = a.per_slot;
  p.n_experts = a.n_experts;
  p.expert_stride = a.expert_stride;
  constexpr bool kMx = fmt_is_mx(FMT);
  // MX: the build sized for three CTAs per SM (72 registers) when each CTA's
  // K range is short (measured on GB300: 2880^2 x 8-16 tokens, 6 steps per
  // CTA, 7-9% faster; 7168^2, 23 steps, slower)
  const int variant = (kMx && p.steps <= kShortKSteps) ? 1 : 0;
  auto kernel = [variant] {
    if constexpr (kMx) {
      return variant ? verify_mx_kernel<FMT, 3> : verify_mx_kernel<FMT, 2>;
    } else {
      return verify_kernel<FMT>;
    }
  }();
  const size_t smem = verify_smem_bytes(kMx, p.steps);
  static std::mutex mu;
  static size_t configured[2][64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (configured[variant][dev] < smem) {
      g_launch_stage = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      configured[variant][dev] = smem;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(row_blocks * split), (unsigned)items);
  cfg.blockDim = dim3(kVThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeClusterDimension;
  attr[na].val.clusterDim.x = (unsigned)split;
  attr[na].val.clusterDim.y = 1;
  attr[na].val.clusterDim.z = 1;
  ++na;
  if (a.stream != nullptr) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  g_launch_stage = "cudaLaunchKernelEx(verify)";
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_verify(const MatvecArgs& a) {
  switch (a.fmt) {
    case MXFP4: return launch_verify_fmt<MXFP4>(a);
    case MXFP8: return launch_verify_fmt<MXFP8>(a);
    case CB2: return launch_verify_fmt<CB2>(a);
    case CB3: return launch_verify_fmt<CB3>(a);
    default: return launch_verify_fmt<CB4>(a);
  }
}

QMV_DEFINE_STATUS_ACCESSOR(status_verify)

}  // namespace qmv
