// qmv_verify.cu -- verify and batched products of the MX formats on the
// fifth-generation tensor cores (tcgen05): dense matvecs of 5..16 tokens, and
// sorted expert gathers of 33..128 routed slots.
//
// A speculative-decoding verify batch applies one weight matrix to several
// tokens at once ("perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on RDNA ...",
// "Depends on": the batched ROCmFPX MMQ that runs the verify batch). With
// more than a few tokens the product is a skinny GEMM, D[n][t] = sum_k W[n][k]
// x[t][k], and the CUDA-core matvec becomes ALU-bound (one FMA per weight and
// token). Here the CUDA cores only decode: each E2M1 / E4M3 code times its
// group's 2^(e-127) is written as an exact bf16 into a shared-memory operand,
// and one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32, M = 128
// rows, N = 16 tokens, K = 16) accumulating in tensor memory. Products of
// bf16 values are exact in fp32, so the result differs from the CUDA-core
// path only in the order of the fp32 additions.
//
// Work decomposition: a CTA owns 128 rows (16 row tiles of the packed
// layout) and one of `split` K ranges; the `split` CTAs of a row block form a
// thread-block cluster and add their partial sums through distributed shared
// memory in rank order (deterministic), each rank storing a share of the
// outputs. Per CTA: 8 decoding warps -- a warp decodes 16 rows (two row
// tiles) of every 64-column step, a lane taking one row and one of the two
// 32-groups, its weight loads issued a window of steps ahead -- and one warp
// that issues the MMAs. Three A buffers, each with a "full" barrier (one
// arrival per decoding warp) and an "empty" one (tcgen05.commit), let the
// warps decode ahead of the tensor core. A sorted gather adds a second grid
// dimension of work items, one (expert, up to 16 of its slots) pair each.
//
// Operand layouts (no swizzle, K-major "canonical" core matrices of 8 rows x
// 16 bytes): A step buffer (128 rows x 64 columns), core matrix (row group
// g, k group kk) at kk * 2048 + g * 128; B (activations, tokens padded to 16
// with zeros), core matrix (token group g, k group kk) at kk * 256 + g * 128. Descriptor
// leading byte offset = the K-direction stride, stride byte offset = the
// row-direction stride.
//
// Range: a weight whose value exceeds bf16 / fp32 range (E8M0 254 with
// |E2M1| >= 2, or E8M0 255 = NaN) decodes to inf / NaN here; the CUDA-core
// path multiplies the scale into the fp32 sum instead.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "qmv_device.cuh"
#include "qmv_internal.h"
#include "qmv_layout.h"

namespace qmv {
namespace cg = cooperative_groups;

namespace {

constexpr int kVRows = 128;      // rows per CTA (MMA M)
constexpr int kVTok = 16;        // MMA N: tokens, padded
constexpr int kDecoders = 256;   // decoding threads: two per row
constexpr int kVThreads = kDecoders + 32;   // plus one warp that issues the MMAs
constexpr int kVStepK = 64;      // columns per step (one A buffer): 2 groups of 32
constexpr int kVBufs = 3;        // A buffers
// Steps of weight loads in flight per thread: 128 bytes (8 MXFP4 or 4
// MXFP8 lane blocks), so two CTAs keep ~64 KB per SM in flight.
template <int FMT>
struct Window {
  static constexpr int value = 128 / lane_code_bytes(FMT);
};
constexpr uint32_t kABytes = kVRows * kVStepK * 2;   // 16 KB
constexpr uint32_t kALbo = kVRows / 8 * 128;          // A: k-group stride (16 row groups of 128 B)
constexpr int kVMaxSplit = 8;    // cluster size limit (portable)
constexpr int kVMaxSlots = 128;  // routed slots of a sorted gather
constexpr int kVMaxSteps = 24;   // activation operand <= 48 KB (two CTAs per SM)

struct VParams {
  const uint8_t* w;
  const __nv_bfloat16* x;
  __nv_bfloat16* y;
  int N, K, T;
  int row_tiles, chunks, last_lanes;
  uint32_t full_tile;
  uint64_t rowtile;
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

// kind::f16 instruction descriptor: fp32 accumulator, bf16 A and B, both
// K-major, N = 16, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kVTok >> 3) << 17) |
                            ((uint32_t)(kVRows >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
  asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
               " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
               :: "r"(tmem), "l"(a), "l"(b), "r"(kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Lane block of one row and one 32-group: codes (LCB bytes) and scale.
template <int FMT>
struct Block {
  static constexpr int kWords = lane_code_bytes(FMT) / 4;
  uint32_t c[kWords];
  uint32_t e;
};

template <int FMT>
__device__ __forceinline__ void load_block(const VParams& p, const uint8_t* w, int rt, int r8, int g, bool valid,
                                           Block<FMT>& b) {
  if (!valid) {
#pragma unroll
    for (int i = 0; i < Block<FMT>::kWords; ++i) b.c[i] = 0;
    b.e = 127;
    return;
  }
  const int c = g >> 5, l = g & 31;
  const int L = (c == p.chunks - 1) ? p.last_lanes : 32;
  const uint8_t* tile = w + (uint64_t)rt * p.rowtile + (uint64_t)c * p.full_tile;
  const uint4* src = reinterpret_cast<const uint4*>(tile + (size_t)(r8 * L + l) * lane_code_bytes(FMT));
#pragma unroll
  for (int q = 0; q < Block<FMT>::kWords / 4; ++q) {
    const uint4 v = __ldg(src + q);
    b.c[4 * q] = v.x; b.c[4 * q + 1] = v.y; b.c[4 * q + 2] = v.z; b.c[4 * q + 3] = v.w;
  }
  b.e = __ldg(tile + tile_code_bytes(FMT, L) + l * kRows + r8);
}

__device__ __forceinline__ uint32_t scaled_bf16x2(uint32_t h2, float s) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * s, f.y * s);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// 32 codes of a lane block -> 32 exact bf16 values (code value x 2^(e-127)),
// written as four 16-byte core-matrix rows (k groups kk0 .. kk0 + 3, kALbo
// bytes apart).
template <int FMT>
__device__ __forceinline__ void decode_store(const Block<FMT>& b, uint8_t* a_row, int kk0) {
  const float s = e8m0_to_f32(b.e);
  uint32_t out[16];
  if constexpr (FMT == MXFP4) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t h[4];
      e2m1x8_to_f16x2(b.c[q], h);
#pragma unroll
      for (int i = 0; i < 4; ++i) out[4 * q + i] = scaled_bf16x2(h[i], s);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t h[2];
      e4m3x4_to_f16x2(b.c[q], h);
      out[2 * q] = scaled_bf16x2(h[0], s);
      out[2 * q + 1] = scaled_bf16x2(h[1], s);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    *reinterpret_cast<uint4*>(a_row + (size_t)(kk0 + j) * kALbo) =
        make_uint4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
  }
}

template <int FMT>
__global__ void __launch_bounds__(kVThreads, 2) verify_kernel(const __grid_constant__ VParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kVBufs + 1];   // empty (MMAs done) x kVBufs, final
  __shared__ __align__(8) uint64_t full[kVBufs];        // A buffer written by all decoding warps
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = (int)(blockIdx.x % (unsigned)p.split);
  const int rb = (int)(blockIdx.x / (unsigned)p.split);
  const int g0 = (int)((long)rank * p.groups / p.split);
  const int g1 = (int)((long)(rank + 1) * p.groups / p.split);
  const int steps = (g1 - g0 + 1) / 2;

  // Sorted gather: work item blockIdx.y is the (expert, group of <= 16 of
  // its slots) pair of that index, experts in order of their first slot and
  // slots in slot order. Each CTA derives it from the ids in shared memory:
  // thread s finds its expert's slot count and its rank among them; the
  // first slot of each expert counts the work items of the experts before
  // it. An index past the last item leaves the CTA idle (every CTA of a
  // cluster shares blockIdx.y, so a cluster exits as a whole, before it
  // allocates tensor memory). Slots with an invalid id get zero rows.
  __shared__ int s_ids[kVMaxSlots];
  __shared__ int s_cnt[kVMaxSlots];
  __shared__ int s_slot[kVTok];
  __shared__ int s_item[3];   // expert, first rank, tokens
  int T = p.T;
  const uint8_t* w = p.w;
  if (p.ids != nullptr) {
    if (!p.prefetch) pdl_wait();
    if (tid == 0) s_item[0] = -1;
    int e = -1;
    if (tid < p.nslots) {
      e = p.ids[tid];
      if (e < 0 || e >= p.n_experts) e = -1;
      s_ids[tid] = e;
    }
    __syncthreads();
    int cnt = 0, rk = 0;
    bool first = false;
    if (tid < p.nslots && e >= 0) {
      for (int q = 0; q < p.nslots; ++q) {
        const int eq = s_ids[q];
        cnt += (eq == e);
        rk += (eq == e && q < tid);
      }
      first = (rk == 0);
    }
    if (tid < p.nslots) s_cnt[tid] = first ? cnt : 0;
    __syncthreads();
    if (first) {
      int before = 0;
      for (int q = 0; q < tid; ++q) before += (s_cnt[q] + kVTok - 1) / kVTok;
      const int mine = (cnt + kVTok - 1) / kVTok;
      const int y = (int)blockIdx.y;
      if (y >= before && y < before + mine) {
        s_item[0] = e;
        s_item[1] = (y - before) * kVTok;
        s_item[2] = min(kVTok, cnt - (y - before) * kVTok);
      }
    }
    __syncthreads();
    if (s_item[0] >= 0 && e == s_item[0] && rk >= s_item[1] && rk < s_item[1] + s_item[2]) s_slot[rk - s_item[1]] = tid;
    if (blockIdx.y == 0) {
      if (p.prefetch) pdl_wait();   // outputs are written only after the preceding kernel completed
      for (int i = rank * kVThreads + tid; i < p.nslots * kVRows; i += p.split * kVThreads) {
        const int sl = i / kVRows, orow = rb * kVRows + i % kVRows;
        if (s_ids[sl] < 0 && orow < p.N) p.y[(size_t)sl * p.N + orow] = __float2bfloat16_rn(0.f);
      }
    }
    __syncthreads();
    if (s_item[0] < 0) return;
    T = s_item[2];
    w = p.w + (uint64_t)s_item[0] * p.expert_stride;
  }
  uint8_t* abuf = smem;                                   // kVBufs x 16 KB
  uint8_t* bbuf = smem + kVBufs * kABytes;                // steps x 64 columns x 16 tokens
  float* part = reinterpret_cast<float*>(smem);           // 16 x 128 fp32, after the MMAs

  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;" :: "r"(smem_addr(&tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int i = 0; i <= kVBufs; ++i) mbar_init(smem_addr(&bars[i]), 1);
    for (int i = 0; i < kVBufs; ++i) mbar_init(smem_addr(&full[i]), kDecoders / 32);
    fence_mbar_init();
  }
  // Weight stream: decoding warp w takes row tiles 2w and 2w + 1 of the
  // block; lane (i, r8, h) takes row r8 of tile 2w + i and group
  // 2 * step + h, so one warp load covers 16 rows x 32 contiguous bytes
  // (16 full sectors).
  // The first window of loads goes out first (before griddepcontrol.wait
  // when the caller guarantees the weights are not the preceding kernel's
  // output), then the activations, whose loads are all issued before any of
  // them is stored.
  const bool decoder = tid < kDecoders;
  const int h = lane & 1;
  const int r = (warp & 7) * 16 + (lane >> 1);   // row of the block: tile 2w + (lane >> 4), row (lane >> 1) & 7
  const int row = rb * kVRows + r;
  const int rt = row >> 3, r8 = row & 7;
  const bool row_ok = decoder && rt < p.row_tiles;
  uint8_t* a_row = abuf + (r >> 3) * 128 + (r & 7) * 16;
  constexpr int kWindow = Window<FMT>::value;
  Block<FMT> win[kWindow];
  if (!p.prefetch) pdl_wait();
#pragma unroll
  for (int u = 0; u < kWindow; ++u) {
    const int g = g0 + 2 * u + h;
    load_block<FMT>(p, w, rt, r8, g, row_ok && u < steps && g < g1, win[u]);
  }
  if (p.prefetch) pdl_wait();
  pdl_launch_dependents();

  // Activation operand: tokens t < T of columns [32 g0, 32 g0 + 64 steps),
  // zero beyond the CTA's range and for padding tokens.
  {
    constexpr int kU = 4;
    const int kk_n = steps * (kVStepK / 8);
    const int k_end = g1 * 32;
    const int n_units = decoder ? kk_n * kVTok : 0;
    for (int u0 = tid; u0 < n_units; u0 += kU * kDecoders) {
      uint4 v[kU];
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int u = u0 + j * kDecoders;
        const int t = u % kVTok, kk = u / kVTok;
        const int k = g0 * 32 + kk * 8;
        v[j] = make_uint4(0, 0, 0, 0);
        if (u < n_units && t < T && k < k_end) {
          const int vec = (p.ids == nullptr) ? t : (p.per_slot ? s_slot[t] : s_slot[t] / p.top_k);
          v[j] = *reinterpret_cast<const uint4*>(p.x + (size_t)vec * p.K + k);
        }
      }
#pragma unroll
      for (int j = 0; j < kU; ++j) {
        const int u = u0 + j * kDecoders;
        const int t = u % kVTok, kk = u / kVTok;
        if (u < n_units) *reinterpret_cast<uint4*>(bbuf + (size_t)kk * 256 + (t >> 3) * 128 + (t & 7) * 16) = v[j];
      }
    }
  }

  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  bool ok = true;

  if (decoder) {
    for (int s0 = 0; s0 < steps; s0 += kWindow) {
#pragma unroll
      for (int u = 0; u < kWindow; ++u) {
        const int st = s0 + u;
        if (st < steps) {
          const int b = st % kVBufs;
          if (st >= kVBufs) {
            // the MMAs that read this buffer kVBufs steps ago are done
            ok &= mbar_wait_bounded(smem_addr(&bars[b]), (uint32_t)((st / kVBufs) - 1) & 1u, kWaitLimitNs);
          }
          decode_store<FMT>(win[u], a_row + (size_t)b * kABytes, 4 * h);
          const int gn = g0 + 2 * (st + kWindow) + h;
          load_block<FMT>(p, w, rt, r8, gn, row_ok && st + kWindow < steps && gn < g1, win[u]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&full[b]));
        }
      }
    }
  } else if (lane == 0) {
    // MMA issue: step st once every decoding warp has written its A buffer.
    for (int st = 0; st < steps; ++st) {
      const int b = st % kVBufs;
      ok &= mbar_wait_bounded(smem_addr(&full[b]), (uint32_t)(st / kVBufs) & 1u, kWaitLimitNs);
      tc_fence_after();
      const uint32_t a0 = smem_addr(abuf + (size_t)b * kABytes);
      const uint32_t b0 = smem_addr(bbuf + (size_t)st * (kVStepK / 8) * 256);
#pragma unroll
      for (int j = 0; j < kVStepK / 16; ++j) {
        mma_bf16(tmem, mma_desc(a0 + j * 2 * kALbo, kALbo, 128), mma_desc(b0 + j * 2 * 256, 256, 128),
                 (st > 0 || j > 0) ? 1u : 0u);
      }
      mma_commit(smem_addr(&bars[b]));
    }
    mma_commit(smem_addr(&bars[kVBufs]));
  }
  __syncwarp();
  ok &= mbar_wait_bounded(smem_addr(&bars[kVBufs]), 0u, kWaitLimitNs);
  tc_fence_after();
  if (!__all_sync(0xffffffffu, ok) && lane == 0) set_status(kStatusWaitTile);

  // Accumulator rows 32 w .. 32 w + 31 (tensor-memory lanes of warp w) ->
  // partial sums part[t][row], t < 16. The A buffers are free: every MMA that
  // read them has completed.
  if (warp < 4) {
    uint32_t v[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                   "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                   "=r"(v[15])
                 : "r"(tmem + ((uint32_t)(warp * 32) << 16)));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int t = 0; t < kVTok; ++t) part[t * kVRows + warp * 32 + lane] = __uint_as_float(v[t]);
  }
  tc_fence_before();

  // K ranges meet in rank order; rank q stores outputs q, q + split, ...
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  for (int i = rank * kVThreads + tid; i < kVRows * T; i += p.split * kVThreads) {  // all 9 warps
    const int t = i / kVRows, rr = i % kVRows;
    const int orow = rb * kVRows + rr;
    if (orow >= p.N) continue;
    float v[kVMaxSplit];
#pragma unroll
    for (int q = 0; q < kVMaxSplit; ++q) v[q] = (q < p.split) ? cluster.map_shared_rank(part, q)[t * kVRows + rr] : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int q = 0; q < kVMaxSplit; ++q) acc += v[q];   // rank order; absent ranks add +0
    const int oslot = (p.ids == nullptr) ? t : s_slot[t];
    p.y[(size_t)oslot * p.N + orow] = __float2bfloat16_rn(acc);
  }
  cluster.sync();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;" :: "r"(tmem));
  }
}

}  // namespace

// Verify-batch plan: rows in blocks of 128, K cut into `split` ranges (one
// cluster rank each) so that the grid covers about two CTAs per SM.
bool verify_supported(const MatvecArgs& a) {
  if (!fmt_is_mx(a.fmt) || a.x_f16 || a.glu || a.dbg != nullptr) return false;
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

size_t verify_smem_bytes(int steps) { return (size_t)kVBufs * kABytes + (size_t)steps * (kVStepK / 8) * 256; }

template <int FMT>
static cudaError_t launch_verify_fmt(const MatvecArgs& a) {
  const Geometry g = make_geometry(a.fmt, a.N, a.K);
  VParams p;
  p.w = static_cast<const uint8_t*>(a.w);
  p.x = static_cast<const __nv_bfloat16*>(a.x);
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.N = a.N;
  p.K = a.K;
  p.T = a.ntok;
  p.row_tiles = g.row_tiles;
  p.chunks = g.chunks;
  p.last_lanes = g.last_lanes;
  p.full_tile = g.full_tile;
  p.rowtile = g.rowtile;
  p.groups = a.K / 32;
  const int row_blocks = (a.N + kVRows - 1) / kVRows;
  // One wave of at most two CTAs per SM; a sorted gather has many work items
  // (grid.y), so it splits K only as far as the activation operand needs.
  const int nslots = a.ids ? a.ntok * a.top_k : 0;
  const int items = a.ids ? (nslots + kVTok - 1) / kVTok + (a.n_experts < nslots ? a.n_experts : nslots) : 1;
  int split = a.ids ? 1 : (2 * device_sm_count()) / row_blocks;
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
  const size_t smem = verify_smem_bytes(p.steps);
  static std::mutex mu;
  static size_t configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (configured[dev] < smem) {
      g_launch_stage = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
      err = cudaFuncSetAttribute(verify_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
      configured[dev] = smem;
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
  return cudaLaunchKernelEx(&cfg, verify_kernel<FMT>, p);
}

cudaError_t launch_verify(const MatvecArgs& a) {
  return a.fmt == MXFP4 ? launch_verify_fmt<MXFP4>(a) : launch_verify_fmt<MXFP8>(a);
}

QMV_DEFINE_STATUS_ACCESSOR(status_verify)

}  // namespace qmv
