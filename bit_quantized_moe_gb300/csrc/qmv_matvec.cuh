// qmv_matvec.cuh -- the decode matvec kernel (dense and expert-gathered), one
// template for all weight formats.
//
// Work decomposition. A "work item" is one row tile (kRows rows) of one
// matrix applied to up to NV activation vectors (the "entry": an expert and
// the (token, slot) pairs routed to it). Items are shared out evenly over the
// CTAs of a one-wave grid (round-robin, or contiguous ranges for per-slot
// gathers), an item may be cut into K ranges (split-K, for calls with few
// items), and the resulting tasks are dealt over each CTA's warps. A warp
// streams its tasks' tiles -- one tile per K chunk -- through a private ring
// of shared-memory stages (Shape::stages) filled by bulk asynchronous copies
// (one elected lane issues them, an mbarrier per stage tracks completion).
// Lane l of the warp owns columns [32 l, 32 l + 32) of every chunk for all
// kRows rows, so the activations it needs are loaded into registers once per
// chunk and reused for kRows rows. After the task's last chunk a warp
// reduce-scatter (shuffles) leaves each (row, vector) sum in one lane group,
// which stores it (or, under split-K, parks it for the item's last range).
//
// Per format (lane-block encodings are defined in qmv_layout.h):
//   MXFP4: E2M1 nibbles -> f16x2 with cvt.rn.f16x2.e2m1x2, mixed-precision
//          FMA (f16 operands, fp32 product and sum) against the activations
//          staged as group-scaled f16, fp32 group sum times 2^(e-127) per 32
//          weights ("perf(rocm): add an mxfp4 arm to the warp-shared
//          gather_qmv kernel ...", "Proposed Solution" item 1).
//   MXFP8: E4M3 bytes -> f16x2 with cvt.rn.f16x2.e4m3x2, then as MXFP4
//          (the f16 MXFP4 and MXFP8 gathers the same page names as the next
//          scope, "Scope"). The kernels' ALT variant of an MX format takes
//          fp16 activations, staged as they are (unscaled), and stores fp16.
//
// Kernel variants: matvec_kernel<FMT, NV, ALT>. ALT is the integer block-sum
// export (DBG) for the codebook formats and fp16 activations/outputs (XH)
// for the MX formats: a compile-time choice, so the common kernels carry no
// code for either (each launch runs its prologue from a cold instruction
// cache).
//   CB2/CB3/CB4: codes -> int8 through byte permutes (prmt) over the codebook
//          held in registers, dp4a against q8_1 activations, integer sums per
//          16-weight half-block (CB2, CB3) or 32-weight block (CB4), then
//          d_b * 2^(e-127) * isum in fp32 ("perf(ggml/hip): optimize ROCMFPX
//          fp3/fp2 MMVQ on RDNA ...", "Changes" items 1, 2, 4 and the review
//          reply's dot structure).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "qmv_device.cuh"
#include "qmv_internal.h"
#include "qmv_layout.h"

namespace qmv {

// Launch shape of the kernel for entries of up to NV vectors: two CTAs per SM;
// a CTA of `warps` warps, each with a ring of `stages` tiles. One-vector
// kernels (every decode call at one token) run 10 warps with 2-stage rings:
// 20 warps per SM give each warp about one 8-row item of a 2880-row gather,
// and 40 tiles (174 KB) are in flight per SM. Two-vector kernels (<= 128
// registers) run 8 warps with 2-stage rings; 3- and 4-vector kernels need up
// to 160 registers per thread and run 6 warps with 3-stage rings.
template <int NV>
struct Shape {
  static constexpr int warps = (NV == 1) ? 10 : (NV == 2 ? 8 : 6);
  static constexpr int stages = (NV <= 2) ? 2 : 3;
};
constexpr int kCtasPerSm = 2;

// Tile copies per warp issued before griddepcontrol.wait in a prefetching
// launch; the rest follow the activation loads, which would otherwise queue
// behind them. Measured best on GB300 (same-box timings of every workload
// config): none for MXFP4 one- and two-vector kernels, one for the codebook
// ones, all for three- and four-vector kernels (their 3-stage rings and
// heavier arithmetic hide the activation latency). Contiguously dealt
// launches (per-slot gathers: the down projection of a layer) issue every
// ring stage early whatever the format: their CTAs start while the
// preceding gate/up launch drains, about 2 us before its completion releases
// the wait, so the copies have landed before the activation loads go out
// (24-layer MXFP4 sweep: 18.9 -> 17.8 us per layer).
template <int FMT, int NV>
struct EarlyTiles {
  static constexpr int value = (NV >= 3) ? Shape<NV>::stages : (fmt_is_mx(FMT) ? 0 : 1);
};

inline void launch_shape(int nv, int& warps, int& stages) {
  switch (nv) {
    case 1: warps = Shape<1>::warps; stages = Shape<1>::stages; break;
    case 2: warps = Shape<2>::warps; stages = Shape<2>::stages; break;
    default: warps = Shape<4>::warps; stages = Shape<4>::stages; break;
  }
}

// Vectors per entry of a launch's kernel. Dense calls put every token in each
// entry (up to 4). Gathers group the routed pairs of one expert; with
// independently routed tokens that is almost always one pair, so gathers use
// at most the two-vector kernel (its launch shape keeps more warps per SM) and
// an expert shared by more pairs is streamed once per two of them.
inline int launch_vectors(bool gather, int ntok) {
  const int cap = gather ? 2 : 4;
  return ntok < cap ? ntok : cap;
}
constexpr int kMaxEntries = 32;  // routed slots (ntok * top_k) of a gather; dense entries <= 16 / 4

#ifdef QMV_PHASE_PROBE
static __device__ unsigned long long g_phase[kProbeSlots * kProbeCtas * kProbeWarps * kPhases];
#endif
constexpr int kMaxDevices = 64;

struct Entry {
  int expert;
  int nv;
  int vec[4];   // activation vector index per routed pair
  int slot[4];  // output slot (t for dense, t * top_k + j for gather)
};

struct KParams {
  const uint8_t* w;
  uint64_t expert_stride;
  const uint8_t* x;
  uint32_t x_vec_bytes;   // bytes per activation vector (global and shared)
  int nvec;
  int x_slots;            // vectors the shared activation region holds (<= nvec)
  const int32_t* ids;
  int ntok, top_k, per_slot, n_experts;
  int contig;             // deal contiguous item ranges and stage only the vectors they use
  int N, K, row_tiles, chunks, last_lanes;
  uint32_t full_tile, last_tile;
  uint64_t rowtile;
  void* y;
  int32_t* dbg;
  uint32_t lut[4];
  uint32_t flags;
  int out_n;              // rows of each output vector (N, or N / 2 rounded for gate/up fusion)
  int splits;             // K ranges per item (split-K inside a CTA), >= 1
  int split_chunks;       // chunks per K range (the last may be shorter)
  int items_per_cta;      // upper bound on items per CTA (split-K partial slots)
  FastDiv fd_rt, fd_split, fd_grid, fd_grp, fd_per;   // row_tiles, splits, grid, K / 32, x_vec_bytes / 16
#ifdef QMV_PHASE_PROBE
  int probe_slot;         // launch slot of the phase probe, -1 = not recorded
#endif
};

__device__ __forceinline__ void probe_phase(const KParams& p, int k) {
#ifdef QMV_PHASE_PROBE
  if ((threadIdx.x & 31) == 0 && p.probe_slot >= 0 && blockIdx.x < kProbeCtas && (threadIdx.x >> 5) < kProbeWarps) {
    g_phase[(((size_t)p.probe_slot * kProbeCtas + blockIdx.x) * kProbeWarps + (threadIdx.x >> 5)) * kPhases + k] =
        global_timer_ns();
  }
#else
  (void)p;
  (void)k;
#endif
}

// KParams::flags
constexpr uint32_t kFlagPrefetch = 1u;   // weights and ids are not written by the preceding kernel
constexpr uint32_t kFlagGlu = 2u;        // gate/up-interleaved matrix: store silu(gate) * up
constexpr uint32_t kFlagXF32 = 4u;       // codebooks: x is fp32, quantized to q8_1 while staged

// Largest number of activation vectors one work item applies a tile to.
template <int FMT>
struct MaxVectors {
  static constexpr int value = 4;
};

__host__ __device__ constexpr uint32_t round_up_u32(uint32_t v, uint32_t a) {
  return (v + a - 1) / a * a;
}

struct SmemLayout {
  uint32_t x_off, xinv_off, ring_off, bar_off, ent_off, part_off, cnt_off, total;
};

// Split-K partial sums: 32 floats (8 rows x up to 4 vectors, after the
// warp reduction) per (item of the CTA, K range), and one counter per item.
constexpr uint32_t kPartFloats = 32;
constexpr int kMaxSplits = 8;

// x region: the staged activation vectors, x_slots of them (per-slot gathers
// stage only the vectors of the CTA's items, at consecutive positions); for
// the MX formats they are f16 (see stage_x_mxfp4) and xinv holds one float
// per 32-group.
__host__ __device__ inline SmemLayout smem_layout(int fmt, uint32_t nvec, uint32_t x_vec_bytes,
                                                  uint32_t full_tile, int K, int warps, int stages,
                                                  int splits, int items_per_cta) {
  SmemLayout L;
  L.x_off = 0;
  L.xinv_off = round_up_u32(nvec * x_vec_bytes, 16);
  const uint32_t xinv_bytes = fmt_is_mx(fmt) ? nvec * (uint32_t)(K / 32) * 4u : 0u;
  L.ring_off = round_up_u32(L.xinv_off + xinv_bytes, 128);
  L.bar_off = L.ring_off + (uint32_t)(warps * stages) * full_tile;
  L.ent_off = round_up_u32(L.bar_off + (uint32_t)(warps * stages) * 8, 16);
  L.part_off = L.ent_off + kMaxEntries * (uint32_t)sizeof(Entry);
  const uint32_t slots = (splits > 1) ? (uint32_t)items_per_cta : 0u;
  L.cnt_off = L.part_off + slots * (uint32_t)splits * kPartFloats * 4u;
  L.total = L.cnt_off + slots * 4u;
  return L;
}

// ---------------------------------------------------------------------------
// Work list
// ---------------------------------------------------------------------------

// Work list, built by the 32 lanes of one warp (lane s = routed slot s):
// entries in order of their first slot, an expert's slots grouped NV at a time
// (repeated experts share one tile stream for up to NV vectors). Unused vec /
// slot positions repeat the entry's first member. Also copies the ids to
// s_ids. Returns the entry count on every lane.
template <int NV>
__device__ int build_entries_warp(const KParams& p, Entry* ent, int* s_ids) {
  const int lane = threadIdx.x & 31;
  if (p.ids == nullptr) {
    const int n = (p.ntok + NV - 1) / NV;
    if (lane < n) {
      const int t = lane * NV;
      Entry e;
      e.expert = 0;
      e.nv = min(NV, p.ntok - t);
      for (int i = 0; i < 4; ++i) e.vec[i] = e.slot[i] = t + min(i, e.nv - 1);
      ent[lane] = e;
    }
    __syncwarp();
    return n;
  }
  const int nslots = p.ntok * p.top_k;
  const bool in = lane < nslots;
  const int ex = in ? p.ids[lane] : -1;
  if (in) s_ids[lane] = ex;
  const bool valid = in && ex >= 0 && ex < p.n_experts;
  // invalid slots get keys no valid id or other slot can have
  const unsigned key = valid ? (unsigned)ex : (0x80000000u | (unsigned)lane);
  const unsigned match = __match_any_sync(0xffffffffu, key);
  const int r = __popc(match & ((1u << lane) - 1u));   // rank among the slots of this expert
  const int c = r / NV, m = r % NV;                    // chunk of NV slots, position in it
  const unsigned leaders = __ballot_sync(0xffffffffu, valid && m == 0);
  unsigned rest = match;                               // drop the c * NV earlier slots
  for (int i = 0; i < c * NV; ++i) rest &= rest - 1u;
  const int leader_lane = __ffs(rest) - 1;             // first slot of this chunk
  const int eid = __popc(leaders & ((1u << leader_lane) - 1u));
  const int v = p.per_slot ? lane : lane / p.top_k;
  if (valid && m == 0) {
    ent[eid].expert = ex;
    ent[eid].nv = min(NV, __popc(match) - c * NV);
    for (int i = 0; i < 4; ++i) {
      ent[eid].vec[i] = v;
      ent[eid].slot[i] = lane;
    }
  }
  __syncwarp();
  if (valid && m != 0) {
    ent[eid].vec[m] = v;
    ent[eid].slot[m] = lane;
  }
  __syncwarp();
  return __popc(leaders);
}

// ---------------------------------------------------------------------------
// Tile loads
// ---------------------------------------------------------------------------

// Work of a CTA: its share of the n items, the same number within one for
// every CTA (and, with a full grid, every SM). Calls whose vectors are shared
// by all slots (dense, gate/up) deal items round-robin (CTA b: b, b + G,
// ...), so that at any moment the grid streams neighbouring row tiles.
// Per-slot gathers, and dense calls of more than one entry (over 4 tokens),
// give each CTA a contiguous range (p.contig), which lies within one or two
// entries, so the CTA stages only those entries' vectors; the entries of a
// dense call then stream the same row tiles at about the same time, and all
// but the first read them from L2. Item k of the
// CTA is split into `splits` K ranges, and task lt = k * splits + r (range r
// of item k) goes to warp lt % W. A warp streams the tiles of its tasks, in
// order, through its ring. Lane 0 keeps the issue cursor (the next task and
// chunk to copy).
struct WarpPipe {
  const KParams* p;   // the matrix (points into kernel parameter space)
  const Entry* ent;   // the work list
  uint32_t ring;      // shared address of this warp's stage 0
  uint32_t bars;      // shared address of this warp's mbarrier 0
  const uint8_t* ring_ptr;
  int first;          // the CTA's first item
  int stride;         // between the CTA's items (G round-robin, 1 contiguous)
  int n_tasks;        // tasks of this CTA
  int warps;          // W
  int iss_n;          // tiles issued so far
  int iss_lt, iss_c, iss_c1;  // issue cursor: task, next chunk, end chunk
  const uint8_t* iss_base;    // global address of the cursor task's row tile
  uint64_t policy;
};

__device__ __forceinline__ int task_item(const KParams& p, const WarpPipe& wp, int lt) {
  return wp.first + (int)fast_div((uint32_t)lt, p.fd_split) * wp.stride;
}

// The CTA's items first, first + stride, ... (count of them) out of n.
__device__ __forceinline__ void cta_items(const KParams& p, int n, int& first, int& stride, int& count) {
  const int b = blockIdx.x, G = gridDim.x;
  if (p.contig) {
    const int per = (int)fast_div((uint32_t)n, p.fd_grid), rem = n - per * G;
    first = b * per + (b < rem ? b : rem);
    count = per + (b < rem ? 1 : 0);
    stride = 1;
  } else {
    first = b;
    stride = G;
    count = (b < n) ? (int)fast_div((uint32_t)(n - b + G - 1), p.fd_grid) : 0;
  }
}

__device__ __forceinline__ void task_chunks(const KParams& p, int lt, int& c0, int& c1) {
  c0 = (int)fast_mod((uint32_t)lt, p.fd_split) * p.split_chunks;
  c1 = min(p.chunks, c0 + p.split_chunks);
}

// Moves the issue cursor to task lt (the divisions happen once per task).
__device__ __forceinline__ void cursor_to(WarpPipe& wp, int lt) {
  wp.iss_lt = lt;
  if (lt >= wp.n_tasks) return;
  const KParams& p = *wp.p;
  task_chunks(p, lt, wp.iss_c, wp.iss_c1);
  const int item = task_item(p, wp, lt);
  const int ei = (int)fast_div((uint32_t)item, p.fd_rt);
  const Entry& e = wp.ent[ei];
  wp.iss_base = p.w + (uint64_t)e.expert * p.expert_stride + (uint64_t)(item - ei * p.row_tiles) * p.rowtile;
}

// Lane 0: copies the next tile of this warp's task sequence into ring stage
// (tiles issued) % ST, if there is one.
template <int ST>
__device__ __forceinline__ void issue_next(WarpPipe& wp) {
  if (wp.iss_lt >= wp.n_tasks) return;
  const KParams& p = *wp.p;
  const int c = wp.iss_c;
  const uint8_t* src = wp.iss_base + (uint64_t)c * p.full_tile;
  const uint32_t bytes = (c == p.chunks - 1) ? p.last_tile : p.full_tile;
  const int s = wp.iss_n % ST;
  const uint32_t bar = wp.bars + 8u * s;
  mbar_arrive_expect_tx(bar, bytes);
  bulk_copy_g2s_hint(wp.ring + (uint32_t)s * p.full_tile, src, bytes, bar, wp.policy);
  ++wp.iss_n;
  if (++wp.iss_c == wp.iss_c1) cursor_to(wp, wp.iss_lt + wp.warps);
}

// ---------------------------------------------------------------------------
// Decoders: 32 codes of one lane and one row -> 8 words of int8x4 (CB) in
// column order: word i holds columns 4i..4i+3.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void decode_cb2(uint32_t w0, uint32_t w1, uint32_t l0, uint32_t (&v)[8]) {
  uint32_t s;
  s = w0 & 0x33333333u;
  v[0] = prmt(l0, l0, s);
  v[1] = prmt(l0, l0, s >> 16);
  s = (w0 >> 2) & 0x33333333u;
  v[2] = prmt(l0, l0, s);
  v[3] = prmt(l0, l0, s >> 16);
  s = w1 & 0x33333333u;
  v[4] = prmt(l0, l0, s);
  v[5] = prmt(l0, l0, s >> 16);
  s = (w1 >> 2) & 0x33333333u;
  v[6] = prmt(l0, l0, s);
  v[7] = prmt(l0, l0, s >> 16);
}

__device__ __forceinline__ void decode_cb3(uint32_t a, uint32_t b, uint32_t c, uint32_t l0,
                                           uint32_t l1, uint32_t (&v)[8]) {
  uint32_t s;
  s = (a & 0x33333333u) | ((c << 2) & 0x44444444u);
  v[0] = prmt(l0, l1, s);
  v[1] = prmt(l0, l1, s >> 16);
  s = ((a >> 2) & 0x33333333u) | ((c << 1) & 0x44444444u);
  v[2] = prmt(l0, l1, s);
  v[3] = prmt(l0, l1, s >> 16);
  s = (b & 0x33333333u) | (c & 0x44444444u);
  v[4] = prmt(l0, l1, s);
  v[5] = prmt(l0, l1, s >> 16);
  s = ((b >> 2) & 0x33333333u) | ((c >> 1) & 0x44444444u);
  v[6] = prmt(l0, l1, s);
  v[7] = prmt(l0, l1, s >> 16);
}

// 16-entry codebook: two 8-entry lookups (codes 0..7 and 8..15) and a byte
// select by bit 3 of each code.
__device__ __forceinline__ uint32_t cb4_quad(uint32_t sel_lo, uint32_t hi_bits, const uint32_t (&t)[4]) {
  const uint32_t a = prmt(t[0], t[1], sel_lo);
  const uint32_t b = prmt(t[2], t[3], sel_lo);
  const uint32_t pick = (hi_bits & 0x4444u) | 0x3210u;
  return prmt(a, b, pick);
}

__device__ __forceinline__ void decode_cb4(const uint32_t (&w)[4], const uint32_t (&t)[4], uint32_t (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0x77777777u;
    v[2 * i] = cb4_quad(lo, w[i] >> 1, t);
    v[2 * i + 1] = cb4_quad(lo >> 16, w[i] >> 17, t);
  }
}

// ---------------------------------------------------------------------------
// Per-chunk compute
// ---------------------------------------------------------------------------

// acc + w * x with f16 operands, product and sum in fp32 (mixed-precision FMA,
// sm_100 and later).
__device__ __forceinline__ float fma_f16_f32(uint16_t w, uint16_t x, float acc) {
  asm("fma.rn.f32.f16 %0, %1, %2, %0;" : "+f"(acc) : "h"(w), "h"(x));
  return acc;
}

// Exact 2^e as an fp32 for e in [-149, 127].
__device__ __forceinline__ float pow2f(int e) {
  return (e >= -126) ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// Activation staging. Every thread issues the global loads of several units
// (kStageU MXFP4 groups, one fp32 block, four 16-byte pieces) before it
// converts or stores any of them: at the start of a launch the loads queue
// behind the weight tiles just requested, so each extra dependent round of
// loads costs a full queued round trip. (One fp32 block, 32 registers, keeps
// the one-vector codebook kernels within 102 registers per thread.)
constexpr int kStageU = 2;

// MXFP4 activations are staged once per CTA: each 32-element group (one E8M0
// group of the weights) is scaled by 2^s, s chosen so that the group's largest
// magnitude lands in [2^14, 2^15), and stored as f16; xinv holds 2^-s. A bf16
// value v of the group is then exact in f16 whenever |v| >= max|group| * 2^-31,
// so every product w * x' (E2M1 times f16) and its fp32 accumulation match
// fp32 arithmetic on the bf16 input, and dot * 2^-s undoes the shift exactly.
// One thread converts one group (64 bytes of bf16).
// Converts one group (32 bf16 values in 16 words) in place to shifted f16
// and returns 2^-s.
__device__ __forceinline__ float shift_group_to_f16(uint32_t (&w)[16]) {
  uint32_t m8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a = w[2 * i] & 0x7fff7fffu, b = w[2 * i + 1] & 0x7fff7fffu;
    m8[i] = max(max(a & 0xffffu, a >> 16), max(b & 0xffffu, b >> 16));
  }
  const uint32_t mx = max(max(max(m8[0], m8[1]), max(m8[2], m8[3])), max(max(m8[4], m8[5]), max(m8[6], m8[7])));
  int sh = 0;
  if (mx != 0 && mx < 0x7f80u) {
    const int ex = (int)(mx >> 7);
    const int lg = (ex != 0) ? ex - 127 : -133 + (31 - __clz((int)(mx & 0x7fu)));   // floor(log2 max)
    sh = 14 - lg;                                                                  // in [-113, 147]
  }
  const float m1 = pow2f(sh > 127 ? 127 : sh);
  const float m2 = pow2f(sh > 127 ? sh - 127 : 0);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float lo = __fmul_rn(__fmul_rn(__uint_as_float(w[i] << 16), m1), m2);
    const float hi = __fmul_rn(__fmul_rn(__uint_as_float(w[i] & 0xffff0000u), m1), m2);
    const __half2 h2 = __floats2half2_rn(lo, hi);
    w[i] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  return pow2f(-sh);
}

__device__ __forceinline__ void convert_group_mxfp4(uint32_t (&w)[16], uint8_t* dst_bytes, float* xinv_slot) {
  const float inv = shift_group_to_f16(w);
  uint4* dst = reinterpret_cast<uint4*>(dst_bytes);
#pragma unroll
  for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  *xinv_slot = inv;
}

// Each staging function issues the loads of its first round (every thread's
// first units), then calls mid() -- uniformly, from every thread -- and only
// then converts and stores: loads issued before the caller's tile copies sit
// ahead of them in the memory queue.
// Units are numbered over the CTA's list of vectors: unit u is group (or
// block, or piece) u % per_vec of vector vlist[u / per_vec], staged at that
// vector's index, or at list position u / per_vec in a compact region.
__device__ __forceinline__ void load_groups_mxfp4(const uint8_t* x, const int* vlist, int g0, int n,
                                                  const FastDiv& groups, uint32_t vec_bytes,
                                                  uint32_t (&w)[kStageU][16]) {
#pragma unroll
  for (int u = 0; u < kStageU; ++u) {
    const int gi = g0 + u * blockDim.x;
    if (gi < n) {
      const int vi = (int)fast_div((uint32_t)gi, groups), g = gi - vi * (int)groups.d;
      const int v = vlist ? vlist[vi] : vi;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)v * vec_bytes + (size_t)g * 64);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = src[q];
        w[u][4 * q] = v.x; w[u][4 * q + 1] = v.y; w[u][4 * q + 2] = v.z; w[u][4 * q + 3] = v.w;
      }
    }
  }
}

__device__ __forceinline__ void store_groups_mxfp4(uint8_t* xs, float* xinv, const int* vlist, bool compact,
                                                   int g0, int n, const FastDiv& groups, uint32_t vec_bytes,
                                                   uint32_t (&w)[kStageU][16]) {
#pragma unroll
  for (int u = 0; u < kStageU; ++u) {
    const int gi = g0 + u * blockDim.x;
    if (gi < n) {
      const int vi = (int)fast_div((uint32_t)gi, groups), g = gi - vi * (int)groups.d;
      const int v = compact ? vi : (vlist ? vlist[vi] : vi);
      convert_group_mxfp4(w[u], xs + (size_t)v * vec_bytes + (size_t)g * 64, xinv + v * (int)groups.d + g);
    }
  }
}

template <class Mid>
__device__ __forceinline__ void stage_x_mxfp4(const uint8_t* x, uint8_t* xs, float* xinv, const int* vlist,
                                              bool compact, int nvl, const FastDiv& groups, uint32_t vec_bytes,
                                              Mid&& mid) {
  const int n = nvl * (int)groups.d;
  const int step = kStageU * blockDim.x;
  uint32_t w[kStageU][16];
  load_groups_mxfp4(x, vlist, threadIdx.x, n, groups, vec_bytes, w);
  mid();
  store_groups_mxfp4(xs, xinv, vlist, compact, threadIdx.x, n, groups, vec_bytes, w);
  for (int g0 = threadIdx.x + step; g0 < n; g0 += step) {
    load_groups_mxfp4(x, vlist, g0, n, groups, vec_bytes, w);
    store_groups_mxfp4(xs, xinv, vlist, compact, g0, n, groups, vec_bytes, w);
  }
}

// q8_1 quantization of fp32 vectors straight into the shared-memory
// activation layout (codebook formats with kFlagXF32): one thread per
// 32-element block, amax = max|x|, d = amax / 127,
// q = round_half_away(x * (1 / d)) clamped to +-127, d stored as fp16 (RNE);
// the same IEEE-rounded fp32 operations as the standalone quantizer, so the
// result equals quantizing first and passing q8_1.
__device__ __forceinline__ float q8_block(const float (&f)[32], uint32_t (&qw)[8]) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  const float d = __fdiv_rn(amax, 127.0f);
  const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float r = roundf(__fmul_rn(f[4 * i + j], id));
      r = fminf(fmaxf(r, -127.0f), 127.0f);
      word |= ((uint32_t)(uint8_t)(int8_t)(int)r) << (8 * j);
    }
    qw[i] = word;
  }
  return d;
}

__device__ __forceinline__ void quantize_block_q8(const float (&f)[32], uint8_t* out, int K, int blk) {
  uint32_t qw[8];
  const float d = q8_block(f, qw);
  uint4* dst = reinterpret_cast<uint4*>(out + (size_t)blk * 32);
  dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
  reinterpret_cast<__half*>(out + K)[blk] = __float2half_rn(d);
}

__device__ __forceinline__ void load_block_f32(const float* x, const int* vlist, int bi, int n,
                                               const FastDiv& blocks, int K, float (&f)[32]) {
  if (bi < n) {
    const int vi = (int)fast_div((uint32_t)bi, blocks), b = bi - vi * (int)blocks.d;
    const int v = vlist ? vlist[vi] : vi;
    const float4* src = reinterpret_cast<const float4*>(x + (size_t)v * K + (size_t)b * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = src[i];
      f[4 * i] = v.x; f[4 * i + 1] = v.y; f[4 * i + 2] = v.z; f[4 * i + 3] = v.w;
    }
  }
}

template <class Mid>
__device__ __forceinline__ void stage_q8_from_f32(const float* x, uint8_t* xs, const int* vlist, bool compact,
                                                  int nvl, int K, const FastDiv& blocks, uint32_t vec_bytes,
                                                  Mid&& mid) {
  const int n = nvl * (int)blocks.d;
  float f[32];
  int bi = threadIdx.x;
  load_block_f32(x, vlist, bi, n, blocks, K, f);
  mid();
  for (;;) {
    if (bi < n) {
      const int vi = (int)fast_div((uint32_t)bi, blocks), b = bi - vi * (int)blocks.d;
      const int v = compact ? vi : (vlist ? vlist[vi] : vi);
      quantize_block_q8(f, xs + (size_t)v * vec_bytes, K, b);
    }
    bi += blockDim.x;
    if (bi >= n) break;
    load_block_f32(x, vlist, bi, n, blocks, K, f);
  }
}

// Codebook activations (q8_1 vectors), and fp16 activations of the MX
// formats, are copied to shared memory as they are, four 16-byte loads per
// thread in flight.
template <class Mid>
__device__ __forceinline__ void stage_x_copy(const uint8_t* x, uint8_t* xs, const int* vlist, bool compact,
                                             int nvl, const FastDiv& pieces, Mid&& mid) {
  const uint4* src = reinterpret_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(xs);
  const int per = (int)pieces.d;
  const int n = nvl * per;
  const int step = 4 * blockDim.x;
  uint4 v[4];
  size_t at[4];
  bool first = true;
  for (int i0 = threadIdx.x;; i0 += step) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      at[u] = 0;
      if (i < n) {
        if (vlist) {
          const int vi = (int)fast_div((uint32_t)i, pieces);
          at[u] = (size_t)vlist[vi] * per + (i - vi * per);
        } else {
          at[u] = (size_t)i;
        }
        v[u] = src[at[u]];
      }
    }
    if (first) {
      mid();
      first = false;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i < n) dst[compact ? (size_t)i : at[u]] = v[u];
    }
    if (i0 + step >= n) break;
  }
}

template <int NVV, int NVP>
__device__ __forceinline__ void chunk_mxfp4(const KParams& p, const Entry& e, int c, int L,
                                            const uint8_t* st, const uint8_t* xs, const float* xinv,
                                            float* acc) {
  const int lane = threadIdx.x & 31;
  // The lane's 32 activations as separate f16 values, unpacked once per chunk
  // and reused for all kRows rows.
  uint16_t xv16[NVV][32];
  float inv[NVV];
#pragma unroll
  for (int v = 0; v < NVV; ++v) {
    const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)e.vec[v] * p.x_vec_bytes +
                                                     (size_t)(c * kChunkK + lane * kLaneK) * 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = xp[q];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv16[v][8 * q + 2 * i] = (uint16_t)(w4[i] & 0xffffu);
        xv16[v][8 * q + 2 * i + 1] = (uint16_t)(w4[i] >> 16);
      }
    }
    inv[v] = xinv[e.vec[v] * (p.K / 32) + c * 32 + lane];
  }
  const uint2 sc = *reinterpret_cast<const uint2*>(st + tile_code_bytes(MXFP4, L) + lane * kRows);
  const uint32_t scw[2] = {sc.x, sc.y};
  uint4 cw[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) cw[r] = *reinterpret_cast<const uint4*>(st + (size_t)(r * L + lane) * 16);
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const uint32_t w4[4] = {cw[r].x, cw[r].y, cw[r].z, cw[r].w};
    float d0[NVV], d1[NVV];   // even / odd columns: two independent chains
#pragma unroll
    for (int v = 0; v < NVV; ++v) d0[v] = d1[v] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t h[4];
      e2m1x8_to_f16x2(w4[q], h);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int k = 8 * q + 2 * b;
        const uint16_t wl = (uint16_t)(h[b] & 0xffffu), wh = (uint16_t)(h[b] >> 16);
#pragma unroll
        for (int v = 0; v < NVV; ++v) {
          d0[v] = fma_f16_f32(wl, xv16[v][k], d0[v]);
          d1[v] = fma_f16_f32(wh, xv16[v][k + 1], d1[v]);
        }
      }
    }
    const float s = e8m0_to_f32((scw[r >> 2] >> (8 * (r & 3))) & 0xffu);
#pragma unroll
    for (int v = 0; v < NVV; ++v) acc[r * NVP + v] = fmaf(s, (d0[v] + d1[v]) * inv[v], acc[r * NVP + v]);
  }
}

// MXFP8: the lane's 32 E4M3 codes of a row are 32 bytes; each byte pair
// becomes an f16x2 (exact), then the same mixed-precision FMA chains and
// group scale as MXFP4.
template <int NVV, int NVP>
__device__ __forceinline__ void chunk_mxfp8(const KParams& p, const Entry& e, int c, int L,
                                            const uint8_t* st, const uint8_t* xs, const float* xinv,
                                            float* acc) {
  const int lane = threadIdx.x & 31;
  uint16_t xv16[NVV][32];
  float inv[NVV];
#pragma unroll
  for (int v = 0; v < NVV; ++v) {
    const uint4* xp = reinterpret_cast<const uint4*>(xs + (size_t)e.vec[v] * p.x_vec_bytes +
                                                     (size_t)(c * kChunkK + lane * kLaneK) * 2);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = xp[q];
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv16[v][8 * q + 2 * i] = (uint16_t)(w4[i] & 0xffffu);
        xv16[v][8 * q + 2 * i + 1] = (uint16_t)(w4[i] >> 16);
      }
    }
    inv[v] = xinv[e.vec[v] * (p.K / 32) + c * 32 + lane];
  }
  const uint2 sc = *reinterpret_cast<const uint2*>(st + tile_code_bytes(MXFP8, L) + lane * kRows);
  const uint32_t scw[2] = {sc.x, sc.y};
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const uint4* cp = reinterpret_cast<const uint4*>(st + (size_t)(r * L + lane) * 32);
    const uint4 a = cp[0], b = cp[1];
    const uint32_t w8[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float d0[NVV], d1[NVV];
#pragma unroll
    for (int v = 0; v < NVV; ++v) d0[v] = d1[v] = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      uint32_t h[2];
      e4m3x4_to_f16x2(w8[q], h);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int k = 4 * q + 2 * hb;
        const uint16_t wl = (uint16_t)(h[hb] & 0xffffu), wh = (uint16_t)(h[hb] >> 16);
#pragma unroll
        for (int v = 0; v < NVV; ++v) {
          d0[v] = fma_f16_f32(wl, xv16[v][k], d0[v]);
          d1[v] = fma_f16_f32(wh, xv16[v][k + 1], d1[v]);
        }
      }
    }
    const float s = e8m0_to_f32((scw[r >> 2] >> (8 * (r & 3))) & 0xffu);
#pragma unroll
    for (int v = 0; v < NVV; ++v) acc[r * NVP + v] = fmaf(s, (d0[v] + d1[v]) * inv[v], acc[r * NVP + v]);
  }
}

template <int FMT, int NVV, int NVP, bool DBG>
__device__ __forceinline__ void chunk_cb(const KParams& p, const Entry& e, int rt, int c, int L,
                                         const uint8_t* st, const uint8_t* xs, float* acc) {
  const int lane = threadIdx.x & 31;
  constexpr int SPL = lane_scale_bytes(FMT);  // 2 (half-blocks) or 1
  uint32_t qx[NVV][8];
  float dv[NVV];
#pragma unroll
  for (int v = 0; v < NVV; ++v) {
    const uint8_t* xv = xs + (size_t)e.vec[v] * p.x_vec_bytes;
    const uint4* qp = reinterpret_cast<const uint4*>(xv + c * kChunkK + lane * kLaneK);
    const uint4 a = qp[0], b = qp[1];
    qx[v][0] = a.x; qx[v][1] = a.y; qx[v][2] = a.z; qx[v][3] = a.w;
    qx[v][4] = b.x; qx[v][5] = b.y; qx[v][6] = b.z; qx[v][7] = b.w;
    dv[v] = __half2float(reinterpret_cast<const __half*>(xv + p.K)[c * 32 + lane]);
  }
  const uint8_t* scl = st + tile_code_bytes(FMT, L) + lane * kRows * SPL;
  static_assert(kRows * SPL == 8 || kRows * SPL == 16, "scale block of 8 or 16 bytes");
  uint32_t sw[kRows * SPL / 4];
  if constexpr (kRows * SPL == 16) {
    const uint4 u = *reinterpret_cast<const uint4*>(scl);
    sw[0] = u.x; sw[1] = u.y; sw[2] = u.z; sw[3] = u.w;
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(scl);
    sw[0] = u.x; sw[1] = u.y;
  }
  uint32_t t[4] = {p.lut[0], p.lut[1], p.lut[2], p.lut[3]};
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    uint32_t wv[8];
    if constexpr (FMT == CB2) {
      const uint2 u = *reinterpret_cast<const uint2*>(st + (size_t)(r * L + lane) * 8);
      decode_cb2(u.x, u.y, t[0], wv);
    } else if constexpr (FMT == CB3) {
      const uint2 u = *reinterpret_cast<const uint2*>(st + (size_t)(r * L + lane) * 8);
      const uint32_t hc = *reinterpret_cast<const uint32_t*>(st + (size_t)kRows * L * 8 +
                                                             (size_t)(r * L + lane) * 4);
      decode_cb3(u.x, u.y, hc, t[0], t[1], wv);
    } else {
      const uint4 u = *reinterpret_cast<const uint4*>(st + (size_t)(r * L + lane) * 16);
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
      decode_cb4(w4, t, wv);
    }
    const int row = r + rt * kRows;
    if constexpr (SPL == 2) {
      const uint32_t sb = sw[r >> 1] >> (16 * (r & 1));
      const float s0 = e8m0_to_f32(sb & 0xffu);
      const float s1 = e8m0_to_f32((sb >> 8) & 0xffu);
#pragma unroll
      for (int v = 0; v < NVV; ++v) {
        int i0 = 0, i1 = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          i0 = dp4a(wv[i], qx[v][i], i0);
          i1 = dp4a(wv[4 + i], qx[v][4 + i], i1);
        }
        acc[r * NVP + v] = fmaf(dv[v], fmaf(s0, (float)i0, s1 * (float)i1), acc[r * NVP + v]);
        if constexpr (DBG) {
          if (row < p.N) {
            int32_t* o = p.dbg + ((size_t)e.slot[v] * p.N + row) * (p.K / 16) + (c * kChunkK + lane * kLaneK) / 16;
            o[0] = i0;
            o[1] = i1;
          }
        }
      }
    } else {
      const float s = e8m0_to_f32((sw[r >> 2] >> (8 * (r & 3))) & 0xffu);
#pragma unroll
      for (int v = 0; v < NVV; ++v) {
        int i0 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) i0 = dp4a(wv[i], qx[v][i], i0);
        acc[r * NVP + v] = fmaf(dv[v], s * (float)i0, acc[r * NVP + v]);
        if constexpr (DBG) {
          if (row < p.N) {
            p.dbg[((size_t)e.slot[v] * p.N + row) * (p.K / 32) + (c * kChunkK + lane * kLaneK) / 32] = i0;
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Warp reduce-scatter: after rs_step<M, 16>, lane l holds value index
// l / (32 / M) when M <= 32, or 2 l + i (i = 0, 1) when M = 64, each summed
// over all 32 lanes.
// ---------------------------------------------------------------------------

template <int M, int O>
__device__ __forceinline__ void rs_step(float* v, int lane) {
  if constexpr (O >= 1) {
    if constexpr (M >= 2) {
      constexpr int H = M / 2;
      const bool up = (lane & O) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float send = up ? v[i] : v[i + H];
        const float keep = up ? v[i + H] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      rs_step<H, O / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      rs_step<1, O / 2>(v, lane);
    }
  }
}

// SwiGLU h = silu(z) * u, silu(z) = z / (1 + exp(-z)), in fp32 with no
// intermediate that overflows or falls into fp32's subnormal range (where
// exp(z) keeps only a few significant bits, and multiplying by z * u would
// magnify that loss): for z < 0 as z * t / (1 + t) * u with t = exp(z); for
// z <= -80, where 1 + t rounds to 1, as (z * exp(z + 80)) * (u * e^-80) --
// z + 80 is exact (z <= -80 has an ulp of at least 2^-17, which z + 80 keeps)
// and both factors stay normal, so only the final product rounds into the
// subnormals.
__device__ __forceinline__ float swiglu_f32(float z, float u) {
  if (z >= 0.0f) return z / (1.0f + expf(-z)) * u;
  if (z > -80.0f) {
    const float t = expf(z);
    return z * t / (1.0f + t) * u;
  }
  return (z * expf(z + 80.0f)) * (u * 1.8048513878454153e-35f);   // e^-80
}

template <int FMT, bool XH>
__device__ __forceinline__ void store_out(const KParams& p, size_t o, float val) {
  if constexpr (fmt_is_mx(FMT) && XH) {
    reinterpret_cast<__half*>(p.y)[o] = __float2half_rn(val);
  } else if constexpr (fmt_is_mx(FMT)) {
    reinterpret_cast<__nv_bfloat16*>(p.y)[o] = __float2bfloat16_rn(val);
  } else {
    reinterpret_cast<float*>(p.y)[o] = val;
  }
}

// After the reduce-scatter (rs_step), each group of 32 / M lanes holds the
// sum of (row, vector) index l / (32 / M), M = kRows * NVP.
template <int NVP>
__device__ __forceinline__ float reduce_lanes(float* acc) {
  constexpr int M = kRows * NVP;
  static_assert(M <= 32, "one value per lane group after the reduce-scatter");
  rs_step<M, 16>(acc, threadIdx.x & 31);
  return acc[0];
}

// Stores the reduced value of this lane's (row, vector). Plain: y[slot][rt *
// kRows + row]. Gate/up fusion (kFlagGlu): rows 0..3 of the tile are gate rows
// 4 rt .. 4 rt + 3 and rows 4..7 the matching up rows; the lane of gate row r
// takes up row r from lane l + 16 and stores silu(g) * u at h[slot][4 rt + r]
// (mlxcel-2178, "Problem / Background": gate, up and down per layer, SwiGLU
// between them). All lanes of the warp call it.
template <int FMT, int NVV, int NVP, bool XH>
__device__ __forceinline__ void store_lanes(const KParams& p, const Entry& e, int rt, float val) {
  const int lane = threadIdx.x & 31;
  constexpr int M = kRows * NVP;
  constexpr int S = 32 / M;
  const int idx = lane / S;
  const int r = idx / NVP, v = idx % NVP;
  if (p.flags & kFlagGlu) {
    const float up = __shfl_xor_sync(0xffffffffu, val, 16);   // row r + 4 (same vector) lives 16 lanes up
    const int row = rt * (kRows / 2) + r;
    if (lane % S == 0 && r < kRows / 2 && v < NVV && row < p.out_n) {
      store_out<FMT, XH>(p, (size_t)e.slot[v] * p.out_n + row, swiglu_f32(val, up));
    }
  } else {
    const int row = rt * kRows + r;
    if (lane % S == 0 && v < NVV && row < p.out_n) store_out<FMT, XH>(p, (size_t)e.slot[v] * p.out_n + row, val);
  }
}

// ---------------------------------------------------------------------------
// One task: chunks [c0, c1) of one row tile, applied to NVV vectors; then the
// warp reduction and either the store (one K range per item) or the split-K
// combine: the warp parks its reduced values in shared memory, and the warp
// that completes an item's last range adds the ranges in range order (the
// same order every run) and stores.
// ---------------------------------------------------------------------------

template <int FMT, int NVV, bool ALT, int ST>
__device__ __forceinline__ bool run_task(const KParams& p, const Entry& e, int rt, int k, int range, int c0,
                                         int c1, int& q, WarpPipe& wp, const uint8_t* xs, const float* xinv,
                                         float* part, int* cnt) {
  constexpr int NVP = (NVV == 3) ? 4 : NVV;
  constexpr bool DBG = ALT && !fmt_is_mx(FMT);
  constexpr bool XH = ALT && fmt_is_mx(FMT);
  const int lane = threadIdx.x & 31;
  float acc[kRows * NVP];
#pragma unroll
  for (int i = 0; i < kRows * NVP; ++i) acc[i] = 0.f;
  for (int c = c0; c < c1; ++c, ++q) {
    const int s = q % ST;
    const uint32_t parity = (uint32_t)(q / ST) & 1u;
    bool ok = mbar_wait_bounded(wp.bars + 8u * s, parity, kWaitLimitNs);
    if (!__all_sync(0xffffffffu, ok)) return false;
    if (q == 0) probe_phase(p, kPhTile0Ready);
    if (q == 1) probe_phase(p, kPhTile1Ready);
    if (q == 2) probe_phase(p, kPhTile2Ready);
    const int L = (c == p.chunks - 1) ? p.last_lanes : 32;
    const uint8_t* st = wp.ring_ptr + (size_t)s * p.full_tile;
    if (lane < L) {
      if constexpr (FMT == MXFP4) {
        chunk_mxfp4<NVV, NVP>(p, e, c, L, st, xs, xinv, acc);
      } else if constexpr (FMT == MXFP8) {
        chunk_mxfp8<NVV, NVP>(p, e, c, L, st, xs, xinv, acc);
      } else {
        chunk_cb<FMT, NVV, NVP, DBG>(p, e, rt, c, L, st, xs, acc);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (q == 0) probe_phase(p, kPhTile0Done);
    if (lane == 0) issue_next<ST>(wp);
  }
  probe_phase(p, kPhLastDone);
  float val = reduce_lanes<NVP>(acc);
  if (p.splits > 1) {
    constexpr int M = kRows * NVP;
    constexpr int S = 32 / M;
    volatile float* slot = part + (size_t)k * p.splits * kPartFloats;
    if (lane % S == 0) slot[range * kPartFloats + lane / S] = val;
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = (atomicAdd(&cnt[k], 1) == p.splits - 1) ? 1 : 0;
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) return true;
    __threadfence_block();
    val = 0.f;
    for (int r = 0; r < p.splits; ++r) val += slot[r * kPartFloats + lane / S];
  }
  store_lanes<FMT, NVV, NVP, XH>(p, e, rt, val);
  return true;
}

// All tasks of this warp. False if a tile wait gave up.
template <int FMT, int NV, bool ALT, int ST>
__device__ __forceinline__ bool run_tasks(const KParams& p, int& q, WarpPipe& wp, const uint8_t* xs,
                                          const float* xinv, float* part, int* cnt) {
  const int warp = threadIdx.x >> 5;
  for (int lt = warp; lt < wp.n_tasks; lt += wp.warps) {
    const int item = task_item(p, wp, lt);
    const int ei = (int)fast_div((uint32_t)item, p.fd_rt);
    const Entry& e = wp.ent[ei];
    const int rt = item - ei * p.row_tiles;
    const int k = (int)fast_div((uint32_t)lt, p.fd_split), range = lt - k * p.splits;
    int c0, c1;
    task_chunks(p, lt, c0, c1);
    bool ok = true;
    switch (e.nv) {
      case 1: ok = run_task<FMT, 1, ALT, ST>(p, e, rt, k, range, c0, c1, q, wp, xs, xinv, part, cnt); break;
      case 2:
        if constexpr (NV >= 2) ok = run_task<FMT, 2, ALT, ST>(p, e, rt, k, range, c0, c1, q, wp, xs, xinv, part, cnt);
        break;
      case 3:
        if constexpr (NV >= 3) ok = run_task<FMT, 3, ALT, ST>(p, e, rt, k, range, c0, c1, q, wp, xs, xinv, part, cnt);
        break;
      case 4:
        if constexpr (NV >= 4) ok = run_task<FMT, 4, ALT, ST>(p, e, rt, k, range, c0, c1, q, wp, xs, xinv, part, cnt);
        break;
      default: break;
    }
    if (!ok) return false;
  }
  return true;
}

// After a failed wait: let every copy this warp still has in flight (tiles q
// up to the number issued) land, bounded, before the CTA's shared memory can
// be released. Lane 0 holds the issue count.
template <int ST>
__device__ __forceinline__ void drain_ring(const WarpPipe& wp, int q) {
  const int lane = threadIdx.x & 31;
  const int issued = __shfl_sync(0xffffffffu, wp.iss_n, 0);
  for (int qq = q; qq < issued; ++qq) {
    const int s = qq % ST;
    if (!mbar_wait_bounded(wp.bars + 8u * s, (uint32_t)(qq / ST) & 1u, kDrainLimitNs)) {
      if (lane == 0) set_status(kStatusDrain);
    }
  }
}

template <int FMT, int NV, bool ALT>
__global__ void __launch_bounds__(Shape<NV>::warps * 32, kCtasPerSm)
    matvec_kernel(const __grid_constant__ KParams p) {
  constexpr int W = Shape<NV>::warps;
  constexpr int ST = Shape<NV>::stages;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const SmemLayout sl = smem_layout(FMT, (uint32_t)p.x_slots, p.x_vec_bytes, p.full_tile, p.K, W, ST, p.splits,
                                    p.items_per_cta);
  uint8_t* xs = smem + sl.x_off;
  float* xinv = reinterpret_cast<float*>(smem + sl.xinv_off);
  uint8_t* ring = smem + sl.ring_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sl.bar_off);
  Entry* ent = reinterpret_cast<Entry*>(smem + sl.ent_off);
  float* part = reinterpret_cast<float*>(smem + sl.part_off);
  int* cnt = reinterpret_cast<int*>(smem + sl.cnt_off);
  __shared__ int s_nent;

  __shared__ int s_ids[kMaxEntries];
  __shared__ int s_vlist[kMaxEntries];   // activation vectors this CTA's items use
  __shared__ int s_nvl;
  probe_phase(p, kPhStart);
  if (threadIdx.x == 0) {
    for (int i = 0; i < W * ST; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_mbar_init();
  }
  if (p.splits > 1) {
    for (int i = threadIdx.x; i < p.items_per_cta; i += blockDim.x) cnt[i] = 0;
  }
  // Programmatic dependent launch. Activations may be produced by the kernel
  // that precedes this one in the stream, so they are read only after
  // griddepcontrol.wait. Without kFlagPrefetch the ids are read after the wait
  // too. With it, the caller guarantees that the weights and ids were not
  // written by that preceding kernel; every kernel of this library signals its
  // dependents only after its own wait, so everything older is complete, and
  // the ids and the first weight tiles are fetched while the preceding kernel
  // drains.
  const bool early = (p.flags & kFlagPrefetch) != 0;
  if (!early) pdl_wait();
  if (warp == 0) {
    const int n = build_entries_warp<NV>(p, ent, s_ids);
    if (lane == 0) s_nent = n;
  }
  __syncthreads();
  probe_phase(p, kPhWorkList);

  WarpPipe wp;
  wp.p = &p;
  wp.ent = ent;
  wp.warps = W;
  int items_here = 0;
  cta_items(p, s_nent * p.row_tiles, wp.first, wp.stride, items_here);
  wp.n_tasks = items_here * p.splits;
  wp.ring_ptr = ring + (size_t)warp * ST * p.full_tile;
  wp.ring = smem_addr(wp.ring_ptr);
  wp.bars = smem_addr(&bars[warp * ST]);
  wp.policy = l2_evict_first_policy();
  wp.iss_n = 0;
  cursor_to(wp, warp);
  // Tile copies go out stage-major (every warp's first tile, then every
  // warp's second, ...) so that each warp's first tile arrives early. With
  // kFlagPrefetch the first kEarlyTiles per warp go out before the wait, the
  // rest right after the activation loads (which must not queue behind them).
  const int pre = early ? (p.contig ? ST : EarlyTiles<FMT, NV>::value) : 0;
  for (int q = 0; q < pre; ++q) {
    if (lane == 0) issue_next<ST>(wp);
    __syncthreads();
  }
  probe_phase(p, kPhEarlyTiles);
  // Per-slot gathers stage only the vectors of the entries the CTA's
  // contiguous item range touches (listed here, after the first tile copies
  // are out); other calls stage all vectors. A vector is staged at its own
  // index, unless the host planned a compact region (x_slots < nvec: all
  // vectors would not fit beside the tile ring); then the listed vectors sit
  // at consecutive positions and the CTA's entries are pointed at them. The
  // compact region holds the most vectors a CTA's range can touch; a longer
  // list is recorded in the status word and cut (a planning error).
  if (p.contig) {
    if (warp == 0) {
      uint32_t used = 0;
      if (items_here > 0) {
        const int e0 = (int)fast_div((uint32_t)wp.first, p.fd_rt);
        const int e1 = (int)fast_div((uint32_t)(wp.first + items_here - 1), p.fd_rt);
        for (int e = e0 + lane; e <= e1; e += 32) {
          for (int m = 0; m < ent[e].nv; ++m) used |= 1u << ent[e].vec[m];
        }
      }
      used = __reduce_or_sync(0xffffffffu, used);
      int n_used = __popc(used);
      if (n_used > p.x_slots) {
        if (lane == 0) set_status(kStatusPlan);
        n_used = p.x_slots;
      }
      const int pos = __popc(used & ((1u << lane) - 1u));
      if ((used & (1u << lane)) && pos < n_used) s_vlist[pos] = lane;
      if (lane == 0) s_nvl = n_used;
      if (p.x_slots < p.nvec && items_here > 0) {
        __syncwarp();
        const int e0 = (int)fast_div((uint32_t)wp.first, p.fd_rt);
        const int e1 = (int)fast_div((uint32_t)(wp.first + items_here - 1), p.fd_rt);
        for (int e = e0 + lane; e <= e1; e += 32) {
          for (int m = 0; m < 4; ++m) {
            const int at = __popc(used & ((1u << ent[e].vec[m]) - 1u));
            ent[e].vec[m] = at < n_used ? at : 0;
          }
        }
      }
    }
    __syncthreads();
  }
  const int* vlist = p.contig ? s_vlist : nullptr;
  const int nvl = p.contig ? s_nvl : p.nvec;
  const bool compact = p.x_slots < p.nvec;
  if (early) pdl_wait();
  probe_phase(p, kPhDepWait);
  // Dependents are released only after this kernel's own wait, so when one
  // starts, every kernel before this one is complete (what
  // QMV_FLAG_PREFETCH_INPUTS relies on).
  pdl_launch_dependents();

  // Gather slots with an invalid id produce zero rows.
  if (p.ids != nullptr) {
    const int nslots = p.ntok * p.top_k;
    for (int s = 0; s < nslots; ++s) {
      const int ex = s_ids[s];
      if (ex >= 0 && ex < p.n_experts) continue;
      for (int row = blockIdx.x * blockDim.x + threadIdx.x; row < p.out_n; row += gridDim.x * blockDim.x) {
        store_out<FMT, ALT>(p, (size_t)s * p.out_n + row, 0.f);
      }
    }
  }

  // Activations: plain 16-byte loads by every thread (they do not queue
  // behind the tile copies), converted on the way for MXFP4.
  // Contiguously dealt launches (their copies went out early) issue the rest
  // of the ring here; the others one stage per warp, and the remaining
  // stages once the activations are staged: fewer copies queued ahead of the
  // activation loads of the SM's other CTA (24-layer MXFP4 sweep: 17.75 ->
  // 17.46 us per layer; no copy before the activations: 18.4).
  const int first_round = p.contig ? ST : (pre > 1 ? pre : 1);
  auto issue_rest = [&]() {
    probe_phase(p, kPhActLoads);
    for (int q = pre; q < first_round; ++q) {
      if (lane == 0) issue_next<ST>(wp);
      __syncthreads();
    }
    probe_phase(p, kPhRingIssued);
  };
  if constexpr (fmt_is_mx(FMT) && ALT) {
    stage_x_copy(p.x, xs, vlist, compact, nvl, p.fd_per, issue_rest);
    for (int i = threadIdx.x; i < p.x_slots * (p.K / 32); i += blockDim.x) xinv[i] = 1.0f;
  } else if constexpr (fmt_is_mx(FMT)) {
    stage_x_mxfp4(p.x, xs, xinv, vlist, compact, nvl, p.fd_grp, p.x_vec_bytes, issue_rest);
  } else if (p.flags & kFlagXF32) {
    stage_q8_from_f32(reinterpret_cast<const float*>(p.x), xs, vlist, compact, nvl, p.K, p.fd_grp, p.x_vec_bytes,
                      issue_rest);
  } else {
    stage_x_copy(p.x, xs, vlist, compact, nvl, p.fd_per, issue_rest);
  }
  __syncthreads();
  for (int q = first_round; q < ST; ++q) {
    if (lane == 0) issue_next<ST>(wp);
  }
  probe_phase(p, kPhActStaged);

  int q = 0;
  if (!run_tasks<FMT, NV, ALT, ST>(p, q, wp, xs, xinv, part, cnt)) {
    if (lane == 0) set_status(kStatusWaitTile);
    drain_ring<ST>(wp, q);
  }
  probe_phase(p, kPhEnd);
}

// ---------------------------------------------------------------------------
// Host launcher
// ---------------------------------------------------------------------------

// The kernel of a launch: NV vectors per entry, ALT variant or not.
template <int FMT, int NV>
void* kernel_for(bool alt) {
  return alt ? reinterpret_cast<void*>(&matvec_kernel<FMT, NV, true>)
             : reinterpret_cast<void*>(&matvec_kernel<FMT, NV, false>);
}

// Host plan of a launch: kernel (vectors per entry), launch shape, split-K
// and shared memory. Items are upper-bounded by one entry per routed pair.
// Split-K: when a full grid has at least 3 warps per item (or 2, for items of
// 4 or more chunks), each item is cut into floor(warps / items) K ranges (at
// most one per chunk, at most kMaxSplits), so that more warps stream at once.
// Measured on GB300: dense CB4 2048x7168 7.7 -> 4.4 us, 7168x7168 11.9 ->
// 9.5 us; splitting the 3-chunk items of a 1440-item gather in two was slower.
// Shared memory per CTA beyond the dynamic region: the runtime's 1 KB
// reserve plus the kernel's static variables, rounded up.
constexpr size_t kSmemReserve = 1024 + 512;

struct LaunchPlan {
  int nv, warps, stages;
  long items;              // upper bound
  long grid;               // CTAs of a full grid (ctas_per_sm per SM), at most `items`
  int splits, split_chunks, items_per_cta;
  int x_slots;             // activation vectors staged per CTA
  int contig;              // contiguous dealing (per-slot gathers, dense calls of several entries)
  SmemLayout smem;
};

inline LaunchPlan plan_launch(const MatvecArgs& a, int sm_count, int ctas_per_sm, size_t smem_per_sm) {
  const Geometry g = make_geometry(a.fmt, a.N, a.K);
  LaunchPlan L;
  L.nv = launch_vectors(a.ids != nullptr, a.ntok);
  launch_shape(L.nv, L.warps, L.stages);
  const long entries = a.ids ? (long)a.ntok * a.top_k : (a.ntok + L.nv - 1) / L.nv;
  L.items = entries * g.row_tiles;
  L.contig = (a.ids != nullptr) ? (a.per_slot ? 1 : 0) : (entries > 1 ? 1 : 0);
  L.grid = (long)sm_count * ctas_per_sm;
  if (L.grid > L.items) L.grid = L.items;
  if (L.grid < 1) L.grid = 1;
  const long warps_total = (long)sm_count * ctas_per_sm * L.warps;
  long splits = warps_total / L.items;
  if (splits < 3 && !(splits == 2 && g.chunks >= 4)) splits = 1;
  if (splits > g.chunks) splits = g.chunks;
  if (splits > kMaxSplits) splits = kMaxSplits;
  if (splits < 1) splits = 1;
  L.split_chunks = (int)((g.chunks + splits - 1) / splits);
  L.splits = (g.chunks + L.split_chunks - 1) / L.split_chunks;
  L.items_per_cta = (int)((L.items + L.grid - 1) / L.grid);
  // Every vector gets its own slot of the activation region, unless that
  // leaves a contiguously dealt CTA more than its share of the SM's shared
  // memory: then the region holds only the most vectors a CTA's range can
  // touch -- a range of at most items_per_cta items covers at most
  // (items_per_cta - 1) / row_tiles + 2 entries of up to nv vectors.
  const uint32_t xvb = fmt_is_mx(a.fmt) ? (uint32_t)a.K * 2u : (uint32_t)q8_vec_bytes(a.K);
  L.x_slots = a.nvec;
  L.smem = smem_layout(a.fmt, (uint32_t)L.x_slots, xvb, g.full_tile, a.K, L.warps, L.stages, L.splits,
                       L.items_per_cta);
  const size_t share = smem_per_sm / (size_t)ctas_per_sm;
  if (L.contig && (size_t)L.smem.total + kSmemReserve > share) {
    const long touch = ((long)L.items_per_cta - 1) / g.row_tiles + 2;
    if (touch * L.nv < L.x_slots) {
      L.x_slots = (int)(touch * L.nv);
      L.smem = smem_layout(a.fmt, (uint32_t)L.x_slots, xvb, g.full_tile, a.K, L.warps, L.stages, L.splits,
                           L.items_per_cta);
    }
  }
  return L;
}

inline KParams make_params(const MatvecArgs& a) {
  const Geometry g = make_geometry(a.fmt, a.N, a.K);
  KParams p;
  p.w = static_cast<const uint8_t*>(a.w);
  p.expert_stride = a.expert_stride;
  p.x = static_cast<const uint8_t*>(a.x);
  p.x_vec_bytes = fmt_is_mx(a.fmt) ? (uint32_t)a.K * 2u : (uint32_t)q8_vec_bytes(a.K);
  p.nvec = a.nvec;
  p.x_slots = a.nvec;
  p.ids = a.ids;
  p.ntok = a.ntok;
  p.top_k = a.ids ? a.top_k : 1;
  p.per_slot = a.per_slot;
  p.contig = 0;
  p.n_experts = a.n_experts;
  p.N = a.N;
  p.K = a.K;
  p.row_tiles = g.row_tiles;
  p.chunks = g.chunks;
  p.last_lanes = g.last_lanes;
  p.full_tile = g.full_tile;
  p.last_tile = g.last_tile;
  p.rowtile = g.rowtile;
  p.y = a.y;
  p.dbg = a.dbg;
  for (int i = 0; i < 4; ++i) p.lut[i] = a.lut[i];
  p.flags = (a.prefetch ? kFlagPrefetch : 0u) | (a.glu ? kFlagGlu : 0u) | (a.x_f32 ? kFlagXF32 : 0u);
  p.out_n = a.out_n > 0 ? a.out_n : a.N;
  p.splits = 1;
  p.split_chunks = g.chunks;
  p.items_per_cta = 0;
  p.fd_rt = make_fastdiv((uint32_t)g.row_tiles);
  p.fd_split = make_fastdiv(1);
  p.fd_grid = make_fastdiv(1);
  p.fd_grp = make_fastdiv((uint32_t)(a.K / 32));
  p.fd_per = make_fastdiv(p.x_vec_bytes / 16u);
#ifdef QMV_PHASE_PROBE
  p.probe_slot = -1;
#endif
  return p;
}

template <int FMT>
cudaError_t launch_matvec(const MatvecArgs& a) {
  constexpr int NVMAX = MaxVectors<FMT>::value;
  static_assert(NVMAX == 4, "kernels exist for 1 to 4 vectors per entry");
  KParams p = make_params(a);
  LaunchPlan plan = plan_launch(a, device_sm_count(), kCtasPerSm, device_smem_per_sm());
  const int want_nv = plan.nv;
  const int warps = plan.warps;
  void* fn = nullptr;
  // ALT: block sums (codebooks) or fp16 activations (MX formats)
  const bool alt = fmt_is_mx(FMT) ? a.x_f16 : (a.dbg != nullptr);
  switch (want_nv) {
    case 1: fn = kernel_for<FMT, 1>(alt); break;
    case 2: fn = kernel_for<FMT, 2>(alt); break;
    case 3: fn = kernel_for<FMT, 3>(alt); break;
    default: fn = kernel_for<FMT, 4>(alt); break;
  }
  g_launch_stage = "kernel selection";
  if (fn == nullptr) return cudaErrorInvalidValue;

  // Opt in to the shared memory this launch needs, once per kernel and size.
  static std::mutex mu;
  static size_t configured[kMaxDevices][5][2] = {};
  int dev = 0;
  cudaError_t derr = cudaGetDevice(&dev);
  if (derr != cudaSuccess) return derr;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = configured[dev][want_nv][alt ? 1 : 0];
    if (have < plan.smem.total) {
      // The opt-in limit covers static plus dynamic shared memory.
      cudaFuncAttributes fa;
      g_launch_stage = "cudaFuncGetAttributes";
      cudaError_t err = cudaFuncGetAttributes(&fa, fn);
      if (err != cudaSuccess) return err;
      const size_t target = device_max_smem_optin() - fa.sharedSizeBytes;
      if (target < plan.smem.total) {
        g_launch_stage = "shared memory limit";
        return cudaErrorInvalidValue;
      }
      g_launch_stage = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
      err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)target);
      if (err != cudaSuccess) return err;
      have = target;
    }
  }
  int per_sm = 0;
  g_launch_stage = "cudaOccupancyMaxActiveBlocksPerMultiprocessor";
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, warps * 32, plan.smem.total);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  if (per_sm < kCtasPerSm) {
    // fewer CTAs fit: more items per CTA (the plan's smem only grows by the
    // split-K slots, which the opt-in above already covers up to its limit)
    plan = plan_launch(a, device_sm_count(), per_sm, device_smem_per_sm());
    g_launch_stage = "shared memory limit";
    if (plan.smem.total > device_max_smem_optin()) return cudaErrorInvalidValue;
  }
#ifdef QMV_PHASE_PROBE
  {
    static std::atomic<int> next_slot{0};
    if (g_phase_probe_on) p.probe_slot = next_slot.fetch_add(1) % kProbeSlots;
  }
#endif
  p.splits = plan.splits;
  p.fd_split = make_fastdiv((uint32_t)plan.splits);
  p.fd_grid = make_fastdiv((uint32_t)plan.grid);
  p.split_chunks = plan.split_chunks;
  p.items_per_cta = plan.items_per_cta;
  p.x_slots = plan.x_slots;
  p.contig = plan.contig;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.grid);
  cfg.blockDim = dim3(warps * 32);
  cfg.dynamicSmemBytes = plan.smem.total;
  cfg.stream = a.stream;
  // Programmatic dependent launch lets this grid start while the previous
  // kernel in the stream drains; the kernel waits (griddepcontrol.wait) before
  // it reads any input. Not used on the legacy NULL stream.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (a.stream != nullptr) ? 1 : 0;
  void* args[] = {const_cast<KParams*>(&p)};
  g_launch_stage = "cudaLaunchKernelExC";
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// ---------------------------------------------------------------------------
// Compute-rate probe (diagnostic export qmv_debug_chunk_rate): every warp
// applies the format's chunk routine, `iters` times, to a tile resident in
// shared memory -- the matvec's inner loop with no copies and no waits -- so
// that the weights per clock per SM of the arithmetic alone can be set beside
// the rate the HBM stream delivers. An opaque zero offset per iteration (a
// volatile load) keeps the loads and the decode inside the loop.
// ---------------------------------------------------------------------------

template <int FMT, int NV>
__global__ void __launch_bounds__(Shape<NV>::warps * 32, kCtasPerSm)
    chunk_rate_kernel(const __grid_constant__ KParams p, int iters, float* sink) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint32_t s_zero;
  constexpr int NVP = (NV == 3) ? 4 : NV;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_zero = 0;
  uint8_t* xs = smem;
  float* xinv = reinterpret_cast<float*>(smem + NV * p.x_vec_bytes);
  uint8_t* tiles = smem + round_up_u32(NV * p.x_vec_bytes + NV * 32 * 4, 128);
  const uint32_t code_bytes = tile_code_bytes(FMT, 32);
  for (uint32_t i = threadIdx.x; i < NV * p.x_vec_bytes; i += blockDim.x) {
    // activations: f16 near 1 (MX formats), q8_1 codes in [-63, 63] and d = 1/64 (codebooks)
    if constexpr (fmt_is_mx(FMT)) {
      xs[i] = (i & 1) ? 0x3c : (uint8_t)(i * 29);
    } else {
      const uint32_t k = i % p.x_vec_bytes;
      xs[i] = (k < (uint32_t)p.K) ? (uint8_t)((int8_t)((int)(k * 37 % 127) - 63)) : ((k & 1) ? 0x24 : 0x00);
    }
  }
  for (int i = threadIdx.x; i < NV * 32; i += blockDim.x) xinv[i] = 1.0f / 16384.0f;
  for (uint32_t i = threadIdx.x; i < Shape<NV>::warps * p.full_tile; i += blockDim.x) {
    const uint32_t k = i % p.full_tile;
    tiles[i] = (k >= code_bytes) ? 127 : (uint8_t)(i * 37 + 11);   // scale bytes 2^0
  }
  __syncthreads();
  Entry e;
  e.expert = 0;
  e.nv = NV;
  for (int v = 0; v < 4; ++v) e.vec[v] = e.slot[v] = (v < NV) ? v : 0;
  float acc[kRows * NVP];
#pragma unroll
  for (int i = 0; i < kRows * NVP; ++i) acc[i] = 0.f;
  for (int it = 0; it < iters; ++it) {
    // an offset the compilers cannot see through (a volatile shared-memory
    // load of a word that holds 0): every iteration reloads and decodes the
    // tile instead of the loop-invariant work being hoisted
    uint32_t z;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(z) : "r"(smem_addr(&s_zero)));
    const uint8_t* st = tiles + (size_t)warp * p.full_tile + z;
    const uint8_t* xz = xs + z;
    const float* iz = xinv + z;
    if constexpr (FMT == MXFP4) {
      chunk_mxfp4<NV, NVP>(p, e, 0, 32, st, xz, iz, acc);
    } else if constexpr (FMT == MXFP8) {
      chunk_mxfp8<NV, NVP>(p, e, 0, 32, st, xz, iz, acc);
    } else {
      chunk_cb<FMT, NV, NVP, false>(p, e, 0, 0, 32, st, xz, acc);
    }
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < kRows * NVP; ++i) sum += acc[i];
  sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = sum;
}

// Launches sms x ctas_per_sm CTAs of the production launch shape for NV
// vectors; *weights = matrix weights the launch processes (each applied to
// NV vectors), *threads = threads launched (sink entries).
template <int FMT, int NV>
cudaError_t launch_chunk_rate_nv(int ctas_per_sm, int iters, float* sink, int64_t* weights, int64_t* threads,
                                 cudaStream_t s) {
  KParams p{};
  const Geometry g = make_geometry(FMT, kRows, kChunkK);
  p.K = kChunkK;
  p.x_vec_bytes = fmt_is_mx(FMT) ? (uint32_t)kChunkK * 2u : (uint32_t)q8_vec_bytes(kChunkK);
  p.full_tile = g.full_tile;
  p.chunks = 1;
  p.last_lanes = 32;
  for (int i = 0; i < 4; ++i) p.lut[i] = 0xfd02fe01u * (uint32_t)(i + 1);   // int8 codebook values
  constexpr int W = Shape<NV>::warps;
  const size_t smem = round_up_u32(NV * p.x_vec_bytes + NV * 32 * 4, 128) + (size_t)W * p.full_tile;
  cudaError_t err = cudaFuncSetAttribute(chunk_rate_kernel<FMT, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = device_sm_count() * ctas_per_sm;
  *weights = (int64_t)grid * W * iters * kRows * kChunkK;
  *threads = (int64_t)grid * W * 32;
  if (sink == nullptr) return cudaSuccess;
  chunk_rate_kernel<FMT, NV><<<grid, W * 32, smem, s>>>(p, iters, sink);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_chunk_rate(int nv, int ctas_per_sm, int iters, float* sink, int64_t* weights, int64_t* threads,
                              cudaStream_t s) {
  switch (nv) {
    case 1: return launch_chunk_rate_nv<FMT, 1>(ctas_per_sm, iters, sink, weights, threads, s);
    case 2: return launch_chunk_rate_nv<FMT, 2>(ctas_per_sm, iters, sink, weights, threads, s);
    case 3: return launch_chunk_rate_nv<FMT, 3>(ctas_per_sm, iters, sink, weights, threads, s);
    default: return launch_chunk_rate_nv<FMT, 4>(ctas_per_sm, iters, sink, weights, threads, s);
  }
}

}  // namespace qmv

// Defines `int NAME(unsigned long long* out, size_t n, int clear)`: copies this
// translation unit's phase-probe buffer (kProbeSlots x kProbeCtas x
// kProbeWarps x kPhases stamps) to the host and optionally clears it; -1 in
// a build without the probe.
#ifdef QMV_PHASE_PROBE
#define QMV_DEFINE_PHASE_ACCESSOR(NAME)                                                        \
  int NAME(unsigned long long* out, size_t n, int clear) {                                     \
    const size_t bytes = sizeof(qmv::g_phase);                                                 \
    if (n * sizeof(unsigned long long) < bytes) return -1;                                     \
    if (cudaMemcpyFromSymbol(out, qmv::g_phase, bytes) != cudaSuccess) return -1;               \
    if (clear) {                                                                               \
      void* a = nullptr;                                                                       \
      if (cudaGetSymbolAddress(&a, qmv::g_phase) != cudaSuccess) return -1;                    \
      if (cudaMemset(a, 0, bytes) != cudaSuccess) return -1;                                   \
    }                                                                                          \
    return 0;                                                                                  \
  }
#else
#define QMV_DEFINE_PHASE_ACCESSOR(NAME) \
  int NAME(unsigned long long*, size_t, int) { return -1; }
#endif
