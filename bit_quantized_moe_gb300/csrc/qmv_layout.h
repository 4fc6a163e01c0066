// qmv_layout.h -- the GPU weight layout shared by the host packer and the kernels.
//
// A matrix of N rows x K columns is cut into row tiles of kRows rows and K
// chunks of kChunkK columns. One (row tile, chunk) pair is a "tile": a
// contiguous, 16-byte aligned block that one bulk copy moves into shared
// memory. Inside a chunk, lane l of the consuming warp owns the 32 columns
// [32 l, 32 l + 32) -- exactly one E8M0 group for MXFP4/MXFP8/CB4 and one
// q8_1 block of activations -- for all kRows rows of the tile.
//
// Tile of a chunk with L active lanes (L = 32 except for a ragged last chunk):
//   codes  : kRows x L lane blocks, row-major ([row][lane][lane block]);
//            CB3 splits its 12-byte lane block into an 8-byte plane
//            [row][lane][8] followed by a 4-byte plane [row][lane][4]
//   scales : [lane][row][scales per lane] E8M0 bytes
// The code region is a multiple of 16 bytes; the tile is padded to a multiple
// of 16 bytes, so every tile starts 16-byte aligned. Row tiles past N and the
// padding are zero-filled. Experts follow one another at a stride rounded up
// to 256 bytes.
//
// The bit order of codes inside a lane block is chosen for the device decode
// (see the per-format notes below) and is not the canonical storage order.
#pragma once

#include <cstddef>
#include <cstdint>

namespace qmv {

constexpr int kRows = 8;           // rows per tile
constexpr int kLaneK = 32;         // columns per lane per chunk
constexpr int kChunkK = 32 * kLaneK;  // columns per chunk (one warp)
constexpr int kExpertAlign = 256;

enum Fmt : int { MXFP4 = 0, CB2 = 1, CB3 = 2, CB4 = 3, MXFP8 = 4 };
constexpr int kNumFmts = 5;

#if defined(__CUDACC__)
#define QMV_HD __host__ __device__
#else
#define QMV_HD
#endif

QMV_HD constexpr int fmt_bits(int f) { return f == CB2 ? 2 : (f == CB3 ? 3 : (f == MXFP8 ? 8 : 4)); }
// MX formats: floating-point elements times bf16 / fp16 activations
QMV_HD constexpr bool fmt_is_mx(int f) { return f == MXFP4 || f == MXFP8; }
QMV_HD constexpr int fmt_group(int f) { return (f == CB2 || f == CB3) ? 16 : 32; }
// bytes of codes per lane per row (32 codes)
QMV_HD constexpr int lane_code_bytes(int f) { return 32 * fmt_bits(f) / 8; }
// E8M0 bytes per lane per row
QMV_HD constexpr int lane_scale_bytes(int f) { return kLaneK / fmt_group(f); }

QMV_HD constexpr uint32_t tile_code_bytes(int f, int lanes) {
  return (uint32_t)kRows * lanes * lane_code_bytes(f);
}
QMV_HD constexpr uint32_t tile_scale_bytes(int f, int lanes) {
  return (uint32_t)lanes * kRows * lane_scale_bytes(f);
}
// Padded to 16 bytes: the bulk copy size must be a multiple of 16.
QMV_HD constexpr uint32_t tile_bytes(int f, int lanes) {
  return (tile_code_bytes(f, lanes) + tile_scale_bytes(f, lanes) + 15u) / 16u * 16u;
}

struct Geometry {
  int fmt, N, K;
  int row_tiles;        // ceil(N / kRows)
  int chunks;           // ceil(K / kChunkK)
  int last_lanes;       // active lanes of the last chunk
  uint32_t full_tile;   // bytes of a 32-lane tile
  uint32_t last_tile;   // bytes of the last chunk's tile
  uint64_t rowtile;     // bytes of one row tile (all chunks)
  uint64_t expert;      // expert stride, multiple of kExpertAlign
};

QMV_HD inline Geometry make_geometry(int f, int N, int K) {
  Geometry g{};
  g.fmt = f;
  g.N = N;
  g.K = K;
  g.row_tiles = (N + kRows - 1) / kRows;
  g.chunks = (K + kChunkK - 1) / kChunkK;
  int rem = K - (g.chunks - 1) * kChunkK;
  g.last_lanes = rem / kLaneK;
  g.full_tile = tile_bytes(f, 32);
  g.last_tile = tile_bytes(f, g.last_lanes);
  g.rowtile = (uint64_t)(g.chunks - 1) * g.full_tile + g.last_tile;
  uint64_t e = (uint64_t)g.row_tiles * g.rowtile;
  g.expert = (e + kExpertAlign - 1) / kExpertAlign * kExpertAlign;
  return g;
}

// Division by a divisor fixed for a launch, without a division instruction:
// q = (n * m) >> 40 with m = ceil(2^40 / d). Writing m = (2^40 + r) / d
// (0 <= r < d), n * m / 2^40 = n / d + n r / (d 2^40), so the floor is exact
// whenever n * d <= 2^40; every quotient taken with it has n < 2^23 and
// d < 2^17.
struct FastDiv {
  uint64_t m;
  uint32_t d;
};

QMV_HD inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f;
  f.d = d;
  f.m = ((1ull << 40) + d - 1) / d;
  return f;
}

QMV_HD inline uint32_t fast_div(uint32_t n, const FastDiv& f) { return (uint32_t)(((uint64_t)n * f.m) >> 40); }
QMV_HD inline uint32_t fast_mod(uint32_t n, const FastDiv& f) { return n - fast_div(n, f) * f.d; }

// Byte offset of tile (row tile rt, chunk c) inside one expert.
QMV_HD inline uint64_t tile_offset(const Geometry& g, int rt, int c) {
  return (uint64_t)rt * g.rowtile + (uint64_t)c * g.full_tile;
}

// ---------------------------------------------------------------------------
// Lane-block encodings. `c` are the 32 codes of one lane for one row, c[i]
// belonging to column 32 l + i of the chunk.
//
// MXFP4 / CB4 (16 bytes): byte b = c[2b] | c[2b+1] << 4; word w holds c[8w..8w+7]
//   in nibbles 0..7.
// MXFP8 (32 bytes): byte i = c[i].
// CB2 (8 bytes, words W0, W1): nibble n of W0 holds c[n] in bits 0-1 and
//   c[n+8] in bits 2-3 (n = 0..7); W1 the same for c[16+n], c[24+n]. So
//   (W >> 2s) & 0x33333333 has one code per nibble.
// CB3 (12 bytes: plane words A, B and C): A and B carry the low two bits of
//   each code exactly as CB2's W0 and W1; bit 4n + j of C is the high bit of
//   c[8 j + n] (j = 0..3, n = 0..7).
// ---------------------------------------------------------------------------

inline void encode_lane(int f, const uint8_t* c, uint8_t* out /* lane_code_bytes */) {
  if (f == MXFP8) {
    for (int i = 0; i < 32; ++i) out[i] = c[i];
    return;
  }
  if (f == MXFP4 || f == CB4) {
    for (int b = 0; b < 16; ++b) out[b] = (uint8_t)((c[2 * b] & 15) | ((c[2 * b + 1] & 15) << 4));
    return;
  }
  uint32_t w[3] = {0, 0, 0};
  for (int half = 0; half < 2; ++half)
    for (int n = 0; n < 8; ++n) {
      w[half] |= (uint32_t)(c[16 * half + n] & 3) << (4 * n);
      w[half] |= (uint32_t)(c[16 * half + n + 8] & 3) << (4 * n + 2);
    }
  if (f == CB3)
    for (int j = 0; j < 4; ++j)
      for (int n = 0; n < 8; ++n) w[2] |= (uint32_t)((c[8 * j + n] >> 2) & 1) << (4 * n + j);
  const int words = (f == CB3) ? 3 : 2;
  for (int i = 0; i < words; ++i)
    for (int b = 0; b < 4; ++b) out[4 * i + b] = (uint8_t)(w[i] >> (8 * b));
}

inline void decode_lane(int f, const uint8_t* in, uint8_t* c /* 32 codes */) {
  if (f == MXFP8) {
    for (int i = 0; i < 32; ++i) c[i] = in[i];
    return;
  }
  if (f == MXFP4 || f == CB4) {
    for (int b = 0; b < 16; ++b) {
      c[2 * b] = in[b] & 15;
      c[2 * b + 1] = in[b] >> 4;
    }
    return;
  }
  uint32_t w[3] = {0, 0, 0};
  const int words = (f == CB3) ? 3 : 2;
  for (int i = 0; i < words; ++i)
    for (int b = 0; b < 4; ++b) w[i] |= (uint32_t)in[4 * i + b] << (8 * b);
  for (int half = 0; half < 2; ++half)
    for (int n = 0; n < 8; ++n) {
      c[16 * half + n] = (w[half] >> (4 * n)) & 3;
      c[16 * half + n + 8] = (w[half] >> (4 * n + 2)) & 3;
    }
  if (f == CB3)
    for (int j = 0; j < 4; ++j)
      for (int n = 0; n < 8; ++n) c[8 * j + n] |= ((w[2] >> (4 * n + j)) & 1) << 2;
}

// q8_1 activation vector: K int8 codes, then K/32 fp16 scales, padded to 16 bytes.
QMV_HD inline uint64_t q8_vec_bytes(int K) {
  uint64_t b = (uint64_t)K + (uint64_t)(K / 32) * 2;
  return (b + 15) / 16 * 16;
}

}  // namespace qmv
