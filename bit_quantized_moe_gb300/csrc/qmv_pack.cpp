// qmv_pack.cpp -- host packer: canonical codes + E8M0 scales <-> GPU weight layout.
//
// Canonical storage order (per row): MXFP8 element k in byte k; MXFP4/CB4
// element k in byte k/2, low nibble first; CB2 code j of a byte at bits [2j, 2j+2); CB3 eight codes per
// three bytes, code j at bits [3j, 3j+3) of the little-endian 24-bit word.
// The GPU layout is described in qmv_layout.h.
#include <cstring>
#include <vector>

#include "qmv_layout.h"

namespace qmv {

static inline uint8_t canon_get(int fmt, const uint8_t* row, int k) {
  switch (fmt) {
    case MXFP8:
      return row[k];
    case CB2:
      return (row[k >> 2] >> (2 * (k & 3))) & 3;
    case CB3: {
      const uint8_t* g = row + 3 * (k >> 3);
      const uint32_t word = (uint32_t)g[0] | ((uint32_t)g[1] << 8) | ((uint32_t)g[2] << 16);
      return (word >> (3 * (k & 7))) & 7;
    }
    default:
      return (row[k >> 1] >> (4 * (k & 1))) & 15;
  }
}

static inline void canon_set(int fmt, uint8_t* row, int k, uint8_t c) {
  switch (fmt) {
    case MXFP8:
      row[k] = c;
      return;
    case CB2:
      row[k >> 2] = (uint8_t)(row[k >> 2] | ((c & 3) << (2 * (k & 3))));
      return;
    case CB3: {
      uint8_t* g = row + 3 * (k >> 3);
      uint32_t word = (uint32_t)g[0] | ((uint32_t)g[1] << 8) | ((uint32_t)g[2] << 16);
      word |= (uint32_t)(c & 7) << (3 * (k & 7));
      g[0] = (uint8_t)word;
      g[1] = (uint8_t)(word >> 8);
      g[2] = (uint8_t)(word >> 16);
      return;
    }
    default:
      row[k >> 1] = (uint8_t)(row[k >> 1] | ((c & 15) << (4 * (k & 1))));
      return;
  }
}

// Location of lane l's code block (row r) inside a tile with L lanes.
static inline void lane_block_offsets(int fmt, int L, int r, int l, size_t* off_a, size_t* off_b) {
  const int lb = lane_code_bytes(fmt);
  if (fmt == CB3) {
    *off_a = (size_t)(r * L + l) * 8;
    *off_b = (size_t)kRows * L * 8 + (size_t)(r * L + l) * 4;
  } else {
    *off_a = (size_t)(r * L + l) * lb;
    *off_b = 0;
  }
}

void pack_expert(const Geometry& g, const uint8_t* codes, const uint8_t* scales, uint8_t* out) {
  const int fmt = g.fmt;
  const size_t row_code_bytes = (size_t)g.K * fmt_bits(fmt) / 8;
  const int groups = g.K / fmt_group(fmt);
  const int spl = lane_scale_bytes(fmt);
  std::memset(out, 0, g.expert);
  uint8_t c32[32];
  uint8_t lb[32];
  for (int rt = 0; rt < g.row_tiles; ++rt) {
    for (int c = 0; c < g.chunks; ++c) {
      const int L = (c == g.chunks - 1) ? g.last_lanes : 32;
      uint8_t* tile = out + tile_offset(g, rt, c);
      uint8_t* scl = tile + tile_code_bytes(fmt, L);
      for (int r = 0; r < kRows; ++r) {
        const int row = rt * kRows + r;
        if (row >= g.N) break;
        const uint8_t* crow = codes + (size_t)row * row_code_bytes;
        const uint8_t* srow = scales + (size_t)row * groups;
        for (int l = 0; l < L; ++l) {
          const int k0 = c * kChunkK + l * kLaneK;
          for (int i = 0; i < 32; ++i) c32[i] = canon_get(fmt, crow, k0 + i);
          encode_lane(fmt, c32, lb);
          size_t oa, ob;
          lane_block_offsets(fmt, L, r, l, &oa, &ob);
          if (fmt == CB3) {
            std::memcpy(tile + oa, lb, 8);
            std::memcpy(tile + ob, lb + 8, 4);
          } else {
            std::memcpy(tile + oa, lb, lane_code_bytes(fmt));
          }
          for (int i = 0; i < spl; ++i) {
            scl[(size_t)(l * kRows + r) * spl + i] = srow[k0 / fmt_group(fmt) + i];
          }
        }
      }
    }
  }
}

void unpack_expert(const Geometry& g, const uint8_t* in, uint8_t* codes, uint8_t* scales) {
  const int fmt = g.fmt;
  const size_t row_code_bytes = (size_t)g.K * fmt_bits(fmt) / 8;
  const int groups = g.K / fmt_group(fmt);
  const int spl = lane_scale_bytes(fmt);
  std::memset(codes, 0, row_code_bytes * g.N);
  uint8_t c32[32];
  uint8_t lb[32];
  for (int rt = 0; rt < g.row_tiles; ++rt) {
    for (int c = 0; c < g.chunks; ++c) {
      const int L = (c == g.chunks - 1) ? g.last_lanes : 32;
      const uint8_t* tile = in + tile_offset(g, rt, c);
      const uint8_t* scl = tile + tile_code_bytes(fmt, L);
      for (int r = 0; r < kRows; ++r) {
        const int row = rt * kRows + r;
        if (row >= g.N) break;
        uint8_t* crow = codes + (size_t)row * row_code_bytes;
        uint8_t* srow = scales + (size_t)row * groups;
        for (int l = 0; l < L; ++l) {
          const int k0 = c * kChunkK + l * kLaneK;
          size_t oa, ob;
          lane_block_offsets(fmt, L, r, l, &oa, &ob);
          if (fmt == CB3) {
            std::memcpy(lb, tile + oa, 8);
            std::memcpy(lb + 8, tile + ob, 4);
          } else {
            std::memcpy(lb, tile + oa, lane_code_bytes(fmt));
          }
          decode_lane(fmt, lb, c32);
          for (int i = 0; i < 32; ++i) canon_set(fmt, crow, k0 + i, c32[i]);
          for (int i = 0; i < spl; ++i) {
            srow[k0 / fmt_group(fmt) + i] = scl[(size_t)(l * kRows + r) * spl + i];
          }
        }
      }
    }
  }
}

// Gate and up projections of one expert (each N x K, canonical) packed as one
// matrix of 2 * round_up(N, 4) rows whose 8-row tile i holds gate rows
// 4i..4i+3 then up rows 4i..4i+3 (rows past N are zero). `g` is the geometry
// of that interleaved matrix.
void pack_gate_up_expert(const Geometry& g, int N, const uint8_t* gate_codes, const uint8_t* gate_scales,
                         const uint8_t* up_codes, const uint8_t* up_scales, uint8_t* out) {
  const size_t rcb = (size_t)g.K * fmt_bits(g.fmt) / 8;
  const size_t rsb = (size_t)(g.K / fmt_group(g.fmt));
  std::vector<uint8_t> codes((size_t)g.N * rcb, 0), scales((size_t)g.N * rsb, 0);
  for (int row = 0; row < g.N; ++row) {
    const int tile = row / kRows, r = row % kRows;
    const int src = tile * (kRows / 2) + (r % (kRows / 2));
    if (src >= N) continue;
    const bool up = r >= kRows / 2;
    std::memcpy(&codes[(size_t)row * rcb], (up ? up_codes : gate_codes) + (size_t)src * rcb, rcb);
    std::memcpy(&scales[(size_t)row * rsb], (up ? up_scales : gate_scales) + (size_t)src * rsb, rsb);
  }
  pack_expert(g, codes.data(), scales.data(), out);
}

}  // namespace qmv
