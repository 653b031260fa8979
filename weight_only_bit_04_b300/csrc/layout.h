// Device layout of the packed blob, shared by the host API and the kernels.
//
// The blob holds, each on a 256-byte boundary:
//   qweight  [NR][KB] tiles of 128 rows x 64 columns of codes: 3072 bytes
//            (3-bit), 4096 bytes (4-bit) or 8192 bytes (8-bit)
//   scales   [NR][G][8 r16][8 g][2] fp16: for 16-row tile r16 and lane group g
//            the pair (row r16*16+g, row r16*16+g+8); a row block's 128 rows
//            of one group are 256 contiguous bytes (one copy for the GEMM),
//            a 32-row group's are 64 (the decode stream's unit)
//   zeros    (asymmetric formats only) 3- and 4-bit: [NR][G][8 r16][8 g]
//            bytes, low nibble row r16*16+g, high nibble row r16*16+g+8; 8-bit:
//            [NR][G][8 r16][8 g][2] bytes, row r16*16+g then row r16*16+g+8
//   perm     [K] int32: packed column -> original column (act order only)
//   ascale   [K] fp16: per-input-channel activation divisor (unfolded AWQ
//            only), in packed column order
//
// 8-bit codes: the 2048 words of a tile are ordered [r16 (8)][p (2)][lane (32)]
// [jj (2)][h (2)]: lane L = 4*g + t loads its eight words as two 16-byte parts
// p (each part of a warp is 512 contiguous bytes); word (r16, p, L, jj, h)
// holds the codes of row r16*16 + g + 8h, columns 16*j + 4*t + {0, 1, 2, 3}
// with j = 2p + jj (byte kk = column 4t + kk).
//
// 3-bit codes: the 768 words of a tile are ordered [pair (4)][A: lane (32) x 4]
// [B: lane (32) x 2], pair p holding 16-row tiles r16 = 2p (h = 0) and 2p + 1
// (h = 1): a warp's two tiles are one 16-byte and one 8-byte load per lane.
// Lane L = 4*g + t owns three words of each tile: h = 0: A.x, A.y, A.z;
// h = 1: A.w, B.x, B.y. The two 16-bit halves of a word belong to the two
// columns of one m16n8k16 register; each half holds five 3-bit codes at bits
// 0, 3, 6, 9, 12 and one bit of a sixteenth code at bit 15. Fragment register
// a of 16-column step j (a = 0: row g, columns 4t, 4t+1; 1: row g+8, same
// columns; 2: row g, columns 4t+2, 4t+3; 3: row g+8, same) sits in
//   j < 3: word j at bit {0, 9, 3, 12}[a]
//   j = 3: a < 3: word a at bit 6; a = 3: bit 15 of words 0, 1, 2 (code bits
//          0, 1, 2)
// so (w >> shift) & 0x00070007 is the register's pair of codes.
//
// 4-bit codes:
// Inside a 4096-byte tile the 1024 32-bit words are ordered [r16 (8)][lane (32)][j (4)]:
// lane L = 4*g + t of the warp owning 16-row tile r16 loads its four words (j = 0..3,
// one per 16-column step) with one 16-byte load. Word (r16, L, j) holds the codes of
// rows r16*16 + {g, g+8} and columns 16*j + 4*t + {0, 1, 2, 3} of the tile:
//   nibble (kk & 1) * 4 + (kk >> 1) * 2 + h   <->   column 4t + kk, row g + 8h
// so that (w & 0x000f000f) and (w & 0x00f000f0) give the half2 pairs of the
// m16n8k16 A fragment (rows g / g+8, column pairs {4t, 4t+1}; after w >> 8 the
// pairs {4t+2, 4t+3}), and the same four registers are the 16x256b tensor-memory
// fragment of a 16-row x 16-column fp16 tile.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/w4a16.h"

namespace w4a16 {

constexpr int kRowsPerBlock = 128;
constexpr int kColsPerBlock = 64;
constexpr int kTileBytes = 4096;   // 4-bit codes; 8-bit tiles are twice as large
constexpr int kTileWords = 1024;
constexpr int kScaleBytesPerGroupBlock = 256;
constexpr int kZeroBytesPerGroupBlock = 64;  // 4-bit; 8-bit zero points take twice as much

__host__ __device__ constexpr int tile_bytes(int bits) { return kTileBytes * bits / 4; }
__host__ __device__ constexpr int zero_bytes(int bits) { return bits == 8 ? 2 * kZeroBytesPerGroupBlock : kZeroBytesPerGroupBlock; }

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

__host__ __device__ inline int nibble_index(int kk, int h) { return (kk & 1) * 4 + (kk >> 1) * 2 + h; }

// Index of the scale pair (and of the zero-point byte, or byte pair) of
// 16-row tile r16 of row block R, group gi, lane group g.
__host__ __device__ inline int64_t meta_index(int64_t R, int64_t gi, int r16, int g, int64_t G) {
  return ((R * G + gi) * 8 + r16) * 8 + g;
}
// Entries between the same (r16, g) of consecutive groups.
constexpr int kMetaGroupStride = 64;

// 3-bit codes: index, inside a tile, of word wi (0..2) of 16-row tile r16 for a lane.
__host__ __device__ inline int w3_word_index(int r16, int lane, int wi) {
  const int base = (r16 >> 1) * 192;
  if ((r16 & 1) == 0) return base + lane * 4 + wi;
  return wi == 0 ? base + lane * 4 + 3 : base + 128 + lane * 2 + (wi - 1);
}
// Word and bit of fragment register a of step j (in each 16-bit half of the
// word). Steps 0..2 use word j, registers 0..3 at bits 0, 3, 6 and 9: the
// row-(g+8) registers 1 and 3 then come out of a mask alone, at 8x scale, and
// registers 2 and 3 out of one shift by 6. Step 3 uses bits 12..15: registers
// 0..2 at bit 12 of words 0..2, register 3 spread over bit 15 of words 0..2
// (returns wi = -1 for it).
__host__ __device__ inline void w3_field(int j, int a, int* wi, int* shift) {
  if (j < 3) {
    *wi = j;
    *shift = 3 * a;
  } else if (a < 3) {
    *wi = a;
    *shift = 12;
  } else {
    *wi = -1;
    *shift = 15;
  }
}

struct Layout {
  int64_t N, K, NR, KB, G;
  int gsize;
  int bits;  // 3, 4 or 8
  bool sym, act, awq;
  size_t q_off, q_bytes, s_off, s_bytes, z_off, z_bytes, p_off, p_bytes, a_off, a_bytes, total;
};

inline Layout make_layout(const w4a16_format& f) {
  Layout L{};
  L.N = f.N;
  L.K = f.K;
  L.gsize = f.group_size;
  L.bits = f.bits;
  L.sym = f.symmetric != 0;
  L.act = f.has_g_idx != 0;
  L.awq = f.has_act_scale != 0;
  L.NR = (f.N + kRowsPerBlock - 1) / kRowsPerBlock;
  L.KB = (f.K + kColsPerBlock - 1) / kColsPerBlock;
  L.G = f.K / f.group_size;
  L.q_off = 0;
  L.q_bytes = size_t(L.NR) * size_t(L.KB) * tile_bytes(f.bits);
  L.s_off = align256(L.q_off + L.q_bytes);
  L.s_bytes = size_t(L.NR) * size_t(L.G) * kScaleBytesPerGroupBlock;
  L.z_off = align256(L.s_off + L.s_bytes);
  L.z_bytes = L.sym ? 0 : size_t(L.NR) * size_t(L.G) * zero_bytes(f.bits);
  L.p_off = align256(L.z_off + L.z_bytes);
  L.p_bytes = L.act ? size_t(L.K) * 4 : 0;
  L.a_off = align256(L.p_off + L.p_bytes);
  L.a_bytes = L.awq ? size_t(L.K) * 2 : 0;
  L.total = align256(L.a_off + L.a_bytes);
  return L;
}

// Pointers into one blob, as the kernels see it.
struct BlobView {
  const uint32_t* qweight;
  const uint16_t* scales;   // fp16 bits
  const uint8_t* zeros;     // nullptr when symmetric
  const int32_t* perm;      // nullptr without act order
  const uint16_t* ascale;   // fp16 bits, packed order; nullptr without an act scale
};

inline BlobView view_of(const Layout& L, const void* blob) {
  const char* b = static_cast<const char*>(blob);
  BlobView v;
  v.qweight = reinterpret_cast<const uint32_t*>(b + L.q_off);
  v.scales = reinterpret_cast<const uint16_t*>(b + L.s_off);
  v.zeros = L.sym ? nullptr : reinterpret_cast<const uint8_t*>(b + L.z_off);
  v.perm = L.act ? reinterpret_cast<const int32_t*>(b + L.p_off) : nullptr;
  v.ascale = L.awq ? reinterpret_cast<const uint16_t*>(b + L.a_off) : nullptr;
  return v;
}

}  // namespace w4a16
