// Decode-sized W4A16 product y[M][N] = x[M][K] . W_hat^T, 1 <= M <= 16.
//
// At batch one every packed weight is read once and used for about two flops
// ("AWQ + GPTQ Quantization, in depth", section "What W4A16 buys and why
// decoding gets faster"), so the kernel is an HBM stream whose instruction
// count per weight must stay small:
//
//  * Each warp owns two 16-row tiles (32 rows) and a contiguous run of
//    64-column blocks. Per block it issues one coalesced 16-byte load per lane
//    and tile (1 KiB contiguous per warp). The loads of four blocks, with the
//    scales and zero points of their groups, stay in flight in a register
//    ring; the loop structure follows the group size at compile time. The
//    asynchronous-copy variant (WB) lands the same loads with cp.async in a
//    shared-memory ring instead, so more bytes stay in flight per SM.
//  * A 32-bit word holds the codes of one lane's m16n8k16 A fragment. Masking
//    its nibbles with AND gives fp16 bit patterns 0x000q (= q * 2^-24) and
//    0x00q0 (= q * 2^-20): exact subnormal values, so four ANDs and one shift
//    expand eight weights. The tensor cores multiply them with the activations
//    (B fragment, tokens in the n dimension, read through L1) into fp32
//    accumulators.
//  * Per (row, group) the accumulator holds sum_k x_k q_k scaled by 2^-24
//    (rows g) or 2^-20 (rows g+8); one more MMA per 16 columns with a constant
//    all-2^-24 operand gives the group's activation sum X. The dequantization
//    (q - z) * s is applied once per group: y += s * (sum x q - z * X).
//    Summation order differs from the dequantize-then-multiply definition;
//    the error stays within the stated tolerance (products are exact, sums
//    are fp32).
//  * Under act order, with an unfolded AWQ act scale, and when K is not a
//    multiple of 64, a thread block first gathers its columns of x into
//    shared memory in packed order (divided by the act scale), with the
//    padding columns zero.
//  * Warps sharing rows reduce through shared memory; thread blocks of a
//    cluster that split K reduce through distributed shared memory in rank
//    order (deterministic, no atomics).
//  * Programmatic dependent launch: the next kernel's blocks become resident
//    while this one finishes. By default a block waits for the previous kernel
//    before its first global read. With kGemvWeightsReady (the caller vouches
//    that no kernel still in flight writes the packed weights) it issues its
//    first weight loads before that wait; activations are always read after.
//
// This header holds the kernels, templated on the code width (4 or 8 bits);
// k_gemv_b4.cu and k_gemv_b8.cu instantiate them, k_gemv.cu plans and
// dispatches. 8-bit codes: a lane's fragment of a 16-column step is two words
// (row g, row g+8), one byte per column; PRMT with a zero operand turns each
// into the fp16 patterns 0x00qq = q * 2^-24 (exact) for both rows.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <type_traits>

#include "device_util.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace w4a16 {
namespace {  // internal linkage: each including translation unit has its own copy

constexpr int kWarps = 8;
constexpr int kMaxGroup = 4;  // layers per grouped launch
constexpr int kThreads = kWarps * 32;
constexpr int kTilesPerWarp = 2;
constexpr uint64_t kTWaitLimitNs = 1000ull * 1000ull * 1000ull;  // every pipeline wait gives up after 1 s
// bounded waits that gave up (see w4a16_pipeline_timeouts); one per translation unit
static __device__ unsigned int g_gemv_timeouts;

// Debug builds (-DW4A16_DEBUG_CHECKS): index checks on the decode stream's
// shared- and global-memory accesses. A failed check records its code (the
// first one wins) in this word and the access is skipped; nothing traps. In
// other builds every check is the constant true.
static __device__ unsigned int g_debug_error;
#ifdef W4A16_DEBUG_CHECKS
__device__ __forceinline__ bool debug_check(bool ok, unsigned int code) {
  if (!ok) atomicCAS(&g_debug_error, 0u, code);
  return ok;
}
#define W4A16_CHECK(cond, code) debug_check(bool(cond), (code))
#else
#define W4A16_CHECK(cond, code) true
#endif

struct GemvArgs {
  const uint32_t* qweight;
  const uint32_t* scales2;  // scale pairs (row g, row g+8)
  const uint8_t* zeros;     // nullptr when symmetric
  const int32_t* perm;      // packed -> original column, or nullptr
  const uint16_t* ascale;   // activation divisor per packed column (unfolded AWQ), or nullptr
  const uint16_t* x;
  uint16_t* y;
  int M, N, K, G, KB;
  int rows16;      // 16-row tiles per thread block (2, 4 or 8)
  int kb_per_cta;  // 64-column blocks per thread block (the last blocks of a cluster may get fewer)
  uint32_t flags;  // kGemvWeightsReady
  int depth;       // asynchronous-copy ring: units in flight per thread
  int wb_off;      // asynchronous-copy ring: byte offset of the ring in shared memory
  int slot_bytes;  // asynchronous-copy ring: bytes of one slot
  // Grouped launch: up to kMaxGroup layers with the same K, format and input
  // x, their 128-row blocks one after another along gridDim.x (group m owns
  // blocks [gstart[m], gstart[m+1])). ngroup == 1: the fields above.
  int ngroup;
  int gstart[kMaxGroup + 1];
  const uint32_t* gq[kMaxGroup];
  const uint32_t* gs[kMaxGroup];
  const uint8_t* gz[kMaxGroup];
  uint16_t* gy[kMaxGroup];
  int gN[kMaxGroup];
};

// Scale and zero for the rows (g, g+8) of one tile and one group, folded into
// the two per-element factors of the finalisation.
struct GroupFactors {
  float sa, sb;  // s_g * 2^24, s_{g+8} * 2^20 / 2^21 / 2^24 (4 / 3 / 8 bits): acc holds q-sums at the inverse scales
  float za, zb;  // -s_g * z_g * 2^24, -s_{g+8} * z_{g+8} * 2^24   (cx holds x-sums at 2^-24)
};

// Exact float of a 4-bit value without an int-to-float conversion.
__device__ __forceinline__ float nib_to_float(uint32_t v) { return __uint_as_float(0x4B000000u | v) - 8388608.f; }

// zraw: 3 and 4 bits: one byte, row g in the low nibble, row g+8 in the high
// one; 8 bits: two bytes, row g then row g+8. Rows g+8 sit at 2^-20 (4-bit
// high nibbles) or 2^-21 (3-bit codes at bits 3..5), everything else at 2^-24.
template <bool SYM, int BITS>
__device__ __forceinline__ GroupFactors make_factors(uint32_t s2, uint32_t zraw) {
  const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&s2));
  constexpr float kSymZero = float(1 << (BITS - 1));
  const float zg = SYM ? kSymZero : nib_to_float(BITS != 8 ? (zraw & 0xFu) : (zraw & 0xFFu));
  const float zh = SYM ? kSymZero : nib_to_float(BITS != 8 ? (zraw >> 4) & 0xFu : (zraw >> 8) & 0xFFu);
  GroupFactors f;
  f.sa = sf.x * 16777216.f;
  f.sb = sf.y * (BITS == 4 ? 1048576.f : BITS == 3 ? 2097152.f : 16777216.f);
  f.za = f.sa * -zg;
  f.zb = sf.y * -zh * 16777216.f;
  return f;
}

template <int NB>
__device__ __forceinline__ void finalize(const float acc[NB][4], const float cx[NB][4], const GroupFactors& f,
                                         float tot[NB][4]) {
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    tot[nb][0] = fmaf(f.sa, acc[nb][0], fmaf(f.za, cx[nb][0], tot[nb][0]));
    tot[nb][1] = fmaf(f.sa, acc[nb][1], fmaf(f.za, cx[nb][1], tot[nb][1]));
    tot[nb][2] = fmaf(f.sb, acc[nb][2], fmaf(f.zb, cx[nb][2], tot[nb][2]));
    tot[nb][3] = fmaf(f.sb, acc[nb][3], fmaf(f.zb, cx[nb][3], tot[nb][3]));
  }
}

// a[0..3] of one word as q * 2^-24 (rows g) and q * 2^-20 (rows g+8).
__device__ __forceinline__ void extract_word(uint32_t w, uint32_t a[4]) {
  a[0] = w & 0x000F000Fu;
  a[1] = w & 0x00F000F0u;
  const uint32_t w8 = w >> 8;
  a[2] = w8 & 0x000F000Fu;
  a[3] = w8 & 0x00F000F0u;
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// 16-byte parts a lane loads per tile and 64-column block: 4 bits one, 8 bits
// two; 3 bits one per warp tile pair and block (tile 0: a 16-byte part, tile
// 1: an 8-byte part), read together.
template <int BITS>
constexpr int kParts = BITS == 8 ? 2 : 1;

// The four A-fragment registers of 16-column step j of tile tt from the codes
// the lane loaded for its two tiles: values q * 2^-24, or for the rows g+8
// (registers 1 and 3) q * 2^-20 with 4-bit codes (high nibbles) and q * 2^-21
// with 3-bit codes (bits 3..5 of each half, see w3_field).
template <int BITS>
__device__ __forceinline__ void extract_step(const uint4 (&wb)[2][kParts<BITS>], int tt, int j, uint32_t a[4]) {
  if (BITS == 4) {
    extract_word(word_of(wb[tt][0], j), a);
  } else if (BITS == 8) {
    const uint4& v = wb[tt][(kParts<BITS> - 1) & (j >> 1)];
    const uint32_t wg = word_of(v, 2 * (j & 1)), wh = word_of(v, 2 * (j & 1) + 1);
    a[0] = prmt(wg, 0u, 0x4140u);  // row g,   columns 4t, 4t+1
    a[1] = prmt(wh, 0u, 0x4140u);  // row g+8
    a[2] = prmt(wg, 0u, 0x4342u);  // row g,   columns 4t+2, 4t+3
    a[3] = prmt(wh, 0u, 0x4342u);  // row g+8
  } else {
    // the tile's three words: tile 0 A.x, A.y, A.z; tile 1 A.w, B.x, B.y
    const uint4& A = wb[0][0];
    const uint4& Bp = wb[1][0];
    const uint32_t w0 = tt == 0 ? A.x : A.w, w1 = tt == 0 ? A.y : Bp.x, w2 = tt == 0 ? A.z : Bp.y;
    // rows g at q * 2^-24 (codes at bits 0..2), rows g+8 at q * 2^-21 (bits 3..5)
    constexpr uint32_t M = 0x00070007u, M8 = 0x00380038u;
    if (j < 3) {
      const uint32_t w = j == 0 ? w0 : j == 1 ? w1 : w2;
      const uint32_t w6 = w >> 6;
      a[0] = w & M;
      a[1] = w & M8;
      a[2] = w6 & M;
      a[3] = w6 & M8;
    } else {
      const uint32_t w0s = w0 >> 12;
      a[0] = w0s & M;
      a[1] = (w1 >> 9) & M8;
      a[2] = (w2 >> 12) & M;
      a[3] = (w0s & 0x00080008u) | ((w1 >> 11) & 0x00100010u) | ((w2 >> 10) & 0x00200020u);
    }
  }
}

// Where the activations are read from: the read-only path (x is constant for
// the kernel), shared memory (staged), or ordinary global loads (x may have
// been written earlier by other blocks of the same chained launch, so the
// read-only path is not allowed; these loads follow an acquire of the
// producer's counter by thread 0 and a block barrier, which makes the
// producer's writes visible to them).
constexpr int kXGlobal = 0, kXShared = 1, kXCoherent = 2;
template <int XM>
__device__ __forceinline__ uint2 ld_x(const uint16_t* p) {
  if (XM == kXShared) return *reinterpret_cast<const uint2*>(p);
  uint2 v;
  if (XM == kXCoherent)
    asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p) : "memory");
  else
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Unit of the weight stream: the blocks of one group (two 64-column blocks for
// 128-column groups), or one block holding one (64) or two (32) groups.
template <int GS>
struct Unit {
  static constexpr int kBlocks = GS == 128 ? 2 : 1;
  static constexpr int kGroups = GS == 32 ? 2 : 1;
  static constexpr int kInFlight = GS == 128 ? 2 : 4;  // units in flight per warp (4 blocks)
};

template <int GS, int BITS>
struct UnitRegs {
  uint4 w[Unit<GS>::kBlocks][kTilesPerWarp][kParts<BITS>];  // a lane's codes
  uint32_t s[Unit<GS>::kGroups][kTilesPerWarp];
  uint32_t z[Unit<GS>::kGroups][kTilesPerWarp];
};

// Words of one 64-column block of codes, and of one 16-row tile of it.
template <int BITS>
struct CodeWords {
  static constexpr int kBlock = kTileWords * BITS / 4;
  static constexpr int kRow16 = 128 * BITS / 4;
  static constexpr int kPart = 128;  // 8 bits: words between a lane's two 16-byte parts
  // words from a lane's first code word to part `part` of tile tt; 3 bits:
  // tile 1 is the 8-byte part after the pair's 512 bytes of 16-byte parts
  __device__ static __forceinline__ int off(int tt, int part, int lane) {
    return BITS == 3 ? (tt == 0 ? 0 : 128 - 2 * lane) : tt * kRow16 + part * kPart;
  }
  static constexpr bool narrow(int tt) { return BITS == 3 && tt == 1; }  // an 8-byte part
};

__device__ __forceinline__ int lane_id() { return int(threadIdx.x & 31); }

// Zero-point bytes per (row pair, group): a nibble pair, or two bytes.
template <int BITS>
constexpr int kZeroMul = BITS == 8 ? 2 : 1;

__device__ __forceinline__ uint4 ldg_stream_u2(const uint32_t* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return make_uint4(v.x, v.y, 0u, 0u);
}

__device__ __forceinline__ uint32_t ldg_nc_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Issue the loads of one unit: codes of both tiles, scale pairs and zero bytes.
template <int GS, bool SYM, int BITS>
__device__ __forceinline__ void load_unit(UnitRegs<GS, BITS>& r, const uint32_t* qp, const uint32_t* sp,
                                          const uint8_t* zp, int unit, int gmax) {
  using U = Unit<GS>;
  using CW = CodeWords<BITS>;
#pragma unroll
  for (int bb = 0; bb < U::kBlocks; ++bb)
#pragma unroll
    for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
      for (int part = 0; part < kParts<BITS>; ++part) {
        const uint32_t* src = qp + (unit * U::kBlocks + bb) * CW::kBlock + CW::off(tt, part, lane_id());
        r.w[bb][tt][part] = CW::narrow(tt) ? ldg_stream_u2(src) : ldg_stream_u4(src);
      }
#pragma unroll
  for (int gg = 0; gg < U::kGroups; ++gg) {
    // (32-column groups only: a ragged last block's second half has no group;
    // its codes and staged activations are zero, any scale will do)
    const int gi = GS == 32 ? min(unit * U::kGroups + gg, gmax) : unit * U::kGroups + gg;
#pragma unroll
    for (int tt = 0; tt < kTilesPerWarp; ++tt) {
      r.s[gg][tt] = ldg_nc_u32(sp + gi * kMetaGroupStride + tt * 8);
      r.z[gg][tt] = SYM ? 0u
                    : BITS != 8 ? ldg_nc_u8(zp + gi * kMetaGroupStride + tt * 8)
                                : ldg_nc_u16(zp + (gi * kMetaGroupStride + tt * 8) * 2);
    }
  }
}

// Multiply-accumulate one unit. xl0 / xl1 point at this lane's x fragment
// (token rows g and g+8, column 4t) for the unit's first column.
// SPLIT: even and odd 16-column steps accumulate into separate sets, twice
// the independent MMA chains (consecutive MMAs into one accumulator wait for
// each other). Measured on B300, it pays only in the 4-bit register ring
// (4096x11008: 8.63 -> 7.84 us). It is slower in the asynchronous-copy ring
// (28672x8192: 30.3 -> 32.3 us) and in the 8-bit register ring (4096x4096:
// 5.48 -> 7.88 us), and 3-bit codes lose 2.5 % of the decode step with it.
// XSUM: the group activation sums come from the caller (xsg[gg][nb][e] =
// sum of the group's activations for token nb * 8 + 2t + e, plain units)
// instead of the all-2^-24 MMA. ONE: a single token; only the accumulator
// elements of token 0 (0 and 2) are finalized.
template <int NB, int GS, bool SYM, int XM, int BITS, bool SPLIT, bool XSUM = false, bool ONE = false>
__device__ __forceinline__ void compute_unit(const UnitRegs<GS, BITS>& r, const uint16_t* xl0, const uint16_t* xl1,
                                             float tot[kTilesPerWarp][NB][4],
                                             const float (*xsg)[NB][2] = nullptr) {
  using U = Unit<GS>;
  const uint32_t ones[4] = {0x00010001u, 0x00010001u, 0x00010001u, 0x00010001u};  // 2^-24 each
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  constexpr int NS = SPLIT ? 2 : 1;
  float acc[NS][kTilesPerWarp][NB][4];
  float cx[NS][NB][4];
#pragma unroll
  for (int bb = 0; bb < U::kBlocks; ++bb) {
    uint2 bx[4][NB];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int off = bb * 64 + j * 16;
      bx[j][0] = ld_x<XM>(xl0 + off);
      if (NB > 1) bx[j][NB - 1] = ld_x<XM>(xl1 + off);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ph = SPLIT ? (j & 1) : 0;
      // first step of the group (of this parity, with SPLIT): start the set fresh
      const bool fresh = SPLIT ? ((GS == 32) ? true : (j < 2 && bb == 0))
                               : ((GS == 32) ? (j == 0 || j == 2) : (j == 0 && bb == 0));
      if (!XSUM) {
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
          mma_16816(cx[ph][nb], ones, bx[j][nb].x, bx[j][nb].y, fresh ? zero4 : cx[ph][nb]);
      }
#pragma unroll
      for (int tt = 0; tt < kTilesPerWarp; ++tt) {
        uint32_t af[4];
        extract_step<BITS>(r.w[bb], tt, j, af);
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
          mma_16816(acc[ph][tt][nb], af, bx[j][nb].x, bx[j][nb].y, fresh ? zero4 : acc[ph][tt][nb]);
      }
      const bool group_end = (GS == 32) ? (j == 1 || j == 3) : (j == 3 && bb == U::kBlocks - 1);
      if (XSUM && group_end) {
        // tot += s * (2^k acc - z xs) per row, 2^k undoing the accumulator's
        // scale (2^24; 2^20 for the high-nibble rows of 4-bit codes). The zero
        // point enters as f = 2^23 + z, exact from its bits with one OR, and
        // -z xs = fma(f, -xs, 2^23 xs) with one rounding.
        const int gg = (GS == 32) ? (j >> 1) : 0;
        constexpr float kA = 16777216.f;
        constexpr float kB = BITS == 4 ? 1048576.f : BITS == 3 ? 2097152.f : 16777216.f;
        constexpr float kSymZero = float(1 << (BITS - 1));
        float xs[NB][2], x23[NB][2];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            xs[nb][e] = xsg[gg][nb][e];
            x23[nb][e] = SYM ? -kSymZero * xs[nb][e] : xs[nb][e] * 8388608.f;
          }
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt) {
          float a2[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              a2[nb][i] = SPLIT ? acc[0][tt][nb][i] + acc[NS - 1][tt][nb][i] : acc[0][tt][nb][i];
          const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&r.s[gg][tt]));
          const uint32_t zr = r.z[gg][tt];
          const float fg = __uint_as_float(0x4B000000u | (BITS != 8 ? (zr & 0xFu) : (zr & 0xFFu)));
          const float fh = __uint_as_float(0x4B000000u | (BITS != 8 ? ((zr >> 4) & 0xFu) : ((zr >> 8) & 0xFFu)));
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              if (ONE && (nb > 0 || e > 0)) continue;  // a single token: elements 0 and 2 only
              const float zg = SYM ? x23[nb][e] : fmaf(fg, -xs[nb][e], x23[nb][e]);
              const float zh = SYM ? x23[nb][e] : fmaf(fh, -xs[nb][e], x23[nb][e]);
              tot[tt][nb][e] = fmaf(sf.x, fmaf(a2[nb][e], kA, zg), tot[tt][nb][e]);
              tot[tt][nb][e + 2] = fmaf(sf.y, fmaf(a2[nb][e + 2], kB, zh), tot[tt][nb][e + 2]);
            }
        }
      } else if (group_end) {
        const int gg = (GS == 32) ? (j >> 1) : 0;
        float c2[NB][4];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
          for (int i = 0; i < 4; ++i) c2[nb][i] = SPLIT ? cx[0][nb][i] + cx[NS - 1][nb][i] : cx[0][nb][i];
        }
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt) {
          float a2[NB][4];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              a2[nb][i] = SPLIT ? acc[0][tt][nb][i] + acc[NS - 1][tt][nb][i] : acc[0][tt][nb][i];
          const GroupFactors f = make_factors<SYM, BITS>(r.s[gg][tt], r.z[gg][tt]);
          finalize<NB>(a2, c2, f, tot[tt]);
        }
      }
    }
  }
}

// Copy columns [p0, p0 + span) of every token row of x into xs[tok][c] (row
// stride `stride` halves), in packed order (through perm when given), with
// zeros beyond K. Without perm the copy moves 16 bytes per thread and step.
__device__ __forceinline__ void stage_activations(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                                  const uint16_t* __restrict__ ascale, uint16_t* xs, int M, int K,
                                                  int p0, int span, int stride, int tid, int nthreads) {
  if (perm == nullptr) {
    const int chunks = span / 8;  // span is a multiple of 64
    for (int e = tid; e < M * chunks; e += nthreads) {
      const int tok = e / chunks, c = (e - tok * chunks) * 8;
      const int p = p0 + c;
      uint4 v;
      if (p + 8 <= K && ascale == nullptr) {
        v = *reinterpret_cast<const uint4*>(x + size_t(tok) * K + p);
      } else {
        uint16_t h[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          h[i] = p + i < K ? x[size_t(tok) * K + p + i] : uint16_t(0);
          if (ascale != nullptr && p + i < K) h[i] = div_act(h[i], ascale[p + i]);
        }
        v = make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16), h[4] | (uint32_t(h[5]) << 16),
                       h[6] | (uint32_t(h[7]) << 16));
      }
      *reinterpret_cast<uint4*>(xs + tok * stride + c) = v;
    }
  } else {
    for (int e = tid; e < M * span; e += nthreads) {
      const int tok = e / span, c = e - tok * span;
      const int p = p0 + c;
      uint16_t v = p < K ? x[size_t(tok) * K + perm[p]] : uint16_t(0);
      if (ascale != nullptr && p < K) v = div_act(v, ascale[p]);
      xs[tok * stride + c] = v;
    }
  }
}

// Asynchronous-copy ring (WB): instead of holding the next units in
// registers, every thread lands its own 16-byte code loads, scale pairs and
// zero-point words with cp.async (LDGSTS) in a ring of shared-memory slots and
// reads back only what it copied itself: the bytes in flight no longer cost
// registers, and no thread waits for another (cp.async.wait_group only).
// Slot layout, per field, one entry per thread of the block (conflict-free):
//   codes [kBlocks][2 tiles] 16 B, scales [kGroups][2 tiles] 4 B,
//   zero words [kGroups][2 tiles] 4 B (the word holding this row pair's byte).
template <int GS, int BITS>
struct WbSlot {
  static constexpr int kCodeFields = Unit<GS>::kBlocks * kTilesPerWarp * kParts<BITS>;
  static constexpr int kMetaFields = Unit<GS>::kGroups * kTilesPerWarp;
  static constexpr int kScaleOff = kCodeFields * kThreads * 16;
  static constexpr int kZeroOff = kScaleOff + kMetaFields * kThreads * 4;
  static constexpr int kBytes = kZeroOff + kMetaFields * kThreads * 4;
};
// Ring depth: 4 units of 4-bit codes, 2 of 8-bit codes -- the same bytes in
// flight, and a ring small enough for three thread blocks per SM.
template <int BITS>
constexpr int kWbSlots = BITS == 8 ? 2 : 4;

__host__ __device__ inline int wb_slot_bytes(int GS, int bits) {
  if (bits == 8) return GS == 128 ? WbSlot<128, 8>::kBytes : GS == 64 ? WbSlot<64, 8>::kBytes : WbSlot<32, 8>::kBytes;
  static_assert(WbSlot<128, 3>::kBytes == WbSlot<128, 4>::kBytes, "3-bit slots reuse the 4-bit size");
  return GS == 128 ? WbSlot<128, 4>::kBytes : GS == 64 ? WbSlot<64, 4>::kBytes : WbSlot<32, 4>::kBytes;
}

__device__ __forceinline__ void cp_async_8(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gmem_src) : "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// STAGED: gather x into shared memory first (act order, K not a multiple of
// 64, or on request).
template <int MP, int GS, bool SYM, bool STAGED, bool WB, int BITS>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NB = MP > 8 ? 2 : 1;
  using U = Unit<GS>;
  constexpr int PF = WB ? 1 : U::kInFlight;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int RT = a.rows16;
  const int WR = RT / kTilesPerWarp;  // warp row groups per block
  const int WK = kWarps / WR;         // warps splitting K per row group
  const int wr = warp % WR;
  const int wk = warp / WR;
  // this block's layer (grouped launch) and its block index within it
  int bx = int(blockIdx.x);
  const uint32_t* qweight = a.qweight;
  const uint32_t* scales2 = a.scales2;
  const uint8_t* zeros = a.zeros;
  uint16_t* yout = a.y;
  int Nl = a.N;
  if (a.ngroup > 1) {
    int m = 0;
    while (m + 1 < a.ngroup && bx >= a.gstart[m + 1]) ++m;
    bx -= a.gstart[m];
    qweight = a.gq[m];
    scales2 = a.gs[m];
    zeros = a.gz[m];
    yout = a.gy[m];
    Nl = a.gN[m];
  }
  const int Tc = bx * RT;  // first 16-row tile of the block
  const int R = Tc >> 3;
  const int r16 = (Tc & 7) + wr * kTilesPerWarp;

  // Block column range (whole units), then this warp's contiguous share of it.
  const int kb_lo = int(blockIdx.y) * a.kb_per_cta;
  const int kb_hi = min(kb_lo + a.kb_per_cta, a.KB);
  const int span_blk = max(kb_hi - kb_lo, 0);
  const int cta_units = (span_blk + U::kBlocks - 1) / U::kBlocks;
  const int u0 = kb_lo / U::kBlocks + (cta_units * wk) / WK;
  const int nunit = (cta_units * (wk + 1)) / WK - (cta_units * wk) / WK;

  const int G = a.G;
  const int gmax = G - 1 - u0 * U::kGroups;  // last group, relative to this warp's first
  using CW = CodeWords<BITS>;
  const uint32_t* qp = qweight + (size_t(R) * a.KB * 8 + r16) * CW::kRow16 + lane * 4 +
                       size_t(u0) * U::kBlocks * CW::kBlock;
  // the warp's row group (r16 is even) from the unit's first group on; entries per group: [tt][g]
  const uint32_t* sp = scales2 + meta_index(R, int64_t(u0) * U::kGroups, r16, g, G);
  const uint8_t* zp = SYM ? nullptr : zeros + meta_index(R, int64_t(u0) * U::kGroups, r16, g, G) * kZeroMul<BITS>;

  const bool early = (a.flags & kGemvWeightsReady) != 0;
  const int M = a.M;

  // ---- asynchronous-copy ring: this thread's entries of every slot
  using SL = WbSlot<GS, BITS>;
  constexpr int D = kWbSlots<BITS>;  // units in flight per thread
  const int tid = int(threadIdx.x);
  unsigned char* ringb = smem + a.wb_off;
  auto issue_unit = [&](int i) {  // unit u0 + i into slot i % D, one commit group
    if (i < nunit) {
      unsigned char* slot = ringb + size_t(i % D) * SL::kBytes;
#pragma unroll
      for (int bb = 0; bb < U::kBlocks; ++bb)
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
          for (int part = 0; part < kParts<BITS>; ++part) {
            unsigned char* dst = slot + (((bb * kTilesPerWarp + tt) * kParts<BITS> + part) * kThreads + tid) * 16;
            const uint32_t* src = qp + (i * U::kBlocks + bb) * CW::kBlock + CW::off(tt, part, lane);
            if (CW::narrow(tt))
              cp_async_8(dst, src);
            else
              cp_async_16(dst, src);
          }
#pragma unroll
      for (int gg = 0; gg < U::kGroups; ++gg) {
        const int gi = GS == 32 ? min(i * U::kGroups + gg, gmax) : i * U::kGroups + gg;
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt) {
          const int f = gg * kTilesPerWarp + tt;
          cp_async_4(slot + SL::kScaleOff + (f * kThreads + tid) * 4, sp + gi * kMetaGroupStride + tt * 8);
          if (!SYM)  // the aligned word holding this lane's zero point(s)
            cp_async_4(slot + SL::kZeroOff + (f * kThreads + tid) * 4,
                       reinterpret_cast<const uint32_t*>(
                           reinterpret_cast<uintptr_t>(zp + (gi * kMetaGroupStride + tt * 8) * kZeroMul<BITS>) & ~uintptr_t(3)));
        }
      }
    }
    cp_async_commit();
  };

  // The next kernel may be scheduled right away: its griddepcontrol.wait still
  // waits for this grid to complete, but its blocks can become resident and
  // start their own weight stream while this one runs.
  pdl_launch_dependents();
  const bool inputs_ready = (a.flags & kGemvInputsReady) != 0;  // nothing in flight writes x: no wait at all
  if (!early && !inputs_ready) pdl_wait();
  UnitRegs<GS, BITS> ring[PF];
  if (WB) {
#pragma unroll
    for (int i = 0; i < D; ++i) issue_unit(i);
  } else {
#pragma unroll
    for (int s = 0; s < PF; ++s)
      if (s < nunit) load_unit<GS, SYM, BITS>(ring[s], qp, sp, zp, s, gmax);
  }
  if (early && !inputs_ready) pdl_wait();

  // Activations: lanes of absent tokens read a real row (their outputs are
  // never stored), so no masking is needed.
  const int tok0 = min(g, M - 1);
  const int tok1 = min(g + 8, M - 1);
  const uint16_t* xl0;
  const uint16_t* xl1;
  if (STAGED) {
    // Gather this block's columns of x in packed order: xs[tok][c], row stride
    // span + 8 halves (keeps the lanes' reads on distinct banks).
    const int span = span_blk * kColsPerBlock;
    const int stride = span + 8;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
    stage_activations(a.x, a.perm, a.ascale, xs, M, a.K, kb_lo * kColsPerBlock, span, stride, int(threadIdx.x), kThreads);
    __syncthreads();
    const int c0 = (u0 * U::kBlocks - kb_lo) * kColsPerBlock + 4 * t;
    xl0 = xs + tok0 * stride + c0;
    xl1 = xs + tok1 * stride + c0;
  } else {
    const int c0 = u0 * U::kBlocks * kColsPerBlock + 4 * t;
    xl0 = a.x + size_t(tok0) * a.K + c0;
    xl1 = a.x + size_t(tok1) * a.K + c0;
  }

  float tot[kTilesPerWarp][NB][4];
#pragma unroll
  for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) tot[tt][nb][i] = 0.f;

  if (WB) {
    const int zshift = int((reinterpret_cast<uintptr_t>(zp) & 3u) * 8);  // this lane's byte in its zero word
    for (int i = 0; i < nunit; ++i) {
      cp_async_wait_group<D - 1>();  // unit i has landed (this thread's copies)
      const unsigned char* slot = ringb + size_t(i % D) * SL::kBytes;
      UnitRegs<GS, BITS> r;
#pragma unroll
      for (int bb = 0; bb < U::kBlocks; ++bb)
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
          for (int part = 0; part < kParts<BITS>; ++part)
            r.w[bb][tt][part] = *reinterpret_cast<const uint4*>(
                slot + (((bb * kTilesPerWarp + tt) * kParts<BITS> + part) * kThreads + tid) * 16);
#pragma unroll
      for (int gg = 0; gg < U::kGroups; ++gg)
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt) {
          const int f = gg * kTilesPerWarp + tt;
          r.s[gg][tt] = *reinterpret_cast<const uint32_t*>(slot + SL::kScaleOff + (f * kThreads + tid) * 4);
          r.z[gg][tt] = SYM ? 0u
                            : (*reinterpret_cast<const uint32_t*>(slot + SL::kZeroOff + (f * kThreads + tid) * 4) >>
                               zshift) & (BITS != 8 ? 0xFFu : 0xFFFFu);
        }
      const int xo = i * U::kBlocks * kColsPerBlock;
      compute_unit<NB, GS, SYM, STAGED ? kXShared : kXGlobal, BITS, !WB && BITS == 4>(r, xl0 + xo, xl1 + xo, tot);
      issue_unit(i + D);  // refills the slot just read (this thread's own entries)
    }
    cp_async_wait_all();
  } else {
    for (int i0 = 0; i0 < nunit; i0 += PF) {
#pragma unroll
      for (int s = 0; s < PF; ++s) {
        const int i = i0 + s;
        if (i < nunit) {
          const int xo = i * U::kBlocks * kColsPerBlock;
          compute_unit<NB, GS, SYM, STAGED ? kXShared : kXGlobal, BITS, !WB && BITS == 4>(ring[s], xl0 + xo, xl1 + xo, tot);
          if (i + PF < nunit) load_unit<GS, SYM, BITS>(ring[s], qp, sp, zp, i + PF, gmax);
        }
      }
    }
  }

  // Reduce: per-warp partials -> per-block partials (fixed order) -> cluster.
  // The buffers sit at offset 0 in every block of the cluster (peers read red_c).
  if (STAGED) __syncthreads();  // the staged activations are no longer needed
  float* red_w = reinterpret_cast<float*>(smem);  // [warp][32 rows][16 tokens]
  float* red_c = red_w + kWarps * 512;            // [tok][RT*16 rows]
#pragma unroll
  for (int tt = 0; tt < kTilesPerWarp; ++tt) {
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      const int tk = nb * 8 + 2 * t;
      float* rw = red_w + warp * 512 + tt * 256;
      rw[g * 16 + tk] = tot[tt][nb][0];
      rw[g * 16 + tk + 1] = tot[tt][nb][1];
      rw[(g + 8) * 16 + tk] = tot[tt][nb][2];
      rw[(g + 8) * 16 + tk + 1] = tot[tt][nb][3];
    }
  }
  __syncthreads();
  const int rows = RT * 16;
  const int nout = rows * M;
  for (int e = threadIdx.x; e < nout; e += kThreads) {
    const int tok = e / rows;
    const int row = e - tok * rows;           // (wr * 2 + tt) * 16 + r
    const int w_r = row >> 5, rr = row & 31;  // warp row group, row within its 32
    float acc = 0.f;
    for (int k = 0; k < WK; ++k) acc += red_w[(k * WR + w_r) * 512 + rr * 16 + tok];
    red_c[e] = acc;
  }
  const int KS = int(gridDim.y);
  if (KS > 1) {
    cluster_sync_all();
    const int rank = int(cluster_ctarank());
    const int per = (nout + KS - 1) / KS;
    const int e_lo = rank * per;
    const int e_hi = min(e_lo + per, nout);
    for (int e = e_lo + threadIdx.x; e < e_hi; e += kThreads) {
      float acc = 0.f;
      for (int rk = 0; rk < KS; ++rk) acc += ld_dsmem_f32(red_c + e, uint32_t(rk));
      const int tok = e / rows;
      const int n = bx * rows + (e - tok * rows);
      if (n < Nl) yout[size_t(tok) * Nl + n] = __half_as_ushort(__float2half_rn(acc));
    }
    cluster_sync_all();  // keep this block's shared memory alive until peers are done
  } else {
    __syncthreads();
    for (int e = threadIdx.x; e < nout; e += kThreads) {
      const int tok = e / rows;
      const int n = bx * rows + (e - tok * rows);
      if (n < Nl) yout[size_t(tok) * Nl + n] = __half_as_ushort(__float2half_rn(red_c[e]));
    }
  }
}

size_t gemv_smem_bytes(int M, int kb_per_cta, bool staged) {
  const size_t red = size_t(kWarps) * 512 * 4 + size_t(8) * 256 * 4;
  const size_t xs = staged ? size_t(M) * (size_t(kb_per_cta) * kColsPerBlock + 8) * 2 : 0;
  return xs > red ? xs : red;
}

template <int MP, int GS, bool SYM, bool STAGED, bool WB, int BITS>
cudaError_t launch_typed(const GemvArgs& a, int KS, size_t smem_bytes, cudaStream_t stream) {
  auto kern = gemv_kernel<MP, GS, SYM, STAGED, WB, BITS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes));
  if (e != cudaSuccess) return e;
  if (KS > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  const int ntiles = a.ngroup > 1 ? a.gstart[a.ngroup] * a.rows16 : ((a.N + kRowsPerBlock - 1) / kRowsPerBlock) * 8;
  cfg.gridDim = dim3(unsigned(ntiles / a.rows16), unsigned(KS), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int na = 0;
  attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (KS > 1) {
    attrs[na].id = cudaLaunchAttributeClusterDimension;
    attrs[na].val.clusterDim.x = 1;
    attrs[na].val.clusterDim.y = unsigned(KS);
    attrs[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MP, int GS, bool WB, int BITS>
cudaError_t launch_flags(const GemvArgs& a, bool sym, bool staged, int KS, size_t smem, cudaStream_t stream) {
  if (staged) {
    return sym ? launch_typed<MP, GS, true, true, WB, BITS>(a, KS, smem, stream)
               : launch_typed<MP, GS, false, true, WB, BITS>(a, KS, smem, stream);
  }
  return sym ? launch_typed<MP, GS, true, false, WB, BITS>(a, KS, smem, stream)
             : launch_typed<MP, GS, false, false, WB, BITS>(a, KS, smem, stream);
}

template <int MP, int BITS>
cudaError_t launch_gs(const GemvArgs& a, int gs, bool sym, bool staged, bool wb, int KS, size_t smem,
                      cudaStream_t stream) {
  if (wb) {
    switch (gs) {
      case 32: return launch_flags<MP, 32, true, BITS>(a, sym, staged, KS, smem, stream);
      case 64: return launch_flags<MP, 64, true, BITS>(a, sym, staged, KS, smem, stream);
      default: return launch_flags<MP, 128, true, BITS>(a, sym, staged, KS, smem, stream);
    }
  }
  switch (gs) {
    case 32: return launch_flags<MP, 32, false, BITS>(a, sym, staged, KS, smem, stream);
    case 64: return launch_flags<MP, 64, false, BITS>(a, sym, staged, KS, smem, stream);
    default: return launch_flags<MP, 128, false, BITS>(a, sym, staged, KS, smem, stream);
  }
}

// Shared memory of the register / warp-bulk kernel: staged activations or the
// reduction buffers at offset 0, then (WB) the warps' rings and barriers.
struct RingSmem {
  size_t total;
  int wb_off, slot_bytes;
};
RingSmem ring_smem(const Layout& L, int M, int kb_per_cta, bool staged, bool wb, int depth) {
  RingSmem r{};
  const size_t base = gemv_smem_bytes(M, kb_per_cta, staged);
  if (!wb) {
    r.total = base;
    return r;
  }
  r.wb_off = int((base + 127) / 128 * 128);
  r.slot_bytes = wb_slot_bytes(L.gsize, L.bits);
  r.total = size_t(r.wb_off) + size_t(L.bits == 8 ? kWbSlots<8> : kWbSlots<4>) * r.slot_bytes;
  (void)depth;
  return r;
}

constexpr size_t kMaxGemvSmem = 200 * 1024;

// Activations go through shared memory under act order, with an act scale
// (divided on the way), or when the last 64-column block is ragged (its
// padding columns must read as zero).
bool gemv_staged(const Layout& L) { return L.act || L.awq || (L.K % kColsPerBlock) != 0; }

// 64-column blocks per thread block of a K split: whole groups.
int kb_per_cta_of(const Layout& L, int ksplit) {
  const int unit = L.gsize == 128 ? 2 : 1;
  const int kbc = int((L.KB + ksplit - 1) / ksplit);
  return (kbc + unit - 1) / unit * unit;
}

bool valid_ksplit(int ks) { return ks == 1 || ks == 2 || ks == 4 || ks == 8 || ks == 16; }

template <int BITS>
cudaError_t launch_gemv_bits(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                        const GemvPlan& plan, uint32_t flags, cudaStream_t stream) {
  const BlobView B = view_of(L, blob);
  const bool staged = gemv_staged(L);
  const int gs = L.gsize;
  GemvArgs a;
  a.qweight = B.qweight;
  a.scales2 = reinterpret_cast<const uint32_t*>(B.scales);
  a.zeros = B.zeros;
  a.perm = B.perm;
  a.ascale = B.ascale;
  a.x = x;
  a.y = y;
  a.M = M;
  a.N = int(L.N);
  a.K = int(L.K);
  a.G = int(L.G);
  a.KB = int(L.KB);
  a.rows16 = plan.rows16;
  a.kb_per_cta = kb_per_cta_of(L, plan.ksplit);
  a.flags = flags;
  a.ngroup = 1;
  const bool ring_staged = staged || plan.stage_x;
  const bool wb = plan.kind == kGemvAsyncCopy;
  const RingSmem rs = ring_smem(L, M, a.kb_per_cta, ring_staged, wb, plan.stages);
  a.depth = wb ? plan.stages : 1;
  a.wb_off = rs.wb_off;
  a.slot_bytes = rs.slot_bytes;
  const size_t smem = rs.total;
  if (M <= 1) return launch_gs<1, BITS>(a, gs, L.sym, ring_staged, wb, plan.ksplit, smem, stream);
  if (M <= 2) return launch_gs<2, BITS>(a, gs, L.sym, ring_staged, wb, plan.ksplit, smem, stream);
  if (M <= 4) return launch_gs<4, BITS>(a, gs, L.sym, ring_staged, wb, plan.ksplit, smem, stream);
  if (M <= 8) return launch_gs<8, BITS>(a, gs, L.sym, ring_staged, wb, plan.ksplit, smem, stream);
  return launch_gs<16, BITS>(a, gs, L.sym, ring_staged, wb, plan.ksplit, smem, stream);
}

// Grouped launch: Lc describes the group as one layer (the sum of the row
// blocks, the shared K and format); layer m has its own blob and output.
template <int BITS>
cudaError_t launch_gemv_group_bits(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M,
                                   const GemvPlan& plan, uint32_t flags, cudaStream_t stream) {
  GemvArgs a = {};
  a.perm = nullptr;
  a.ascale = nullptr;
  a.x = x;
  a.M = M;
  a.N = int(Lc.N);
  a.K = int(Lc.K);
  a.G = int(Lc.G);
  a.KB = int(Lc.KB);
  a.rows16 = plan.rows16;
  a.kb_per_cta = kb_per_cta_of(Lc, plan.ksplit);
  a.flags = flags;
  a.ngroup = grp.n;
  a.gstart[0] = 0;
  for (int m = 0; m < grp.n; ++m) {
    a.gq[m] = grp.views[m].qweight;
    a.gs[m] = reinterpret_cast<const uint32_t*>(grp.views[m].scales);
    a.gz[m] = grp.views[m].zeros;
    a.gy[m] = grp.y[m];
    a.gN[m] = int(grp.N[m]);
    a.gstart[m + 1] = a.gstart[m] + int(grp.NR[m] * 8 / plan.rows16);
  }
  a.qweight = a.gq[0];
  a.scales2 = a.gs[0];
  a.zeros = a.gz[0];
  a.y = a.gy[0];
  const bool staged = gemv_staged(Lc) || plan.stage_x;
  const bool wb = plan.kind == kGemvAsyncCopy;
  const RingSmem rs = ring_smem(Lc, M, a.kb_per_cta, staged, wb, plan.stages);
  a.depth = wb ? plan.stages : 1;
  a.wb_off = rs.wb_off;
  a.slot_bytes = rs.slot_bytes;
  const size_t smem = rs.total;
  const int gs = Lc.gsize;
  if (M <= 1) return launch_gs<1, BITS>(a, gs, Lc.sym, staged, wb, plan.ksplit, smem, stream);
  if (M <= 2) return launch_gs<2, BITS>(a, gs, Lc.sym, staged, wb, plan.ksplit, smem, stream);
  if (M <= 4) return launch_gs<4, BITS>(a, gs, Lc.sym, staged, wb, plan.ksplit, smem, stream);
  if (M <= 8) return launch_gs<8, BITS>(a, gs, Lc.sym, staged, wb, plan.ksplit, smem, stream);
  return launch_gs<16, BITS>(a, gs, Lc.sym, staged, wb, plan.ksplit, smem, stream);
}

// This translation unit's timeout counter (read and cleared).
cudaError_t take_local_debug_error(unsigned int* word) {
  unsigned int w = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&w, g_debug_error, sizeof(w));
  if (e != cudaSuccess) return e;
  if (w != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_debug_error, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *word = w;
  return cudaSuccess;
}

cudaError_t take_local_gemv_timeouts(unsigned int* count) {
  unsigned int c = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&c, g_gemv_timeouts, sizeof(c));
  if (e != cudaSuccess) return e;
  if (c != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_gemv_timeouts, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  *count = c;
  return cudaSuccess;
}

}  // namespace
}  // namespace w4a16
