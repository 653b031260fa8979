// Prefill-sized W4A16 product y[M][N] = x[M][K] . W_hat^T on the tcgen05
// tensor cores.
//
// With many tokens the product is a dense contraction and the tensor cores set
// the pace ("AWQ + GPTQ Quantization, in depth", section "What W4A16 buys and
// why decoding gets faster": 4-bit weights are expanded to 16 bits before the
// multiply). The weights enter the MMA from tensor memory:
//
//  * One thread block owns WR x 128 weight rows and NT tokens. A TMA warp
//    streams, per 64-column step, the activations (NT tokens x 64 columns,
//    128-byte swizzle: the MMA's B operand) and the 4 KiB packed tile of each
//    128-row block with its scales and zero points (bulk copies) into a ring
//    of shared-memory stages, several steps ahead.
//  * Dequantization warps read a stage's packed tile from shared memory,
//    expand the nibbles to w_hat = fp16((q - z) * s) -- the same rounding as
//    w4a16_dequant -- and store them into tensor memory with tcgen05.st: they
//    are the MMA's A operand (lane = weight row, two fp16 per 32-bit column).
//  * One thread issues tcgen05.mma (M = 128 weight rows, N = NT tokens,
//    K = 16) into fp32 accumulators in tensor memory and releases each
//    stage with tcgen05.commit.
//  * The epilogue reads the accumulators back (tcgen05.ld), rounds to fp16,
//    transposes through shared memory (one slice per warp) and writes y with
//    16-byte stores.
//  * Under act order the packed columns are in group order; a gather kernel
//    first writes x with its columns in that order to the caller's workspace.
//    With an unfolded AWQ act scale the same kernel divides x by it on the
//    way (and runs without act order too).
//  * Every wait is bounded in time: a wait that gives up raises the device's
//    pipeline-timeout count (w4a16_pipeline_timeouts), the block drains what
//    it has in flight and returns without writing y.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "device_util.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace w4a16 {

__device__ unsigned int g_pipeline_timeouts;

namespace {

// Limit of the waits that let copies and MMAs already issued land before the
// block exits after an abort; the pipeline's own waits use GemmArgs::wait_ns.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// WR: 128-row weight blocks per thread block; NT: tokens per thread block;
// SA: tensor-memory stages of dequantized weights; SB: shared-memory stages of
// activations; DS: dequantization warp sets, set d producing the 64-column
// steps kb = d (mod DS), so that each scheduler interleaves DS independent
// dequantization streams.
// Packed-weight part of a stage, per 128-row tile: the code tile (3, 4 or
// 8 KiB of 3-, 4- or 8-bit codes), then up to two groups of scale pairs (256 B
// each) and of zero points (64 B of nibble pairs or 128 B of byte pairs each).
template <int BITS>
struct WTile {
  static constexpr int kCodes = 4096 * BITS / 4;
  static constexpr int kR16 = kCodes / 8;  // bytes of one 16-row tile (3 bits: half a tile pair)
  static constexpr int kScaleOff = kCodes;
  static constexpr int kZeroGroup = BITS == 8 ? 128 : 64;
  static constexpr int kZeroOff = kScaleOff + 2 * 256;
  static constexpr int kBytes = kZeroOff + 2 * kZeroGroup;
};

constexpr int kMaxSmem = 232448;
constexpr int stage_bytes(int WR, int NT, int BITS) {
  return (NT * 128 + WR * (4096 * BITS / 4 + 512 + 2 * (BITS == 8 ? 128 : 64)) + 1023) / 1024 * 1024;
}
// Activation stages of a tile, reduced for 8-bit codes until the block's
// shared memory fits.
constexpr int fit_sb(int WR, int NT, int SA, int SB, int BITS) {
  int s = SB;
  while (s > 2 && s * stage_bytes(WR, NT, BITS) + 1024 + 8 * (SA * 2 + s * 2 + 1) + 16 > kMaxSmem) --s;
  return s;
}

template <int WR, int NT, int SA, int SB, int DS, int BITS>
struct Cfg {
  static constexpr int kSetWarps = 4 * WR;        // one warp per (128-row tile, lane quarter)
  static constexpr int kDeqWarps = kSetWarps * DS;
  static constexpr int kTmaWarp = kDeqWarps;
  static constexpr int kMmaWarp = kDeqWarps + 1;
  static constexpr int kThreads = (kDeqWarps + 2) * 32;
  static constexpr int kDCols = WR * NT;          // fp32 accumulators
  static constexpr int kACol0 = kDCols;           // first A column
  static constexpr int kBStage = NT * 128;        // activations: NT rows x 64 fp16 (128-byte swizzle)
  static constexpr int kStage = stage_bytes(WR, NT, BITS);  // + packed weights
  static_assert(kStage == (kBStage + WR * WTile<BITS>::kBytes + 1023) / 1024 * 1024, "stage layout");
  static constexpr int kBarBytes = 8 * (SA * 2 + SB * 2 + 1) + 16;
  static constexpr int kSmem = SB * kStage + 1024 + kBarBytes;
  static constexpr int kEpiTokens = NT / DS;      // tokens each set writes back
  // tensor-memory columns allocated: 256 lets two blocks share an SM
  static constexpr int kTmemCols = kDCols + SA * WR * 32 <= 256 ? 256 : 512;
  static_assert(kDCols + SA * WR * 32 <= 512, "tensor memory budget");
  static_assert(kSmem <= kMaxSmem, "shared memory per block");
  static_assert(NT * WR * 128 * 4 <= SB * kStage, "split-K partial sums must fit in the stages");
  static_assert(SA % DS == 0, "each tensor-memory stage belongs to one set");
  static_assert(kEpiTokens % 32 == 0, "epilogue in 32-token chunks");
  static_assert(kDeqWarps * kEpiTokens * 32 * 2 <= SB * kStage, "epilogue staging must fit in the stages");
  static_assert(NT % 32 == 0 && NT >= 32 && NT <= 256, "MMA N");
};

struct GemmArgs {
  const uint32_t* qweight;
  const uint32_t* scales2;  // scale pairs (row g, row g+8)
  const uint8_t* zeros;     // nullptr when symmetric
  uint16_t* y;
  int M, N, NR, G, KB;
  int tok_blocks;
  unsigned long long wait_ns;  // limit of the pipeline's bounded waits
  // K split over the blocks of a cluster (gridDim.y): block r takes the
  // 64-column steps [KB*r/ks, KB*(r+1)/ks); the partial sums are added
  // through distributed shared memory in rank order.
};

// Instruction descriptor of tcgen05.mma kind::f16: fp32 D, fp16 A and B, both
// K-major, M = 128, N = NT.
template <int NT>
__device__ __forceinline__ uint32_t idesc_f16() {
  return (1u << 4)                      // D format: f32
         | (0u << 7) | (0u << 10)       // A, B format: f16
         | (uint32_t(NT >> 3) << 17)    // N / 8
         | (uint32_t(128 >> 4) << 24);  // M / 16
}

// Shared-memory descriptor of a K-major operand stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return uint64_t((saddr & 0x3FFFFu) >> 4)  // start address
         | (uint64_t(1) << 16)              // leading byte offset (unused with this swizzle)
         | (uint64_t(1024 >> 4) << 32)      // stride byte offset: 8 rows
         | (uint64_t(1) << 46)              // descriptor version
         | (uint64_t(2) << 61);             // 128-byte swizzle
}

__device__ __forceinline__ void note_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicAdd(&g_pipeline_timeouts, 1u);
}

// Bounded wait that also gives up once another role of the block has.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint64_t limit_ns) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity, limit_ns)) return true;
  note_timeout(abort_flag);
  return false;
}

// 16-byte parts of packed codes per 16-row tile (3 bits: tile 0 a 16-byte
// part, tile 1 an 8-byte part, read together).
template <int BITS>
constexpr int kGemmParts = BITS == 8 ? 2 : 1;

template <int GS, bool SYM, int BITS>
struct StepRegs {
  static constexpr int kGroups = GS == 32 ? 2 : 1;  // groups in one 64-column step
  uint4 w[2][kGemmParts<BITS>];  // packed words of the warp's two 16-row tiles
  uint32_t s[2][kGroups];     // scale pairs
  uint32_t z[2][kGroups];     // zero points (nibble pair, or byte pair)
};

__device__ __forceinline__ uint32_t prmt_u32(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Groups whose metadata a 64-column step carries: one, or two for 32-column
// groups (one at a ragged end of K).
template <int GS>
__device__ __forceinline__ int step_groups(int kb, int G) {
  return GS == 32 ? min(2, G - 2 * kb) : 1;
}

// Dequantize one step of one 16-row tile into the 16 registers of a
// tcgen05.st 16x256b.x4: per 16-column group j, (row g, columns 4t..4t+1),
// (row g, 4t+2..4t+3), (row g+8, 4t..4t+1), (row g+8, 4t+2..4t+3).
// 8-bit codes: PRMT places code bytes under the exponent byte 0x64, giving
// fp16 1024 + q; subtracting 1024 + z leaves the exact q - z. 3-bit codes: the
// register's pair of fields, shifted down and masked, ORed under 0x6400.
template <int GS, bool SYM, int BITS>
__device__ __forceinline__ void dequant_tile(const StepRegs<GS, SYM, BITS>& r, int i, uint32_t (&v)[16]) {
  constexpr int NG = StepRegs<GS, SYM, BITS>::kGroups;
  uint32_t za[NG], zb[NG], sg[NG], sh[NG];
#pragma unroll
  for (int gg = 0; gg < NG; ++gg) {
    if (BITS == 4) {
      const uint32_t zlo = SYM ? 8u : (r.z[i][gg] & 0xFu);
      const uint32_t zhi = SYM ? 8u : (r.z[i][gg] >> 4);
      za[gg] = zero_lo_const(zlo);
      zb[gg] = zero_hi_const(zhi);
    } else if (BITS == 3) {
      const uint32_t zg = SYM ? 4u : (r.z[i][gg] & 0xFu);
      const uint32_t zh = SYM ? 4u : (r.z[i][gg] >> 4);
      za[gg] = (0x6400u + zg) * 0x00010001u;
      zb[gg] = (0x6400u + zh) * 0x00010001u;
    } else {
      const uint32_t zg = SYM ? 128u : (r.z[i][gg] & 0xFFu);
      const uint32_t zh = SYM ? 128u : (r.z[i][gg] >> 8);
      za[gg] = (0x6400u + zg) * 0x00010001u;
      zb[gg] = (0x6400u + zh) * 0x00010001u;
    }
    sg[gg] = (r.s[i][gg] & 0xFFFFu) * 0x00010001u;
    sh[gg] = (r.s[i][gg] >> 16) * 0x00010001u;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int gg = NG == 2 ? (j >> 1) : 0;
    if (BITS == 4) {
      const uint4& wv = r.w[i][0];
      const uint32_t w = j == 0 ? wv.x : j == 1 ? wv.y : j == 2 ? wv.z : wv.w;
      uint32_t a[4];
      expand_word(w, za[gg], zb[gg], a);  // exact (q - z) in fp16
      v[4 * j + 0] = hmul2_u32(a[0], sg[gg]);
      v[4 * j + 1] = hmul2_u32(a[2], sg[gg]);
      v[4 * j + 2] = hmul2_u32(a[1], sh[gg]);
      v[4 * j + 3] = hmul2_u32(a[3], sh[gg]);
    } else if (BITS == 3) {
      const uint4& A = r.w[0][0];
      const uint4& Bp = r.w[1][0];
      const uint32_t w0 = i == 0 ? A.x : A.w, w1 = i == 0 ? A.y : Bp.x, w2 = i == 0 ? A.z : Bp.y;
      constexpr uint32_t M = 0x00070007u;
      uint32_t c[4];  // fragment registers a0..a3 (row g / g+8, column pairs 4t, 4t+2)
      if (j < 3) {  // the bit positions of w3_field
        const uint32_t w = j == 0 ? w0 : j == 1 ? w1 : w2;
        c[0] = w & M;
        c[1] = (w >> 3) & M;
        c[2] = (w >> 6) & M;
        c[3] = (w >> 9) & M;
      } else {
        c[0] = (w0 >> 12) & M;
        c[1] = (w1 >> 12) & M;
        c[2] = (w2 >> 12) & M;
        c[3] = ((w0 >> 15) & 0x00010001u) | ((w1 >> 14) & 0x00020002u) | ((w2 >> 13) & 0x00040004u);
      }
      v[4 * j + 0] = hmul2_u32(hsub2_u32(c[0] | 0x64006400u, za[gg]), sg[gg]);
      v[4 * j + 1] = hmul2_u32(hsub2_u32(c[2] | 0x64006400u, za[gg]), sg[gg]);
      v[4 * j + 2] = hmul2_u32(hsub2_u32(c[1] | 0x64006400u, zb[gg]), sh[gg]);
      v[4 * j + 3] = hmul2_u32(hsub2_u32(c[3] | 0x64006400u, zb[gg]), sh[gg]);
    } else {
      const uint4& wv = r.w[i][(kGemmParts<BITS> - 1) & (j >> 1)];
      const uint32_t wg = (j & 1) ? wv.z : wv.x;  // row g, columns 4t .. 4t+3
      const uint32_t wh = (j & 1) ? wv.w : wv.y;  // row g+8
      v[4 * j + 0] = hmul2_u32(hsub2_u32(prmt_u32(wg, 0x64646464u, 0x5150u), za[gg]), sg[gg]);
      v[4 * j + 1] = hmul2_u32(hsub2_u32(prmt_u32(wg, 0x64646464u, 0x5352u), za[gg]), sg[gg]);
      v[4 * j + 2] = hmul2_u32(hsub2_u32(prmt_u32(wh, 0x64646464u, 0x5150u), zb[gg]), sh[gg]);
      v[4 * j + 3] = hmul2_u32(hsub2_u32(prmt_u32(wh, 0x64646464u, 0x5352u), zb[gg]), sh[gg]);
    }
  }
}

// One 64-column step of a warp's 32 weight rows (two 16-row tiles, lane
// quarter q4 of the 128-row tile): read the packed codes, scales and zero
// points of the step from the stage's weight tile `ws`, expand them and store
// the fp16 A operand into tensor memory at column `col`. ng: groups the step
// carries; a dead tile (rows beyond N) stores zeros.
template <int GS, bool SYM, int BITS>
__device__ __forceinline__ void dequant_step(const unsigned char* ws, int ng, bool live, int q4, int lane,
                                             uint32_t col) {
  using WT = WTile<BITS>;
  const int g = lane >> 2;
  StepRegs<GS, SYM, BITS> r;
  if (live) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r16 = 2 * q4 + h;
      if (BITS == 3) {
        // the pair's 16-byte parts, then its 8-byte parts (768 bytes per pair)
        if (h == 0) {
          r.w[0][0] = *reinterpret_cast<const uint4*>(ws + q4 * 768 + lane * 16);
        } else {
          const uint2 b2 = *reinterpret_cast<const uint2*>(ws + q4 * 768 + 512 + lane * 8);
          r.w[1][0] = make_uint4(b2.x, b2.y, 0u, 0u);
        }
      } else {
#pragma unroll
        for (int part = 0; part < kGemmParts<BITS>; ++part)
          r.w[h][part] = *reinterpret_cast<const uint4*>(ws + r16 * WT::kR16 + part * 512 + lane * 16);
      }
#pragma unroll
      for (int gg = 0; gg < StepRegs<GS, SYM, BITS>::kGroups; ++gg) {
        const int gs = min(gg, ng - 1);  // the padding half of a ragged last step reuses the last group
        r.s[h][gg] = *reinterpret_cast<const uint32_t*>(ws + WT::kScaleOff + gs * 256 + (r16 * 8 + g) * 4);
        r.z[h][gg] = SYM ? 0u
                     : BITS != 8
                         ? uint32_t(ws[WT::kZeroOff + gs * 64 + r16 * 8 + g])
                         : uint32_t(*reinterpret_cast<const uint16_t*>(ws + WT::kZeroOff + gs * 128 + (r16 * 8 + g) * 2));
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t v[16];
    if (live) {
      dequant_tile<GS, SYM, BITS>(r, h, v);
    } else {
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = 0u;
    }
    tmem_st_16x256b_x4(col + (uint32_t(32 * q4 + 16 * h) << 16), v);
  }
}

// Bulk copies of one step's packed weights of 128-row block R (codes, then
// the scale pairs and zero points of its ng groups from group g0, four row
// groups each) to the stage's weight tile at wdst, completing on barrier bar.
template <bool SYM, int BITS>
__device__ __forceinline__ void load_weight_step(uint32_t wdst, const GemmArgs& a, int R, int kbg, int g0, int ng,
                                                 uint32_t bar) {
  using WT = WTile<BITS>;
  const unsigned char* qbytes = reinterpret_cast<const unsigned char*>(a.qweight);
  const unsigned char* sbytes = reinterpret_cast<const unsigned char*>(a.scales2);
  bulk_copy_g2s(wdst, qbytes + (size_t(R) * a.KB + kbg) * WT::kCodes, WT::kCodes, bar);
  // the step's groups of this row block are contiguous in the blob
  // ([group][16-row tile][lane group]): one copy for the scales, one for the zeros
  const size_t mi = size_t(meta_index(R, g0, 0, 0, a.G));
  bulk_copy_g2s(wdst + WT::kScaleOff, sbytes + mi * 4, uint32_t(ng * 256), bar);
  if (!SYM)
    bulk_copy_g2s(wdst + WT::kZeroOff, a.zeros + mi * (WT::kZeroGroup / 64), uint32_t(ng * WT::kZeroGroup), bar);
}

template <int WR, int NT, int SA, int SB, int DS, int GS, bool SYM, int BITS>
__global__ void __launch_bounds__(Cfg<WR, NT, SA, SB, DS, BITS>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmArgs a) {
  using C = Cfg<WR, NT, SA, SB, DS, BITS>;
  using WT = WTile<BITS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-byte aligned for the swizzle
  const uint32_t sbase = smem_addr(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SB * C::kStage);
  // barriers: full_a[SA], empty_a[SA], full_b[SB], empty_b[SB], acc
  const uint32_t bar0 = smem_addr(bars);
  auto full_a = [&](int s) { return bar0 + 8u * uint32_t(s); };
  auto empty_a = [&](int s) { return bar0 + 8u * uint32_t(SA + s); };
  auto full_b = [&](int s) { return bar0 + 8u * uint32_t(2 * SA + s); };
  auto empty_b = [&](int s) { return bar0 + 8u * uint32_t(2 * SA + SB + s); };
  const uint32_t acc_bar = bar0 + 8u * uint32_t(2 * SA + 2 * SB);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * SA + 2 * SB + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = int(threadIdx.x >> 5), lane = int(threadIdx.x & 31);
  const int tb = int(blockIdx.x) % a.tok_blocks;
  const int rg = int(blockIdx.x) / a.tok_blocks;
  const int m0 = tb * NT;
  const int KS = int(gridDim.y);
  const int kb_lo = int((int64_t(a.KB) * blockIdx.y) / KS);
  const int KB = int((int64_t(a.KB) * (blockIdx.y + 1)) / KS) - kb_lo;  // steps of this block (>= 1)

  if (threadIdx.x == 0) {
    for (int s = 0; s < SA; ++s) {
      mbar_init(full_a(s), C::kSetWarps * 32);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
    }
    mbar_init(acc_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == C::kTmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < C::kDeqWarps) {
    // ---------------- dequantization into tensor memory, then the epilogue
    const int ds = warp / C::kSetWarps;  // warp set: steps kb = ds (mod DS)
    const int at = (warp % C::kSetWarps) >> 2;  // 128-row tile of this block
    const int q4 = warp & 3;   // tensor-memory lane quarter: rows 32*q4 .. 32*q4+31 of the tile
    const int R = rg * WR + at;
    const bool live = R < a.NR;
    const int nsteps = KB > ds ? (KB - ds + DS - 1) / DS : 0;  // steps of this set

    // The packed weights of a step arrive with its activations (TMA warp);
    // this warp only expands them and writes tensor memory.
    bool ok = true;
    for (int i = 0; i < nsteps && ok; ++i) {
      const int kb = ds + i * DS;  // local step
      const int sb = kb % SB, sa = kb % SA;
      if (!wait_or_abort(full_b(sb), uint32_t(kb / SB) & 1u, abort_flag, a.wait_ns)) {
        ok = false;
        break;
      }
      if (kb >= SA && !wait_or_abort(empty_a(sa), uint32_t(kb / SA - 1) & 1u, abort_flag, a.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const unsigned char* ws = smem + size_t(sb) * C::kStage + C::kBStage + at * WT::kBytes;
      dequant_step<GS, SYM, BITS>(ws, step_groups<GS>(kb_lo + kb, a.G), live, q4, lane,
                                  tmem + uint32_t(C::kACol0 + (sa * WR + at) * 32));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(full_a(sa));
    }

    // ---------------- epilogue: set ds writes tokens [ds*NT/DS, (ds+1)*NT/DS).
    // Each warp transposes its 32 rows x NT/DS tokens through a private
    // shared-memory slice (no block-wide barrier, so a warp that gave up
    // cannot stall the others) and writes 64-byte row segments.
    if (ok && wait_or_abort(acc_bar, 0u, abort_flag, a.wait_ns)) {
      tc_fence_after();
      constexpr int ET = C::kEpiTokens;
      const int t0 = ds * ET;  // first token of this set
      if (KS > 1) {
        // split K: this block's fp32 partial sums, part[token][row], for the
        // cluster reduction below (the activation stages are free by now)
        float* part = reinterpret_cast<float*>(smem);
        const int nl = at * 128 + 32 * q4 + lane;
#pragma unroll 1
        for (int c = 0; c < ET / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + (uint32_t(32 * q4) << 16) + uint32_t(at * NT + t0 + c * 32), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) part[(t0 + c * 32 + i) * (WR * 128) + nl] = __uint_as_float(v[i]);
        }
      } else {
        uint16_t* wst = reinterpret_cast<uint16_t*>(smem) + warp * ET * 32;  // [ET tokens][32 rows]
        const int n_warp = (rg * WR + at) * 128 + 32 * q4;
        const int m_live = max(0, min(ET, a.M - m0 - t0));  // tokens of this set that exist
#pragma unroll 1
        for (int c = 0; c < ET / 32; ++c) {
          if (c * 32 >= m_live) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + (uint32_t(32 * q4) << 16) + uint32_t(at * NT + t0 + c * 32), v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            wst[(c * 32 + i) * 32 + lane] = __half_as_ushort(__float2half_rn(__uint_as_float(v[i])));
        }
        __syncwarp();
        const bool vec = (a.N % 8) == 0;
        for (int e = lane; e < m_live * 4; e += 32) {
          const int m = e >> 2, gn = n_warp + (e & 3) * 8;
          if (gn >= a.N) continue;
          const uint16_t* src = wst + m * 32 + (e & 3) * 8;
          uint16_t* dst = a.y + size_t(m0 + t0 + m) * a.N + gn;
          if (vec) {
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
          } else {
            for (int i = 0; i < 8 && gn + i < a.N; ++i) dst[i] = src[i];
          }
        }
      }
    }
  } else if (warp == C::kTmaWarp) {
    // ---------------- activation stream (one thread)
    if (lane == 0) {
      tma_prefetch_desc(&tmap_x);
      pdl_wait();  // x may come from the preceding gather kernel
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % SB;
        const int n = kb / SB;
        if (kb >= SB && !wait_or_abort(empty_b(s), uint32_t(n - 1) & 1u, abort_flag, a.wait_ns)) break;
        const int kbg = kb_lo + kb;  // global 64-column step
        const int g0 = kbg * 64 / GS;
        const int ng = step_groups<GS>(kbg, a.G);
        const uint32_t wbytes = uint32_t(WT::kCodes + ng * 256 + (SYM ? 0 : ng * WT::kZeroGroup));
        int live_tiles = 0;
#pragma unroll
        for (int t = 0; t < WR; ++t) live_tiles += (rg * WR + t < a.NR) ? 1 : 0;
        const uint32_t stage = sbase + uint32_t(s * C::kStage);
        mbar_arrive_expect_tx(full_b(s), uint32_t(C::kBStage) + uint32_t(live_tiles) * wbytes);
        tma_load_2d(stage, &tmap_x, (kb_lo + kb) * 64, m0, full_b(s));
#pragma unroll
        for (int t = 0; t < WR; ++t) {
          const int R = rg * WR + t;
          if (R >= a.NR) continue;
          load_weight_step<SYM, BITS>(stage + uint32_t(C::kBStage + t * WT::kBytes), a, R, kbg, g0, ng, full_b(s));
        }
        ++issued;
      }
      // drain: the last loads issued must land before the block's shared
      // memory goes away (after a normal run they have all been consumed and
      // each test returns at once; another role may abort after this warp's
      // last issue)
      for (int kb = max(issued - SB, 0); kb < issued; ++kb)
        mbar_wait_bounded(full_b(kb % SB), uint32_t(kb / SB) & 1u, kWaitLimitNs);
    }
  } else if (warp == C::kMmaWarp) {
    // ---------------- MMA issue (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_f16<NT>();
      for (int kb = 0; kb < KB; ++kb) {
        const int sa = kb % SA, sb = kb % SB;
        if (!wait_or_abort(full_b(sb), uint32_t(kb / SB) & 1u, abort_flag, a.wait_ns)) break;
        if (!wait_or_abort(full_a(sa), uint32_t(kb / SA) & 1u, abort_flag, a.wait_ns)) break;
        tc_fence_after();
        const uint32_t b_addr = sbase + uint32_t(sb * C::kStage);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t bdesc = sw128_desc(b_addr + uint32_t(kk * 32));
#pragma unroll
          for (int t = 0; t < WR; ++t)
            mma_ts_f16(tmem + uint32_t(t * NT), tmem + uint32_t(C::kACol0 + (sa * WR + t) * 32 + kk * 8), bdesc,
                       idesc, uint32_t(kb | kk));
        }
        mma_commit(empty_a(sa));
        mma_commit(empty_b(sb));
      }
      mma_commit(acc_bar);
      // on abort, let every MMA issued so far finish before tensor memory is freed
      if (*abort_flag) mbar_wait_bounded(acc_bar, 0u, kWaitLimitNs);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (KS > 1) {
    // Every block of the cluster holds its partial sums; rank r adds its
    // share of (token, row) pairs over all ranks in rank order and writes y.
    cluster_sync_all();
    const float* part = reinterpret_cast<const float*>(smem);
    constexpr int kRows = WR * 128;
    const int E = max(0, min(NT, a.M - m0)) * kRows;
    const int rank = int(cluster_ctarank());
    const int e_lo = int((int64_t(E) * rank) / KS), e_hi = int((int64_t(E) * (rank + 1)) / KS);
    for (int e = e_lo + int(threadIdx.x); e < e_hi; e += C::kThreads) {
      float acc = 0.f;
      for (int rk = 0; rk < KS; ++rk) acc += ld_dsmem_f32(part + e, uint32_t(rk));
      const int tok = e / kRows;
      const int n = rg * kRows + (e - tok * kRows);
      if (n < a.N) a.y[size_t(m0 + tok) * a.N + n] = __half_as_ushort(__float2half_rn(acc));
    }
    cluster_sync_all();  // peers are done reading this block's partial sums
  }
  if (warp == C::kTmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// x_perm[m][p] = x[m][perm[p]] / ascale[p]: activations in the packed
// (group-sorted) column order, divided by the act scale when there is one.
// One thread block per token row: the row is staged in shared memory with
// 16-byte loads, then written back permuted with 16-byte stores.
constexpr int kGatherThreads = 256;
__global__ void __launch_bounds__(kGatherThreads) gather_cols_kernel(const uint16_t* __restrict__ x,
                                                                     const int32_t* __restrict__ perm,
                                                                     const uint16_t* __restrict__ ascale,
                                                                     uint16_t* __restrict__ xp, int K) {
  extern __shared__ __align__(16) uint16_t row_s[];
  pdl_launch_dependents();
  const int64_t m = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + m * K);
  const int chunks = K / 8;
  for (int c = threadIdx.x; c < chunks; c += kGatherThreads) reinterpret_cast<uint4*>(row_s)[c] = src[c];
  __syncthreads();
  uint4* dst = reinterpret_cast<uint4*>(xp + m * K);
  const int4* pv = reinterpret_cast<const int4*>(perm);
  for (int c = threadIdx.x; c < chunks; c += kGatherThreads) {
    const int4 p0 = pv[2 * c], p1 = pv[2 * c + 1];
    uint16_t h[8] = {row_s[p0.x], row_s[p0.y], row_s[p0.z], row_s[p0.w],
                     row_s[p1.x], row_s[p1.y], row_s[p1.z], row_s[p1.w]};
    if (ascale != nullptr) {
      const uint4 sv = reinterpret_cast<const uint4*>(ascale)[c];
      const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = div_act(h[i], uint16_t(sw[i >> 1] >> (16 * (i & 1))));
    }
    uint4 o;
    o.x = uint32_t(h[0]) | (uint32_t(h[1]) << 16);
    o.y = uint32_t(h[2]) | (uint32_t(h[3]) << 16);
    o.z = uint32_t(h[4]) | (uint32_t(h[5]) << 16);
    o.w = uint32_t(h[6]) | (uint32_t(h[7]) << 16);
    dst[c] = o;
  }
}

// The same for rows too long to stage in shared memory, and for the act
// scale alone (perm == nullptr: contiguous 16-byte loads).
__global__ void __launch_bounds__(256) gather_cols_global_kernel(const uint16_t* __restrict__ x,
                                                                 const int32_t* __restrict__ perm,
                                                                 const uint16_t* __restrict__ ascale,
                                                                 uint16_t* __restrict__ xp, int64_t M, int K) {
  pdl_launch_dependents();
  const int64_t chunks = int64_t(K) / 8;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= M * chunks) return;
  const int64_t m = i / chunks;
  const int p0 = int(i - m * chunks) * 8;
  const uint16_t* row = x + m * K;
  uint16_t h[8];
  if (perm == nullptr) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + p0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = uint16_t(w[j >> 1] >> (16 * (j & 1)));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = row[perm[p0 + j]];
  }
  if (ascale != nullptr) {
    const uint4 sv = *reinterpret_cast<const uint4*>(ascale + p0);
    const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) h[j] = div_act(h[j], uint16_t(sw[j >> 1] >> (16 * (j & 1))));
  }
  *reinterpret_cast<uint4*>(xp + m * K + p0) =
      make_uint4(uint32_t(h[0]) | (uint32_t(h[1]) << 16), uint32_t(h[2]) | (uint32_t(h[3]) << 16),
                 uint32_t(h[4]) | (uint32_t(h[5]) << 16), uint32_t(h[6]) | (uint32_t(h[7]) << 16));
}
constexpr size_t kGatherMaxSmem = 160 * 1024;

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;

cudaError_t encode_fn(EncodeTiledFn* out) {
  std::call_once(g_encode_once, []() {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && (q != cudaDriverEntryPointSuccess || fn == nullptr))
      g_encode_err = cudaErrorNotSupported;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  *out = g_encode;
  return g_encode_err;
}

// Tensor map of x [M][K] fp16, box of NT rows x 64 columns, 128-byte swizzle;
// rows and columns beyond the tensor read as zero.
cudaError_t make_x_map(CUtensorMap* map, const uint16_t* x, int64_t M, int64_t K, int NT) {
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encode_fn(&enc);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(M)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {64u, cuuint32_t(NT)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int WR, int NT, int SA, int SB, int DS, int GS, bool SYM, int BITS>
cudaError_t launch_cfg(const Layout& L, const GemmArgs& base, const uint16_t* xa, int64_t M, int ks,
                       bool after_gather, cudaStream_t stream) {
  using C = Cfg<WR, NT, SA, SB, DS, BITS>;
  CUtensorMap map;
  cudaError_t e = make_x_map(&map, xa, M, L.K, NT);
  if (e != cudaSuccess) return e;
  auto kern = gemm_kernel<WR, NT, SA, SB, DS, GS, SYM, BITS>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, int(cudaSharedmemCarveoutMaxShared));
  if (e != cudaSuccess) return e;
  if (ks > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  GemmArgs a = base;
  a.tok_blocks = int((M + NT - 1) / NT);
  const int64_t row_groups = (L.NR + WR - 1) / WR;
  const int64_t blocks = row_groups * a.tok_blocks;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks), unsigned(ks), 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (after_gather) {
    // After our own gather kernel (which writes only the workspace), the
    // block's set-up and weight stream may start before the gather ends; the
    // activation loads wait for it.
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (ks > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = unsigned(ks);
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  e = cudaLaunchKernelEx(&cfg, kern, map, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int WR, int NT, int SA, int SB, int DS, int BITS>
cudaError_t launch_scheme(const Layout& L, const GemmArgs& a, const uint16_t* xa, int64_t M, int ks,
                          bool after_gather, cudaStream_t stream) {
  constexpr int S = fit_sb(WR, NT, SA, SB, BITS);
  switch (L.gsize) {
    case 32:
      return L.sym ? launch_cfg<WR, NT, SA, S, DS, 32, true, BITS>(L, a, xa, M, ks, after_gather, stream)
                   : launch_cfg<WR, NT, SA, S, DS, 32, false, BITS>(L, a, xa, M, ks, after_gather, stream);
    case 64:
      return L.sym ? launch_cfg<WR, NT, SA, S, DS, 64, true, BITS>(L, a, xa, M, ks, after_gather, stream)
                   : launch_cfg<WR, NT, SA, S, DS, 64, false, BITS>(L, a, xa, M, ks, after_gather, stream);
    default:
      return L.sym ? launch_cfg<WR, NT, SA, S, DS, 128, true, BITS>(L, a, xa, M, ks, after_gather, stream)
                   : launch_cfg<WR, NT, SA, S, DS, 128, false, BITS>(L, a, xa, M, ks, after_gather, stream);
  }
}

template <int BITS>
cudaError_t launch_tile(int tile, const Layout& L, const GemmArgs& a, const uint16_t* xa, int64_t M, int ks,
                        bool g, cudaStream_t stream) {
  switch (tile) {
    case 1: return launch_scheme<1, 256, 8, 6, 2, BITS>(L, a, xa, M, ks, g, stream);
    case 2: return launch_scheme<2, 128, 4, 8, 2, BITS>(L, a, xa, M, ks, g, stream);
    case 4: return launch_scheme<1, 256, 8, 6, 1, BITS>(L, a, xa, M, ks, g, stream);
    case 5: return launch_scheme<1, 128, 4, 5, 2, BITS>(L, a, xa, M, ks, g, stream);
    case 6: return launch_scheme<1, 64, 4, 8, 2, BITS>(L, a, xa, M, ks, g, stream);
    default: return launch_scheme<1, 256, 8, 6, 4, BITS>(L, a, xa, M, ks, g, stream);
  }
}

// Tokens per block of each tile.
int tile_tokens(int tile) { return tile == 2 ? 128 : tile == 5 ? 128 : tile == 6 ? 64 : 256; }
int tile_rows(int tile) { return tile == 2 ? 256 : 128; }

}  // namespace

cudaError_t encode_tiled_map(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                             const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  EncodeTiledFn enc = nullptr;
  cudaError_t e = encode_fn(&enc);
  if (e != cudaSuccess) return e;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = cuuint64_t(dims[i]);
    bx[i] = cuuint32_t(box[i]);
    es[i] = 1u;
    if (i + 1 < rank) st[i] = cuuint64_t(strides[i]);
  }
  const CUresult r = enc(map, type, cuuint32_t(rank), const_cast<void*>(base), d, st, bx, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

GemmPlan gemm_default_plan(const Layout& L, int64_t M, int sm_count) {
  // Few tokens: a narrow tile (two blocks per SM) and K split over a cluster
  // so that every SM dequantizes; many tokens: the 128 x 256 tile.
  GemmPlan p{M <= 64 ? 6 : M <= 128 ? 5 : 1, 1};
  const int64_t blocks = ((L.NR * 128 + tile_rows(p.tile) - 1) / tile_rows(p.tile)) *
                         ((M + tile_tokens(p.tile) - 1) / tile_tokens(p.tile));
  const double target = (p.tile >= 5 ? 2.0 : 1.0) * sm_count;
  double best = 1e30;
  for (int ks : {1, 2, 4, 8, 16}) {
    if (ks > 1 && L.KB / ks < 8) break;  // at least 8 steps of 64 columns per block
    const double d = std::fabs(std::log(double(blocks * ks) / target));
    if (d < best - 1e-9) {
      best = d;
      p.ksplit = ks;
    }
  }
  return p;
}

bool gemm_plan_ok(const Layout& L, const GemmPlan& p) {
  if (p.tile < 1 || p.tile > 6) return false;
  if (p.ksplit != 1 && p.ksplit != 2 && p.ksplit != 4 && p.ksplit != 8 && p.ksplit != 16) return false;
  return p.ksplit <= L.KB;
}

cudaError_t launch_gemm(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int64_t M,
                        void* workspace, const GemmPlan& plan, cudaStream_t stream) {
  const BlobView B = view_of(L, blob);
  const uint16_t* xa = x;
  if (L.act || L.awq) {
    uint16_t* xp = static_cast<uint16_t*>(workspace);
    const size_t smem = size_t(L.K) * 2;
    cudaError_t e = cudaSuccess;
    if (L.act && smem <= kGatherMaxSmem && M <= 0x7FFFFFFF) {
      if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(gather_cols_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e != cudaSuccess) return e;
      gather_cols_kernel<<<unsigned(M), kGatherThreads, smem, stream>>>(x, B.perm, B.ascale, xp, int(L.K));
    } else {
      const int64_t chunks = M * (L.K / 8);
      gather_cols_global_kernel<<<unsigned((chunks + 255) / 256), 256, 0, stream>>>(x, B.perm, B.ascale, xp, M,
                                                                                  int(L.K));
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    xa = xp;
  }
  GemmArgs a{};
  a.qweight = B.qweight;
  a.scales2 = reinterpret_cast<const uint32_t*>(B.scales);
  a.zeros = B.zeros;
  a.y = y;
  a.M = int(M);
  a.N = int(L.N);
  a.NR = int(L.NR);
  a.G = int(L.G);
  a.KB = int(L.KB);
  a.wait_ns = wait_limit_ns();
  const bool g = L.act || L.awq;
  const int ks = plan.ksplit;
  if (L.bits == 8) return launch_tile<8>(plan.tile, L, a, xa, M, ks, g, stream);
  if (L.bits == 3) return launch_tile<3>(plan.tile, L, a, xa, M, ks, g, stream);
  return launch_tile<4>(plan.tile, L, a, xa, M, ks, g, stream);
}

cudaError_t take_pipeline_timeouts(unsigned int* count) {
  unsigned int c = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&c, g_pipeline_timeouts, sizeof(c));
  if (e != cudaSuccess) return e;
  if (c != 0) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_pipeline_timeouts, &zero, sizeof(zero));
    if (e != cudaSuccess) return e;
  }
  unsigned int cv = 0;
  e = take_gemv_timeouts(&cv);
  if (e != cudaSuccess) return e;
  *count = c + cv;
  return cudaSuccess;
}

}  // namespace w4a16
