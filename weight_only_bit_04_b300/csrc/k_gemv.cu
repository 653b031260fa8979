// Decode-sized W4A16 product y[M][N] = x[M][K] . W_hat^T, 1 <= M <= 16.
//
// At batch one every packed weight is read once and used for about two flops
// ("AWQ + GPTQ Quantization, in depth", section "What W4A16 buys and why
// decoding gets faster"), so the kernel is an HBM stream whose instruction
// count per weight must stay small:
//
//  * Each warp owns two 16-row tiles (32 rows) and a contiguous run of
//    64-column blocks. Per block it issues one coalesced 16-byte load per lane
//    and tile (1 KiB contiguous per warp), kept kPF blocks ahead in registers.
//  * A 32-bit word holds the codes of one lane's m16n8k16 A fragment. Masking
//    its nibbles with AND gives fp16 bit patterns 0x000q (= q * 2^-24) and
//    0x00q0 (= q * 2^-20): exact subnormal values, so four ANDs and one shift
//    expand eight weights. The tensor cores multiply them with the activations
//    (B fragment, tokens in the n dimension) into fp32 accumulators.
//  * Per (row, group) the accumulator holds sum_k x_k q_k scaled by 2^-24
//    (rows g) or 2^-20 (rows g+8); one more MMA per 16 columns with a constant
//    all-2^-24 operand gives the group's activation sum X. The dequantization
//    (q - z) * s is applied once per group: y += s * (sum x q - z * X), from
//    scales and zero points staged in shared memory by cp.async. Summation
//    order differs from the dequantize-then-multiply definition; the error
//    stays within the stated tolerance (products are exact, sums are fp32).
//  * Warps sharing rows reduce through shared memory; CTAs of a thread-block
//    cluster that split K reduce through distributed shared memory in rank
//    order (deterministic, no atomics).
//  * Programmatic dependent launch: the next kernel's CTAs become resident
//    while this one finishes. By default a CTA waits for the previous kernel
//    before its first global read. With kGemvWeightsReady (the caller vouches
//    that no kernel still in flight writes the packed weights) it issues its
//    first weight loads before that wait; activations are always read after.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPF = 4;         // 64-column blocks in flight per warp
constexpr int kTilesPerWarp = 2;

struct GemvArgs {
  const uint32_t* qweight;
  const uint32_t* scales2;  // scale pairs (row g, row g+8)
  const uint8_t* zeros;
  const int32_t* perm;
  const uint16_t* x;
  uint16_t* y;
  int M, N, K, G, KB;
  int rows16;      // 16-row tiles per CTA (2, 4 or 8)
  int kb_per_cta;  // 64-column blocks per CTA (the last CTAs of a cluster may get fewer)
  int gl_per_cta;  // groups a CTA's column range can touch
  int mpad_log2;   // log2 of M rounded up to a power of two
  uint32_t flags;  // kGemvWeightsReady
};

// Scale and zero for the rows (g, g+8) of one tile and one group, folded into
// the two per-element factors of the finalisation.
struct GroupFactors {
  float sa, sb;  // s_g * 2^24, s_{g+8} * 2^20      (acc holds q-sums at 2^-24 / 2^-20)
  float za, zb;  // -s_g * z_g * 2^24, -s_{g+8} * z_{g+8} * 2^24   (cx holds x-sums at 2^-24)
};

template <bool SYM>
__device__ __forceinline__ GroupFactors make_factors(uint32_t s2, uint32_t zbyte) {
  const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&s2));
  const float zg = SYM ? 8.f : float(zbyte & 0xF);
  const float zh = SYM ? 8.f : float(zbyte >> 4);
  GroupFactors f;
  f.sa = sf.x * 16777216.f;
  f.sb = sf.y * 1048576.f;
  f.za = -sf.x * zg * 16777216.f;
  f.zb = -sf.y * zh * 16777216.f;
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

template <int NB, int GS, bool SYM>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  constexpr int kBlocksPerGroup = GS == 128 ? 2 : 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int RT = a.rows16;
  const int WR = RT / kTilesPerWarp;  // warp row groups per CTA
  const int WK = kWarps / WR;         // warps splitting K per row group
  const int wr = warp % WR;
  const int wk = warp / WR;
  const int Tc = int(blockIdx.x) * RT;            // first 16-row tile of the CTA
  const int R = Tc >> 3;
  const int r16c = Tc & 7;
  const int r16 = r16c + wr * kTilesPerWarp;      // this warp's first tile within the row block

  const int kb_lo = int(blockIdx.y) * a.kb_per_cta;
  const int kb_hi = min(kb_lo + a.kb_per_cta, a.KB);
  const int span = max(kb_hi - kb_lo, 0);
  // This warp's contiguous blocks, in whole groups.
  const int units = (span + kBlocksPerGroup - 1) / kBlocksPerGroup;
  const int u_lo = (units * wk) / WK, u_hi = (units * (wk + 1)) / WK;
  const int b_lo = kb_lo + min(u_lo * kBlocksPerGroup, span);
  const int b_hi = kb_lo + min(u_hi * kBlocksPerGroup, span);
  const int nblk = b_hi - b_lo;
  const int G = a.G;
  // Groups touched by this CTA: [g_lo, g_lo + ngl).
  const int g_lo = (kb_lo * kColsPerBlock) / GS;
  const int ngl = span > 0 ? (min(kb_hi * kColsPerBlock, G * GS) - 1) / GS - g_lo + 1 : 0;

  // Shared memory: x fragments [bj][t][tok], then scales [gl][RT*8] and zeros [gl][RT*8].
  const int mp_log = a.mpad_log2;
  const int MP = 1 << mp_log;
  uint2* xs = reinterpret_cast<uint2*>(smem);
  uint32_t* s_sm = reinterpret_cast<uint32_t*>(smem + size_t(a.kb_per_cta) * 16 * MP * 8);
  uint8_t* z_sm = reinterpret_cast<uint8_t*>(s_sm + size_t(a.gl_per_cta) * RT * 8);

  const uint32_t* qp = a.qweight + (size_t(R) * a.KB * 8 + r16) * 128 + lane * 4;  // block 0
  const bool early = (a.flags & kGemvWeightsReady) != 0;
  if (!early) {
    pdl_wait();
    pdl_launch_dependents();
  }
  uint4 wq[kPF][kTilesPerWarp];
#pragma unroll
  for (int u = 0; u < kPF; ++u) {
    if (u < nblk) {
#pragma unroll
      for (int tt = 0; tt < kTilesPerWarp; ++tt)
        wq[u][tt] = ldg_stream_u4(qp + size_t(b_lo + u) * 1024 + tt * 128);
    }
  }
  // Scales and zero points of the CTA's tiles and groups, 16-byte async copies.
  {
    const int s_chunks = RT * 2;            // 32*RT bytes per group
    const int z_chunks = (RT * 8) / 16;     // 8*RT bytes per group (RT >= 2)
    const char* sg = reinterpret_cast<const char*>(a.scales2) + (size_t(R) * G * 8 + r16c) * 32;
    for (int c = threadIdx.x; c < ngl * s_chunks; c += kThreads) {
      const int gl = c / s_chunks, k = c - gl * s_chunks;
      cp_async_16(s_sm + gl * RT * 8 + k * 4, sg + size_t(g_lo + gl) * 256 + k * 16);
    }
    if (!SYM) {
      const char* zg = reinterpret_cast<const char*>(a.zeros) + (size_t(R) * G * 8 + r16c) * 8;
      for (int c = threadIdx.x; c < ngl * z_chunks; c += kThreads) {
        const int gl = c / z_chunks, k = c - gl * z_chunks;
        cp_async_16(z_sm + gl * RT * 8 + k * 16, zg + size_t(g_lo + gl) * 64 + k * 16);
      }
    }
    cp_async_commit();
  }
  if (early) {
    pdl_launch_dependents();
    pdl_wait();
  }

  // Stage this CTA's slice of x (in packed column order) as B fragments:
  // unit (bj = 16-column step, t, token) = 4 consecutive halves.
  const int M = a.M;
  const int nunits = span * 16 << mp_log;
  for (int u = threadIdx.x; u < nunits; u += kThreads) {
    const int tok = u & (MP - 1);
    const int rest = u >> mp_log;
    const int tq = rest & 3;
    const int bj = rest >> 2;
    const int p0 = kb_lo * kColsPerBlock + bj * 16 + 4 * tq;
    uint2 v = make_uint2(0u, 0u);
    if (tok < M && p0 < a.K) {
      if (a.perm == nullptr) {
        v = *reinterpret_cast<const uint2*>(a.x + size_t(tok) * a.K + p0);
      } else {
        const uint16_t* xr = a.x + size_t(tok) * a.K;
        v.x = uint32_t(xr[a.perm[p0]]) | (uint32_t(xr[a.perm[p0 + 1]]) << 16);
        v.y = uint32_t(xr[a.perm[p0 + 2]]) | (uint32_t(xr[a.perm[p0 + 3]]) << 16);
      }
    }
    xs[u] = v;
  }
  cp_async_wait_all();
  __syncthreads();

  float tot[kTilesPerWarp][NB][4];
  float acc[kTilesPerWarp][NB][4];
  float cx[NB][4];  // 2^-24 * (sum of x over the current group), all rows alike
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
    for (int i = 0; i < 4; ++i) cx[nb][i] = 0.f;
#pragma unroll
    for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
      for (int i = 0; i < 4; ++i) tot[tt][nb][i] = 0.f, acc[tt][nb][i] = 0.f;
  }
  const uint32_t ones[4] = {0x00010001u, 0x00010001u, 0x00010001u, 0x00010001u};  // 2^-24 each

  const bool tok_ok0 = g < M;
  const bool tok_ok1 = NB > 1 && g + 8 < M;
  for (int i0 = 0; i0 < nblk; i0 += kPF) {
#pragma unroll
    for (int u = 0; u < kPF; ++u) {
      const int i = i0 + u;
      if (i < nblk) {
        const int b = b_lo + i;
        const uint2* xb = xs + ((b - kb_lo) * 16 << mp_log);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint2 bx[NB];
          bx[0] = tok_ok0 ? xb[((j * 4 + t) << mp_log) + g] : make_uint2(0u, 0u);
          if (NB > 1) bx[NB - 1] = tok_ok1 ? xb[((j * 4 + t) << mp_log) + g + 8] : make_uint2(0u, 0u);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) mma_16816(cx[nb], ones, bx[nb].x, bx[nb].y, cx[nb]);
#pragma unroll
          for (int tt = 0; tt < kTilesPerWarp; ++tt) {
            uint32_t af[4];
            extract_word(word_of(wq[u][tt], j), af);
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) mma_16816(acc[tt][nb], af, bx[nb].x, bx[nb].y, acc[tt][nb]);
          }
          // Group boundary (or end of this warp's run) after this 16-column step?
          const bool last = (j == 3) && (i == nblk - 1);
          const bool group_end = (GS == 32) ? (j == 1 || j == 3) : (j == 3 && (GS == 64 || (b & 1)));
          if (group_end || last) {
            const int gl = min((b * kColsPerBlock + j * 16) / GS, G - 1) - g_lo;
#pragma unroll
            for (int tt = 0; tt < kTilesPerWarp; ++tt) {
              const int mi = gl * RT * 8 + (wr * kTilesPerWarp + tt) * 8 + g;
              const uint32_t s2 = s_sm[mi];
              const uint32_t zb = SYM ? 0u : z_sm[mi];
              const GroupFactors f = make_factors<SYM>(s2, zb);
              finalize<NB>(acc[tt], cx, f, tot[tt]);
#pragma unroll
              for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[tt][nb][q] = 0.f;
            }
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int q = 0; q < 4; ++q) cx[nb][q] = 0.f;
          }
        }
        const int inext = i + kPF;
        if (inext < nblk) {
#pragma unroll
          for (int tt = 0; tt < kTilesPerWarp; ++tt)
            wq[u][tt] = ldg_stream_u4(qp + size_t(b_lo + inext) * 1024 + tt * 128);
        }
      }
    }
  }

  // Reduce: per-warp partials -> per-CTA partials (fixed order) -> cluster.
  // The buffers reuse the staging area (offset 0 in every CTA of the cluster,
  // where peers read red_c).
  __syncthreads();
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
    float s = 0.f;
    for (int k = 0; k < WK; ++k) s += red_w[(k * WR + w_r) * 512 + rr * 16 + tok];
    red_c[e] = s;
  }
  const int KS = int(gridDim.y);
  if (KS > 1) {
    cluster_sync_all();
    const int rank = int(cluster_ctarank());
    const int per = (nout + KS - 1) / KS;
    const int e_lo = rank * per;
    const int e_hi = min(e_lo + per, nout);
    for (int e = e_lo + threadIdx.x; e < e_hi; e += kThreads) {
      float s = 0.f;
      for (int rk = 0; rk < KS; ++rk) s += ld_dsmem_f32(red_c + e, uint32_t(rk));
      const int tok = e / rows;
      const int n = int(blockIdx.x) * rows + (e - tok * rows);
      if (n < a.N) a.y[size_t(tok) * a.N + n] = __half_as_ushort(__float2half_rn(s));
    }
    cluster_sync_all();  // keep this CTA's shared memory alive until peers are done
  } else {
    __syncthreads();
    for (int e = threadIdx.x; e < nout; e += kThreads) {
      const int tok = e / rows;
      const int n = int(blockIdx.x) * rows + (e - tok * rows);
      if (n < a.N) a.y[size_t(tok) * a.N + n] = __half_as_ushort(__float2half_rn(red_c[e]));
    }
  }
}

int mpad_log2_of(int M) {
  int l = 0;
  while ((1 << l) < M) ++l;
  return l;
}

int gl_per_cta_of(int kb_per_cta, int gs) { return (kb_per_cta * kColsPerBlock + gs - 1) / gs + 1; }

size_t gemv_smem_bytes(int M, int kb_per_cta, int gs, int rows16) {
  const size_t xs = size_t(kb_per_cta) * 16 * (size_t(1) << mpad_log2_of(M)) * 8;
  const size_t meta = size_t(gl_per_cta_of(kb_per_cta, gs)) * rows16 * 8 * 5;
  const size_t red = size_t(kWarps) * 512 * 4 + size_t(8) * 256 * 4;
  const size_t stage = (xs + meta + 15) / 16 * 16;
  return stage > red ? stage : red;
}

template <int NB, int GS, bool SYM>
cudaError_t launch_typed(const GemvArgs& a, int KS, size_t smem_bytes, cudaStream_t stream) {
  auto kern = gemv_kernel<NB, GS, SYM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_bytes));
  if (e != cudaSuccess) return e;
  if (KS > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  const int ntiles = ((a.N + kRowsPerBlock - 1) / kRowsPerBlock) * 8;
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

template <int NB, int GS>
cudaError_t launch_sym(const GemvArgs& a, bool sym, int KS, size_t smem, cudaStream_t stream) {
  return sym ? launch_typed<NB, GS, true>(a, KS, smem, stream)
             : launch_typed<NB, GS, false>(a, KS, smem, stream);
}

template <int NB>
cudaError_t launch_gs(const GemvArgs& a, int gs, bool sym, int KS, size_t smem, cudaStream_t stream) {
  switch (gs) {
    case 32: return launch_sym<NB, 32>(a, sym, KS, smem, stream);
    case 64: return launch_sym<NB, 64>(a, sym, KS, smem, stream);
    default: return launch_sym<NB, 128>(a, sym, KS, smem, stream);
  }
}

constexpr size_t kMaxGemvSmem = 100 * 1024;

// 64-column blocks per CTA of a K split; a whole number of groups so that the
// per-CTA group sums line up with the groups.
int kb_per_cta_of(const Layout& L, int ksplit) {
  const int unit = L.gsize == 128 ? 2 : 1;
  const int kbc = int((L.KB + ksplit - 1) / ksplit);
  return (kbc + unit - 1) / unit * unit;
}

}  // namespace

bool gemv_plan_ok(const Layout& L, int M, const GemvPlan& p) {
  if (p.rows16 != 2 && p.rows16 != 4 && p.rows16 != 8) return false;
  if (p.ksplit != 1 && p.ksplit != 2 && p.ksplit != 4 && p.ksplit != 8 && p.ksplit != 16) return false;
  return gemv_smem_bytes(M, kb_per_cta_of(L, p.ksplit), L.gsize, p.rows16) <= kMaxGemvSmem;
}

GemvPlan gemv_default_plan(const Layout& L, int M, const DeviceInfo& dev) {
  // Aim for about four resident CTAs per SM with at least a few 64-column
  // blocks per warp; prefer fewer K splits.
  const int64_t ntiles = L.NR * 8;
  const int64_t target = int64_t(dev.sm_count) * 4;
  GemvPlan best{8, 1};
  int64_t best_score = -1;
  for (int rt : {8, 4, 2}) {
    for (int ks : {1, 2, 4, 8, 16}) {
      GemvPlan p{rt, ks};
      if (!gemv_plan_ok(L, M, p)) continue;
      const int64_t ctas = (ntiles / rt) * ks;
      const int64_t kbc = kb_per_cta_of(L, ks);
      const int64_t per_warp = kbc / (kWarps / (rt / kTilesPerWarp));
      if (per_warp < 2 && !(ks == 1 && rt == 8)) continue;
      int64_t score = ctas >= target ? 4 * target - (ctas - target) / 4 : 4 * ctas;
      score = score * 64 - ks - (8 - rt);
      if (score > best_score) {
        best_score = score;
        best = p;
      }
    }
  }
  return best;
}

cudaError_t launch_gemv(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                        const GemvPlan& plan, uint32_t flags, cudaStream_t stream) {
  const BlobView B = view_of(L, blob);
  GemvArgs a;
  a.qweight = B.qweight;
  a.scales2 = reinterpret_cast<const uint32_t*>(B.scales);
  a.zeros = B.zeros;
  a.perm = B.perm;
  a.x = x;
  a.y = y;
  a.M = M;
  a.N = int(L.N);
  a.K = int(L.K);
  a.G = int(L.G);
  a.KB = int(L.KB);
  a.rows16 = plan.rows16;
  a.kb_per_cta = kb_per_cta_of(L, plan.ksplit);
  a.gl_per_cta = gl_per_cta_of(a.kb_per_cta, L.gsize);
  a.mpad_log2 = mpad_log2_of(M);
  a.flags = flags;
  const size_t smem = gemv_smem_bytes(M, a.kb_per_cta, L.gsize, plan.rows16);
  if (M > 8) return launch_gs<2>(a, L.gsize, L.sym, plan.ksplit, smem, stream);
  return launch_gs<1>(a, L.gsize, L.sym, plan.ksplit, smem, stream);
}

}  // namespace w4a16
