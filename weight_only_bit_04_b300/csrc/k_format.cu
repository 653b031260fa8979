// One-shot kernels around the hot path: round-to-nearest quantization,
// packing into the device blob, and bit-exact dequantization.
//
// Quantization follows "LLM Quantization: INT8, GPTQ, and AWQ Explained",
// section "What quantization actually does" (find the range, pick the scale,
// round to the nearest grid point, clamp) with the linear formula
// q = round(w / s) + z of "LLM Quantization: A Deep Dive into GPTQ, AWQ, and
// Post-Training Quantization", section "The Math of Quantization"; groups of
// input columns per "AWQ + GPTQ Quantization, in depth", section "What W4A16
// buys and why decoding gets faster".
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "internal.h"

namespace w4a16 {
namespace {

// ---------------------------------------------------------------------------
// Round-to-nearest quantization: one warp per (row, group).
// ---------------------------------------------------------------------------
// With an act scale (unfolded AWQ) the group's members are fp16(w * s[col]):
// the fp32 product of two fp16 values is exact and is rounded once.
__global__ void __launch_bounds__(256) quantize_rtn_kernel(Layout L, const uint16_t* __restrict__ w,
                                                           const int32_t* __restrict__ perm,
                                                           const uint16_t* __restrict__ ascale,
                                                           uint8_t* __restrict__ q,
                                                           uint16_t* __restrict__ scales,
                                                           uint8_t* __restrict__ zeros) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (item >= L.N * L.G) return;
  const int64_t n = item / L.G;
  const int64_t t = item - n * L.G;
  const int gs = L.gsize;
  const int per_lane = gs / 32;  // 1, 2 or 4 members per lane

  int64_t col[4];
  float v[4];
  float mn = INFINITY, mx = -INFINITY, amax = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < per_lane) {
      const int64_t p = t * gs + i * 32 + lane;  // position in group-sorted order
      col[i] = perm ? perm[p] : p;
      v[i] = __half2float(__ushort_as_half(w[n * L.K + col[i]]));
      if (ascale) v[i] = __half2float(__float2half_rn(v[i] * __half2float(__ushort_as_half(ascale[col[i]]))));
      mn = fminf(mn, v[i]);
      mx = fmaxf(mx, v[i]);
      amax = fmaxf(amax, fabsf(v[i]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  // fp64 from here on; every fp16 value and difference of two is exact in fp64.
  // b-bit codes, qmax = 2^b - 1. Symmetric: 3, 4 bits s = 2a/qmax, z = 2^(b-1); 8 bits
  // the int8 absmax code, s = a/127, codes clamp(rint(w/s), -127, 127) + 128.
  const double qmax = double((1 << L.bits) - 1);
  const bool sym8 = L.sym && L.bits == 8;
  const double range = L.sym ? (sym8 ? double(amax) / 127.0 : 2.0 * double(amax) / qmax) : (double(mx) - double(mn)) / qmax;
  __half s_h = __double2half(range);  // round to nearest even
  if (__half2float(s_h) == 0.0f) s_h = __float2half(1.0f);
  const double s = double(__half2float(s_h));
  double z;
  if (L.sym) {
    z = double(1 << (L.bits - 1));
  } else {
    z = rint(-double(mn) / s);
    z = fmin(fmax(z, 0.0), qmax);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (i < per_lane) {
      double c;
      if (sym8) {
        c = fmin(fmax(rint(double(v[i]) / s), -127.0), 127.0) + 128.0;
      } else {
        c = rint(double(v[i]) / s) + z;
        c = fmin(fmax(c, 0.0), qmax);
      }
      q[n * L.K + col[i]] = uint8_t(c);
    }
  }
  if (lane == 0) {
    scales[n * L.G + t] = __half_as_ushort(s_h);
    if (zeros) zeros[n * L.G + t] = uint8_t(z);
  }
}

// ---------------------------------------------------------------------------
// Packing: one thread per 32-bit word of the qweight tiles.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pack_qweight_kernel(Layout L, const uint8_t* __restrict__ q,
                                                           const int32_t* __restrict__ perm,
                                                           uint32_t* __restrict__ qweight) {
  const int tile_words = kTileWords * L.bits / 4;
  const int64_t wi = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (wi >= L.NR * L.KB * tile_words) return;
  const int64_t tile = wi / tile_words;
  const int within = int(wi - tile * tile_words);
  const int64_t R = tile / L.KB;
  const int64_t b = tile - R * L.KB;
  uint32_t word = 0;
  if (L.bits == 4) {
    const int r16 = within >> 7;
    const int lane = (within >> 2) & 31;
    const int j = within & 3;
    const int g = lane >> 2, t = lane & 3;
    const int64_t n0 = R * kRowsPerBlock + r16 * 16 + g;
    const int64_t p0 = b * kColsPerBlock + j * 16 + 4 * t;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int64_t p = p0 + kk;
      if (p >= L.K) continue;
      const int64_t c = perm ? perm[p] : p;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t n = n0 + 8 * h;
        if (n < L.N) word |= uint32_t(q[n * L.K + c] & 0xF) << (4 * nibble_index(kk, h));
      }
    }
  } else {
    // word (r16, p, lane, jj, h): row r16*16 + g + 8h, columns 16j + 4t + kk
    // in byte kk, j = 2p + jj
    const int r16 = within >> 8;
    const int lane = (within >> 2) & 31;
    const int j = 2 * ((within >> 7) & 1) + ((within >> 1) & 1);
    const int h = within & 1;
    const int g = lane >> 2, t = lane & 3;
    const int64_t n = R * kRowsPerBlock + r16 * 16 + g + 8 * h;
    const int64_t p0 = b * kColsPerBlock + j * 16 + 4 * t;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int64_t p = p0 + kk;
      if (p >= L.K || n >= L.N) continue;
      const int64_t c = perm ? perm[p] : p;
      word |= uint32_t(q[n * L.K + c]) << (8 * kk);
    }
  }
  qweight[wi] = word;
}

// 3-bit codes: one thread per (tile, 16-row tile, lane) composes that lane's
// three words (the sixteenth code of a step is spread over three words).
__global__ void __launch_bounds__(256) pack_qweight3_kernel(Layout L, const uint8_t* __restrict__ q,
                                                            const int32_t* __restrict__ perm,
                                                            uint32_t* __restrict__ qweight) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= L.NR * L.KB * 256) return;
  const int64_t tile = i >> 8;
  const int r16 = int((i >> 5) & 7), lane = int(i & 31);
  const int64_t R = tile / L.KB;
  const int64_t b = tile - R * L.KB;
  const int g = lane >> 2, t = lane & 3;
  uint32_t w[3] = {0u, 0u, 0u};
  for (int j = 0; j < 4; ++j)
    for (int a = 0; a < 4; ++a) {
      int wi, sh;
      w3_field(j, a, &wi, &sh);
      const int64_t n = R * kRowsPerBlock + r16 * 16 + g + 8 * (a & 1);
      for (int h2 = 0; h2 < 2; ++h2) {
        const int64_t p = b * kColsPerBlock + 16 * j + 4 * t + 2 * (a >> 1) + h2;
        if (p >= L.K || n >= L.N) continue;
        const uint32_t code = q[n * L.K + (perm ? perm[p] : p)] & 7u;
        if (wi >= 0) {
          w[wi] |= code << (sh + 16 * h2);
        } else {
          for (int bt = 0; bt < 3; ++bt) w[bt] |= ((code >> bt) & 1u) << (15 + 16 * h2);
        }
      }
    }
  uint32_t* tw = qweight + tile * 768;
  for (int wi = 0; wi < 3; ++wi) tw[w3_word_index(r16, lane, wi)] = w[wi];
}

// One thread per (row block, group, 16-row tile, lane group): a scale pair and
// the zero points of the two rows (one byte of two nibbles, or two bytes),
// stored at meta_index.
__global__ void __launch_bounds__(256) pack_meta_kernel(Layout L, const uint16_t* __restrict__ scales,
                                                        const uint8_t* __restrict__ zeros,
                                                        uint32_t* __restrict__ s_out,
                                                        uint8_t* __restrict__ z_out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= L.NR * L.G * 64) return;
  const int g = int(i & 7);
  const int r16 = int((i >> 3) & 7);
  const int64_t rg = i >> 6;  // R * G + gi
  const int64_t R = rg / L.G;
  const int64_t gi = rg - R * L.G;
  const int64_t n0 = R * kRowsPerBlock + r16 * 16 + g;
  const int64_t n1 = n0 + 8;
  const int64_t mi = meta_index(R, gi, r16, g, L.G);
  const uint32_t s0 = n0 < L.N ? scales[n0 * L.G + gi] : 0u;
  const uint32_t s1 = n1 < L.N ? scales[n1 * L.G + gi] : 0u;
  s_out[mi] = s0 | (s1 << 16);
  if (z_out) {
    if (L.bits != 8) {
      const uint32_t z0 = n0 < L.N ? (zeros[n0 * L.G + gi] & 0xF) : 0u;
      const uint32_t z1 = n1 < L.N ? (zeros[n1 * L.G + gi] & 0xF) : 0u;
      z_out[mi] = uint8_t(z0 | (z1 << 4));
    } else {
      z_out[2 * mi] = n0 < L.N ? zeros[n0 * L.G + gi] : uint8_t(0);
      z_out[2 * mi + 1] = n1 < L.N ? zeros[n1 * L.G + gi] : uint8_t(0);
    }
  }
}

// The act scale in packed column order: out[p] = ascale[perm[p]].
__global__ void __launch_bounds__(256) pack_act_scale_kernel(Layout L, const uint16_t* __restrict__ ascale,
                                                             const int32_t* __restrict__ perm,
                                                             uint16_t* __restrict__ out) {
  const int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p >= L.K) return;
  out[p] = ascale[perm ? perm[p] : p];
}

// ---------------------------------------------------------------------------
// Dequantization: one thread per packed word, w_hat = fp16_rne((q - z) * s).
// (1024 + q) - (1024 + z) is exact in fp16, the product is rounded once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dequant_kernel(Layout L, BlobView B, uint16_t* __restrict__ out) {
  const int tile_words = kTileWords * L.bits / 4;
  const int64_t wi = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (wi >= L.NR * L.KB * tile_words) return;
  const int64_t tile = wi / tile_words;
  const int within = int(wi - tile * tile_words);
  const int64_t R = tile / L.KB;
  const int64_t b = tile - R * L.KB;
  const bool b8 = L.bits == 8;
  const int r16 = b8 ? within >> 8 : within >> 7;
  const int lane = (within >> 2) & 31;
  const int j = b8 ? 2 * ((within >> 7) & 1) + ((within >> 1) & 1) : within & 3;
  const int hw = b8 ? within & 1 : 0;  // 8-bit: the word's row (g or g+8)
  const int g = lane >> 2, t = lane & 3;
  const int64_t n0 = R * kRowsPerBlock + r16 * 16 + g;
  const int64_t p0 = b * kColsPerBlock + j * 16 + 4 * t;
  const uint32_t word = B.qweight[wi];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const int64_t p = p0 + kk;
    if (p >= L.K) continue;
    const int64_t gi = p / L.gsize;
    const int64_t mi = meta_index(R, gi, r16, g, L.G);
    const int64_t c = B.perm ? B.perm[p] : p;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (b8 && hh != hw) continue;
      const int h = hh;
      const int64_t n = n0 + 8 * h;
      if (n >= L.N) continue;
      uint32_t code, z;
      if (b8) {
        code = (word >> (8 * kk)) & 0xFF;
        z = B.zeros ? B.zeros[2 * mi + h] : 128u;
      } else {
        code = (word >> (4 * nibble_index(kk, h))) & 0xF;
        z = B.zeros ? ((B.zeros[mi] >> (4 * h)) & 0xF) : 8u;
      }
      const __half s = __ushort_as_half(B.scales[2 * mi + h]);
      const __half d = __hsub(__ushort_as_half(uint16_t(0x6400u | code)),
                              __ushort_as_half(uint16_t(0x6400u | z)));
      out[n * L.K + c] = __half_as_ushort(__hmul(d, s));
    }
  }
}

// 3-bit codes: one thread per (tile, 16-row tile, lane), as in the packer.
__global__ void __launch_bounds__(256) dequant3_kernel(Layout L, BlobView B, uint16_t* __restrict__ out) {
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= L.NR * L.KB * 256) return;
  const int64_t tile = i >> 8;
  const int r16 = int((i >> 5) & 7), lane = int(i & 31);
  const int64_t R = tile / L.KB;
  const int64_t b = tile - R * L.KB;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t* tw = B.qweight + tile * 768;
  uint32_t w[3];
  for (int wi = 0; wi < 3; ++wi) w[wi] = tw[w3_word_index(r16, lane, wi)];
  for (int j = 0; j < 4; ++j)
    for (int a = 0; a < 4; ++a) {
      int wi, sh;
      w3_field(j, a, &wi, &sh);
      const int h = a & 1;
      const int64_t n = R * kRowsPerBlock + r16 * 16 + g + 8 * h;
      for (int h2 = 0; h2 < 2; ++h2) {
        const int64_t p = b * kColsPerBlock + 16 * j + 4 * t + 2 * (a >> 1) + h2;
        if (p >= L.K || n >= L.N) continue;
        uint32_t code = 0;
        if (wi >= 0) {
          code = (w[wi] >> (sh + 16 * h2)) & 7u;
        } else {
          for (int bt = 0; bt < 3; ++bt) code |= ((w[bt] >> (15 + 16 * h2)) & 1u) << bt;
        }
        const int64_t gi = p / L.gsize;
        const int64_t mi = meta_index(R, gi, r16, g, L.G);
        const uint32_t z = B.zeros ? ((B.zeros[mi] >> (4 * h)) & 0xF) : 4u;
        const __half s = __ushort_as_half(B.scales[2 * mi + h]);
        const __half d = __hsub(__ushort_as_half(uint16_t(0x6400u | code)),
                                __ushort_as_half(uint16_t(0x6400u | z)));
        out[n * L.K + (B.perm ? B.perm[p] : p)] = __half_as_ushort(__hmul(d, s));
      }
    }
}

inline unsigned blocks_for(int64_t threads, int per_block) {
  return unsigned((threads + per_block - 1) / per_block);
}

}  // namespace

cudaError_t launch_quantize_rtn(const Layout& L, const uint16_t* w, const int32_t* perm_dev,
                                const uint16_t* ascale, uint8_t* q, uint16_t* scales, uint8_t* zeros,
                                cudaStream_t stream) {
  const int64_t threads = L.N * L.G * 32;
  quantize_rtn_kernel<<<blocks_for(threads, 256), 256, 0, stream>>>(L, w, perm_dev, ascale, q, scales, zeros);
  return cudaGetLastError();
}

cudaError_t launch_pack(const Layout& L, const uint8_t* q, const uint16_t* scales,
                        const uint8_t* zeros, const uint16_t* ascale, void* blob, cudaStream_t stream) {
  char* b = static_cast<char*>(blob);
  const int32_t* perm = L.act ? reinterpret_cast<const int32_t*>(b + L.p_off) : nullptr;
  if (L.bits == 3) {
    pack_qweight3_kernel<<<blocks_for(L.NR * L.KB * 256, 256), 256, 0, stream>>>(
        L, q, perm, reinterpret_cast<uint32_t*>(b + L.q_off));
  } else {
    const int64_t words = L.NR * L.KB * kTileWords * L.bits / 4;
    pack_qweight_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(
        L, q, perm, reinterpret_cast<uint32_t*>(b + L.q_off));
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t metas = L.NR * L.G * 64;
  pack_meta_kernel<<<blocks_for(metas, 256), 256, 0, stream>>>(
      L, scales, L.sym ? nullptr : zeros, reinterpret_cast<uint32_t*>(b + L.s_off),
      L.sym ? nullptr : reinterpret_cast<uint8_t*>(b + L.z_off));
  e = cudaGetLastError();
  if (e != cudaSuccess || !L.awq) return e;
  pack_act_scale_kernel<<<blocks_for(L.K, 256), 256, 0, stream>>>(L, ascale, perm,
                                                                  reinterpret_cast<uint16_t*>(b + L.a_off));
  return cudaGetLastError();
}

cudaError_t launch_dequant(const Layout& L, const void* blob, uint16_t* w_out, cudaStream_t stream) {
  if (L.bits == 3) {
    dequant3_kernel<<<blocks_for(L.NR * L.KB * 256, 256), 256, 0, stream>>>(L, view_of(L, blob), w_out);
    return cudaGetLastError();
  }
  const int64_t words = L.NR * L.KB * kTileWords * L.bits / 4;
  dequant_kernel<<<blocks_for(words, 256), 256, 0, stream>>>(L, view_of(L, blob), w_out);
  return cudaGetLastError();
}

}  // namespace w4a16
