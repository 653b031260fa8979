// Small inline-PTX helpers shared by the sm_103a kernels of this library.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace w4a16 {

// (a & b) | c in one LOP3.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// x / s for one fp16 activation and its act scale: the fp32 quotient of two
// fp16 values, correctly rounded, rounds to the same fp16 as the exact
// quotient (24 >= 2 * 11 + 2 bits, so the double rounding is innocuous).
__device__ __forceinline__ uint16_t div_act(uint16_t xv, uint16_t sv) {
  return __half_as_ushort(
      __float2half_rn(__fdiv_rn(__half2float(__ushort_as_half(xv)), __half2float(__ushort_as_half(sv)))));
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// fp16 bit patterns used by the nibble expansion.
constexpr uint32_t kMagic1024x2 = 0x64006400u;   // 1024.0 in both halves
constexpr uint32_t kSixteenthx2 = 0x2C002C00u;   // 1/16 in both halves
constexpr uint32_t kLoMask = 0x000F000Fu;        // nibbles 0 and 4
constexpr uint32_t kHiMask = 0x00F000F0u;        // nibbles 1 and 5

// Operand constants for zero point z of the row pair (g, g+8):
//   za = (1024 + z_g) in both halves       -> (1024 + q) - za      = q - z_g
//   zb = -(64 + z_{g+8}) in both halves    -> (1024 + 16 q)/16 + zb = q - z_{g+8}
__device__ __forceinline__ uint32_t zero_lo_const(uint32_t z) { return (0x6400u | z) * 0x00010001u; }
__device__ __forceinline__ uint32_t zero_hi_const(uint32_t z) { return (0xD400u | (z << 4)) * 0x00010001u; }

// Expand one packed word into the four (q - z) half2 registers of a 16x16 tile
// fragment: a[0] = row g, columns {4t, 4t+1}; a[1] = row g+8, same columns;
// a[2] = row g, columns {4t+2, 4t+3}; a[3] = row g+8, same columns. Exact.
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t za, uint32_t zb, uint32_t a[4]) {
  uint32_t lo = lop3_and_or(w, kLoMask, kMagic1024x2);
  uint32_t hi = lop3_and_or(w, kHiMask, kMagic1024x2);
  a[0] = hsub2_u32(lo, za);
  a[1] = hfma2_u32(hi, kSixteenthx2, zb);
  uint32_t w8 = w >> 8;
  lo = lop3_and_or(w8, kLoMask, kMagic1024x2);
  hi = lop3_and_or(w8, kHiMask, kMagic1024x2);
  a[2] = hsub2_u32(lo, za);
  a[3] = hfma2_u32(hi, kSixteenthx2, zb);
}

// D = A . B + C, m16n8k16, fp16 inputs, fp32 accumulation.
__device__ __forceinline__ void mma_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                          const float c[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

// Read-only 16-byte global load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream_u4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_nc_u8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// 16-byte asynchronous global -> shared copy (L2 only) and its completion.
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait until the previous kernel's writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Thread-block cluster helpers.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ float ld_dsmem_f32(const float* local_smem_ptr, uint32_t rank) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(local_smem_ptr));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

}  // namespace w4a16
