// The decode stream: one persistent launch computes y_i = x_i . W_hat_i^T for
// a list of layers (a decoder's linears for one token step), 1 <= M <= 16.
//
// At batch one every packed weight is read once for about two flops ("AWQ +
// GPTQ Quantization, in depth", section "What W4A16 buys and why decoding gets
// faster"), so a token step is a stream of weight bytes, and the time lost to
// launch ramp-up, drain and dependency waits between layers is lost
// bandwidth. The launch is organised so that the weight stream never waits:
//
//  * One thread block per SM. Every layer is cut into row groups of 32 rows;
//    block b owns a contiguous run of them (the full K of each row group),
//    with the block positions rotated from layer to layer by the number of
//    row groups dealt so far, so that every SM streams the same bytes over
//    the step within about 1 %.
//  * A producer warp streams the block's units -- codes, scales and zero
//    points of one row group over 64 or 128 columns -- layer after layer into
//    a ring of shared-memory slots of up to 32 KiB of codes each. The codes
//    of a slot come by TMA (3-D tensor maps over the blob, no multicast) in
//    one copy, or a few at a row group's end: measured on B300, a stream of
//    8 KiB copies tops out near 4 TB/s and one of 16 KiB copies near
//    6.8 TB/s, so copies must be large. The slot's scales and zero points
//    (64 and 16 bytes per group and row group) come by cp.async from the
//    lanes of a second producer warp (the metadata warp), which keeps small
//    copies off the TMA unit and their instructions off the sub-partition
//    of the warp issuing the codes. Weights never depend on earlier layers,
//    so the producers run ahead across dependency waits for as long as the
//    ring has room.
//  * Eight consumer warps share every slot, one, two or four units each
//    (stream_upw: the most that keep a slot within 32 KiB of codes), all
//    loaded before any is multiplied. Per unit a warp expands the codes into
//    m16n8k16 fragments in registers and multiplies them on the tensor cores
//    with the activations (tokens in the n dimension), as the single-layer
//    product does (gemv_impl.cuh, compute_unit). Each warp keeps one partial
//    sum per row group and writes it to shared memory.
//  * A finishing warp adds a row group's partial sums in warp order
//    (deterministic), releases the partial buffer to the consumers, rounds
//    to fp16 and writes y. When a later layer waits for this one, it then
//    fences and counts the layer as done on a device counter (one per layer
//    slice, 128-byte lines).
//  * A dependency warp walks the layers ahead of the consumers: for a layer
//    that reads earlier layers' outputs it polls their counters (acquire
//    loads) until every block has finished them. The layer's activations
//    are staged in shared memory together with each group's activation sum
//    when they fit (otherwise the consumers read them through L1 after an L1
//    prefetch and get the group sums from the tensor cores): by this warp,
//    ahead of the consumers, when no dependency was just acquired; by the
//    eight consumer warps together, which would otherwise idle, right after
//    one was. The warp then publishes the layer as ready.
//
// Every wait is bounded (1 s by the global timer unless the host set
// another limit, w4a16_set_wait_limit_ns) and also gives up when
// another block has raised the abort flag; a wait that times out is counted
// (w4a16_pipeline_timeouts) and raises the flag, and every role then returns,
// the producer after its copies in flight have landed. Outputs are undefined
// after an abort.
#pragma once

#include "gemv_impl.cuh"
#include "stream_geom.h"

namespace w4a16 {
namespace {

template <int BITS, int GS>
struct SGeo {
  static constexpr int UB = stream_ub(GS);
  static constexpr int GU = stream_gu(GS);
  static constexpr int CB = stream_cb(BITS);
  static constexpr int ZB = stream_zb(BITS);
  static constexpr int kUnitCode = stream_unit_code(BITS, GS);
  static constexpr int UPW = stream_upw(BITS, GS);
  static constexpr int CU = stream_cu(BITS, GS);
  static constexpr int kScaleOff = stream_scale_off(BITS, GS);
  static constexpr int kZeroOff = stream_zero_off(BITS, GS);
  static constexpr int kSlot = stream_slot_bytes(BITS, GS);
  static constexpr int S = stream_slots(BITS, GS);
  static constexpr int kScaleChunks = GU * 4;       // 16-byte pieces of a unit's scales
  static constexpr int kZeroChunks = GU * ZB / 16;  // and of its zero points
  static_assert(Unit<GS>::kBlocks == UB && Unit<GS>::kGroups == GU, "stream units are the GEMV units");
  static_assert((CU & (CU - 1)) == 0 && CU <= 32, "codes copies are power-of-two boxes of at most 32 units");
};

// log2 of a power of two up to 32
__host__ __device__ constexpr int ilog2(int v) {
  return v >= 32 ? 5 : v >= 16 ? 4 : v >= 8 ? 3 : v >= 4 ? 2 : v >= 2 ? 1 : 0;
}

// This block's share of one layer slice.
struct Span {
  int rg0;  // first row group (of the layer) owned by this block
  int n;    // row groups owned
  int NU;   // units per row group
  int T;    // units owned (n * NU)
};

// What the consumer warps need of layer j, written by the dependency warp
// into shared memory (record j % stream_part_depth) before it publishes the layer.
struct alignas(16) LayerRec {
  const uint16_t* x;  // activations in global memory
  int K;
  int T;     // units this block owns
  int NU;    // units per row group
  int xsel;  // byte offset of the staged-activation buffer, | kConsumersStage
  int pad[2];
};
static_assert(sizeof(LayerRec) == kStreamRecBytes, "layer record size");

__device__ __forceinline__ Span span_of(const StreamJob& J, int P, int b, int UB) {
  int p = b - J.rot;
  if (p < 0) p += P;
  // 32-bit: a slice has at most stream_max_rg(MP) row groups per block
  const int lo = int(uint32_t(p) * uint32_t(J.n_rg) / uint32_t(P));
  const int hi = int(uint32_t(p + 1) * uint32_t(J.n_rg) / uint32_t(P));
  Span s;
  s.rg0 = J.rg_first + lo;
  s.n = hi - lo;
  s.NU = J.KB / UB;
  s.T = s.n * s.NU;
  return s;
}

__device__ __forceinline__ StreamJob load_job(const StreamJob* jobs, int j) {
  StreamJob J;
  const uint4* src = reinterpret_cast<const uint4*>(jobs + j);
  uint4* dst = reinterpret_cast<uint4*>(&J);
#pragma unroll
  for (int i = 0; i < int(sizeof(StreamJob) / 16); ++i) dst[i] = __ldg(src + i);
  return J;
}

// Bounded waits. A wait returns kWaitOk when its condition holds, kWaitTimeout
// when its time limit ran out (it then raises the abort flag), kWaitAbort when
// another thread raised the flag first. Warps agree on the outcome with
// warp_outcome, which counts a timeout once per warp.
constexpr int kWaitOk = 0, kWaitTimeout = 1, kWaitAbort = 2;
// A wait looks at another block's abort flag (a global load, one L2 round
// trip during which it would not see its own condition complete) only once it
// has lasted this long; ordinary waits never leave the SM.
constexpr uint64_t kAbortPollNs = 20000;
struct Guard {
  unsigned int* abort_flag;
  uint64_t limit;  // ns
  uint64_t t0;
  uint32_t spins;
  __device__ __forceinline__ void start() {
    t0 = 0;
    spins = 0;
  }
  // kWaitOk: keep waiting. The clock is read on the first spin and then
  // every eighth (a spin is at least an L2 round trip or an mbarrier test).
  __device__ __forceinline__ int check() {
    if ((++spins & 7u) != 1u) return kWaitOk;
    const uint64_t now = global_timer_ns();
    if (t0 == 0) {
      t0 = now;
      return kWaitOk;
    }
    const uint64_t waited = now - t0;
    if (waited > kAbortPollNs && ld_relaxed_gpu_u32(abort_flag) != 0) return kWaitAbort;
    if (waited > limit) {
      atomicExch(abort_flag, 1u);
      return kWaitTimeout;
    }
    return kWaitOk;
  }
};

__device__ __forceinline__ int wait_mbar(uint32_t bar, uint32_t parity, Guard& gd) {
  gd.start();
  while (!mbar_try_wait(bar, parity)) {
    const int st = gd.check();
    if (st != kWaitOk) return st;
  }
  return kWaitOk;
}
// Whole-warp outcome of a wait every lane took part in: true = go on.
__device__ __forceinline__ bool warp_outcome(int st) {
  const bool timed = __any_sync(0xffffffffu, st == kWaitTimeout);
  const bool bad = __any_sync(0xffffffffu, st != kWaitOk);
  if (timed && (threadIdx.x & 31) == 0) atomicAdd(&g_gemv_timeouts, 1u);
  return !bad;
}
// Whole-warp wait for layer j's phase of a set of D per-layer barriers
// (barrier j % D, parity (j / D) & 1); layers below 0 are complete.
template <int D = 2>
__device__ __forceinline__ bool wait_layer(uint32_t bar0, int j, Guard& gd) {
  if (j < 0) return true;
  return warp_outcome(wait_mbar(bar0 + 8 * (j % D), uint32_t(j / D) & 1u, gd));
}

// cp.async of 16 bytes, and the arrival on an mbarrier once this thread's
// cp.async copies so far have landed (.noinc: the arrival is one of the
// barrier's expected arrivals).
__device__ __forceinline__ void cp_async_16_cg(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

constexpr int kConsumersStage = 1 << 30;

// Land the activations of a layer (M rows of K) in a staged buffer and add
// each group of each row (fixed order per group). `tid` / `nt`: this thread's
// index among the `nt` threads that share the work; the caller makes the
// copies visible to all of them (cp.async.wait_all + barrier) between the two.
template <int GS, int MP>
__device__ __forceinline__ void stage_copy(const uint16_t* x, int K, int M, uint16_t* xs, int tid, int nt) {
  const int64_t stride = stream_x_stride(K, M);
  const int cpr = K / 8, total = M * cpr;
  int tok = tid / cpr, kc = tid - tok * cpr;  // chunk (tok, kc) advanced by nt without dividing
  for (int q = tid; q < total; q += nt) {
    cp_async_16_cg(smem_addr(xs + tok * stride + kc * 8), x + size_t(tok) * K + kc * 8);
    kc += nt;
    while (kc >= cpr) {
      kc -= cpr;
      ++tok;
    }
  }
}
// Sum of the eight halves of a 16-byte chunk, in a fixed order.
__device__ __forceinline__ float chunk_sum(const uint4 v) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
  const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&v.z));
  const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&v.w));
  return ((a.x + a.y) + (b.x + b.y)) + ((c.x + c.y) + (d.x + d.y));
}
// Group sums: chunk c of a group is added by lane c of an aligned run of
// GS / 8 lanes, and the run adds its chunk sums as a butterfly (every lane
// gets the same value). The result does not depend on how many threads share
// the work, so the dependency warp alone and the consumer warps together
// produce identical sums.
template <int GS, int MP, int U>  // U: rounds in flight at once
__device__ __forceinline__ void stage_sums(int K, int M, const uint16_t* xs, float* xsum, int tid, int nt) {
  constexpr int CPG = GS / 8;  // 16-byte chunks per group
  const int64_t stride = stream_x_stride(K, M);
  const int cpr = K / 8, total = M * cpr;
  const int lane = tid & 31;
  int tok = tid / cpr, kc = tid - tok * cpr;  // this thread's chunk, advanced by nt without dividing
  for (int q0 = 0; q0 < total; q0 += U * nt) {  // the same trip count for every thread (shuffles below)
    float v[U];
    int tk[U], kk[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      tk[u] = tok;
      kk[u] = kc;
      // a run of CPG lanes is valid or not as a whole: total and nt are multiples of CPG
      v[u] = q0 + u * nt + tid < total ? chunk_sum(*reinterpret_cast<const uint4*>(xs + tok * stride + kc * 8)) : 0.f;
      kc += nt;
      while (kc >= cpr) {
        kc -= cpr;
        ++tok;
      }
    }
#pragma unroll
    for (int o = 1; o < CPG; o <<= 1)
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] += __shfl_xor_sync(0xffffffffu, v[u], o);
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (q0 + u * nt + tid < total && (lane & (CPG - 1)) == 0 && W4A16_CHECK(tk[u] < M && kk[u] < cpr, 0x203u))
        xsum[(kk[u] / CPG) * MP + tk[u]] = v[u];
  }
}

// NU units of one warp multiplied together, 16-column step by 16-column step
// (compute_unit's arithmetic with the group sums from the caller): NU times
// the independent MMA chains between dependent operations. xo[u]: column of
// unit u's first activation; xsg[u]: its group sums.
template <int NU, int NB, int GS, bool SYM, int BITS, bool ONE>
__device__ __forceinline__ void compute_units(const UnitRegs<GS, BITS> (&r)[NU], const uint16_t* xl0,
                                              const uint16_t* xl1, const int (&xo)[NU],
                                              const float (&xsg)[NU][Unit<GS>::kGroups][NB][2],
                                              float tot[kTilesPerWarp][NB][4]) {
  using U = Unit<GS>;
  constexpr bool SPLIT = BITS == 4;  // even and odd steps in separate accumulators
  constexpr int NS = SPLIT ? 2 : 1;
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  float acc[NU][NS][kTilesPerWarp][NB][4];
#pragma unroll
  for (int bb = 0; bb < U::kBlocks; ++bb) {
    uint2 bx[NU][4][NB];
#pragma unroll
    for (int u = 0; u < NU; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int off = xo[u] + bb * 64 + j * 16;
        bx[u][j][0] = ld_x<kXShared>(xl0 + off);
        if (NB > 1) bx[u][j][NB - 1] = ld_x<kXShared>(xl1 + off);
      }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ph = SPLIT ? (j & 1) : 0;
      const bool fresh = SPLIT ? ((GS == 32) ? true : (j < 2 && bb == 0))
                               : ((GS == 32) ? (j == 0 || j == 2) : (j == 0 && bb == 0));
#pragma unroll
      for (int u = 0; u < NU; ++u)
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt) {
          uint32_t af[4];
          extract_step<BITS>(r[u].w[bb], tt, j, af);
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
            mma_16816(acc[u][ph][tt][nb], af, bx[u][j][nb].x, bx[u][j][nb].y, fresh ? zero4 : acc[u][ph][tt][nb]);
        }
      const bool group_end = (GS == 32) ? (j == 1 || j == 3) : (j == 3 && bb == U::kBlocks - 1);
      if (group_end) {
        // tot += s * (2^k acc - z xs) per row, as in compute_unit
        const int gg = (GS == 32) ? (j >> 1) : 0;
        constexpr float kA = 16777216.f;
        constexpr float kB = BITS == 4 ? 1048576.f : BITS == 3 ? 2097152.f : 16777216.f;
        constexpr float kSymZero = float(1 << (BITS - 1));
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          float xs[NB][2], x23[NB][2];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              xs[nb][e] = xsg[u][gg][nb][e];
              x23[nb][e] = SYM ? -kSymZero * xs[nb][e] : xs[nb][e] * 8388608.f;
            }
#pragma unroll
          for (int tt = 0; tt < kTilesPerWarp; ++tt) {
            const float2 sf = __half22float2(*reinterpret_cast<const __half2*>(&r[u].s[gg][tt]));
            const uint32_t zr = r[u].z[gg][tt];
            const float fg = __uint_as_float(0x4B000000u | (BITS != 8 ? (zr & 0xFu) : (zr & 0xFFu)));
            const float fh = __uint_as_float(0x4B000000u | (BITS != 8 ? ((zr >> 4) & 0xFu) : ((zr >> 8) & 0xFFu)));
#pragma unroll
            for (int nb = 0; nb < NB; ++nb)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                if (ONE && (nb > 0 || e > 0)) continue;
                float a_g = acc[u][0][tt][nb][e], a_h = acc[u][0][tt][nb][e + 2];
                if (SPLIT) {
                  a_g += acc[u][NS - 1][tt][nb][e];
                  a_h += acc[u][NS - 1][tt][nb][e + 2];
                }
                const float zg = SYM ? x23[nb][e] : fmaf(fg, -xs[nb][e], x23[nb][e]);
                const float zh = SYM ? x23[nb][e] : fmaf(fh, -xs[nb][e], x23[nb][e]);
                tot[tt][nb][e] = fmaf(sf.x, fmaf(a_g, kA, zg), tot[tt][nb][e]);
                tot[tt][nb][e + 2] = fmaf(sf.y, fmaf(a_h, kB, zh), tot[tt][nb][e + 2]);
              }
          }
        }
      }
    }
  }
}

template <int MP, int GS, bool SYM, int BITS, bool XS>
__global__ void __launch_bounds__(kStreamThreads, 1) decode_stream_kernel(const StreamLaunch c) {
  using SG = SGeo<BITS, GS>;
  constexpr int NB = MP > 8 ? 2 : 1;
  constexpr int NW = kStreamConsumers;
  constexpr int S = SG::S;
  constexpr int CU = SG::CU;
  constexpr int CS = kStreamCounterStride;
  constexpr int RGMAX = stream_max_rg(MP);
  // ring, barriers, records and partial-sum buffers within the block's shared memory
  static_assert(stream_x_off(BITS, GS, MP) <= kStreamSmem, "the stream's shared-memory layout does not fit");
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t ring = smem_addr(smem);
  // mbarriers: full[S], empty[S] (the ring); per layer slot (layer j uses
  // slot j % PD, PD = stream_part_depth(MP)): cdone (the consumer warps have
  // written layer j's partial sums, in partial buffer j % PD), rdy (layer j's
  // activations and record j % PD may be read), fdone (the finishing warp has
  // read layer j's partial sums); then the consumer warps' staging barrier.
  // Layer j's phase is phase (j / PD) & 1 of its slot's barrier. It is never
  // ambiguous: a waiter on a set has seen layer j - PD's phase of the same
  // barrier before it waits for layer j's, and no barrier completes layer
  // j + PD's phase before every waiter has seen layer j's:
  //  * rdy: consumers wait in layer order; the dependency warp publishes
  //    j + PD only after cdone(j), i.e. after every consumer warp saw rdy(j);
  //  * cdone: the finishing warp waits in layer order; the dependency warp
  //    waits for cdone(j - PD) before publishing j, and for cdone(l) of a
  //    staged buffer's last reader l in (j - 1 - PD, j) (it has seen
  //    cdone(l - PD) one publication earlier). The consumers complete
  //    cdone(j + PD) only after rdy(j + PD), which the dependency warp
  //    publishes after fdone(j) (the finishing warp saw cdone(j)) and once it
  //    is past every such wait;
  //  * fdone: the dependency warp waits in layer order (fdone(j - PD) before
  //    publishing j); the finishing warp completes fdone(j + PD) only after
  //    cdone(j + PD), after rdy(j + PD), published after fdone(j) was seen.
  const uint32_t full0 = ring + stream_bar_off(BITS, GS);
  const uint32_t empty0 = full0 + S * 8;
  constexpr int PD = stream_part_depth(MP);  // partial buffers; cdone and fdone barriers
  const uint32_t cdone0 = empty0 + S * 8;   // 4 words
  const uint32_t rdy0 = cdone0 + 32;        // 4 words
  const uint32_t fdone0 = rdy0 + 32;        // 4 words
  const uint32_t stg = fdone0 + 32;         // the consumer warps' staging barrier
  float* part = reinterpret_cast<float*>(smem + stream_part_off(BITS, GS));  // [2][RGMAX][NW][32 rows][MP]
  unsigned char* xbase = smem + stream_x_off(BITS, GS, MP);  // staged-activation buffers (XS)
  LayerRec* rec = reinterpret_cast<LayerRec*>(smem + stream_rec_off(BITS, GS));  // per layer slot

  const int tid = int(threadIdx.x);
  const int warp = tid >> 5, lane = tid & 31;
  const int P = int(gridDim.x), b = int(blockIdx.x);
  const int M = c.M, nj = c.n_jobs;
  unsigned int* done = c.done;
  Guard gd;
  gd.abort_flag = done + size_t(nj) * CS;
  gd.limit = c.wait_ns;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 33);  // the codes warp's expect_tx arrival + one cp.async arrival per metadata-warp lane
      mbar_init(empty0 + 8 * s, NW);
    }
    for (int q = 0; q < PD; ++q) {
      mbar_init(cdone0 + 8 * q, NW);
      mbar_init(rdy0 + 8 * q, 1);
      mbar_init(fdone0 + 8 * q, 1);
    }
    mbar_init(stg, NW);
    fence_mbarrier_init();
  }
  __syncthreads();

  // Every role walks the layer table in order; the next entry is loaded one
  // layer ahead so that its latency hides behind the current layer.
  StreamJob Jn = load_job(c.jobs, 0);

  if (warp == NW || warp == NW + 3) {
    // ---------------- producer warps, walking the ring together: in the codes
    // warp lane 0 issues the TMA copies of the codes; every lane of the
    // metadata warp copies its share of the scales and zero points. The two
    // sit on different SM sub-partitions, each beside two consumer warps
    // (one warp doing both measured slower on B300: its sub-partition issued
    // ~20 % more instructions than the others).
    const bool codes = warp == NW;
    int slot = 0;
    uint32_t phase = 0;
    int issued = 0;  // slots filled (for the drain after an abort)
    bool alive = true;
    for (int j = 0; j < nj && alive; ++j) {
      const StreamJob J = Jn;
      if (j + 1 < nj) Jn = load_job(c.jobs, j + 1);
      const Span s = span_of(J, P, b, SG::UB);
      if (s.T == 0) continue;
      const CUtensorMap* m = c.maps + J.map;
      const int R = (s.T + CU - 1) / CU;
      const uint32_t* sc_base = J.scales2;
      const uint8_t* z_base = J.zeros;
      const int G = J.G, KB = J.KB, NU = s.NU;
      const int64_t ntiles = int64_t((J.N + 127) / 128) * KB;  // 128x64 code tiles of the blob
      const int64_t nmeta = ntiles / KB * G * 64;               // scale pairs of the blob
      int rgl0 = 0, ku0 = 0;  // (row group, unit) of the slot's first unit, advanced without dividing
      for (int k = 0; k < R; ++k) {
        if (!warp_outcome(wait_mbar(empty0 + 8 * slot, phase ^ 1u, gd))) {
          alive = false;
          break;
        }
        const uint32_t full = full0 + 8 * slot;
        const uint32_t sb = ring + uint32_t(slot) * SG::kSlot;
        const int nu_slot = min(CU, s.T - k * CU);
        if (codes && lane == 0) {
          mbar_arrive_expect_tx(full, uint32_t(nu_slot) * SG::kUnitCode);
          int rg = s.rg0 + rgl0, ku = ku0, d = 0;
          while (d < nu_slot) {
            int nu = min(nu_slot - d, NU - ku);  // units of this row group in the slot
            const int rb = rg >> 2, pr = rg & 3;
            const int c1 = BITS == 3 ? pr : 2 * pr;
            int c2 = rb * KB + ku * SG::UB;
            int box = CU;
            while (nu > 0) {  // power-of-two boxes, largest first (one box in the common case)
              while (box > nu) box >>= 1;
              if (W4A16_CHECK(d + box <= CU && int64_t(c2) + box * SG::UB <= ntiles, 0x101u))
                tma_load_3d(sb + d * SG::kUnitCode, m + (ilog2(CU) - ilog2(box)), 0, c1, c2, full);
              c2 += box * SG::UB;
              d += box;
              ku += box;
              nu -= box;
            }
            if (ku == NU) {
              ku = 0;
              ++rg;
            }
          }
        }
        if (!codes) {
          // scales (SG::kScaleChunks 16-byte pieces per unit) and zero points
          // (SG::kZeroChunks per unit): unit d of the slot is (rgl0, ku0 + d),
          // wrapping into the following row groups. A row group's scales of
          // one group are 64 contiguous bytes (its two 16-row tiles in the row
          // block's [group][16-row tile] order), those of the next group
          // kMetaGroupStride entries further on.
          if (NU >= CU) {
            // at most one row-group boundary in the slot: units d < dx lie in
            // row group rg, the rest in rg + 1; an entry is a per-slot base plus
            // a lane constant
            const int rg = s.rg0 + rgl0, dx = NU - ku0;
            const int64_t eA = (int64_t(rg >> 2) * G) * 64 + (rg & 3) * 16 + int64_t(ku0) * SG::GU * 64;
            const int64_t eB = (int64_t((rg + 1) >> 2) * G) * 64 + ((rg + 1) & 3) * 16 +
                               int64_t(ku0 - NU) * SG::GU * 64;
            for (int q = lane; q < nu_slot * SG::kScaleChunks; q += 32) {
              const int d = q / SG::kScaleChunks, p = q % SG::kScaleChunks;
              const int64_t e = (d < dx ? eA : eB) + (d * SG::GU + (p >> 2)) * 64 + (p & 3) * 4;
              const int dst = SG::kScaleOff + (d * SG::GU + (p >> 2)) * 64 + (p & 3) * 16;
              if (W4A16_CHECK(e + 4 <= nmeta && dst + 16 <= SG::kZeroOff, 0x102u)) cp_async_16_cg(sb + dst, sc_base + e);
            }
            if (!SYM) {
              constexpr int ZC = SG::ZB / 16;  // 16-byte pieces of a row group's zero points of one group
              for (int q = lane; q < nu_slot * SG::kZeroChunks; q += 32) {
                const int d = q / SG::kZeroChunks, p = q % SG::kZeroChunks;
                const int gg = p / ZC, h = p % ZC;
                const int64_t e = ((d < dx ? eA : eB) + (d * SG::GU + gg) * 64) * ZC + h * 16;
                const int dst = SG::kZeroOff + (d * SG::GU + gg) * SG::ZB + h * 16;
                if (W4A16_CHECK(e + 16 <= nmeta * ZC && dst + 16 <= SG::kSlot, 0x103u))
                  cp_async_16_cg(sb + dst, z_base + e);
              }
            }
          } else {
            // short row groups (fewer units than a slot): walk each unit's row group
            for (int q = lane; q < nu_slot * SG::kScaleChunks; q += 32) {
              const int d = q / SG::kScaleChunks, p = q - d * SG::kScaleChunks;
              int ku = ku0 + d, rg = s.rg0 + rgl0;
              while (ku >= NU) {
                ku -= NU;
                ++rg;
              }
              const int gg = p >> 2;
              const int64_t e = meta_index(rg >> 2, ku * SG::GU + gg, 2 * (rg & 3), 0, G) + (p & 3) * 4;
              const int dst = SG::kScaleOff + (d * SG::GU + gg) * 64 + (p & 3) * 16;
              if (W4A16_CHECK(e + 4 <= nmeta && dst + 16 <= SG::kZeroOff, 0x102u)) cp_async_16_cg(sb + dst, sc_base + e);
            }
            if (!SYM) {
              for (int q = lane; q < nu_slot * SG::kZeroChunks; q += 32) {
                const int d = q / SG::kZeroChunks, p = q - d * SG::kZeroChunks;
                int ku = ku0 + d, rg = s.rg0 + rgl0;
                while (ku >= NU) {
                  ku -= NU;
                  ++rg;
                }
                const int gg = p / (SG::ZB / 16), h = p - gg * (SG::ZB / 16);
                const int64_t e = meta_index(rg >> 2, ku * SG::GU + gg, 2 * (rg & 3), 0, G) * (SG::ZB / 16) + h * 16;
                const int dst = SG::kZeroOff + (d * SG::GU + gg) * SG::ZB + h * 16;
                if (W4A16_CHECK(e + 16 <= nmeta * (SG::ZB / 16) && dst + 16 <= SG::kSlot, 0x103u))
                  cp_async_16_cg(sb + dst, z_base + e);
              }
            }
          }
          cp_async_arrive_noinc(full);
        }
        ++issued;
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
        ku0 += CU;
        while (ku0 >= NU) {
          ku0 -= NU;
          ++rgl0;
        }
      }
    }
    cp_async_wait_all();
    if (codes && lane == 0) {
      // Let the TMA copies in flight land before the block can exit: the last
      // min(issued, S) fills, each in its own slot. After a normal run every
      // one has been consumed and each test returns at once; after an abort
      // (this warp's or another role's) some may still be landing.
      const int nf = min(issued, S);
      for (int k = 1; k <= nf; ++k) {
        const int q = issued - k;
        const uint32_t bar = full0 + 8 * (q % S);
        const uint32_t par = uint32_t(q / S) & 1u;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar, par) && global_timer_ns() - t0 < kTWaitLimitNs) {
        }
      }
    }
    return;
  }

  if (warp == NW + 1) {
    // ---------------- dependency warp
    int known = -1;     // every layer <= known has been seen complete, and acquired
    bool stale = true;  // the staged activations may be out of date
    const uint16_t* loaded = nullptr;
    int loaded_k = 0;
    int cur = 0;                         // buffer holding the current activations
    int last_use0 = -1, last_use1 = -1;  // last layer that read buffer 0 / 1
    // bytes in use: buffer 0 holds [0, size0) of the area, buffer 1 [room - size1, room)
    const int room = c.x_buf_bytes;
    int size0 = 0, size1 = 0;
    for (int j = 0; j < nj; ++j) {
      const StreamJob J = Jn;
      if (j + 1 < nj) Jn = load_job(c.jobs, j + 1);
      // This warp publishes layer j only once every consumer warp has finished
      // layer j - PD (see the barrier comments above); before that it already
      // polls layer j's dependencies and stages its activations when their
      // buffer is free.
      bool fresh = false;  // a dependency of this layer was acquired just now
      int xmode = 0;
      if (J.wait_lo <= J.wait_hi && J.wait_hi > known) {
        // Every lane polls the counter of the range's last slice with acquire
        // loads (one transaction per poll), so that each lane's later loads
        // see what those layers wrote. The finishing warps count slices in
        // table order, so once every block has counted the last slice of the
        // range, every block has finished (and fenced) all slices up to it.
        int st = kWaitOk;
        gd.start();
        while (ld_acquire_gpu_u32(done + size_t(J.wait_hi) * CS) < unsigned(P)) {
          st = gd.check();
          if (st != kWaitOk) break;
        }
        if (!warp_outcome(st)) return;
        known = J.wait_hi;
        stale = true;
        fresh = true;
      }
      const Span s = span_of(J, P, b, SG::UB);
      if (!W4A16_CHECK(s.n <= RGMAX, 0x402u)) return;
      if (s.n > 0) {
        if (XS) {
          if (stale || J.x != loaded || J.K != loaded_k) {
            // the other buffer. Its last reader finished if that was layer
            // j - 1 - PD or earlier (this warp saw that layer's consumer
            // barrier one publication ago); a later last reader is waited for
            // here, and so is the current buffer's when the two layers'
            // activations do not fit in the area together.
            const int nb = cur ^ 1;
            const int sz = int(stream_x_buf(J.K, M, GS));
            const int lu = nb ? last_use1 : last_use0;
            if (lu > j - 1 - PD && !wait_layer<PD>(cdone0, lu, gd)) return;
            const int lo = nb ? last_use0 : last_use1;
            const bool overlap = nb ? room - sz < size0 : sz > room - size1;
            if (overlap && lo > j - 1 - PD && !wait_layer<PD>(cdone0, lo, gd)) return;
            cur = nb;
            if (nb)
              size1 = sz;
            else
              size0 = sz;
            const int xoff = nb ? room - sz : 0;
            uint16_t* xs = reinterpret_cast<uint16_t*>(xbase + xoff);
            if (!W4A16_CHECK(xoff >= 0 && xoff + sz <= room && stream_x_off(BITS, GS, MP) + room <= kStreamSmem,
                             0x202u))
              return;
            if (!fresh) {
              // ahead of the consumers (no dependency was just acquired):
              // stage here, overlapped with their work on earlier layers
              float* xsum = reinterpret_cast<float*>(xs + stream_xsum_off(J.K, M) / 2);
              stage_copy<GS, MP>(J.x, J.K, M, xs, lane, 32);
              cp_async_wait_all();
              __syncwarp();
              stage_sums<GS, MP, 8>(J.K, M, xs, xsum, lane, 32);
              __syncwarp();
            }
            xmode = fresh ? kConsumersStage : 0;
            loaded = J.x;
            loaded_k = J.K;
            stale = false;
          }
          if (cur)
            last_use1 = j;
          else
            last_use0 = j;
        } else {
          const char* xb = reinterpret_cast<const char*>(J.x);
          const int bytes = M * J.K * 2;
          for (int off = lane * 128; off < bytes; off += 32 * 128) prefetch_l1(xb + off);
        }
      }
      if (!wait_layer<PD>(cdone0, j - PD, gd)) return;  // frees record j % PD
      // and the finishing warp has read layer j - PD's partial sums (buffer j % PD)
      if (!wait_layer<PD>(fdone0, j - PD, gd)) return;
      __syncwarp();
      if (lane == 0) {
        LayerRec r;
        r.x = J.x;
        r.K = J.K;
        r.T = s.T;
        r.NU = s.NU;
        r.xsel = (cur ? room - size1 : 0) + xmode;
        r.pad[0] = r.pad[1] = 0;
        rec[j % PD] = r;
        mbar_arrive(rdy0 + 8 * (j % PD));  // release: the staged rows, sums and the record
      }
    }
    return;
  }

  if (warp == NW + 2) {
    // ---------------- finishing warp: partial sums -> y, then the layer's counter
    for (int j = 0; j < nj; ++j) {
      const StreamJob J = Jn;
      if (j + 1 < nj) Jn = load_job(c.jobs, j + 1);
      // the consumers cannot finish layer j + PD before this warp is done with layer j
      if (!wait_layer<PD>(cdone0, j, gd)) return;
      const Span s = span_of(J, P, b, SG::UB);
      // Row `lane` of each owned row group, every token: the partial sums in
      // warp order (deterministic), kept in registers so that the partial
      // buffer is released before the stores and the fence.
      float acc[RGMAX][MP];
      if (s.n > 0) {
        const float* pb = part + size_t(j % PD) * RGMAX * NW * 32 * MP;
#pragma unroll
        for (int rgl = 0; rgl < RGMAX; ++rgl) {
          if (rgl >= s.n) break;
          // warps holding a piece of this row group: all of them unless it has fewer units than a slot
          uint32_t mask = (1u << NW) - 1u;
          if (s.NU < CU) {
            mask = 0;
            for (int u = rgl * s.NU; u < rgl * s.NU + s.NU; ++u) mask |= 1u << ((u % CU) / SG::UPW);
          }
#pragma unroll
          for (int tok = 0; tok < MP; ++tok) {
            float a = 0.f;
            if (tok < M)
#pragma unroll
              for (int w = 0; w < NW; ++w)
                if (mask & (1u << w)) a += pb[(size_t(rgl * NW + w) * 32 + lane) * MP + tok];
            acc[rgl][tok] = a;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(fdone0 + 8 * (j % PD));  // partial buffer j % PD is free
      if (s.n > 0) {
#pragma unroll
        for (int rgl = 0; rgl < RGMAX; ++rgl) {
          if (rgl >= s.n) break;
          const int n = (s.rg0 + rgl) * 32 + lane;
#pragma unroll
          for (int tok = 0; tok < MP; ++tok)
            if (tok < M && n < J.N) J.y[size_t(tok) * J.N + n] = __half_as_ushort(__float2half_rn(acc[rgl][tok]));
        }
      }
      if (J.signal) {
        // this lane's stores, of this slice and every earlier one, are
        // visible device-wide before the slice is counted
        fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0) red_relaxed_gpu_add_u32(done + size_t(j) * CS, 1u);
      }
    }
    return;
  }

  // ---------------- consumer warps
  const int g = lane >> 2, t = lane & 3;
  const int tok0 = min(g, M - 1), tok1 = min(g + 8, M - 1);
  int slot = 0;
  uint32_t phase = 0;
  bool ready = false;      // the full barrier of ring slot `slot` was seen complete
  bool rdy_ready = false;  // layer j's ready barrier was seen complete
  // Every consumer warp at one point, with a bounded wait (a warp that gave
  // up never arrives, and the others then give up too instead of hanging).
  uint32_t stg_parity = 0;
  auto consumers_sync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(stg);  // release: this warp's copies and stores
    const bool ok = warp_outcome(wait_mbar(stg, stg_parity, gd));
    stg_parity ^= 1u;
    return ok;
  };
  for (int j = 0; j < nj; ++j) {
    // Layer j's activations are readable, and (the dependency warp waited for
    // it before publishing layer j) the finishing warp has read layer j - PD's
    // partial sums, so partial buffer j % PD is free. Every warp waits in
    // every layer, with or without units in it, so that no warp runs ahead of
    // the dependency warp's publication (see the barrier comments above).
    if (!rdy_ready && !wait_layer<PD>(rdy0, j, gd)) return;
    rdy_ready = false;
    const LayerRec L = rec[j % PD];
    if (XS && (L.xsel & kConsumersStage)) {
      // a dependency was just acquired: the consumer warps stage the
      // activations together (the dependency warp's acquire happens before
      // the ready barrier this warp waited on)
      uint16_t* xs_st = reinterpret_cast<uint16_t*>(xbase + (L.xsel & ~kConsumersStage));
      stage_copy<GS, MP>(L.x, L.K, M, xs_st, tid, NW * 32);
      cp_async_wait_all();
      if (!consumers_sync()) return;
      stage_sums<GS, MP, 2>(L.K, M, xs_st, reinterpret_cast<float*>(xs_st + stream_xsum_off(L.K, M) / 2), tid, NW * 32);
      if (!consumers_sync()) return;
    }
    Span s;
    s.T = L.T;
    s.NU = L.NU;
    if (s.T > 0) {
      const int R = (s.T + CU - 1) / CU;
      const uint16_t* xl0;
      const uint16_t* xl1;
      const uint16_t* xs = reinterpret_cast<const uint16_t*>(xbase + (XS ? (L.xsel & ~kConsumersStage) : 0));
      const float* xsum = reinterpret_cast<const float*>(xs + stream_xsum_off(L.K, M) / 2);
      if (XS) {
        const int64_t stride = stream_x_stride(L.K, M);
        xl0 = xs + tok0 * stride + 4 * t;
        xl1 = xs + tok1 * stride + 4 * t;
      } else {
        xl0 = L.x + size_t(tok0) * L.K + 4 * t;
        xl1 = L.x + size_t(tok1) * L.K + 4 * t;
      }
      float* pb = part + size_t(j % PD) * RGMAX * NW * 32 * MP;
      float tot[kTilesPerWarp][NB][4];
      int cur = -1;
      auto flush = [&](int rgl) {
        if (!W4A16_CHECK(rgl >= 0 && rgl < RGMAX, 0x302u)) return;
        float* pe = pb + size_t(rgl * NW + warp) * 32 * MP;
#pragma unroll
        for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int tk = nb * 8 + 2 * t;
            const int r0 = tt * 16 + g, r1 = r0 + 8;
            if (tk < M) {
              pe[r0 * MP + tk] = tot[tt][nb][0];
              pe[r1 * MP + tk] = tot[tt][nb][2];
            }
            if (tk + 1 < M) {
              pe[r0 * MP + tk + 1] = tot[tt][nb][1];
              pe[r1 * MP + tk + 1] = tot[tt][nb][3];
            }
          }
      };
      // (row group, unit) of this warp's first unit in slot k, advanced by CU
      // units per slot without dividing
      int rgl0 = 0, ku0 = warp * SG::UPW;
      while (ku0 >= s.NU) {
        ku0 -= s.NU;
        ++rgl0;
      }
      // registers of unit d of slot sb (codes, scale pairs, zero points, and
      // with staged activations the group sums of the unit's columns ku)
      struct UnitIn {
        UnitRegs<GS, BITS> r;
        float xsg[SG::GU][NB][2];
      };
      auto load_unit_in = [&](const unsigned char* sb, int d, int ku, UnitIn& in) {
        if (!W4A16_CHECK(d >= 0 && d < CU && ku >= 0 && ku < s.NU, 0x301u)) d = 0, ku = 0;
#pragma unroll
        for (int bb = 0; bb < SG::UB; ++bb) {
          const unsigned char* cb = sb + d * SG::kUnitCode + bb * SG::CB;
          if (BITS == 3) {
            in.r.w[bb][0][0] = *reinterpret_cast<const uint4*>(cb + lane * 16);
            const uint2 v = *reinterpret_cast<const uint2*>(cb + 512 + lane * 8);
            in.r.w[bb][1][0] = make_uint4(v.x, v.y, 0u, 0u);
          } else {
#pragma unroll
            for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
              for (int pp = 0; pp < kParts<BITS>; ++pp)
                in.r.w[bb][tt][pp] = *reinterpret_cast<const uint4*>(cb + tt * (SG::CB / 2) + pp * 512 + lane * 16);
          }
        }
#pragma unroll
        for (int gg = 0; gg < SG::GU; ++gg) {
#pragma unroll
          for (int tt = 0; tt < kTilesPerWarp; ++tt) {
            const int gi = d * SG::GU + gg;
            in.r.s[gg][tt] = *reinterpret_cast<const uint32_t*>(sb + SG::kScaleOff + gi * 64 + tt * 32 + g * 4);
            if (SYM)
              in.r.z[gg][tt] = 0u;
            else if (BITS == 8)
              in.r.z[gg][tt] = *reinterpret_cast<const uint16_t*>(sb + SG::kZeroOff + gi * 32 + (tt * 8 + g) * 2);
            else
              in.r.z[gg][tt] = sb[SG::kZeroOff + gi * 16 + tt * 8 + g];
          }
          if (XS) {
#pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const int tk = min(nb * 8 + 2 * t, MP - 1);
              in.xsg[gg][nb][0] = xsum[(ku * SG::GU + gg) * MP + tk];
              in.xsg[gg][nb][1] = xsum[(ku * SG::GU + gg) * MP + min(tk + 1, MP - 1)];
            }
          }
        }
      };
      auto compute_in = [&](const UnitIn& in, int ku) {
        const int xo = ku * SG::UB * kColsPerBlock;
        if (XS)
          compute_unit<NB, GS, SYM, kXShared, BITS, BITS == 4, true, MP == 1>(in.r, xl0 + xo, xl1 + xo, tot, in.xsg);
        else
          compute_unit<NB, GS, SYM, kXCoherent, BITS, BITS == 4>(in.r, xl0 + xo, xl1 + xo, tot);
      };
      for (int k = 0; k < R; ++k) {
        if (!ready && !warp_outcome(wait_mbar(full0 + 8 * slot, phase, gd))) return;
        // the ring's next slot (the next layer's, after this layer's last
        // slot), tested now so that the answer is there after this slot
        {
          const int ns = slot + 1 == S ? 0 : slot + 1;
          ready = mbar_test_wait(full0 + 8 * ns, ns == 0 ? phase ^ 1u : phase);
        }
        // in the layer's last slot, the next layer's ready barrier likewise
        if (k == R - 1 && j + 1 < nj)
          rdy_ready = mbar_test_wait(rdy0 + 8 * ((j + 1) % PD), uint32_t((j + 1) / PD) & 1u);
        const unsigned char* sb = smem + size_t(slot) * SG::kSlot;
        if (k * CU + (warp + 1) * SG::UPW <= s.T && ku0 + SG::UPW <= s.NU) {
          // common case: all of the warp's units exist and lie in one row
          // group -- straight-line code, every load ahead of the arithmetic
          if (rgl0 != cur) {
            if (cur >= 0) flush(cur);
#pragma unroll
            for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
              for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                for (int e = 0; e < 4; ++e) tot[tt][nb][e] = 0.f;
            cur = rgl0;
          }
          UnitIn in[SG::UPW];
#pragma unroll
          for (int i = 0; i < SG::UPW; ++i) load_unit_in(sb, warp * SG::UPW + i, ku0 + i, in[i]);
          if (XS) {
            UnitRegs<GS, BITS> rr[SG::UPW];
            float xg[SG::UPW][SG::GU][NB][2];
            int xo[SG::UPW];
#pragma unroll
            for (int i = 0; i < SG::UPW; ++i) {
              rr[i] = in[i].r;
              xo[i] = (ku0 + i) * SG::UB * kColsPerBlock;
#pragma unroll
              for (int gg = 0; gg < SG::GU; ++gg)
#pragma unroll
                for (int nb = 0; nb < NB; ++nb) {
                  xg[i][gg][nb][0] = in[i].xsg[gg][nb][0];
                  xg[i][gg][nb][1] = in[i].xsg[gg][nb][1];
                }
            }
            compute_units<SG::UPW, NB, GS, SYM, BITS, MP == 1>(rr, xl0, xl1, xo, xg, tot);
          } else {
#pragma unroll
            for (int i = 0; i < SG::UPW; ++i) compute_in(in[i], ku0 + i);
          }
        } else {
          int rgl = rgl0, ku = ku0;
#pragma unroll
          for (int i = 0; i < SG::UPW; ++i) {
            const int d = warp * SG::UPW + i;
            if (k * CU + d < s.T) {
              if (rgl != cur) {
                if (cur >= 0) flush(cur);
#pragma unroll
                for (int tt = 0; tt < kTilesPerWarp; ++tt)
#pragma unroll
                  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                    for (int e = 0; e < 4; ++e) tot[tt][nb][e] = 0.f;
                cur = rgl;
              }
              UnitIn in;
              load_unit_in(sb, d, ku, in);
              compute_in(in, ku);
            }
            if (++ku == s.NU) {  // the warp's next unit in this slot
              ku = 0;
              ++rgl;
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
        ku0 += CU;  // the same position in the next slot
        while (ku0 >= s.NU) {
          ku0 -= s.NU;
          ++rgl0;
        }
      }
      if (cur >= 0) flush(cur);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(cdone0 + 8 * (j % PD));
  }
}

template <int MP, int GS, bool SYM, int BITS, bool XS>
cudaError_t launch_stream_typed(const StreamLaunch& c, int sm_count, cudaStream_t stream) {
  auto kern = decode_stream_kernel<MP, GS, SYM, BITS, XS>;
  const int smem = kStreamSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStreamThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sm_count), 1, 1);
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every block resident at once
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, c);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int GS, bool SYM, int BITS, bool XS>
cudaError_t launch_stream_mp(const StreamLaunch& c, int sm_count, cudaStream_t stream) {
  switch (stream_mp(c.M)) {
    case 1: return launch_stream_typed<1, GS, SYM, BITS, XS>(c, sm_count, stream);
    case 2: return launch_stream_typed<2, GS, SYM, BITS, XS>(c, sm_count, stream);
    case 4: return launch_stream_typed<4, GS, SYM, BITS, XS>(c, sm_count, stream);
    case 8: return launch_stream_typed<8, GS, SYM, BITS, XS>(c, sm_count, stream);
    default: return launch_stream_typed<16, GS, SYM, BITS, XS>(c, sm_count, stream);
  }
}

template <int GS, bool SYM, int BITS>
cudaError_t launch_stream_x(const StreamLaunch& c, int sm_count, cudaStream_t stream) {
  return c.x_nbuf ? launch_stream_mp<GS, SYM, BITS, true>(c, sm_count, stream)
                    : launch_stream_mp<GS, SYM, BITS, false>(c, sm_count, stream);
}

template <int BITS>
cudaError_t launch_stream_bits(const StreamLaunch& c, int gsize, bool sym, int sm_count, cudaStream_t stream) {
  if (gsize == 32)
    return sym ? launch_stream_x<32, true, BITS>(c, sm_count, stream) : launch_stream_x<32, false, BITS>(c, sm_count, stream);
  if (gsize == 64)
    return sym ? launch_stream_x<64, true, BITS>(c, sm_count, stream) : launch_stream_x<64, false, BITS>(c, sm_count, stream);
  return sym ? launch_stream_x<128, true, BITS>(c, sm_count, stream) : launch_stream_x<128, false, BITS>(c, sm_count, stream);
}

}  // namespace
}  // namespace w4a16
