// Geometry of the decode stream (the chained decode products): how a layer's
// packed weights are cut into the units a thread block streams, the
// shared-memory ring that holds them, and the rest of the block's shared
// memory. Shared by the host (tensor-map boxes, shared-memory size, the split
// of large layers, whether activations fit in shared memory) and the kernel.
//
// Terms
//   row group   32 consecutive weight rows (two 16-row tiles of a 128-row
//               block); a thread block always owns whole row groups of a layer,
//               with the full K, so no output row is split between blocks.
//   unit        the codes, scales and zero points of one row group over
//               `stream_ub` 64-column blocks (one group of 128 columns, or one
//               64-column block holding one or two groups of 64 / 32).
//   slot        one ring entry: `stream_cu` consecutive units of the block's
//               share (row group after row group), `stream_upw` for each
//               consumer warp. Its codes arrive by TMA in one to a few copies
//               (24 to 32 KiB together: the TMA stream needs large copies),
//               its scales and zero points by the producer warp's cp.async.
#pragma once

namespace w4a16 {

constexpr int kStreamConsumers = 8;  // consumer warps per thread block
constexpr int kStreamWarps = kStreamConsumers + 4;  // + codes, dependency, finishing and metadata warps
constexpr int kStreamThreads = kStreamWarps * 32;
constexpr int kStreamCounterStride = 32;  // 32-bit words between completion counters (one 128-byte line each)
constexpr int kStreamSmem = 227 * 1024;  // shared memory of one thread block (the opt-in maximum)
constexpr int kStreamRingBudget = 136 * 1024;  // bytes of ring entries

__host__ __device__ constexpr int stream_align128(int v) { return (v + 127) / 128 * 128; }
// 64-column blocks per unit and groups per unit.
__host__ __device__ constexpr int stream_ub(int gs) { return gs == 128 ? 2 : 1; }
__host__ __device__ constexpr int stream_gu(int gs) { return gs == 32 ? 2 : 1; }
// Code bytes of one row group per 64-column block: 768 / 1024 / 2048 for 3 / 4 / 8 bits.
__host__ __device__ constexpr int stream_cb(int bits) { return bits * 256; }
// Zero-point bytes of one row group per group: 3- and 4-bit nibble pairs
// (one byte per row pair), 8-bit byte pairs.
__host__ __device__ constexpr int stream_zb(int bits) { return bits == 8 ? 32 : 16; }
__host__ __device__ constexpr int stream_unit_code(int bits, int gs) { return stream_ub(gs) * stream_cb(bits); }
// Units per consumer warp and slot: the largest power of two that keeps a
// slot's codes within 32 KiB. Measured on B300 (8 x 28672x8192, no
// dependencies): one 2 KiB unit per warp 3.66 TB/s, two 4.92 TB/s -- each
// warp's two units overlap their latency chains, and the per-slot barrier
// waits are paid half as often.
__host__ __device__ constexpr int stream_upw(int bits, int gs) {
  return stream_unit_code(bits, gs) * kStreamConsumers * 4 <= 32768   ? 4
         : stream_unit_code(bits, gs) * kStreamConsumers * 2 <= 32768 ? 2
                                                                      : 1;
}
__host__ __device__ constexpr int stream_cu(int bits, int gs) { return kStreamConsumers * stream_upw(bits, gs); }
// Slot layout: the codes of its units back to back, then their scales (64
// bytes per group), then their zero points (stream_zb bytes per group).
__host__ __device__ constexpr int stream_scale_off(int bits, int gs) {
  return stream_align128(stream_cu(bits, gs) * stream_unit_code(bits, gs));
}
__host__ __device__ constexpr int stream_zero_off(int bits, int gs) {
  return stream_scale_off(bits, gs) + stream_cu(bits, gs) * stream_gu(gs) * 64;
}
__host__ __device__ constexpr int stream_slot_bytes(int bits, int gs) {
  return stream_align128(stream_zero_off(bits, gs) + stream_cu(bits, gs) * stream_gu(gs) * stream_zb(bits));
}
__host__ __device__ constexpr int stream_slots(int bits, int gs) {
  return kStreamRingBudget / stream_slot_bytes(bits, gs) < 3 ? 3 : kStreamRingBudget / stream_slot_bytes(bits, gs);
}
// Padded token count of the kernel instance for M tokens.
__host__ __device__ constexpr int stream_mp(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }
// Row groups one thread block may own in one layer slice; larger layers are
// cut into slices. Each owned row group has one partial-sum entry per consumer
// warp (32 rows x MP tokens of fp32), in stream_part_depth buffers (slice j
// uses buffer j % depth): four at one token, two otherwise. The same depth
// sets how far the dependency warp may publish ahead of the consumer warps.
__host__ __device__ constexpr int stream_max_rg(int mp) { return mp == 1 ? 4 : mp == 2 ? 8 : mp == 4 ? 4 : mp == 8 ? 2 : 1; }
__host__ __device__ constexpr int stream_part_depth(int mp) { return mp == 1 ? 4 : 2; }
__host__ __device__ constexpr int stream_part_bytes(int mp) {
  return stream_part_depth(mp) * stream_max_rg(mp) * kStreamConsumers * 32 * mp * 4;
}

// Shared memory of one thread block: ring | barriers (full and empty per
// slot; consumer-done, ready and finishing-done per layer slot, four words
// each; the consumer warps' staging barrier; a spare word) and four layer
// records (32 bytes each) | the partial-sum buffers | one or two
// staged-activation buffers (rows and group sums; the rest of the block's
// shared memory, up to kStreamSmem). Layer j uses layer slot j % depth
// (stream_part_depth) of each per-layer set.
constexpr int kStreamLayerBars = 14;  // 4 cdone + 4 rdy + 4 fdone + staging + spare
constexpr int kStreamRecs = 4;
__host__ __device__ constexpr int stream_bar_off(int bits, int gs) {
  return stream_slots(bits, gs) * stream_slot_bytes(bits, gs);
}
// after the barriers (16-byte aligned): the kStreamRecs layer records
constexpr int kStreamRecBytes = 32;
__host__ __device__ constexpr int stream_rec_off(int bits, int gs) {
  return stream_bar_off(bits, gs) + (2 * stream_slots(bits, gs) + kStreamLayerBars) * 8;
}
__host__ __device__ constexpr int stream_part_off(int bits, int gs) {
  return stream_bar_off(bits, gs) +
         stream_align128((2 * stream_slots(bits, gs) + kStreamLayerBars) * 8 + kStreamRecs * kStreamRecBytes);
}
__host__ __device__ constexpr int stream_x_off(int bits, int gs, int mp) {
  return stream_part_off(bits, gs) + stream_part_bytes(mp);
}
__host__ __device__ constexpr int stream_x_bytes(int bits, int gs, int mp) { return kStreamSmem - stream_x_off(bits, gs, mp); }
// Row stride (halves) of the staged activations: one row per token; rows
// after the first are offset by 32 bytes so that the lanes of a warp reading
// different tokens fall on different banks. The group sums of the
// activations (fp32 [G][MP]) follow the rows.
__host__ __device__ constexpr long long stream_x_stride(long long K, int M) { return M == 1 ? K : K + 16; }
__host__ __device__ constexpr long long stream_xsum_off(long long K, int M) {  // bytes from the staged rows
  return M * stream_x_stride(K, M) * 2;
}
// Bytes of one staged-activation buffer for a layer (rows, then group sums).
__host__ __device__ constexpr long long stream_x_buf(long long K, int M, int gs) {
  return (stream_xsum_off(K, M) + (K / gs) * stream_mp(M) * 4 + 127) / 128 * 128;
}

}  // namespace w4a16
