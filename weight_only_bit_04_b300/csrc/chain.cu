// w4a16_chain_*: host side of the chained decode products -- validation, the
// table of layer slices with their tensor maps, and the launch of the decode
// stream (decode_stream.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "internal.h"
#include "stream_geom.h"

using namespace w4a16;

namespace {

constexpr int32_t kChainMaxLayers = 1 << 16;
constexpr int kMapsPerLayer = 6;  // the codes as boxes of CU, CU/2, ..., 1 units (CU <= 32)

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int64_t row_groups(const w4a16_format& f) { return (f.N + 31) / 32; }

// Slices of a layer when a thread block may own at most `per_block` row
// groups of a slice and there are `blocks` blocks.
int64_t slices_of(const w4a16_format& f, int64_t blocks, int64_t per_block) {
  const int64_t cap = blocks * per_block;
  return (row_groups(f) + cap - 1) / cap;
}

// Workspace: completion counters (one per slice, then the abort flag; 128-byte
// lines), the slice table, the tensor maps (64-byte aligned).
struct WsLayout {
  size_t counters, jobs, maps, total;
};
WsLayout ws_layout(int64_t n_slices, int32_t n_layers) {
  WsLayout w;
  w.counters = 0;
  w.jobs = align256(size_t(n_slices + 2) * 128);
  w.maps = w.jobs + align256(size_t(n_slices) * sizeof(StreamJob));
  w.total = w.maps + align256(size_t(n_layers) * kMapsPerLayer * sizeof(CUtensorMap));
  return w;
}

w4a16_status check_formats(const w4a16_format* formats, int32_t n) {
  for (int32_t i = 0; i < n; ++i) {
    const w4a16_format& f = formats[i];
    w4a16_status s = w4a16_check_format(&f);
    if (s != W4A16_OK) return s;
    if (f.bits != formats[0].bits || f.group_size != formats[0].group_size || f.symmetric != formats[0].symmetric)
      return W4A16_ERR_UNSUPPORTED;
    if (f.has_g_idx || f.has_act_scale || f.K % kColsPerBlock != 0) return W4A16_ERR_UNSUPPORTED;
  }
  return W4A16_OK;
}

// The tensor maps of one layer's codes (see decode_stream.cuh): a 3-D view
// [tile][16-row tile (8) or tile pair (4)][words of one 16-row tile or pair]
// with boxes of one row group over CU, CU/2, ..., 1 units.
cudaError_t make_maps(const Layout& L, const void* blob, CUtensorMap* maps) {
  const BlobView B = view_of(L, blob);
  const int bits = L.bits, gs = L.gsize;
  const uint32_t ub = uint32_t(stream_ub(gs)), cu = uint32_t(stream_cu(bits, gs));
  const uint64_t tiles = uint64_t(L.NR) * uint64_t(L.KB);
  const uint64_t cw = bits == 3 ? 192 : uint64_t(bits) * 32;  // words per inner row
  const uint64_t c1 = bits == 3 ? 4 : 8;
  const uint64_t cdims[3] = {cw, c1, tiles};
  const uint64_t cstr[2] = {cw * 4, cw * 4 * c1};
  const uint32_t crows = bits == 3 ? 1 : 2;
  cudaError_t e = cudaSuccess;
  for (uint32_t k = 0, box = cu; box >= 1 && e == cudaSuccess; ++k, box >>= 1) {
    const uint32_t b3[3] = {uint32_t(cw), crows, box * ub};
    e = encode_tiled_map(&maps[k], CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, B.qweight, cdims, cstr, b3);
  }
  return e;
}

}  // namespace

extern "C" {

size_t w4a16_chain_workspace_bytes(const w4a16_format* formats, int32_t n_layers, int64_t M) {
  if (formats == nullptr || n_layers < 1 || n_layers > kChainMaxLayers || M < 1 || M > 16) return 0;
  if (check_formats(formats, n_layers) != W4A16_OK) return 0;
  // Bound for any device: as many slices as a single thread block would need.
  const int64_t per_block = stream_max_rg(stream_mp(int(M)));
  int64_t slices = 0;
  for (int32_t i = 0; i < n_layers; ++i) slices += slices_of(formats[i], 1, per_block);
  if (slices > (int64_t(1) << 24)) return 0;
  return ws_layout(slices, n_layers).total;
}

w4a16_status w4a16_chain_prepare(const w4a16_format* formats, const w4a16_chain_layer* layers,
                                 int32_t n_layers, int64_t M, void* workspace, size_t workspace_bytes,
                                 w4a16_chain_info* info) {
  if (formats == nullptr || layers == nullptr || info == nullptr || workspace == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if (n_layers < 1 || n_layers > kChainMaxLayers) return W4A16_ERR_INVALID_ARG;
  if (M < 1 || M > 16) return W4A16_ERR_INVALID_ARG;
  w4a16_status s = check_formats(formats, n_layers);
  if (s != W4A16_OK) return s;
  if (!aligned_to(workspace, 256)) return W4A16_ERR_MISALIGNED;
  const size_t need = w4a16_chain_workspace_bytes(formats, n_layers, M);
  if (need == 0) return W4A16_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return W4A16_ERR_BUFFER_TOO_SMALL;
  for (int32_t i = 0; i < n_layers; ++i) {
    const w4a16_format& f = formats[i];
    const w4a16_chain_layer& l = layers[i];
    if (l.packed == nullptr || l.x == nullptr || l.y == nullptr) return W4A16_ERR_INVALID_ARG;
    if (!aligned_to(l.packed, 256) || !aligned_to(l.x, 16) || !aligned_to(l.y, 16)) return W4A16_ERR_MISALIGNED;
    if (l.packed_bytes < make_layout(f).total) return W4A16_ERR_BUFFER_TOO_SMALL;
    const char* xb = reinterpret_cast<const char*>(l.x);
    const char* yb = reinterpret_cast<const char*>(l.y);
    const size_t xbytes = size_t(M) * size_t(f.K) * 2, ybytes = size_t(M) * size_t(f.N) * 2;
    if (xb < yb + ybytes && yb < xb + xbytes) return W4A16_ERR_INVALID_ARG;  // y overlaps x
    if (l.wait_lo <= l.wait_hi && (l.wait_lo < 0 || l.wait_hi >= i)) return W4A16_ERR_INVALID_ARG;
  }

  // Plan the slices for this device: each block owns at most stream_max_rg
  // row groups of a slice; block positions rotate by the row groups dealt.
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_error_status(e);
  const int64_t P = dev.sm_count;
  const int64_t per_block = stream_max_rg(stream_mp(int(M)));
  std::vector<int64_t> first(size_t(n_layers) + 1, 0);  // first slice of each layer
  for (int32_t i = 0; i < n_layers; ++i) first[size_t(i) + 1] = first[size_t(i)] + slices_of(formats[i], P, per_block);
  const int64_t n_slices = first[size_t(n_layers)];
  const WsLayout wl = ws_layout(n_slices, n_layers);
  std::vector<StreamJob> jobs(static_cast<size_t>(n_slices));
  std::vector<CUtensorMap> maps(size_t(n_layers) * kMapsPerLayer);
  std::memset(maps.data(), 0, maps.size() * sizeof(CUtensorMap));
  int64_t dealt = 0;
  for (int32_t i = 0; i < n_layers; ++i) {
    const w4a16_format& f = formats[i];
    const w4a16_chain_layer& l = layers[i];
    const Layout L = make_layout(f);
    e = make_maps(L, l.packed, &maps[size_t(i) * kMapsPerLayer]);
    if (e != cudaSuccess) return cuda_error_status(e);
    const int64_t nrg = row_groups(f), ns = first[size_t(i) + 1] - first[size_t(i)];
    const bool waits = l.wait_lo <= l.wait_hi;
    for (int64_t k = 0; k < ns; ++k) {
      StreamJob& J = jobs[size_t(first[size_t(i)] + k)];
      std::memset(&J, 0, sizeof(J));
      J.x = l.x;
      J.y = l.y;
      J.scales2 = reinterpret_cast<const uint32_t*>(view_of(L, l.packed).scales);
      J.zeros = view_of(L, l.packed).zeros;
      J.N = int(f.N);
      J.K = int(f.K);
      J.KB = int(L.KB);
      J.G = int(L.G);
      J.rg_first = int(k * nrg / ns);
      J.n_rg = int((k + 1) * nrg / ns) - J.rg_first;
      J.rot = int(dealt % P);
      dealt += J.n_rg;
      J.wait_lo = waits ? int(first[size_t(l.wait_lo)]) : 0;
      J.wait_hi = waits ? int(first[size_t(l.wait_hi) + 1] - 1) : -1;
      J.map = i * kMapsPerLayer;
    }
  }
  // Blocks finish their slices in table order, so "every block counted slice
  // h" means every block finished every slice up to h: a wait for the range
  // [lo, hi] polls slice hi's counter alone, and only such slices are counted.
  for (const StreamJob& J : jobs)
    if (J.wait_lo <= J.wait_hi) jobs[size_t(J.wait_hi)].signal = 1;
  char* ws = static_cast<char*>(workspace);
  e = cudaMemcpy(ws + wl.jobs, jobs.data(), jobs.size() * sizeof(StreamJob), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(ws + wl.maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_error_status(e);
  info->n_layers = n_layers;
  info->bits = formats[0].bits;
  info->group_size = formats[0].group_size;
  info->symmetric = formats[0].symmetric;
  info->M = M;
  info->n_slices = n_slices;
  info->blocks = int32_t(P);
  // Staged activations when every layer's fit the block's activation area:
  // two buffers, one from each end of the area, each sized for the layer it
  // holds (the next layer's activations land while this one computes unless
  // the two layers' together exceed the area).
  long long xbuf = 0;
  for (int32_t i = 0; i < n_layers; ++i)
    xbuf = std::max(xbuf, stream_x_buf(formats[i].K, int(M), formats[0].group_size));
  const long long xroom = stream_x_bytes(formats[0].bits, formats[0].group_size, stream_mp(int(M)));
  const int32_t nbuf = xbuf <= xroom ? 2 : 0;
  info->flags = nbuf;            // staged-activation buffers (0: read through L1)
  info->reserved_x = nbuf ? int32_t(xroom) : 0;
  return W4A16_OK;
}

w4a16_status w4a16_chain_run(const w4a16_chain_info* info, void* workspace, w4a16_stream_t stream) {
  if (info == nullptr || workspace == nullptr) return W4A16_ERR_INVALID_ARG;
  if (info->n_layers < 1 || info->n_layers > kChainMaxLayers || info->M < 1 || info->M > 16 ||
      info->n_slices < info->n_layers || info->n_slices > (int64_t(1) << 24) || info->blocks < 1)
    return W4A16_ERR_INVALID_ARG;
  if (!aligned_to(workspace, 256)) return W4A16_ERR_MISALIGNED;
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_error_status(e);
  if (dev.sm_count != info->blocks) return W4A16_ERR_INVALID_ARG;  // prepared for another device
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  const WsLayout wl = ws_layout(info->n_slices, info->n_layers);
  e = cudaMemsetAsync(ws, 0, size_t(info->n_slices + 2) * 128, st);
  if (e != cudaSuccess) return cuda_error_status(e);
  StreamLaunch c;
  c.jobs = reinterpret_cast<const StreamJob*>(ws + wl.jobs);
  c.maps = reinterpret_cast<const CUtensorMap*>(ws + wl.maps);
  c.done = reinterpret_cast<unsigned int*>(ws);
  c.n_jobs = int(info->n_slices);
  c.M = int(info->M);
  c.x_nbuf = info->flags & 3;
  c.x_buf_bytes = c.x_nbuf ? info->reserved_x : 0;
  c.wait_ns = wait_limit_ns();
  e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_stream(c, info->bits, info->group_size, info->symmetric != 0, info->blocks, st);
  return e == cudaSuccess ? W4A16_OK : cuda_error_status(e);
}

}  // extern "C"
