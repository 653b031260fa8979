// w4a16_chain_*: host-side validation and the layer table of the chained
// decode products; the persistent kernel is in gemv_impl.cuh.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "internal.h"

using namespace w4a16;

namespace {

constexpr int32_t kChainMaxLayers = 1 << 16;

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Workspace: per layer a completion counter, then the abort flag and the
// next-item counter (each in its own 128-byte line), then the layer table.
size_t counters_bytes(int32_t n) { return align256(size_t(n + 2) * 128); }

int64_t items_of(const w4a16_format* formats, int32_t n) {
  int64_t items = 0;
  for (int32_t i = 0; i < n; ++i) items += make_layout(formats[i]).NR * 4;
  return items;
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

}  // namespace

extern "C" {

size_t w4a16_chain_workspace_bytes(const w4a16_format* formats, int32_t n_layers, int64_t M) {
  if (formats == nullptr || n_layers < 1 || n_layers > kChainMaxLayers || M < 1 || M > 16) return 0;
  if (check_formats(formats, n_layers) != W4A16_OK) return 0;
  return counters_bytes(n_layers) + align256(size_t(n_layers) * sizeof(ChainJob));
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
  if (workspace_bytes < counters_bytes(n_layers) + align256(size_t(n_layers) * sizeof(ChainJob)))
    return W4A16_ERR_BUFFER_TOO_SMALL;
  if (items_of(formats, n_layers) > (int64_t(1) << 30)) return W4A16_ERR_UNSUPPORTED;
  std::vector<ChainJob> jobs(static_cast<size_t>(n_layers));
  int64_t items = 0;
  for (int32_t i = 0; i < n_layers; ++i) {
    const w4a16_format& f = formats[i];
    const w4a16_chain_layer& l = layers[i];
    if (l.packed == nullptr || l.x == nullptr || l.y == nullptr) return W4A16_ERR_INVALID_ARG;
    if (!aligned_to(l.packed, 256) || !aligned_to(l.x, 16) || !aligned_to(l.y, 16)) return W4A16_ERR_MISALIGNED;
    const Layout L = make_layout(f);
    if (l.packed_bytes < L.total) return W4A16_ERR_BUFFER_TOO_SMALL;
    const char* xb = reinterpret_cast<const char*>(l.x);
    const char* yb = reinterpret_cast<const char*>(l.y);
    const size_t xbytes = size_t(M) * size_t(f.K) * 2, ybytes = size_t(M) * size_t(f.N) * 2;
    if (xb < yb + ybytes && yb < xb + xbytes) return W4A16_ERR_INVALID_ARG;  // y overlaps x
    if (l.wait_lo <= l.wait_hi && (l.wait_lo < 0 || l.wait_hi >= i)) return W4A16_ERR_INVALID_ARG;
    const BlobView B = view_of(L, l.packed);
    ChainJob& J = jobs[size_t(i)];
    J.qweight = B.qweight;
    J.scales2 = reinterpret_cast<const uint32_t*>(B.scales);
    J.zeros = B.zeros;
    J.x = l.x;
    J.y = l.y;
    J.N = int(f.N);
    J.K = int(f.K);
    J.G = int(L.G);
    J.KB = int(L.KB);
    J.item0 = int(items);
    J.items = int(L.NR * 4);
    J.wait_lo = l.wait_lo <= l.wait_hi ? l.wait_lo : 0;
    J.wait_hi = l.wait_lo <= l.wait_hi ? l.wait_hi : -1;
    items += J.items;
  }
  char* ws = static_cast<char*>(workspace);
  cudaError_t e = cudaMemcpy(ws + counters_bytes(n_layers), jobs.data(), jobs.size() * sizeof(ChainJob),
                             cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_error_status(e);
  info->n_layers = n_layers;
  info->bits = formats[0].bits;
  info->group_size = formats[0].group_size;
  info->symmetric = formats[0].symmetric;
  info->M = M;
  info->total_items = items;
  return W4A16_OK;
}

w4a16_status w4a16_chain_run(const w4a16_chain_info* info, void* workspace, w4a16_stream_t stream) {
  if (info == nullptr || workspace == nullptr) return W4A16_ERR_INVALID_ARG;
  if (info->n_layers < 1 || info->n_layers > kChainMaxLayers || info->M < 1 || info->M > 16 ||
      info->total_items < 1 || info->total_items > (int64_t(1) << 30))
    return W4A16_ERR_INVALID_ARG;
  if (!aligned_to(workspace, 256)) return W4A16_ERR_MISALIGNED;
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_error_status(e);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  e = cudaMemsetAsync(ws, 0, size_t(info->n_layers + 2) * 128, st);
  if (e != cudaSuccess) return cuda_error_status(e);
  ChainLaunch c;
  c.bits = info->bits;
  c.gsize = info->group_size;
  c.M = int(info->M);
  c.sym = info->symmetric != 0;
  c.n_jobs = info->n_layers;
  c.total_items = int(info->total_items);
  c.sm_count = dev.sm_count;
  c.done = reinterpret_cast<unsigned int*>(ws);
  c.jobs = reinterpret_cast<const ChainJob*>(ws + counters_bytes(info->n_layers));
  e = launch_chain(c, st);
  return e == cudaSuccess ? W4A16_OK : cuda_error_status(e);
}

}  // extern "C"
