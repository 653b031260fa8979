// C ABI of libw4a16.so: argument validation on the host, then one launch on
// the caller's stream. See include/w4a16.h for the contract of each call.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"

namespace w4a16 {
namespace {

thread_local int g_last_cuda_error = 0;

w4a16_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = int(e);
  return W4A16_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int kMaxDevices = 64;
std::once_flag g_dev_once[kMaxDevices];
DeviceInfo g_dev[kMaxDevices];
cudaError_t g_dev_err[kMaxDevices];

w4a16_status format_status(const w4a16_format* f) {
  if (f == nullptr) return W4A16_ERR_INVALID_ARG;
  if (f->symmetric != 0 && f->symmetric != 1) return W4A16_ERR_INVALID_ARG;
  if (f->has_g_idx != 0 && f->has_g_idx != 1) return W4A16_ERR_INVALID_ARG;
  if (f->has_act_scale != 0 && f->has_act_scale != 1) return W4A16_ERR_INVALID_ARG;
  if (f->N < 1 || f->K < 1 || f->N > (int64_t(1) << 20) || f->K > (int64_t(1) << 20))
    return W4A16_ERR_INVALID_ARG;
  if (f->bits != 3 && f->bits != 4 && f->bits != 8) return W4A16_ERR_UNSUPPORTED;
  if (f->group_size != 32 && f->group_size != 64 && f->group_size != 128) return W4A16_ERR_UNSUPPORTED;
  if (f->K % f->group_size != 0) return W4A16_ERR_UNSUPPORTED;  // no ragged last group
  return W4A16_OK;
}

// Common checks for calls that read a packed blob.
w4a16_status blob_status(const w4a16_format* f, const void* packed, size_t packed_bytes) {
  w4a16_status s = format_status(f);
  if (s != W4A16_OK) return s;
  if (packed == nullptr) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256)) return W4A16_ERR_MISALIGNED;
  if (packed_bytes < make_layout(*f).total) return W4A16_ERR_BUFFER_TOO_SMALL;
  return W4A16_OK;
}

// Host-side group map check and the stable group-sorted column order.
bool build_perm(const w4a16_format& f, const int32_t* g_idx, std::vector<int32_t>& perm) {
  const int64_t K = f.K, G = f.K / f.group_size;
  std::vector<int64_t> count(static_cast<size_t>(G), 0);
  for (int64_t k = 0; k < K; ++k) {
    const int32_t t = g_idx[k];
    if (t < 0 || t >= G) return false;
    ++count[size_t(t)];
  }
  for (int64_t t = 0; t < G; ++t)
    if (count[size_t(t)] != f.group_size) return false;
  perm.resize(size_t(K));
  std::vector<int64_t> next_slot(static_cast<size_t>(G));
  for (int64_t t = 0; t < G; ++t) next_slot[size_t(t)] = t * f.group_size;
  for (int64_t k = 0; k < K; ++k) perm[size_t(next_slot[size_t(g_idx[k])]++)] = int32_t(k);
  return true;
}

}  // namespace

w4a16_status cuda_error_status(cudaError_t e) { return cuda_fail(e); }

namespace {
constexpr unsigned long long kDefaultWaitNs = 1000ull * 1000ull * 1000ull;  // 1 s
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_injected{0};
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

cudaError_t take_injected_launch_error() {
  if (g_injected.load(std::memory_order_relaxed) == 0) return cudaSuccess;
  return cudaError_t(g_injected.exchange(0));
}

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(g_dev_once[dev], [dev]() {
    DeviceInfo d{};
    cudaError_t err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess)
      err = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    g_dev[dev] = d;
    g_dev_err[dev] = err;
  });
  if (g_dev_err[dev] != cudaSuccess) return g_dev_err[dev];
  *out = g_dev[dev];
  return cudaSuccess;
}

}  // namespace w4a16

using namespace w4a16;

extern "C" {

size_t w4a16_packed_bytes(const w4a16_format* f) {
  if (format_status(f) != W4A16_OK) return 0;
  return make_layout(*f).total;
}

w4a16_status w4a16_check_format(const w4a16_format* f) { return format_status(f); }

const char* w4a16_status_string(w4a16_status s) {
  switch (s) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_INVALID_ARG: return "W4A16_ERR_INVALID_ARG";
    case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED";
    case W4A16_ERR_MISALIGNED: return "W4A16_ERR_MISALIGNED";
    case W4A16_ERR_BUFFER_TOO_SMALL: return "W4A16_ERR_BUFFER_TOO_SMALL";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA";
  }
  return "W4A16_ERR_UNKNOWN";
}

int w4a16_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t w4a16_set_wait_limit_ns(uint64_t ns) {
  return g_wait_ns.exchange(ns == 0 ? kDefaultWaitNs : ns);
}

void w4a16_debug_fail_next_launch(int error) { g_injected.store(error); }

w4a16_status w4a16_debug_check_word(uint32_t* word) {
  if (word == nullptr) return W4A16_ERR_INVALID_ARG;
  *word = 0;
#ifdef W4A16_DEBUG_CHECKS
  cudaError_t e = cudaDeviceSynchronize();
  unsigned int w = 0;
  if (e == cudaSuccess) e = take_debug_error(&w);
  if (e != cudaSuccess) return cuda_fail(e);
  *word = w;
  return W4A16_OK;
#else
  return W4A16_ERR_UNSUPPORTED;
#endif
}

size_t w4a16_quantize_workspace_bytes(const w4a16_format* f) {
  if (format_status(f) != W4A16_OK) return 0;
  return f->has_g_idx ? size_t(f->K) * 4 : 0;
}

static w4a16_status quantize_common(const w4a16_format* f, const uint16_t* w, const uint16_t* act_scale,
                                    const int32_t* g_idx, uint8_t* q, uint16_t* scales, uint8_t* zeros,
                                    void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  w4a16_status s = format_status(f);
  if (s != W4A16_OK) return s;
  if (w == nullptr || q == nullptr || scales == nullptr) return W4A16_ERR_INVALID_ARG;
  if ((zeros == nullptr) != (f->symmetric != 0)) return W4A16_ERR_INVALID_ARG;
  if ((g_idx == nullptr) != (f->has_g_idx == 0)) return W4A16_ERR_INVALID_ARG;
  if ((act_scale == nullptr) != (f->has_act_scale == 0)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(w, 16) || !aligned(scales, 2) || !aligned(act_scale, 2)) return W4A16_ERR_MISALIGNED;
  const size_t need = f->has_g_idx ? size_t(f->K) * 4 : 0;
  if (workspace_bytes < need) return W4A16_ERR_BUFFER_TOO_SMALL;
  if (need > 0 && workspace == nullptr) return W4A16_ERR_INVALID_ARG;
  if (need > 0 && !aligned(workspace, 16)) return W4A16_ERR_MISALIGNED;
  const Layout L = make_layout(*f);
  const int32_t* perm_dev = nullptr;
  if (f->has_g_idx) {
    std::vector<int32_t> perm;
    if (!build_perm(*f, g_idx, perm)) return W4A16_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(workspace, perm.data(), need, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    perm_dev = static_cast<const int32_t*>(workspace);
  }
  cudaError_t e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_quantize_rtn(L, w, perm_dev, act_scale, q, scales, zeros, stream);
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

w4a16_status w4a16_quantize_rtn(const w4a16_format* f, const uint16_t* w, const int32_t* g_idx,
                                uint8_t* q, uint16_t* scales, uint8_t* zeros, void* workspace,
                                size_t workspace_bytes, w4a16_stream_t stream) {
  return quantize_common(f, w, nullptr, g_idx, q, scales, zeros, workspace, workspace_bytes, stream);
}

w4a16_status w4a16_quantize_rtn_awq(const w4a16_format* f, const uint16_t* w, const uint16_t* act_scale,
                                    const int32_t* g_idx, uint8_t* q, uint16_t* scales, uint8_t* zeros,
                                    void* workspace, size_t workspace_bytes, w4a16_stream_t stream) {
  if (f != nullptr && f->has_act_scale != 1) return W4A16_ERR_INVALID_ARG;
  return quantize_common(f, w, act_scale, g_idx, q, scales, zeros, workspace, workspace_bytes, stream);
}

static w4a16_status pack_common(const w4a16_format* f, const uint8_t* q, const uint16_t* scales,
                                const uint8_t* zeros, const int32_t* g_idx, const uint16_t* act_scale,
                                void* packed, size_t packed_bytes, w4a16_stream_t stream) {
  w4a16_status s = format_status(f);
  if (s != W4A16_OK) return s;
  if (q == nullptr || scales == nullptr || packed == nullptr) return W4A16_ERR_INVALID_ARG;
  if ((zeros == nullptr) != (f->symmetric != 0)) return W4A16_ERR_INVALID_ARG;
  if ((g_idx == nullptr) != (f->has_g_idx == 0)) return W4A16_ERR_INVALID_ARG;
  if ((act_scale == nullptr) != (f->has_act_scale == 0)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(packed, 256) || !aligned(scales, 2) || !aligned(act_scale, 2)) return W4A16_ERR_MISALIGNED;
  const Layout L = make_layout(*f);
  if (packed_bytes < L.total) return W4A16_ERR_BUFFER_TOO_SMALL;
  if (f->has_g_idx) {
    std::vector<int32_t> perm;
    if (!build_perm(*f, g_idx, perm)) return W4A16_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(static_cast<char*>(packed) + L.p_off, perm.data(), L.p_bytes,
                                    cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cudaError_t e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_pack(L, q, scales, zeros, act_scale, packed, stream);
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

w4a16_status w4a16_pack(const w4a16_format* f, const uint8_t* q, const uint16_t* scales,
                        const uint8_t* zeros, const int32_t* g_idx, void* packed, size_t packed_bytes,
                        w4a16_stream_t stream) {
  return pack_common(f, q, scales, zeros, g_idx, nullptr, packed, packed_bytes, stream);
}

w4a16_status w4a16_pack_awq(const w4a16_format* f, const uint8_t* q, const uint16_t* scales,
                            const uint8_t* zeros, const int32_t* g_idx, const uint16_t* act_scale,
                            void* packed, size_t packed_bytes, w4a16_stream_t stream) {
  if (f != nullptr && f->has_act_scale != 1) return W4A16_ERR_INVALID_ARG;
  return pack_common(f, q, scales, zeros, g_idx, act_scale, packed, packed_bytes, stream);
}

w4a16_status w4a16_dequant(const w4a16_format* f, const void* packed, size_t packed_bytes,
                           uint16_t* w_out, w4a16_stream_t stream) {
  w4a16_status s = blob_status(f, packed, packed_bytes);
  if (s != W4A16_OK) return s;
  if (w_out == nullptr) return W4A16_ERR_INVALID_ARG;
  if (!aligned(w_out, 16)) return W4A16_ERR_MISALIGNED;
  cudaError_t e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_dequant(make_layout(*f), packed, w_out, stream);
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

static w4a16_status gemv_common(const w4a16_format* f, const void* packed, size_t packed_bytes,
                                const uint16_t* x, uint16_t* y, int64_t M, int32_t shape,
                                int32_t ksplit, uint32_t flags, w4a16_stream_t stream) {
  w4a16_status s = blob_status(f, packed, packed_bytes);
  if (s != W4A16_OK) return s;
  if (x == nullptr || y == nullptr) return W4A16_ERR_INVALID_ARG;
  if (M < 1 || M > 16) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return W4A16_ERR_MISALIGNED;
  const char* xb = reinterpret_cast<const char*>(x);
  const char* yb = reinterpret_cast<const char*>(y);
  const size_t xbytes = size_t(M) * size_t(f->K) * 2, ybytes = size_t(M) * size_t(f->N) * 2;
  if (xb < yb + ybytes && yb < xb + xbytes) return W4A16_ERR_INVALID_ARG;  // overlap
  if ((flags & ~uint32_t(W4A16_GEMV_WEIGHTS_READY | W4A16_GEMV_STAGE_ACTIVATIONS | W4A16_GEMV_ASYNC_COPY |
                         W4A16_GEMV_REGISTER_RING | W4A16_GEMV_INPUTS_READY)) != 0)
    return W4A16_ERR_INVALID_ARG;
  if ((flags & W4A16_GEMV_REGISTER_RING) && (flags & W4A16_GEMV_ASYNC_COPY)) return W4A16_ERR_INVALID_ARG;
  if (shape != 0 && shape != 2 && shape != 4 && shape != 8) return W4A16_ERR_INVALID_ARG;
  const Layout L0 = make_layout(*f);
  // Without a variant flag: the asynchronous-copy ring for layers of 64 or
  // more 128-row blocks (it keeps more bytes in flight), else the register
  // ring (fewer instructions; small layers are bound by launch latency).
  const bool wbulk = (flags & W4A16_GEMV_ASYNC_COPY) != 0 ||
                     ((flags & W4A16_GEMV_REGISTER_RING) == 0 && L0.NR >= 64);
  if (ksplit != 0 && ksplit != 1 && ksplit != 2 && ksplit != 4 && ksplit != 8 && ksplit != 16)
    return W4A16_ERR_INVALID_ARG;
  const Layout L = make_layout(*f);
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  GemvPlan plan = gemv_default_plan(L, int(M), dev, wbulk ? kGemvAsyncCopy : kGemvRegisterRing);
  if (shape != 0) plan.rows16 = shape;
  if ((flags & W4A16_GEMV_STAGE_ACTIVATIONS) != 0) plan.stage_x = true;
  if (ksplit != 0) plan.ksplit = ksplit;
  if (!gemv_plan_ok(L, int(M), plan)) return (shape || ksplit) ? W4A16_ERR_INVALID_ARG : W4A16_ERR_UNSUPPORTED;
  uint32_t kflags = flags & (W4A16_GEMV_WEIGHTS_READY | W4A16_GEMV_INPUTS_READY);
  if (kflags & W4A16_GEMV_INPUTS_READY) kflags |= W4A16_GEMV_WEIGHTS_READY;  // inputs ready implies weights ready
  e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_gemv(L, packed, x, y, int(M), plan, kflags, stream);
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

w4a16_status w4a16_gemv(const w4a16_format* f, const void* packed, size_t packed_bytes,
                        const uint16_t* x, uint16_t* y, int64_t M, w4a16_stream_t stream) {
  return gemv_common(f, packed, packed_bytes, x, y, M, 0, 0, 0, stream);
}

w4a16_status w4a16_gemv_ex(const w4a16_format* f, const void* packed, size_t packed_bytes,
                           const uint16_t* x, uint16_t* y, int64_t M, int32_t shape, int32_t ksplit,
                           uint32_t flags, w4a16_stream_t stream) {
  return gemv_common(f, packed, packed_bytes, x, y, M, shape, ksplit, flags, stream);
}

w4a16_status w4a16_gemv_grouped(const w4a16_format* formats, const void* const* packed, const size_t* packed_bytes,
                                int32_t n, const uint16_t* x, uint16_t* const* y, int64_t M, uint32_t flags,
                                w4a16_stream_t stream) {
  if (formats == nullptr || packed == nullptr || packed_bytes == nullptr || x == nullptr || y == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if (n < 1 || n > 4 || M < 1 || M > 16) return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16)) return W4A16_ERR_MISALIGNED;
  if ((flags & ~uint32_t(W4A16_GEMV_WEIGHTS_READY | W4A16_GEMV_ASYNC_COPY | W4A16_GEMV_REGISTER_RING |
                         W4A16_GEMV_INPUTS_READY)) != 0)
    return W4A16_ERR_INVALID_ARG;
  if ((flags & W4A16_GEMV_REGISTER_RING) && (flags & W4A16_GEMV_ASYNC_COPY)) return W4A16_ERR_INVALID_ARG;
  GemvGroup grp;
  grp.n = n;
  int64_t nr = 0;
  const w4a16_format& f0 = formats[0];
  const char* xb = reinterpret_cast<const char*>(x);
  const size_t xbytes = size_t(M) * size_t(f0.K) * 2;
  for (int32_t m = 0; m < n; ++m) {
    const w4a16_format& f = formats[m];
    w4a16_status s = blob_status(&f, packed[m], packed_bytes[m]);
    if (s != W4A16_OK) return s;
    if (f.bits != f0.bits || f.group_size != f0.group_size || f.symmetric != f0.symmetric || f.K != f0.K)
      return W4A16_ERR_INVALID_ARG;
    if (f.has_g_idx || f.has_act_scale) return W4A16_ERR_UNSUPPORTED;
    if (y[m] == nullptr) return W4A16_ERR_INVALID_ARG;
    if (!aligned(y[m], 16)) return W4A16_ERR_MISALIGNED;
    const char* yb = reinterpret_cast<const char*>(y[m]);
    const size_t ybytes = size_t(M) * size_t(f.N) * 2;
    if (xb < yb + ybytes && yb < xb + xbytes) return W4A16_ERR_INVALID_ARG;  // y overlaps x
    const Layout L = make_layout(f);
    grp.views[m] = view_of(L, packed[m]);
    grp.NR[m] = L.NR;
    grp.N[m] = L.N;
    grp.y[m] = y[m];
    nr += L.NR;
  }
  w4a16_format fc = f0;  // the group as one layer: its row blocks one after another
  fc.N = nr * 128;
  if (format_status(&fc) != W4A16_OK) return W4A16_ERR_UNSUPPORTED;
  const Layout Lc = make_layout(fc);
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool wbulk = (flags & W4A16_GEMV_ASYNC_COPY) != 0 ||
                     ((flags & W4A16_GEMV_REGISTER_RING) == 0 && Lc.NR >= 64);
  const GemvPlan plan = gemv_default_plan(Lc, int(M), dev, wbulk ? kGemvAsyncCopy : kGemvRegisterRing);
  if (!gemv_plan_ok(Lc, int(M), plan)) return W4A16_ERR_UNSUPPORTED;
  uint32_t kflags = flags & (W4A16_GEMV_WEIGHTS_READY | W4A16_GEMV_INPUTS_READY);
  if (kflags & W4A16_GEMV_INPUTS_READY) kflags |= W4A16_GEMV_WEIGHTS_READY;
  e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_gemv_group(Lc, grp, x, int(M), plan, kflags, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

size_t w4a16_gemm_workspace_bytes(const w4a16_format* f, int64_t M) {
  if (format_status(f) != W4A16_OK || M < 1) return 0;
  return (f->has_g_idx || f->has_act_scale) ? size_t(M) * size_t(f->K) * 2 : 0;
}

static w4a16_status gemm_common(const w4a16_format* f, const void* packed, size_t packed_bytes,
                                const uint16_t* x, uint16_t* y, int64_t M, void* workspace,
                                size_t workspace_bytes, int32_t tile, int32_t ksplit, w4a16_stream_t stream) {
  w4a16_status s = blob_status(f, packed, packed_bytes);
  if (s != W4A16_OK) return s;
  if (x == nullptr || y == nullptr) return W4A16_ERR_INVALID_ARG;
  if (M < 1 || M > (int64_t(1) << 20)) return W4A16_ERR_INVALID_ARG;
  if (tile < 0 || tile > 6) return W4A16_ERR_INVALID_ARG;
  if (ksplit != 0 && ksplit != 1 && ksplit != 2 && ksplit != 4 && ksplit != 8 && ksplit != 16)
    return W4A16_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16)) return W4A16_ERR_MISALIGNED;
  const size_t xbytes = size_t(M) * size_t(f->K) * 2, ybytes = size_t(M) * size_t(f->N) * 2;
  const char* xb = reinterpret_cast<const char*>(x);
  const char* yb = reinterpret_cast<const char*>(y);
  if (xb < yb + ybytes && yb < xb + xbytes) return W4A16_ERR_INVALID_ARG;
  const size_t need = w4a16_gemm_workspace_bytes(f, M);
  if (workspace_bytes < need) return W4A16_ERR_BUFFER_TOO_SMALL;
  if (need > 0 && workspace == nullptr) return W4A16_ERR_INVALID_ARG;
  if (need > 0 && !aligned(workspace, 16)) return W4A16_ERR_MISALIGNED;
  if (need > 0) {
    const char* wb = static_cast<const char*>(workspace);
    if ((wb < yb + ybytes && yb < wb + need) || (wb < xb + xbytes && xb < wb + need)) return W4A16_ERR_INVALID_ARG;
  }
  DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev.cc_major != 10) return W4A16_ERR_UNSUPPORTED;  // tcgen05 needs a Blackwell datacenter GPU
  const Layout L = make_layout(*f);
  GemmPlan plan = gemm_default_plan(L, M, dev.sm_count);
  if (tile != 0) {
    plan.tile = tile;
    if (ksplit == 0) plan.ksplit = 1;
  }
  if (ksplit != 0) plan.ksplit = ksplit;
  if (!gemm_plan_ok(L, plan)) return W4A16_ERR_INVALID_ARG;
  e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_gemm(L, packed, x, y, M, workspace, plan, stream);
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

w4a16_status w4a16_gemm(const w4a16_format* f, const void* packed, size_t packed_bytes,
                        const uint16_t* x, uint16_t* y, int64_t M, void* workspace,
                        size_t workspace_bytes, w4a16_stream_t stream) {
  return gemm_common(f, packed, packed_bytes, x, y, M, workspace, workspace_bytes, 0, 0, stream);
}

w4a16_status w4a16_gemm_ex(const w4a16_format* f, const void* packed, size_t packed_bytes,
                           const uint16_t* x, uint16_t* y, int64_t M, void* workspace,
                           size_t workspace_bytes, int32_t tile, int32_t ksplit, w4a16_stream_t stream) {
  return gemm_common(f, packed, packed_bytes, x, y, M, workspace, workspace_bytes, tile, ksplit, stream);
}

size_t w4a16_gptq_workspace_bytes(const w4a16_format* f) {
  if (format_status(f) != W4A16_OK || f->has_act_scale) return 0;
  return gptq_workspace_bytes(f->N, f->K);
}

w4a16_status w4a16_gptq(const w4a16_format* f, const uint16_t* w, const uint16_t* x, int64_t T, double damp,
                        uint8_t* q, uint16_t* scales, uint8_t* zeros, int32_t* g_idx, void* workspace,
                        size_t workspace_bytes, w4a16_stream_t stream) {
  w4a16_status s = format_status(f);
  if (s != W4A16_OK) return s;
  if (f->has_act_scale) return W4A16_ERR_UNSUPPORTED;
  if (w == nullptr || x == nullptr || q == nullptr || scales == nullptr || workspace == nullptr)
    return W4A16_ERR_INVALID_ARG;
  if ((zeros == nullptr) != (f->symmetric != 0)) return W4A16_ERR_INVALID_ARG;
  if ((g_idx == nullptr) != (f->has_g_idx == 0)) return W4A16_ERR_INVALID_ARG;
  if (T < 1 || T > (int64_t(1) << 24) || !(damp >= 0.0) || !std::isfinite(damp)) return W4A16_ERR_INVALID_ARG;
  if (!aligned(w, 2) || !aligned(x, 2) || !aligned(scales, 2) || !aligned(g_idx, 4) || !aligned(workspace, 256))
    return W4A16_ERR_MISALIGNED;
  if (workspace_bytes < gptq_workspace_bytes(f->N, f->K)) return W4A16_ERR_BUFFER_TOO_SMALL;
  cudaError_t e = take_injected_launch_error();
  if (e == cudaSuccess) e = launch_gptq(make_layout(*f), w, x, T, damp, q, scales, zeros, g_idx, workspace,
                              static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? W4A16_OK : cuda_fail(e);
}

w4a16_status w4a16_pipeline_timeouts(uint32_t* count) {
  if (count == nullptr) return W4A16_ERR_INVALID_ARG;
  unsigned int c = 0;
  cudaError_t e = take_pipeline_timeouts(&c);
  if (e != cudaSuccess) return cuda_fail(e);
  *count = c;
  return W4A16_OK;
}

}  // extern "C"
