// w4a16_quantize_rtn_noalloc: the round-to-nearest quantizer for callers that
// cannot allocate device memory.
//
// w4a16_quantize_rtn needs a caller-provided workspace under act order (the
// group-sorted column list, K int32). Some callers cannot obtain one: code that
// runs where cudaMalloc is not allowed or not available (inside a framework or
// plugin that owns every device allocation, a process whose allocator is
// already at its limit, a real-time path that must not allocate). This variant
// keeps that scratch in a fixed array in device memory that belongs to the
// library instead, and its host side uses only fixed static buffers too.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace w4a16 {
namespace {

// Largest K the fixed scratch holds: 65536 columns = 256 KiB of device memory,
// held by every GPU that loads the library until the process exits.
constexpr int64_t kNoAllocMaxK = 65536;
constexpr int64_t kNoAllocMaxGroups = kNoAllocMaxK / 32;

static __device__ __align__(256) int32_t g_rtn_scratch[kNoAllocMaxK];

// Device address of g_rtn_scratch per device, looked up with that device
// current (in host code the symbol's name is only a host-side stand-in). A
// successful lookup is kept; a failed one is tried again on the next call.
constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
int32_t* g_addr[kMaxDevices];

// Host staging for the column list and the group counts: static, shared by
// all calls, serialised by this mutex, which is held until the call's copy
// and its kernel have both been queued (so that on one stream every copy is
// followed by its own kernel).
std::mutex g_host_mutex;
int32_t g_host_perm[kNoAllocMaxK];
int32_t g_host_count[kNoAllocMaxGroups];

cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_rtn_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" {

w4a16_status w4a16_quantize_rtn_noalloc(const w4a16_format* f, const uint16_t* w, const int32_t* g_idx,
                                        uint8_t* q, uint16_t* scales, uint8_t* zeros,
                                        w4a16_stream_t stream) {
  w4a16_status s = w4a16_check_format(f);
  if (s != W4A16_OK) return s;
  if (w == nullptr || q == nullptr || scales == nullptr) return W4A16_ERR_INVALID_ARG;
  if ((zeros == nullptr) != (f->symmetric != 0)) return W4A16_ERR_INVALID_ARG;
  if ((g_idx == nullptr) != (f->has_g_idx == 0)) return W4A16_ERR_INVALID_ARG;
  if (f->has_act_scale) return W4A16_ERR_INVALID_ARG;  // the AWQ quantizer takes the scale
  if ((reinterpret_cast<uintptr_t>(w) & 15) != 0 || (reinterpret_cast<uintptr_t>(scales) & 1) != 0)
    return W4A16_ERR_MISALIGNED;
  if (f->has_g_idx && f->K > kNoAllocMaxK) return W4A16_ERR_BUFFER_TOO_SMALL;  // beyond the fixed scratch
  const Layout L = make_layout(*f);
  if (!f->has_g_idx) {
    cudaError_t e = take_injected_launch_error();
    if (e == cudaSuccess) e = launch_quantize_rtn(L, w, nullptr, nullptr, q, scales, zeros, stream);
    return e == cudaSuccess ? W4A16_OK : cuda_error_status(e);
  }
  int32_t* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return cuda_error_status(e);
  std::lock_guard<std::mutex> lock(g_host_mutex);
  const int64_t K = f->K, G = f->K / f->group_size;
  for (int64_t t = 0; t < G; ++t) g_host_count[t] = 0;
  for (int64_t k = 0; k < K; ++k) {
    const int32_t t = g_idx[k];
    if (t < 0 || t >= G) return W4A16_ERR_INVALID_ARG;
    ++g_host_count[t];
  }
  // Every group has exactly group_size members; stable group-sorted order.
  for (int64_t t = 0; t < G; ++t) {
    if (g_host_count[t] != f->group_size) return W4A16_ERR_INVALID_ARG;
    g_host_count[t] = int32_t(t * f->group_size);  // next free slot of group t
  }
  for (int64_t k = 0; k < K; ++k) g_host_perm[g_host_count[g_idx[k]]++] = int32_t(k);
  e = take_injected_launch_error();
  if (e != cudaSuccess) return cuda_error_status(e);
  // Pageable source: the copy has read the host buffer when it returns.
  e = cudaMemcpyAsync(scratch, g_host_perm, size_t(K) * 4, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return cuda_error_status(e);
  // Queued while the lock is held: the next call's copy lands after this kernel on the same stream.
  e = launch_quantize_rtn(L, w, scratch, nullptr, q, scales, zeros, stream);
  return e == cudaSuccess ? W4A16_OK : cuda_error_status(e);
}

}  // extern "C"
