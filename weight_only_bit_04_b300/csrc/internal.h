// Launchers implemented in the kernel files and called by the C ABI (api.cu).
// Every launcher only enqueues work on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>

#include "layout.h"

namespace w4a16 {

// Device attributes cached per device.
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
  int cc_major, cc_minor;
};
cudaError_t device_info(DeviceInfo* out);

// Record e for w4a16_last_cuda_error() (calling thread) and return W4A16_ERR_CUDA.
w4a16_status cuda_error_status(cudaError_t e);

// ascale: per-input-channel scale (original column order) applied to the
// weights before quantizing, or nullptr.
cudaError_t launch_quantize_rtn(const Layout& L, const uint16_t* w, const int32_t* perm_dev,
                                const uint16_t* ascale, uint8_t* q, uint16_t* scales, uint8_t* zeros,
                                cudaStream_t stream);

// ascale: the act scale to store (original column order) when L.awq.
cudaError_t launch_pack(const Layout& L, const uint8_t* q, const uint16_t* scales,
                        const uint8_t* zeros, const uint16_t* ascale, void* blob, cudaStream_t stream);

cudaError_t launch_dequant(const Layout& L, const void* blob, uint16_t* w_out,
                           cudaStream_t stream);

constexpr int kGemvRegisterRing = 1; // weights loaded straight into a register ring
constexpr int kGemvAsyncCopy = 2;    // each thread lands its own weight loads in a shared-memory ring (cp.async)
struct GemvPlan {
  int kind;     // kGemvRegisterRing or kGemvAsyncCopy
  int rows16;   // 16-row tiles per CTA (2, 4, 8), both kernels
  int stages;   // not read by the kernels: the ring depth is fixed per code width (kWbSlots)
  int ksplit;   // CTAs per cluster along K
  bool stage_x; // register ring: copy the block's activations to shared memory first
};
GemvPlan gemv_default_plan(const Layout& L, int M, const DeviceInfo& dev, int kind);
bool gemv_plan_ok(const Layout& L, int M, const GemvPlan& p);
constexpr uint32_t kGemvWeightsReady = W4A16_GEMV_WEIGHTS_READY;
constexpr uint32_t kGemvStageActivationsFlag = W4A16_GEMV_STAGE_ACTIVATIONS;
constexpr uint32_t kGemvAsyncCopyFlag = W4A16_GEMV_ASYNC_COPY;
constexpr uint32_t kGemvInputsReady = W4A16_GEMV_INPUTS_READY;
cudaError_t launch_gemv(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y,
                        int M, const GemvPlan& plan, uint32_t flags, cudaStream_t stream);

// GEMM plan. tile: 1 = 128 weight rows x 256 tokens per thread block (2
// dequantization warp sets), 2 = 256 rows x 128 tokens (2 sets), 3 = 128 x 256
// with 4 sets, 4 = 128 x 256 with 1 set, 5 = 128 x 128 (2 sets, two blocks per
// SM), 6 = 128 x 64 (2 sets, two blocks per SM). ksplit: blocks of a cluster
// splitting K (1, 2, 4, 8, 16).
struct GemmPlan {
  int tile;
  int ksplit;
};
GemmPlan gemm_default_plan(const Layout& L, int64_t M, int sm_count);
bool gemm_plan_ok(const Layout& L, const GemmPlan& p);
cudaError_t launch_gemm(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y,
                        int64_t M, void* workspace, const GemmPlan& plan, cudaStream_t stream);

// Grouped decode product: up to 4 layers with the same K, format and input,
// in one launch (their row blocks one after another).
struct GemvGroup {
  int n;
  BlobView views[4];
  int64_t NR[4];
  int64_t N[4];
  uint16_t* y[4];
};
cudaError_t launch_gemv_group(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M, const GemvPlan& plan,
                              uint32_t flags, cudaStream_t stream);

// GPTQ (k_gptq.cu): workspace for an N x K layer, and the whole calibration
// on `stream` (all fp64 on the device).
size_t gptq_workspace_bytes(int64_t N, int64_t K);
cudaError_t launch_gptq(const Layout& L, const uint16_t* w, const uint16_t* x, int64_t T, double damp, uint8_t* q,
                        uint16_t* scales, uint8_t* zeros, int32_t* g_idx, void* workspace, cudaStream_t stream);

// Chained decode products (w4a16_chain_*): one persistent launch runs a list
// of layers. Work item = one 32-row group of a layer (the full K); a layer's
// items wait for the completion counters of the layers whose outputs they
// read.
struct ChainJob {
  const uint32_t* qweight;
  const uint32_t* scales2;
  const uint8_t* zeros;  // nullptr when symmetric
  const uint16_t* x;
  uint16_t* y;
  int N, K, G, KB;
  int item0, items;      // first global work item and count (32-row groups)
  int wait_lo, wait_hi;  // layers this layer waits for (none when wait_lo > wait_hi)
};
struct ChainLaunch {
  int bits, gsize, M;
  bool sym;
  int n_jobs;
  int total_items;
  int sm_count;
  const ChainJob* jobs;  // device table
  unsigned int* done;    // per layer a count of finished items, then the abort flag and the next-item
                         // counter, each in its own 128-byte line
};
cudaError_t launch_chain(const ChainLaunch& c, cudaStream_t stream);

// Device-side counts of bounded pipeline waits that gave up, read and reset
// (k_gemm.cu for the GEMM; the GEMV translation units for the GEMV's and the
// chained launch's waits).
cudaError_t take_pipeline_timeouts(unsigned int* count);
cudaError_t take_gemv_timeouts(unsigned int* count);

}  // namespace w4a16
