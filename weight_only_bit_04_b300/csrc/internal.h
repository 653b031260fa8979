// Launchers implemented in the kernel files and called by the C ABI (api.cu).
// Every launcher only enqueues work on `stream` and returns the launch status.
#pragma once

#include <cuda.h>
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

// Limit of the kernels' bounded waits for launches issued now (w4a16_set_wait_limit_ns).
unsigned long long wait_limit_ns();
// The error w4a16_debug_fail_next_launch left for the next launch, taken
// (cudaSuccess when none): every entry point calls this just before it
// launches and reports a non-success value as if the launch had failed.
cudaError_t take_injected_launch_error();

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

// Chained decode products (w4a16_chain_*), run by the decode stream
// (decode_stream.cuh): one persistent launch over a table of layer slices.
// A slice is a run of row groups (32 rows) of one layer; thread block b owns
// a contiguous share of every slice's row groups (positions rotated by `rot`)
// and, before it reads the slice's activations, waits until every block has
// counted slice wait_hi: blocks finish slices in table order, so that covers
// the whole range [wait_lo, wait_hi].
struct StreamJob {
  const uint16_t* x;        // fp16 [M][K]
  uint16_t* y;              // fp16 [M][N]
  const uint32_t* scales2;  // the blob's scale pairs
  const uint8_t* zeros;     // the blob's zero points (nullptr when symmetric)
  int N, K, KB, G;          // the layer's shape (KB 64-column blocks, G groups)
  int rg_first, n_rg;       // this slice's row groups
  int rot;                  // block position of the slice's first share
  int wait_lo, wait_hi;     // slices to wait for (none when wait_lo > wait_hi)
  int map;                  // index of the layer's first tensor map (the codes as boxes of
                            // CU, CU/2, ..., 1 units, CU = units per ring slot, at most 32)
  int signal;               // 1: a later slice waits for this one as the last of its range,
                            // so every block counts it as done (fenced); 0: not counted
  int pad;
};
static_assert(sizeof(StreamJob) == 80, "the layer table is read as 16-byte vectors");
struct StreamLaunch {
  const StreamJob* jobs;    // device table
  const CUtensorMap* maps;  // device array, 64-byte aligned
  unsigned int* done;       // per slice a count of finished blocks (128-byte stride), then the abort flag
  int n_jobs, M;
  int x_buf_bytes;          // bytes of the staged-activation area (0: activations not staged)
  int x_nbuf;               // 2: two staged-activation buffers, the first at the start of the area
                            // and the second ending at its end, each sized for its layer; 0: none
  unsigned long long wait_ns;  // limit of every bounded wait (wait_limit_ns() at launch)
};
cudaError_t launch_stream(const StreamLaunch& c, int bits, int gsize, bool sym, int sm_count, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (k_gemm.cu):
// a tensor of `rank` dimensions (dims[0] innermost), byte strides of the
// outer dimensions, a box per copy; no interleave, no swizzle, 256-byte L2
// promotion, out-of-range elements read as zero.
cudaError_t encode_tiled_map(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                             const uint64_t* dims, const uint64_t* strides, const uint32_t* box);

// Device-side counts of bounded pipeline waits that gave up, read and reset
// (k_gemm.cu for the GEMM; the GEMV translation units for the GEMV's and the
// chained launch's waits).
cudaError_t take_pipeline_timeouts(unsigned int* count);
cudaError_t take_gemv_timeouts(unsigned int* count);
// First failed index check of a debug build (-DW4A16_DEBUG_CHECKS), read and reset.
cudaError_t take_debug_error(unsigned int* word);

}  // namespace w4a16
