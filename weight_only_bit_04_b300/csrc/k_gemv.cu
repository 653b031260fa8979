// Planning and dispatch of the decode-sized product. The kernels live in
// gemv_impl.cuh (one layer or a group) and decode_stream.cuh (a list of layers); k_gemv_b3.cu, k_gemv_b4.cu and k_gemv_b8.cu compile them for
// 3-, 4- and 8-bit codes.
#include "gemv_impl.cuh"

namespace w4a16 {

cudaError_t launch_gemv_b3(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                           const GemvPlan& plan, uint32_t flags, cudaStream_t stream);
cudaError_t launch_gemv_b4(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                           const GemvPlan& plan, uint32_t flags, cudaStream_t stream);
cudaError_t launch_gemv_b8(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                           const GemvPlan& plan, uint32_t flags, cudaStream_t stream);
cudaError_t launch_gemv_group_b3(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M,
                                 const GemvPlan& plan, uint32_t flags, cudaStream_t stream);
cudaError_t launch_gemv_group_b4(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M,
                                 const GemvPlan& plan, uint32_t flags, cudaStream_t stream);
cudaError_t launch_gemv_group_b8(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M,
                                 const GemvPlan& plan, uint32_t flags, cudaStream_t stream);
cudaError_t launch_stream_b3(const StreamLaunch& c, int gsize, bool sym, int sm_count, cudaStream_t stream);
cudaError_t launch_stream_b4(const StreamLaunch& c, int gsize, bool sym, int sm_count, cudaStream_t stream);
cudaError_t launch_stream_b8(const StreamLaunch& c, int gsize, bool sym, int sm_count, cudaStream_t stream);
cudaError_t take_gemv_timeouts_b3(unsigned int* count);
cudaError_t take_gemv_timeouts_b4(unsigned int* count);
cudaError_t take_gemv_timeouts_b8(unsigned int* count);
cudaError_t take_debug_error_b3(unsigned int* word);
cudaError_t take_debug_error_b4(unsigned int* word);
cudaError_t take_debug_error_b8(unsigned int* word);

bool gemv_plan_ok(const Layout& L, int M, const GemvPlan& p) {
  if (!valid_ksplit(p.ksplit)) return false;
  if (p.kind == kGemvRegisterRing || p.kind == kGemvAsyncCopy) {
    if (p.rows16 != 2 && p.rows16 != 4 && p.rows16 != 8) return false;
    const bool wb = p.kind == kGemvAsyncCopy;
    return ring_smem(L, M, kb_per_cta_of(L, p.ksplit), gemv_staged(L) || p.stage_x, wb, p.stages).total <=
           kMaxGemvSmem;
  }
  return false;
}

GemvPlan gemv_default_plan(const Layout& L, int M, const DeviceInfo& dev, int kind) {
  if (kind == kGemvRegisterRing || kind == kGemvAsyncCopy) {
    // Measured on B300 (graph-replayed sweeps of 4096..28672-row layers): the
    // register-ring stream runs best with about 1.35 thread blocks per SM,
    // each warp keeping at least two 64-column blocks; among equally close
    // plans, fewer K splits and then fewer rows per block win.
    const int64_t ntiles = L.NR * 8;
    const double target = 1.35 * dev.sm_count;
    const int depth = kind == kGemvAsyncCopy ? 4 : 0;
    GemvPlan best{kind, 8, depth, 1, false};
    double best_dist = 1e30;
    for (int ks : {1, 2, 4, 8, 16}) {
      for (int rt : {2, 4, 8}) {
        GemvPlan p{kind, rt, depth, ks, false};
        if (!gemv_plan_ok(L, M, p)) continue;
        const int64_t ctas = (ntiles / rt) * ks;
        const int64_t kbc = kb_per_cta_of(L, ks);
        const int64_t per_warp = kbc / (kWarps / (rt / kTilesPerWarp));
        if (per_warp < 2) continue;
        const double d = std::fabs(std::log(double(ctas) / target));
        if (d < best_dist - 1e-9) {
          best_dist = d;
          best = p;
        }
      }
    }
    return best;
  }
  return GemvPlan{kGemvRegisterRing, 8, 0, 1, false};
}

cudaError_t launch_gemv(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                        const GemvPlan& plan, uint32_t flags, cudaStream_t stream) {
  if (L.bits == 8) return launch_gemv_b8(L, blob, x, y, M, plan, flags, stream);
  if (L.bits == 3) return launch_gemv_b3(L, blob, x, y, M, plan, flags, stream);
  return launch_gemv_b4(L, blob, x, y, M, plan, flags, stream);
}

cudaError_t launch_gemv_group(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M, const GemvPlan& plan,
                              uint32_t flags, cudaStream_t stream) {
  if (Lc.bits == 8) return launch_gemv_group_b8(Lc, grp, x, M, plan, flags, stream);
  if (Lc.bits == 3) return launch_gemv_group_b3(Lc, grp, x, M, plan, flags, stream);
  return launch_gemv_group_b4(Lc, grp, x, M, plan, flags, stream);
}

cudaError_t launch_stream(const StreamLaunch& c, int bits, int gsize, bool sym, int sm_count, cudaStream_t stream) {
  if (bits == 8) return launch_stream_b8(c, gsize, sym, sm_count, stream);
  if (bits == 3) return launch_stream_b3(c, gsize, sym, sm_count, stream);
  return launch_stream_b4(c, gsize, sym, sm_count, stream);
}

cudaError_t take_debug_error(unsigned int* word) {
  unsigned int w[3] = {0, 0, 0};
  cudaError_t e = take_debug_error_b4(&w[0]);
  if (e == cudaSuccess) e = take_debug_error_b8(&w[1]);
  if (e == cudaSuccess) e = take_debug_error_b3(&w[2]);
  if (e != cudaSuccess) return e;
  *word = w[0] ? w[0] : w[1] ? w[1] : w[2];
  return cudaSuccess;
}

cudaError_t take_gemv_timeouts(unsigned int* count) {
  unsigned int a = 0, b = 0, c = 0;
  cudaError_t e = take_gemv_timeouts_b4(&a);
  if (e != cudaSuccess) return e;
  e = take_gemv_timeouts_b8(&b);
  if (e != cudaSuccess) return e;
  e = take_gemv_timeouts_b3(&c);
  if (e != cudaSuccess) return e;
  *count = a + b + c;
  return cudaSuccess;
}

}  // namespace w4a16
