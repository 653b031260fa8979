// The decode-sized product compiled for 8-bit codes.
#include "decode_stream.cuh"

namespace w4a16 {

cudaError_t launch_gemv_b8(const Layout& L, const void* blob, const uint16_t* x, uint16_t* y, int M,
                           const GemvPlan& plan, uint32_t flags, cudaStream_t stream) {
  return launch_gemv_bits<8>(L, blob, x, y, M, plan, flags, stream);
}

cudaError_t launch_gemv_group_b8(const Layout& Lc, const GemvGroup& grp, const uint16_t* x, int M,
                                 const GemvPlan& plan, uint32_t flags, cudaStream_t stream) {
  return launch_gemv_group_bits<8>(Lc, grp, x, M, plan, flags, stream);
}

cudaError_t launch_stream_b8(const StreamLaunch& c, int gsize, bool sym, int sm_count, cudaStream_t stream) {
  return launch_stream_bits<8>(c, gsize, sym, sm_count, stream);
}

cudaError_t take_gemv_timeouts_b8(unsigned int* count) { return take_local_gemv_timeouts(count); }
cudaError_t take_debug_error_b8(unsigned int* word) { return take_local_debug_error(word); }

}  // namespace w4a16
