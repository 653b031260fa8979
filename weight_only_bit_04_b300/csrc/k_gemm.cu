// Prefill-sized W4A16 product on the tcgen05 tensor cores (not built yet).
#include <cuda_runtime.h>

#include "internal.h"

namespace w4a16 {

cudaError_t launch_gemm(const Layout&, const void*, const uint16_t*, uint16_t*, int64_t, void*,
                        cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace w4a16
