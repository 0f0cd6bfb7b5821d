// tc.cu -- tcgen05 tensor-core path (bf16 I/O, fp32 accumulation in TMEM).
#include "common.cuh"
#include "launch.h"

namespace zeco {

bool tc_supported(const Dims& d) {
  (void)d;
  return false;
}

cudaError_t tc_forward(const Dims&, const void*, const void*, const void*, const void*,
                       const float*, void*, float*, float*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

cudaError_t tc_backward(const Dims&, const void*, const void*, const void*, const void*,
                        const float*, const float*, const void*, const float*, void*, void*,
                        void*, void*, float*, float*, float*, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace zeco
