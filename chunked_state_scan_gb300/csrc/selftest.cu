// selftest.cu -- a diagnostic that exercises the bounded mbarrier waits of the
// tensor-core kernels on the GPU: four warps each wait kWaits times on
// barriers that nothing will ever complete.  The first wait to reach its time
// limit gives up and sets the CTA's abort word; every other wait then gives up
// within 64 polls, so the kernel ends after about one time limit (not one per wait),
// records the timeout in this file's status flag and leaves the context usable.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
namespace {

constexpr int kWarps = 4;
constexpr int kWaits = 64;  // waits per thread, all on barriers that never complete

__device__ int g_selftest_status = 0;

__global__ void __launch_bounds__(kWarps * 32) bounded_wait_kernel() {
  __shared__ uint64_t bar[kWarps];
  __shared__ int abort_word;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w) tc::mbar_init(&bar[w], 1);  // one arrive each, never made
    abort_word = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  const tc::Waits wait{tc::smem_u32(&abort_word), &g_selftest_status};
  // parity 0 is the phase in progress, which never completes
  for (int i = 0; i < kWaits; ++i) (void)wait(&bar[threadIdx.x >> 5], 0u);
  __syncthreads();
}

}  // namespace

int selftest_take_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_status, sizeof(v)) != cudaSuccess) return -1;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace zeco

extern "C" int zeco_selftest_bounded_wait(zeco_stream_t stream) {
  zeco::bounded_wait_kernel<<<1, zeco::kWarps * 32, 0, (cudaStream_t)stream>>>();
  return cudaGetLastError() == cudaSuccess ? ZECO_OK : ZECO_ERR_CUDA;
}
