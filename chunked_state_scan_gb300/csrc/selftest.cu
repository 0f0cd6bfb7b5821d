// selftest.cu -- a diagnostic that exercises the bounded mbarrier wait of the
// tensor-core kernels on the GPU: one thread waits on a barrier that nothing
// will ever complete, gives up after the wait's time limit, records the
// timeout in this file's status flag and returns, leaving the context usable.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
namespace {

__device__ int g_selftest_status = 0;

__global__ void bounded_wait_kernel() {
  __shared__ uint64_t bar;
  tc::mbar_init(&bar, 1);  // expects one arrive, which never comes
  tc::fence_mbar_init();
  if (!tc::mbar_wait(&bar, 0u)) atomicExch(&g_selftest_status, 1);
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
  zeco::bounded_wait_kernel<<<1, 1, 0, (cudaStream_t)stream>>>();
  return cudaGetLastError() == cudaSuccess ? ZECO_OK : ZECO_ERR_CUDA;
}
