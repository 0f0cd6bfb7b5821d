// decay_forms.cu -- the scalar-decay and no-decay forms of the recurrence.
//
// The ZeCO pages study the diagonal (per-d_k-row) decay of gated linear
// attention and leave other linear-attention forms to future work (ZeCO,
// Limitations); the LASP page's linear attention has no decay.  A per-token
// scalar decay (RetNet / Lightning style) is the diagonal recurrence with the
// same log-decay in every d_k row, and no decay is log-decay 0, so both run the
// diagonal kernels on a broadcast log-decay.  By the chain rule through the
// broadcast, the gradient of a scalar log-decay is the sum over d_k of the
// per-row gradient.  Where every kernel that reads the log-decay has the form
// built in (the tensor-core path: the decay pass and the dq/dk sweeps), no
// broadcast is made; the dq/dk reverse sweep leaves fp32 sums over blocks of 32
// d_k rows, which the last kernel here adds up per token.
#include "common.cuh"
#include "launch.h"

namespace zeco {
namespace {

// one thread per 4 consecutive elements of a [rows, dk] matrix (dk % 16 == 0)
template <typename T>
__global__ void expand_kernel(const T* __restrict__ g, T* __restrict__ gx, int64_t rows, int dk,
                              bool scalar) {
  const int64_t n4 = rows * dk / 4;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n4;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = e * 4 / dk;
    const float x = scalar ? ld(g + r) : 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) st(gx + e * 4 + u, x);
  }
}

// one warp per row: fp32 sum of the row's dk values
template <typename T>
__global__ void reduce_kernel(const T* __restrict__ dgx, T* __restrict__ dg, int64_t rows, int dk) {
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float s = 0.f;
  for (int i = lane; i < dk; i += 32) s += ld(dgx + r * dk + i);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) st(dg + r, s);
}

// one thread per token: the sum of its nparts partials (partial c at c * rows)
__global__ void sum_parts_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ dg,
                                 int64_t rows, int nparts) {
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int c = 0; c < nparts; ++c) s += part[(size_t)c * rows + r];
    dg[r] = __float2bfloat16_rn(s);
  }
}

}  // namespace

cudaError_t launch_sum_dlog_alpha_parts(const Dims& d, const float* part, void* dg,
                                        cudaStream_t st) {
  const int64_t rows = d.B * d.H * d.T;
  const int64_t nb = (rows + 255) / 256;
  const unsigned blocks = (unsigned)(nb < 65535 * 16 ? nb : 65535 * 16);
  prof_start(st);
  sum_parts_kernel<<<blocks, 256, 0, st>>>(part, (__nv_bfloat16*)dg, rows, (int)(d.dk / 32));
  prof_mark("sum_dlog_alpha_parts", st);
  return cudaGetLastError();
}

cudaError_t launch_expand_log_alpha(const Dims& d, const void* g, void* gx, cudaStream_t st) {
  const int64_t rows = d.B * d.H * d.T;
  const int64_t n4 = rows * d.dk / 4;
  const unsigned blocks = (unsigned)((n4 + 255) / 256 < 65535 * 16 ? (n4 + 255) / 256 : 65535 * 16);
  const bool scalar = d.decay == ZECO_DECAY_SCALAR;
  prof_start(st);
  if (d.bf16)
    expand_kernel<<<blocks, 256, 0, st>>>((const __nv_bfloat16*)g, (__nv_bfloat16*)gx, rows,
                                          (int)d.dk, scalar);
  else
    expand_kernel<<<blocks, 256, 0, st>>>((const float*)g, (float*)gx, rows, (int)d.dk, scalar);
  prof_mark("expand_log_alpha", st);
  return cudaGetLastError();
}

cudaError_t launch_reduce_dlog_alpha(const Dims& d, const void* dgx, void* dg, cudaStream_t st) {
  const int64_t rows = d.B * d.H * d.T;
  const unsigned blocks = (unsigned)((rows * 32 + 255) / 256);
  prof_start(st);
  if (d.bf16)
    reduce_kernel<<<blocks, 256, 0, st>>>((const __nv_bfloat16*)dgx, (__nv_bfloat16*)dg, rows,
                                          (int)d.dk);
  else
    reduce_kernel<<<blocks, 256, 0, st>>>((const float*)dgx, (float*)dg, rows, (int)d.dk);
  prof_mark("reduce_dlog_alpha", st);
  return cudaGetLastError();
}

}  // namespace zeco
