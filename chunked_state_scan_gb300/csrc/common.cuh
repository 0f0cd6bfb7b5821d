// common.cuh -- shared definitions of the CUDA library (internal).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/zeco_gla.h"

namespace zeco {

// Problem description handed from the C ABI to the kernel launchers.
struct Dims {
  int64_t B, H, T, dk, dv;
  int P, K, C;
  int64_t L;  // tokens per segment
  bool bf16;
  int decay;  // zeco_decay
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Operands of the tensor-core sweeps computed once by the forward and kept in
// `saved` for the backward: Q~, K~ [B,H,T,dk] bf16, e^{b_last} of every chunk
// [B,H,T/64,dk] fp32 (tc_decay.cu) and the masked intra-chunk scores A
// [B,H,T,64] bf16 (tc_scores.cu).
struct DecayLayout {
  size_t Qt_off, Kt_off, Eb_off, A_off, total;
};
// One [B,H,T,64] bf16 score array (A, or the backward's dA).
inline size_t scores_bytes(const Dims& d) { return (size_t)d.B * d.H * d.T * 64 * 2; }
inline DecayLayout decay_layout(const Dims& d, size_t base) {
  DecayLayout l;
  const size_t n = (size_t)d.B * d.H * d.T * d.dk;
  l.Qt_off = align_up(base, 256);
  l.Kt_off = align_up(l.Qt_off + n * 2, 256);
  l.Eb_off = align_up(l.Kt_off + n * 2, 256);
  l.A_off = align_up(l.Eb_off + n / 64 * sizeof(float), 256);
  l.total = align_up(l.A_off + scores_bytes(d), 256);
  return l;
}

// Byte layout of the `saved` buffer (with `ops`: followed by the operands
// above) and of the backward workspace.
struct SavedLayout {
  size_t S_in_off, gamma_off;
  DecayLayout ops;
  size_t total;
};
struct BwdWsLayout {
  size_t D_off, carry_off, qdq_off, dAf_off, total;
};

inline SavedLayout saved_layout(const Dims& d, bool ops) {
  SavedLayout s;
  const size_t bh = (size_t)d.B * d.H;
  s.S_in_off = 0;
  s.gamma_off = align_up(bh * (d.P + 1) * d.dk * d.dv * sizeof(float), 256);
  const size_t end = align_up(s.gamma_off + bh * d.P * d.dk * sizeof(float), 256);
  s.ops = decay_layout(d, end);
  s.total = ops ? s.ops.total : end;
  return s;
}

// simt_dA: the backward runs the CUDA-core dq/dk kernel, which reads the
// intra-chunk score gradient dA [B,H,T,C] fp32 from here (at dAf_off).
inline BwdWsLayout bwd_ws_layout(const Dims& d, bool simt_dA) {
  BwdWsLayout w;
  const size_t bh = (size_t)d.B * d.H;
  w.D_off = 0;
  w.carry_off = align_up(bh * (d.P + 1) * d.dk * d.dv * sizeof(float), 256);
  w.qdq_off = align_up(w.carry_off + bh * d.P * d.dk * sizeof(float), 256);
  w.dAf_off = align_up(w.qdq_off + bh * d.T * d.dk * sizeof(float), 256);
  w.total = simt_dA ? align_up(w.dAf_off + bh * d.T * d.C * sizeof(float), 256) : w.dAf_off;
  return w;
}

// SCALAR / NONE decay forms (decay_forms.cu): the log-decay broadcast to
// [B,H,T,dk] and, backward, the per-row gradient [B,H,T,dk] (I/O dtype).
struct FormsLayout {
  size_t gx_off, dgx_off, total;
};
// native: the form is read in its own layout (tc_native_forms); then only the
// SCALAR backward needs scratch, the fp32 partial sums [dk / 32][B,H,T] of its
// gradient (at dgx_off).
inline FormsLayout forms_layout(const Dims& d, size_t base, bool bwd, bool native) {
  FormsLayout l;
  const size_t rows = (size_t)d.B * d.H * d.T;
  const size_t n = rows * d.dk * (d.bf16 ? 2 : 4);
  l.gx_off = align_up(base, 256);
  if (native) {
    l.dgx_off = l.gx_off;
    l.total = (bwd && d.decay == ZECO_DECAY_SCALAR)
                  ? align_up(l.dgx_off + rows * (size_t)(d.dk / 32) * 4, 256)
                  : base;
    return l;
  }
  l.dgx_off = align_up(l.gx_off + n, 256);
  l.total = d.decay == ZECO_DECAY_DIAG ? base : (bwd ? align_up(l.dgx_off + n, 256) : l.dgx_off);
  return l;
}

// ------------------------------------------------------------ element I/O

template <typename T>
__device__ __forceinline__ float ld(const T* p);
template <>
__device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void st(T* p, float x);
template <>
__device__ __forceinline__ void st<float>(float* p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

// ------------------------------------------------------- launch bookkeeping

// Per-kernel timing marks (see zeco_set_profile_events); no-ops when off.
// prof_start right before a kernel's launch, prof_mark(name) right after it,
// both on the stream the kernel is launched on.
void prof_start(cudaStream_t st);
void prof_mark(const char* kernel, cudaStream_t st);

// Sets the dynamic shared-memory limit of a kernel once per process.
template <typename F>
inline cudaError_t allow_smem(F* kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace zeco
