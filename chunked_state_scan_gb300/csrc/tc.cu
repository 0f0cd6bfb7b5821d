// tc.cu -- the tcgen05 tensor-core path (bf16 I/O, fp32 accumulation):
// launch sequence of the forward and backward.  Steps without a tensor-core
// kernel for the shape run their CUDA-core (SIMT) kernel.
#include "common.cuh"
#include "launch.h"

namespace zeco {

bool tc_supported(const Dims& d) { return tc_state_supported(d); }

bool tc_uses_decay(const Dims& d) { return tc_supported(d) && tc_fwd_supported(d); }

bool tc_uses_dA(const Dims& d) {
  return tc_uses_decay(d) && tc_bwd_qk_supported(d) && tc_dA_supported(d);
}

bool tc_native_forms(const Dims& d, bool bwd) { return bwd ? tc_uses_dA(d) : tc_uses_decay(d); }

// Forward: the decay pass, then pass 1 (on its K~ and e^{b_last}) and the scan on
// the caller's stream while the scores run on the auxiliary stream (they do not
// depend on the scan); pass 2 joins both.  In overlap mode 2 the scan runs on the
// auxiliary stream instead, beside the scores (the pages' schedule).
cudaError_t tc_forward(const Dims& d, const void* q, const void* k, const void* v,
                       const void* g, const float* S0, void* o, float* S_final, float* S_in,
                       float* gamma, const TcOps& ops, cudaStream_t st) {
  if (!tc_fwd_supported(d)) {
    cudaError_t e = tc_chunk_state(d, k, v, g, nullptr, nullptr, S_in, gamma, st);
    if (e != cudaSuccess) return e;
    e = launch_seg_scan_fwd(d, S_in, gamma, S0, S_final, st);
    if (e != cudaSuccess) return e;
    return simt_fwd_out_bf16(d, q, k, v, g, S_in, o, st);
  }
  void* Qt = ops.Qt;
  void* Kt = ops.Kt;
  float* Eb = ops.Eb;
  void* A = ops.A;
  const int mode = overlap_mode(d);
  cudaError_t e = tc_decay(d, q, k, g, Qt, Kt, Eb, st);
  if (e != cudaSuccess) return e;
  if (mode == 3) {
    // pass 2 of a block of segments starts as soon as the scan has given that block
    // its incoming states: the scan runs block by block on the caller's stream, and
    // pass 2 of each block on the auxiliary stream after the scores and after the
    // scan of its block
    const Fork f = fork_begin(st, mode);
    e = tc_A(d, Qt, Kt, A, f.aux);
    if (e == cudaSuccess) e = tc_chunk_state(d, k, v, g, Kt, Eb, S_in, gamma, st);
    const int nb = d.P < kStepEvents ? d.P : kStepEvents;
    for (int b = 0; e == cudaSuccess && b < nb; ++b) {
      const int p0 = (int)((int64_t)d.P * b / nb), p1 = (int)((int64_t)d.P * (b + 1) / nb);
      e = launch_seg_scan_fwd(d, S_in, gamma, S0, S_final, st, p0, p1);
      if (e == cudaSuccess) e = fork_follow(f, st, b);
      if (e == cudaSuccess) e = tc_fwd_out(d, Qt, Kt, v, A, Eb, S_in, o, f.aux, p0, p1 - p0);
    }
    if (e == cudaSuccess) e = fork_mark(f, 0);
    if (e == cudaSuccess) e = fork_join(f, st, 0);
    return e;
  }
  if (mode == 2) {
    // the pages' schedule: the scan on the second stream beside the scores
    e = tc_chunk_state(d, k, v, g, Kt, Eb, S_in, gamma, st);
    if (e != cudaSuccess) return e;
    const Fork f = fork_begin(st, mode);
    e = launch_seg_scan_fwd(d, S_in, gamma, S0, S_final, f.aux);
    if (e == cudaSuccess) e = fork_mark(f, 0);
    if (e == cudaSuccess) e = tc_A(d, Qt, Kt, A, st);
    if (e == cudaSuccess) e = fork_join(f, st, 0);
    if (e != cudaSuccess) return e;
    return tc_fwd_out(d, Qt, Kt, v, A, Eb, S_in, o, st);
  }
  const Fork f = fork_begin(st, mode);
  e = tc_A(d, Qt, Kt, A, f.aux);
  if (e == cudaSuccess) e = fork_mark(f, 0);
  if (e != cudaSuccess) return e;
  e = tc_chunk_state(d, k, v, g, Kt, Eb, S_in, gamma, st);
  if (e == cudaSuccess) e = launch_seg_scan_fwd(d, S_in, gamma, S0, S_final, st);
  if (e == cudaSuccess) e = fork_join(f, st, 0);
  if (e != cudaSuccess) return e;
  return tc_fwd_out(d, Qt, Kt, v, A, Eb, S_in, o, st);
}

// Backward: Q~, K~, e^{b_last} and the masked scores A are the forward's (kept in
// `saved`); the pre-pass, the reverse scan and the dv sweep run on the caller's
// stream while the score gradient dA runs on the auxiliary stream; in overlap mode 4
// (the default) the dq/dk sweeps then run on the high-priority stream beside the dv
// sweep (mode 2: the reverse scan on the auxiliary stream beside dA).
cudaError_t tc_backward(const Dims& d, const void* q, const void* k, const void* v,
                        const void* g, const float* S_in, const float* gamma, const void* d_o,
                        const float* dS_final, void* dq, void* dk, void* dv, void* dg,
                        float* dS0, float* D, float* carry, float* qdq, float* dAf,
                        const TcOps& ops, cudaStream_t st) {
  if (!tc_fwd_supported(d)) {
    cudaError_t e = tc_dstate_local(d, q, d_o, g, nullptr, nullptr, D, st);
    if (e != cudaSuccess) return e;
    e = launch_seg_scan_rev(d, D, S_in, gamma, dS_final, dS0, carry, st);
    if (e != cudaSuccess) return e;
    return simt_bwd_main_bf16(d, q, k, v, g, S_in, d_o, dq, dk, dv, dg, D, carry, qdq, dAf, st);
  }
  const void* Qt = ops.Qt;
  const void* Kt = ops.Kt;
  const float* Eb = ops.Eb;
  const void* A = ops.A;
  const bool qk_tc = tc_uses_dA(d);
  void* dA = ops.dA;
  const int mode = overlap_mode(d);
  cudaError_t e = cudaSuccess;
  if (mode == 4 && qk_tc) {
    // dq/dk on a high-priority stream, dv on the caller's: the dq/dk CTAs are
    // scheduled first and the dv sweep's fill the SMs their last waves leave idle
    const Fork f = fork_begin(st, mode);
    e = tc_dA(d, d_o, v, dA, f.aux);
    if (e == cudaSuccess) e = fork_mark(f, 0);
    if (e == cudaSuccess) e = tc_dstate_local(d, q, d_o, g, Qt, Eb, D, st);
    if (e == cudaSuccess) e = launch_seg_scan_rev(d, D, S_in, gamma, dS_final, dS0, carry, st);
    if (e == cudaSuccess) e = fork_follow_to(f, st, f.hi, 0);  // after the reverse scan
    if (e == cudaSuccess) e = fork_join(f, f.hi, 0);           // and after dA
    if (e == cudaSuccess)
      e = tc_bwd_qk(d, Qt, Kt, v, g, Eb, dA, S_in, d_o, dq, dk, dg, D, carry, qdq, f.hi);
    if (e == cudaSuccess) e = fork_mark_on(f, f.hi, 1);
    if (e == cudaSuccess) e = tc_bwd_dv(d, Qt, Kt, d_o, A, Eb, D, dv, st);
    if (e == cudaSuccess) e = fork_join(f, st, 1);
    return e;
  }
  if (mode == 2) {
    // the pages' schedule: the reverse scan on the second stream beside dA
    e = tc_dstate_local(d, q, d_o, g, Qt, Eb, D, st);
    if (e != cudaSuccess) return e;
    const Fork f = fork_begin(st, mode);
    e = launch_seg_scan_rev(d, D, S_in, gamma, dS_final, dS0, carry, f.aux);
    if (e == cudaSuccess) e = fork_mark(f, 0);
    if (e == cudaSuccess && qk_tc) e = tc_dA(d, d_o, v, dA, st);
    if (e == cudaSuccess) e = fork_join(f, st, 0);
    if (e == cudaSuccess) e = tc_bwd_dv(d, Qt, Kt, d_o, A, Eb, D, dv, st);
  } else {
    const Fork f = fork_begin(st, mode);
    e = qk_tc ? tc_dA(d, d_o, v, dA, f.aux) : cudaSuccess;
    if (e == cudaSuccess) e = fork_mark(f, 0);
    if (e != cudaSuccess) return e;
    e = tc_dstate_local(d, q, d_o, g, Qt, Eb, D, st);
    if (e == cudaSuccess) e = launch_seg_scan_rev(d, D, S_in, gamma, dS_final, dS0, carry, st);
    if (e == cudaSuccess) e = tc_bwd_dv(d, Qt, Kt, d_o, A, Eb, D, dv, st);
    if (e == cudaSuccess) e = fork_join(f, st, 0);
  }
  if (e != cudaSuccess) return e;
  if (qk_tc) return tc_bwd_qk(d, Qt, Kt, v, g, Eb, dA, S_in, d_o, dq, dk, dg, D, carry, qdq, st);
  return simt_bwd_dqk_bf16(d, q, k, v, g, S_in, d_o, dq, dk, dg, D, carry, qdq, dAf, st);
}

}  // namespace zeco
