// launch.h -- internal kernel launchers (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace zeco {

// ---- auxiliary stream for the scan-independent passes (overlap.cu) -----
struct Fork {
  cudaStream_t aux;   // where the forked kernels go (the caller's stream when off)
  cudaStream_t hi;    // a second one at the highest priority (the caller's when off)
  cudaEvent_t ev[2];  // recorded on aux by fork_mark, waited on by fork_join
  cudaEvent_t* step;  // recorded on the caller's stream by fork_follow
  bool on;
};
// Forks from st (aux waits for st's work so far); off in schedule 0.
Fork fork_begin(cudaStream_t st, int mode);
// The schedule chosen with zeco_set_overlap: 0 one stream, 1 the scan-independent
// passes on the auxiliary stream, 2 the segment scan on the auxiliary stream, 3 pass 2
// per block of segments as soon as the scan has reached it, 4 (default) mode 1 with
// the dq/dk sweeps on the high-priority stream beside the dv sweep.  The schedule
// a call of shape d runs: the one set, except that the default (4) runs on one
// stream (0) when the segments hold fewer than 4 chunks -- there every kernel is
// bound by its segment-state traffic and the streams only contend (measured: at 2
// chunks per segment 84.0 ms on one stream against 87.3 ms).
int overlap_mode(const Dims& d);
// Records event i (of 2) on the auxiliary stream, or on stream s (f.aux or f.hi).
cudaError_t fork_mark(const Fork& f, int i);
cudaError_t fork_mark_on(const Fork& f, cudaStream_t s, int i);
// Makes st wait for event i.
cudaError_t fork_join(const Fork& f, cudaStream_t st, int i);
// Makes the auxiliary stream (or stream `to`) wait for st's work so far (event i
// of kStepEvents).
constexpr int kStepEvents = 8;
cudaError_t fork_follow(const Fork& f, cudaStream_t st, int i);
cudaError_t fork_follow_to(const Fork& f, cudaStream_t st, cudaStream_t to, int i);

// ---- bounded-wait flags of the tensor-core kernels: read and clear; -1 when
//      the flag cannot be read
int tc_bwd_qk_take_status();
int tc_fwd_take_status();
int tc_scores_take_status();
int tc_state_take_status();
int selftest_take_status();

// ---- decay forms (decay_forms.cu) --------------------------------------
// gx[b,h,t,i] = g[b,h,t] (SCALAR) or 0 (NONE)
cudaError_t launch_expand_log_alpha(const Dims& d, const void* g, void* gx, cudaStream_t st);
// dg[b,h,t] = sum_i dgx[b,h,t,i] (SCALAR)
cudaError_t launch_reduce_dlog_alpha(const Dims& d, const void* dgx, void* dg, cudaStream_t st);
// dg[b,h,t] = sum_c part[c][b,h,t], c < d_k / 32 (SCALAR on the tensor-core path:
// part holds the dq/dk reverse sweep's fp32 sums over blocks of 32 rows)
cudaError_t launch_sum_dlog_alpha_parts(const Dims& d, const float* part, void* dg,
                                        cudaStream_t st);

// ---- segment scans (scan.cu) ------------------------------------------
// segments [p_begin, p_end) (p_end < 0: to the last); S_final when p_end is the last
cudaError_t launch_seg_scan_fwd(const Dims& d, float* S_in, const float* gamma, const float* S0,
                                float* S_final, cudaStream_t st, int p_begin = 0,
                                int p_end = -1);
cudaError_t launch_seg_scan_rev(const Dims& d, float* D, const float* S_in, const float* gamma,
                                const float* dS_final, float* dS0, float* carry,
                                cudaStream_t st);

// ---- fp32 SIMT path (simt.cu) -----------------------------------------
// Shared memory the SIMT kernels need for this shape (bytes, max over kernels).
size_t simt_smem_bytes(const Dims& d);
cudaError_t simt_forward(const Dims& d, const void* q, const void* k, const void* v,
                         const void* g, const float* S0, void* o, float* S_final, float* S_in,
                         float* gamma, cudaStream_t st);
cudaError_t simt_backward(const Dims& d, const void* q, const void* k, const void* v,
                          const void* g, const float* S_in, const float* gamma, const void* d_o,
                          const float* dS_final, void* dq, void* dk, void* dv, void* dg,
                          float* dS0, float* D, float* carry, float* qdq, float* dA,
                          cudaStream_t st);

cudaError_t simt_fwd_out_bf16(const Dims& d, const void* q, const void* k, const void* v,
                              const void* g, const float* S_in, void* o, cudaStream_t st);
cudaError_t simt_bwd_main_bf16(const Dims& d, const void* q, const void* k, const void* v,
                               const void* g, const float* S_in, const void* d_o, void* dq,
                               void* dk, void* dv, void* dg, float* D, float* carry, float* qdq,
                               float* dA, cudaStream_t st);

cudaError_t simt_bwd_dqk_bf16(const Dims& d, const void* q, const void* k, const void* v,
                              const void* g, const float* S_in, const void* d_o, void* dq,
                              void* dk, void* dg, float* D, float* carry, float* qdq, float* dA,
                              cudaStream_t st);

// ---- tcgen05 tensor-core path (tc_*.cu) --------------------------------
bool tc_state_supported(const Dims& d);
// Segment states; with Eb != NULL the operand is the decay pass's K~ (resp. Q~)
// and the per-chunk e^{b_last} replaces log_alpha (tc_state.cu, PRE).
cudaError_t tc_chunk_state(const Dims& d, const void* k, const void* v, const void* g,
                           const void* Kt, const float* Eb, float* S_in, float* gamma,
                           cudaStream_t st);
cudaError_t tc_dstate_local(const Dims& d, const void* q, const void* d_o, const void* g,
                            const void* Qt, const float* Eb, float* D, cudaStream_t st);
bool tc_fwd_supported(const Dims& d);
// Q~ = bf16(q e^{b}), K~ = bf16(k e^{-b}) and e^{b_last} per chunk (tc_decay.cu);
// g in the layout of d.decay: [B,H,T,dk] (DIAG), [B,H,T] (SCALAR), unread (NONE)
cudaError_t tc_decay(const Dims& d, const void* q, const void* k, const void* g, void* Qt,
                     void* Kt, float* Eb, cudaStream_t st);
// segments [p_begin, p_begin + p_count) (p_count < 0: all)
cudaError_t tc_fwd_out(const Dims& d, const void* Qt, const void* Kt, const void* v,
                       const void* A, const float* Eb, const float* S_in, void* o,
                       cudaStream_t st, int p_begin = 0, int p_count = -1);
cudaError_t tc_bwd_dv(const Dims& d, const void* Qt, const void* Kt, const void* d_o,
                      const void* A, const float* Eb, const float* D, void* dv,
                      cudaStream_t st);
// masked bf16 A = Q~ K~^T and dA = do v^T of every chunk (tc_scores.cu)
bool tc_A_supported(const Dims& d);
cudaError_t tc_A(const Dims& d, const void* Qt, const void* Kt, void* P, cudaStream_t st);
bool tc_dA_supported(const Dims& d);
cudaError_t tc_dA(const Dims& d, const void* d_o, const void* v, void* P, cudaStream_t st);
bool tc_bwd_qk_supported(const Dims& d);
// g and dg by d.decay: DIAG [B,H,T,dk] bf16 both; SCALAR g [B,H,T] bf16, dg the
// fp32 partial sums [dk / 32][B,H,T]; NONE neither is used
cudaError_t tc_bwd_qk(const Dims& d, const void* Qt, const void* Kt, const void* v,
                      const void* g, const float* Eb, const void* dA, const float* S_in,
                      const void* d_o, void* dq, void* dk, void* dg, float* D, float* carry,
                      float* qdq, cudaStream_t st);
bool tc_supported(const Dims& d);
// Whether the tensor-core path of this shape runs the decay pass (its forward
// then keeps decay_layout's operands in `saved` for the backward).
bool tc_uses_decay(const Dims& d);
// Whether its backward also runs tc_dA (and so needs a dA buffer in its workspace).
bool tc_uses_dA(const Dims& d);
// Whether the tensor-core forward (bwd = false) or backward (bwd = true) of this
// shape reads the SCALAR / NONE log-decay in its own layout ([B,H,T] or none)
// rather than broadcast to [B,H,T,dk]: every kernel of that direction that reads
// the log-decay is one with the form built in (tc_decay, tc_bwd_qk).
bool tc_native_forms(const Dims& d, bool bwd);
// Device buffers of the operands computed once per forward (decay_layout) and
// of the backward's score gradient dA [B,H,T,64] bf16.
struct TcOps {
  void* Qt;
  void* Kt;
  float* Eb;
  void* A;
  void* dA;
};
cudaError_t tc_forward(const Dims& d, const void* q, const void* k, const void* v,
                       const void* g, const float* S0, void* o, float* S_final, float* S_in,
                       float* gamma, const TcOps& ops, cudaStream_t st);
cudaError_t tc_backward(const Dims& d, const void* q, const void* k, const void* v,
                        const void* g, const float* S_in, const float* gamma, const void* d_o,
                        const float* dS_final, void* dq, void* dk, void* dv, void* dg,
                        float* dS0, float* D, float* carry, float* qdq, float* dAf,
                        const TcOps& ops, cudaStream_t st);

}  // namespace zeco
