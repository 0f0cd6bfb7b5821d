// api.cu -- the C ABI: argument checks, buffer layout, and the launch sequence.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace {

using zeco::Dims;

// Per-thread profiling state (zeco_set_profile_events): events[2i] and
// events[2i + 1] bracket kernel i on its own stream.
constexpr int kMaxProf = 256;  // events (two per kernel)
struct ProfState {
  void* const* events = nullptr;
  int cap = 0;
  int count = 0;      // events recorded
  bool open = false;  // a start event waits for its kernel's end event
  const char* names[kMaxProf / 2] = {};
};
thread_local ProfState g_prof;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Largest B*H*P_eff: the kernels launch at most 32 blocks per (b, h, segment) along
// grid x, whose limit is 2^31 - 1 blocks.
constexpr int64_t kMaxBHP = ((1LL << 31) - 1) / 32;

// Shape checks.  Returns ZECO_OK and fills d, or an error code.
int check_shape(const zeco_shape* s, Dims* d) {
  if (!s) return ZECO_ERR_ARG;
  if (s->B < 1 || s->H < 1 || s->T < 1 || s->dk < 1 || s->dv < 1 || s->P < 1 || s->K < 1 ||
      s->C < 1)
    return ZECO_ERR_ARG;
  if (s->dtype != ZECO_F32 && s->dtype != ZECO_BF16) return ZECO_ERR_ARG;
  if (s->path < ZECO_PATH_AUTO || s->path > ZECO_PATH_TC) return ZECO_ERR_ARG;
  if (s->decay < ZECO_DECAY_DIAG || s->decay > ZECO_DECAY_NONE) return ZECO_ERR_ARG;
  if (s->T % s->P != 0 || s->dk % s->K != 0) return ZECO_ERR_ARG;
  const int64_t L = s->T / s->P;
  if (L % s->C != 0) return ZECO_ERR_ARG;
  if (s->C != 16 && s->C != 32 && s->C != 64 && s->C != 128) return ZECO_ERR_UNSUPPORTED;
  if (s->dk % 16 != 0 || s->dk > 256) return ZECO_ERR_UNSUPPORTED;
  if (s->dv % 32 != 0 || s->dv > 512) return ZECO_ERR_UNSUPPORTED;
  // grid limits: the segment scans put B*H on grid z (at most 65,535 blocks); every
  // other kernel puts (b, h, segment) times at most 32 tiles on grid x (2^31 - 1)
  if (s->B * s->H > 65535LL || s->B * s->H * s->P > kMaxBHP) return ZECO_ERR_UNSUPPORTED;
  d->B = s->B;
  d->H = s->H;
  d->T = s->T;
  d->dk = s->dk;
  d->dv = s->dv;
  d->P = s->P;
  d->K = s->K;
  d->C = s->C;
  d->L = L;
  d->bf16 = s->dtype == ZECO_BF16;
  d->decay = s->decay;
  // Chunk length.  The chunked form is exact for any chunk length (results are
  // the token recurrence's, up to rounding), and a 128-token chunk's decay range
  // (the sum of log_alpha over a chunk above -80) implies that of its 64-token
  // halves, so a call asking for C = 128 that does not force the CUDA-core path
  // is evaluated with C = 64 where that is what runs it: bf16 (the tensor-core
  // kernels' chunk), and fp32 where a 128-token chunk does not fit the CUDA-core
  // kernels' shared memory (d_k above 128).  (Shorter chunks are kept: their
  // range may be what the caller needs.)
  if (s->path != ZECO_PATH_SIMT && s->C == 128 &&
      (d->bf16 || zeco::simt_smem_bytes(*d) > 227 * 1024))
    d->C = 64;
  // Segments on one GPU.  The P segments of the method exchange their states
  // through the segment scan; the decomposition is exact for any split, so when
  // B*H*P is too small to give the chunk sweeps a wave of CTAs (one per 128 d_v
  // columns of a segment; 152 SMs), each segment is split further into 2^m equal
  // sub-segments of at least 4 chunks (at most 64 per segment).  Everything
  // below, the `saved` layout included, uses the effective count.
  constexpr int64_t kWave = 152;
  const int64_t tiles = (s->dv + 127) / 128;
  const int64_t C = d->C;
  int64_t m = 1;
  while (s->B * s->H * s->P * m * tiles < kWave && m < 64 && s->T % (s->P * m * 2 * C) == 0 &&
         s->T / (s->P * m * 2) >= 4 * C && s->B * s->H * s->P * m * 2 <= kMaxBHP)
    m *= 2;
  d->P = (int)(s->P * m);
  d->L = s->T / d->P;
  return ZECO_OK;
}

int resolve(const zeco_shape* s, const Dims& d) {
  // the tensor-core path runs CUDA-core kernels for the steps it has no
  // tensor-core kernel for (C != 64): their shared memory must fit one CTA too
  const bool tc = zeco::tc_supported(d) &&
                  (zeco::tc_uses_dA(d) || zeco::simt_smem_bytes(d) <= 227 * 1024);
  if (s->path == ZECO_PATH_TC) return tc ? (int)ZECO_PATH_TC : (int)ZECO_ERR_UNSUPPORTED;
  if (s->path == ZECO_PATH_AUTO && tc) return ZECO_PATH_TC;
  // SIMT: shared memory must fit one CTA
  if (zeco::simt_smem_bytes(d) > 227 * 1024) return ZECO_ERR_UNSUPPORTED;
  return ZECO_PATH_SIMT;
}

// Scratch layout of one call: the backward's own buffers (bwd only; with the
// CUDA-core dq/dk kernel also its fp32 dA), then, for
// the backward on the tensor-core path, the score gradient dA, then, for the
// SCALAR / NONE decay forms, the broadcast log-decay and its per-row gradient,
// or, where the kernels read the form in its own layout, the SCALAR gradient's
// partial sums (forms_layout).  The operands the forward computes once
// (decay_layout) live in `saved`, not here.
struct WsPlan {
  zeco::BwdWsLayout bwd;
  size_t dA_off;  // backward on the tensor-core path: the score gradient dA
  bool native;    // the decay form is read in its own layout (tc_native_forms)
  zeco::FormsLayout forms;
  size_t total;
};

WsPlan plan_ws(const Dims& d, int path, bool bwd) {
  WsPlan w;
  w.bwd = zeco::bwd_ws_layout(d, path != ZECO_PATH_TC || !zeco::tc_uses_dA(d));
  size_t base = bwd ? w.bwd.total : 0;
  w.dA_off = zeco::align_up(base, 256);
  if (bwd && path == ZECO_PATH_TC && zeco::tc_uses_dA(d))
    base = zeco::align_up(w.dA_off + zeco::scores_bytes(d), 256);
  w.native = path == ZECO_PATH_TC && zeco::tc_native_forms(d, bwd);
  w.forms = zeco::forms_layout(d, base, bwd, w.native);
  w.total = w.forms.total;
  return w;
}

// Whether the forward keeps the tensor-core operands (Q~, K~, e^{b_last}, A) in
// `saved` for the backward.
bool keeps_ops(const Dims& d, int path) {
  return path == ZECO_PATH_TC && zeco::tc_uses_decay(d);
}

zeco::TcOps tc_ops(const zeco::SavedLayout& sl, const void* saved, void* ws, size_t dA_off) {
  char* b = (char*)saved;
  zeco::TcOps o;
  o.Qt = b + sl.ops.Qt_off;
  o.Kt = b + sl.ops.Kt_off;
  o.Eb = (float*)(b + sl.ops.Eb_off);
  o.A = b + sl.ops.A_off;
  o.dA = ws ? (char*)ws + dA_off : nullptr;
  return o;
}

}  // namespace

namespace zeco {

void prof_start(cudaStream_t st) {
  g_prof.open = false;
  if (!g_prof.events || g_prof.count + 2 > g_prof.cap) return;
  if (cudaEventRecord((cudaEvent_t)g_prof.events[g_prof.count], st) == cudaSuccess)
    g_prof.open = true;
}

void prof_mark(const char* kernel, cudaStream_t st) {
  if (!g_prof.events || !g_prof.open) return;
  g_prof.open = false;
  if (cudaEventRecord((cudaEvent_t)g_prof.events[g_prof.count + 1], st) != cudaSuccess) return;
  g_prof.names[g_prof.count / 2] = kernel;
  g_prof.count += 2;
}

}  // namespace zeco

extern "C" {

int zeco_set_profile_events(void* const* events, int n) {
  g_prof.events = (n > 0) ? events : nullptr;
  g_prof.cap = (n > 0 && events) ? (n < kMaxProf ? n : kMaxProf) : 0;
  g_prof.count = 0;
  g_prof.open = false;
  return ZECO_OK;
}

int zeco_profile_event_count(void) { return g_prof.count; }

const char* zeco_profile_kernel_name(int i) {
  return (i >= 0 && i < g_prof.count / 2) ? g_prof.names[i] : nullptr;
}

size_t zeco_gla_saved_bytes(const zeco_shape* shape) {
  Dims d;
  if (check_shape(shape, &d) != ZECO_OK) return 0;
  const int path = resolve(shape, d);
  if (path < 0) return 0;
  return zeco::saved_layout(d, keeps_ops(d, path)).total;
}

size_t zeco_gla_workspace_bytes(const zeco_shape* shape, int bwd) {
  Dims d;
  if (check_shape(shape, &d) != ZECO_OK) return 0;
  const int path = resolve(shape, d);
  if (path < 0) return 0;
  return plan_ws(d, path, bwd != 0).total;
}

int64_t zeco_gla_segments(const zeco_shape* shape) {
  Dims d;
  const int rc = check_shape(shape, &d);
  return rc != ZECO_OK ? rc : d.P;
}

int zeco_gla_resolve_path(const zeco_shape* shape) {
  Dims d;
  const int rc = check_shape(shape, &d);
  if (rc != ZECO_OK) return rc;
  return resolve(shape, d);
}

int zeco_gla_fwd(const zeco_shape* shape, const void* q, const void* k, const void* v,
                 const void* log_alpha, const float* S0, void* o, float* S_final, void* saved,
                 void* workspace, size_t ws_bytes, zeco_stream_t stream) {
  Dims d;
  int rc = check_shape(shape, &d);
  if (rc != ZECO_OK) return rc;
  const void* req[] = {q, k, v, o, saved};
  for (const void* p : req)
    if (!p || !aligned16(p)) return ZECO_ERR_ARG;
  if ((S0 && !aligned16(S0)) || (S_final && !aligned16(S_final))) return ZECO_ERR_ARG;
  if (d.decay != ZECO_DECAY_NONE && (!log_alpha || !aligned16(log_alpha))) return ZECO_ERR_ARG;
  const int path = resolve(shape, d);
  if (path < 0) return path;
  const WsPlan wp = plan_ws(d, path, false);
  if (wp.total > 0 && (!workspace || !aligned16(workspace))) return ZECO_ERR_ARG;
  if (ws_bytes < wp.total) return ZECO_ERR_WORKSPACE;
  const zeco::SavedLayout sl = zeco::saved_layout(d, keeps_ops(d, path));
  float* S_in = (float*)((char*)saved + sl.S_in_off);
  float* gamma = (float*)((char*)saved + sl.gamma_off);
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  const void* g = log_alpha;
  if (d.decay != ZECO_DECAY_DIAG && !wp.native) {
    g = (char*)workspace + wp.forms.gx_off;
    e = zeco::launch_expand_log_alpha(d, log_alpha, (void*)g, st);
  }
  if (e == cudaSuccess)
    e = path == ZECO_PATH_TC
            ? zeco::tc_forward(d, q, k, v, g, S0, o, S_final, S_in, gamma,
                               tc_ops(sl, saved, nullptr, 0), st)
            : zeco::simt_forward(d, q, k, v, g, S0, o, S_final, S_in, gamma, st);
  return e == cudaSuccess ? ZECO_OK : ZECO_ERR_CUDA;
}

int zeco_gla_bwd(const zeco_shape* shape, const void* q, const void* k, const void* v,
                 const void* log_alpha, const void* saved, const void* d_o,
                 const float* dS_final, void* dq, void* dk, void* dv, void* dlog_alpha,
                 float* dS0, void* workspace, size_t ws_bytes, zeco_stream_t stream) {
  Dims d;
  int rc = check_shape(shape, &d);
  if (rc != ZECO_OK) return rc;
  const void* req[] = {q, k, v, saved, d_o, dq, dk, dv, workspace};
  for (const void* p : req)
    if (!p || !aligned16(p)) return ZECO_ERR_ARG;
  if (d.decay != ZECO_DECAY_NONE && (!log_alpha || !aligned16(log_alpha) || !dlog_alpha ||
                                     !aligned16(dlog_alpha)))
    return ZECO_ERR_ARG;
  if ((dS_final && !aligned16(dS_final)) || (dS0 && !aligned16(dS0))) return ZECO_ERR_ARG;
  const int path = resolve(shape, d);
  if (path < 0) return path;
  const WsPlan wp = plan_ws(d, path, true);
  const zeco::BwdWsLayout& wl = wp.bwd;
  if (ws_bytes < wp.total) return ZECO_ERR_WORKSPACE;
  const zeco::SavedLayout sl = zeco::saved_layout(d, keeps_ops(d, path));
  const float* S_in = (const float*)((const char*)saved + sl.S_in_off);
  const float* gamma = (const float*)((const char*)saved + sl.gamma_off);
  float* D = (float*)((char*)workspace + wl.D_off);
  float* carry = (float*)((char*)workspace + wl.carry_off);
  float* qdq = (float*)((char*)workspace + wl.qdq_off);
  float* dAf = (float*)((char*)workspace + wl.dAf_off);  // CUDA-core dq/dk only
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  const void* g = log_alpha;
  void* dg = dlog_alpha;
  if (d.decay == ZECO_DECAY_SCALAR || (d.decay == ZECO_DECAY_NONE && !wp.native))
    dg = (char*)workspace + wp.forms.dgx_off;  // NONE: a gradient nobody reads
  else if (d.decay == ZECO_DECAY_NONE)
    dg = nullptr;
  if (d.decay != ZECO_DECAY_DIAG && !wp.native) {
    g = (char*)workspace + wp.forms.gx_off;
    e = zeco::launch_expand_log_alpha(d, log_alpha, (void*)g, st);
  }
  if (e == cudaSuccess)
    e = path == ZECO_PATH_TC
            ? zeco::tc_backward(d, q, k, v, g, S_in, gamma, d_o, dS_final, dq, dk, dv, dg, dS0, D,
                                carry, qdq, dAf, tc_ops(sl, saved, workspace, wp.dA_off), st)
            : zeco::simt_backward(d, q, k, v, g, S_in, gamma, d_o, dS_final, dq, dk, dv, dg,
                                  dS0, D, carry, qdq, dAf, st);
  if (e == cudaSuccess && d.decay == ZECO_DECAY_SCALAR)
    e = wp.native ? zeco::launch_sum_dlog_alpha_parts(d, (const float*)dg, dlog_alpha, st)
                  : zeco::launch_reduce_dlog_alpha(d, dg, dlog_alpha, st);
  return e == cudaSuccess ? ZECO_OK : ZECO_ERR_CUDA;
}

int zeco_check_device_status(void) {
  const int v[] = {zeco::tc_state_take_status(), zeco::tc_fwd_take_status(),
                   zeco::tc_scores_take_status(), zeco::tc_bwd_qk_take_status(),
                   zeco::selftest_take_status()};
  int rc = ZECO_OK;
  for (int x : v) {
    if (x < 0) return ZECO_ERR_CUDA;
    if (x > 0) rc = ZECO_ERR_TIMEOUT;
  }
  return rc;
}

int zeco_last_device_status(zeco_stream_t stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ZECO_ERR_CUDA;
  return zeco_check_device_status();
}

const char* zeco_strerror(int code) {
  switch (code) {
    case ZECO_OK:
      return "success";
    case ZECO_ERR_ARG:
      return "invalid argument (null or misaligned pointer, or inconsistent shape)";
    case ZECO_ERR_UNSUPPORTED:
      return "shape outside the supported set";
    case ZECO_ERR_WORKSPACE:
      return "workspace too small";
    case ZECO_ERR_CUDA:
      return "CUDA kernel launch failed";
    case ZECO_ERR_TIMEOUT:
      return "a bounded device wait gave up (results of that call are not valid)";
    default:
      return "unknown error code";
  }
}

}  // extern "C"
