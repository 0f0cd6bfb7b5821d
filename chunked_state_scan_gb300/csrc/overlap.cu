// overlap.cu -- a second stream for work that runs beside the segment scan.
//
// The pages' central claim is that the state exchange between segments (the
// All-Scan) hides behind work that does not need it (ZeCO: Pith review, "What
// carries the argument"; Algorithm 1 runs the All-Scan and the intra-chunk
// diagonal attention on two streams, Eq. 11).  The schedules that use auxiliary
// streams:
//   1: the passes that do not depend on the scan -- the intra-chunk
//     scores A (forward) and their gradient dA (backward) -- go to the
//     auxiliary stream as soon as their inputs exist, concurrently with pass 1
//     and the scan (forward) or with the backward pre-pass, the reverse scan
//     and the dv sweep;
//   2 (the pages' schedule): the segment scan itself goes to the auxiliary
//     stream, concurrently with the diagonal-attention pass (A, or dA) on the
//     caller's stream;
//   3 (forward): pass 2 of each block of segments starts as soon as the scan has
//     produced that block's incoming states (the scan runs block by block on the
//     caller's stream, pass 2 of each block on the auxiliary stream);
//   4 (default): mode 1, and in the backward the dq/dk sweeps on a second
//     auxiliary stream of the highest priority while the dv sweep runs on the
//     caller's: the two are independent, so the dv sweep's CTAs take the SMs
//     that the dq/dk sweeps' last waves leave idle.
// The caller's stream forks to the auxiliary streams with events and joins them
// with others before the first kernel that needs the forked work, so the call
// stays ordered on the caller's stream.
//
// The auxiliary stream and its events are created on first use, once per host
// thread and device, and live until the thread exits.  zeco_set_overlap(0)
// turns the fork off (everything on the caller's stream).
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace zeco {
namespace {

constexpr int kMaxDevices = 128;
constexpr int kEvents = 3 + kStepEvents;

struct AuxState {
  cudaStream_t stream = nullptr;
  cudaStream_t hi = nullptr;  // the device's highest stream priority
  cudaEvent_t ev[kEvents] = {};
  bool ok = false;
  bool tried = false;
};

struct ThreadAux {
  AuxState dev[kMaxDevices];
  ~ThreadAux() {
    for (auto& a : dev) {
      if (!a.ok) continue;
      for (auto& e : a.ev) cudaEventDestroy(e);
      cudaStreamDestroy(a.stream);
      cudaStreamDestroy(a.hi);
    }
  }
};

std::atomic<int> g_overlap{ZECO_OVERLAP_DEFAULT};
thread_local ThreadAux t_aux;

AuxState* aux_for_current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  AuxState& a = t_aux.dev[d];
  if (!a.tried) {
    a.tried = true;
    int lo_pri = 0, hi_pri = 0;
    bool ok = cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking) == cudaSuccess &&
              cudaDeviceGetStreamPriorityRange(&lo_pri, &hi_pri) == cudaSuccess &&
              cudaStreamCreateWithPriority(&a.hi, cudaStreamNonBlocking, hi_pri) == cudaSuccess;
    for (int i = 0; ok && i < kEvents; ++i)
      ok = cudaEventCreateWithFlags(&a.ev[i], cudaEventDisableTiming) == cudaSuccess;
    a.ok = ok;
  }
  return a.ok ? &a : nullptr;
}

}  // namespace

int overlap_mode(const Dims& d) {
  const int m = g_overlap.load(std::memory_order_relaxed);
  return (m == 4 && d.L / d.C < 4) ? 0 : m;
}

Fork fork_begin(cudaStream_t st, int mode) {
  Fork f;
  f.aux = st;
  f.hi = st;
  f.step = nullptr;
  f.on = false;
  if (!mode) return f;
  AuxState* a = aux_for_current_device();
  if (!a) return f;
  if (cudaEventRecord(a->ev[0], st) != cudaSuccess) return f;
  if (cudaStreamWaitEvent(a->stream, a->ev[0], 0) != cudaSuccess) return f;
  f.aux = a->stream;
  f.hi = a->hi;
  f.ev[0] = a->ev[1];
  f.ev[1] = a->ev[2];
  f.step = a->ev + 3;
  f.on = true;
  return f;
}

cudaError_t fork_mark_on(const Fork& f, cudaStream_t s, int i) {
  return f.on ? cudaEventRecord(f.ev[i], s) : cudaSuccess;
}

cudaError_t fork_mark(const Fork& f, int i) { return fork_mark_on(f, f.aux, i); }

cudaError_t fork_join(const Fork& f, cudaStream_t st, int i) {
  return f.on ? cudaStreamWaitEvent(st, f.ev[i], 0) : cudaSuccess;
}

cudaError_t fork_follow_to(const Fork& f, cudaStream_t st, cudaStream_t to, int i) {
  if (!f.on) return cudaSuccess;
  cudaError_t e = cudaEventRecord(f.step[i], st);
  return e == cudaSuccess ? cudaStreamWaitEvent(to, f.step[i], 0) : e;
}

cudaError_t fork_follow(const Fork& f, cudaStream_t st, int i) {
  return fork_follow_to(f, st, f.aux, i);
}

}  // namespace zeco

extern "C" int zeco_set_overlap(int mode) {
  if (mode < 0 || mode > 4) return ZECO_ERR_ARG;
  zeco::g_overlap.store(mode, std::memory_order_relaxed);
  return ZECO_OK;
}
