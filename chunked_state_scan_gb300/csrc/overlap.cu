// overlap.cu -- a second stream for the steps that do not depend on the
// segment scan.
//
// The pages' central claim is that the state exchange between segments (the
// All-Scan) hides behind work that does not need it (ZeCO: Pith review,
// "What carries the argument"; the diagonal attention overlaps the All-Scan).
// On one GPU the scan itself is short, but the passes that build the
// scan-independent operands -- the decay-weighted Q~, K~ (tc_decay.cu), the
// intra-chunk scores A and their gradient dA (tc_scores.cu) -- run on an
// auxiliary stream concurrently with pass 1 and the scan (forward) or with the
// backward pre-pass, the reverse scan and the dv sweep (backward).  The caller's
// stream forks to the auxiliary stream with an event and joins it with another
// before the first kernel that reads those operands, so the call stays ordered
// on the caller's stream (and capturable into a CUDA graph).
//
// The auxiliary stream and its events are created on first use, once per host
// thread and device, and live until the thread exits.  zeco_set_overlap(0)
// turns the fork off (everything on the caller's stream); so does an active
// zeco_set_profile_events, whose per-kernel marks assume one stream.
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace zeco {
namespace {

constexpr int kMaxDevices = 128;
constexpr int kEvents = 3;

struct AuxState {
  cudaStream_t stream = nullptr;
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
    }
  }
};

std::atomic<int> g_overlap{1};
thread_local ThreadAux t_aux;

AuxState* aux_for_current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  AuxState& a = t_aux.dev[d];
  if (!a.tried) {
    a.tried = true;
    bool ok = cudaStreamCreateWithFlags(&a.stream, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i < kEvents; ++i)
      ok = cudaEventCreateWithFlags(&a.ev[i], cudaEventDisableTiming) == cudaSuccess;
    a.ok = ok;
  }
  return a.ok ? &a : nullptr;
}

}  // namespace

Fork fork_begin(cudaStream_t st) {
  Fork f;
  f.aux = st;
  f.on = false;
  if (!g_overlap.load(std::memory_order_relaxed) || prof_active()) return f;
  AuxState* a = aux_for_current_device();
  if (!a) return f;
  if (cudaEventRecord(a->ev[0], st) != cudaSuccess) return f;
  if (cudaStreamWaitEvent(a->stream, a->ev[0], 0) != cudaSuccess) return f;
  f.aux = a->stream;
  f.ev[0] = a->ev[1];
  f.ev[1] = a->ev[2];
  f.on = true;
  return f;
}

cudaError_t fork_mark(const Fork& f, int i) {
  return f.on ? cudaEventRecord(f.ev[i], f.aux) : cudaSuccess;
}

cudaError_t fork_join(const Fork& f, cudaStream_t st, int i) {
  return f.on ? cudaStreamWaitEvent(st, f.ev[i], 0) : cudaSuccess;
}

}  // namespace zeco

extern "C" int zeco_set_overlap(int on) {
  zeco::g_overlap.store(on ? 1 : 0, std::memory_order_relaxed);
  return ZECO_OK;
}
