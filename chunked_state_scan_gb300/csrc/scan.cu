// scan.cu -- segment scans over the P segment states (forward and reverse).
//
// Forward (the All-Scan update; Pith review of ZeCO, "What carries the
// argument"):   S_in[0] = S0,  S_in[p+1] = (gamma_p^T 1) .* S_in[p] + S_loc[p].
// The state rows are cut into K contiguous d_k blocks and every block is
// scanned on its own (blockIdx.y), as in the pages' pipelined All-Scan; the
// carried value is the accumulated state (Pith review of ZeCO, referee major
// comment 4 on Algorithm 2).  On one GPU the "devices" are the P segment
// slots of the `saved` buffer, so the scan reads each local state once and
// writes each global state once, in place: pass 1 leaves S_loc[p] in slot p+1.
//
// Reverse (the adjoint scan, the dKV pass of Linear Attention Sequence
// Parallelism, summary):  D[P] = dS_final,  D[p] = dS_loc[p] + gamma_p .* D[p+1],
// dS0 = D[0], where D[p] is the adjoint of S_in[p].  It also forms the
// per-segment carry of d log_alpha,  c_p[i] = sum_j D[p+1][i,j] S_in[p+1][i,j],
// which is the gradient of log_alpha at the first token after segment p
// (equivalently: the dlog_alpha suffix sum of all later segments plus
// rowsum(dS_final .* S_final)).
//
// Layout: one warp owns one d_k row of one (b,h); lane l holds the float4
// columns l, l+32, ... of that row, so every access is a coalesced 512-byte
// warp transaction and the row sums of the carry are warp-shuffle reductions.
// The p loop is sequential, but the loads of a step do not depend on the steps
// before it: they are issued kBatch steps at a time and only the FMA chain is
// serial, so the scan streams at memory bandwidth even for very many segments
// (a tree scan would move at least as many bytes).
#include "common.cuh"
#include "launch.h"

namespace zeco {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxU = 4;  // dv <= 512: at most 4 float4 per lane
constexpr int kBatch = 4;  // segment steps whose loads are issued together

__device__ __forceinline__ float4 fma4(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

__global__ void __launch_bounds__(kWarps * 32)
seg_scan_fwd_kernel(float* __restrict__ S_in, const float* __restrict__ gamma,
                    const float* __restrict__ S0, float* __restrict__ S_final, int P, int dk,
                    int dv, int rows_per_kblock, int p_begin, int p_end) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int local_row = blockIdx.x * kWarps + warp;
  if (local_row >= rows_per_kblock) return;
  const int i = blockIdx.y * rows_per_kblock + local_row;
  const int64_t bh = blockIdx.z;
  const int nv4 = dv >> 2;
  const size_t slot = (size_t)dk * dv;
  float4* base = reinterpret_cast<float4*>(S_in + (size_t)bh * (P + 1) * slot + (size_t)i * dv);
  const float* gam = gamma + (size_t)bh * P * dk + i;

  // segments [p_begin, p_end): the state entering p_begin is S0 (p_begin = 0) or the
  // one an earlier launch left in slot p_begin
  float4 s[kMaxU];
#pragma unroll
  for (int u = 0; u < kMaxU; ++u) {
    const int j4 = lane + 32 * u;
    s[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j4 < nv4) {
      if (p_begin == 0) {
        s[u] = S0 ? reinterpret_cast<const float4*>(S0 + ((size_t)bh * dk + i) * dv)[j4]
                  : make_float4(0.f, 0.f, 0.f, 0.f);
        base[j4] = s[u];
      } else {
        s[u] = base[(size_t)p_begin * (slot >> 2) + j4];
      }
    }
  }
  for (int p0 = p_begin; p0 < p_end; p0 += kBatch) {
    // the loads of kBatch steps go out together; only the FMA chain is serial
    float4 x[kBatch][kMaxU];
    float gm[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int p = p0 + b;
      gm[b] = p < p_end ? gam[(size_t)p * dk] : 0.f;
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const int j4 = lane + 32 * u;
        x[b][u] = (p < p_end && j4 < nv4) ? base[(size_t)(p + 1) * (slot >> 2) + j4]
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int p = p0 + b;
      if (p >= p_end) break;
      float4* dst = base + (size_t)(p + 1) * (slot >> 2);
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const int j4 = lane + 32 * u;
        if (j4 < nv4) {
          s[u] = fma4(gm[b], s[u], x[b][u]);  // gamma_p * S_in[p] + S_loc[p]
          dst[j4] = s[u];
        }
      }
    }
  }
  if (S_final && p_end == P) {
    float4* sf = reinterpret_cast<float4*>(S_final + ((size_t)bh * dk + i) * dv);
#pragma unroll
    for (int u = 0; u < kMaxU; ++u) {
      const int j4 = lane + 32 * u;
      if (j4 < nv4) sf[j4] = s[u];
    }
  }
}

__global__ void __launch_bounds__(kWarps * 32)
seg_scan_rev_kernel(float* __restrict__ D, const float* __restrict__ S_in,
                    const float* __restrict__ gamma, const float* __restrict__ dS_final,
                    float* __restrict__ dS0, float* __restrict__ carry, int P, int dk, int dv,
                    int rows_per_kblock) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int local_row = blockIdx.x * kWarps + warp;
  if (local_row >= rows_per_kblock) return;
  const int i = blockIdx.y * rows_per_kblock + local_row;
  const int64_t bh = blockIdx.z;
  const int nv4 = dv >> 2;
  const size_t slot4 = (size_t)dk * dv / 4;
  float4* Db = reinterpret_cast<float4*>(D + (size_t)bh * (P + 1) * dk * dv + (size_t)i * dv);
  const float4* Sb =
      reinterpret_cast<const float4*>(S_in + (size_t)bh * (P + 1) * dk * dv + (size_t)i * dv);
  const float* gam = gamma + (size_t)bh * P * dk + i;

  float4 s[kMaxU];
#pragma unroll
  for (int u = 0; u < kMaxU; ++u) {
    const int j4 = lane + 32 * u;
    s[u] = make_float4(0.f, 0.f, 0.f, 0.f);  // columns past dv stay 0 (they enter the carry)
    if (j4 < nv4) {
      s[u] = dS_final ? reinterpret_cast<const float4*>(dS_final + ((size_t)bh * dk + i) * dv)[j4]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      Db[(size_t)P * slot4 + j4] = s[u];
    }
  }
  for (int p0 = P - 1; p0 >= 0; p0 -= kBatch) {
    // the loads of kBatch steps (S_in[p+1], dS_loc[p], gamma_p) go out together
    float4 y[kBatch][kMaxU], x[kBatch][kMaxU];
    float gm[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int p = p0 - b;
      gm[b] = p >= 0 ? gam[(size_t)p * dk] : 0.f;
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const int j4 = lane + 32 * u;
        const bool ok = p >= 0 && j4 < nv4;
        y[b][u] = ok ? Sb[(size_t)(p + 1) * slot4 + j4] : make_float4(0.f, 0.f, 0.f, 0.f);
        x[b][u] = ok ? Db[(size_t)p * slot4 + j4] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int p = p0 - b;
      if (p < 0) break;
      // carry c_p = rowsum(D[p+1] .* S_in[p+1])
      float part = 0.f;
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const float4 yy = y[b][u];
        part = fmaf(s[u].x, yy.x, fmaf(s[u].y, yy.y, fmaf(s[u].z, yy.z, fmaf(s[u].w, yy.w, part))));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0) carry[((size_t)bh * P + p) * dk + i] = part;
#pragma unroll
      for (int u = 0; u < kMaxU; ++u) {
        const int j4 = lane + 32 * u;
        if (j4 < nv4) {
          s[u] = fma4(gm[b], s[u], x[b][u]);  // dS_loc[p] + gamma_p * D[p+1]
          Db[(size_t)p * slot4 + j4] = s[u];
        }
      }
    }
  }
  if (dS0) {
    float4* o = reinterpret_cast<float4*>(dS0 + ((size_t)bh * dk + i) * dv);
#pragma unroll
    for (int u = 0; u < kMaxU; ++u) {
      const int j4 = lane + 32 * u;
      if (j4 < nv4) o[j4] = s[u];
    }
  }
}

}  // namespace

cudaError_t launch_seg_scan_fwd(const Dims& d, float* S_in, const float* gamma, const float* S0,
                                float* S_final, cudaStream_t st, int p_begin, int p_end) {
  const int rows = (int)(d.dk / d.K);
  if (p_end < 0) p_end = d.P;
  dim3 grid((rows + kWarps - 1) / kWarps, d.K, (unsigned)(d.B * d.H));
  prof_start(st);
  seg_scan_fwd_kernel<<<grid, kWarps * 32, 0, st>>>(S_in, gamma, S0, S_final, d.P, (int)d.dk,
                                                    (int)d.dv, rows, p_begin, p_end);
  prof_mark("seg_scan_fwd", st);
  return cudaGetLastError();
}

cudaError_t launch_seg_scan_rev(const Dims& d, float* D, const float* S_in, const float* gamma,
                                const float* dS_final, float* dS0, float* carry,
                                cudaStream_t st) {
  const int rows = (int)(d.dk / d.K);
  dim3 grid((rows + kWarps - 1) / kWarps, d.K, (unsigned)(d.B * d.H));
  prof_start(st);
  seg_scan_rev_kernel<<<grid, kWarps * 32, 0, st>>>(D, S_in, gamma, dS_final, dS0, carry, d.P,
                                                    (int)d.dk, (int)d.dv, rows);
  prof_mark("seg_scan_rev", st);
  return cudaGetLastError();
}

}  // namespace zeco
