// tc_scores.cu -- masked intra-chunk products P = X Y^T (s <= t) for every chunk
// of C = 64 tokens, in bf16 ([B,H,T,64]: row t of a chunk holds its 64 values
// over s).  Neither depends on the state, so each is computed once per chunk
// here and read by the sweeps (chunkwise form of the diagonal attention: Pith
// review of ZeCO, referee major comment 3 on Algorithm 1):
//
//   A  = Q~ K~^T   (X = Q~, Y = K~, K = d_k): the intra-chunk scores, read by
//                  the forward sweep (o += A v) and the dv sweep (dv += A^T do);
//   dA = do v^T    (X = do, Y = v,  K = d_v): their gradient, read by the dq/dk
//                  sweeps (dq~ += dA K~, dk~ += dA^T Q~).
//
// A persistent kernel, one CTA per SM, bound by reading X and Y once from HBM.
// Warp 4 streams X/Y tiles of 64 tokens x 128 columns through a 4-stage ring
// (TMA, 128B swizzle); warp 5 issues the tcgen05 MMAs (M = 64 t, N = 64 s,
// K) into one of two TMEM accumulators; warps 0-3 read a finished accumulator
// (the M = 64 layout puts row t in lane 32 (t / 16) + t % 16), mask, round and
// store it while the next chunk accumulates.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);

namespace {

using namespace tc;

constexpr int kC = 64;
constexpr int kQ = 128;                     // columns of K per stage
constexpr int kStages = 4;
constexpr int kHalf = kC * kQ * 2;          // X or Y part of a stage (16 KB)
constexpr int kStageBytes = 2 * kHalf;
constexpr int kThreads = 192;

__device__ int g_scores_status = 0;

__global__ void __launch_bounds__(kThreads, 1)
tc_masked_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                 __nv_bfloat16* __restrict__ P, int64_t nchunks, int K) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = align1024(smraw);
  __shared__ uint64_t full[kStages], empty[kStages], accfull[2], accempty[2], fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_word;  // set when a bounded wait of this CTA gives up
  const Waits wait{smem_u32(&abort_word), &g_scores_status};
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // K slices of kQ columns; a last partial slice reads zeros past column K (the
  // copy of a box past the end of a tensor fills it with zeros)
  const int nq = (K + kQ - 1) / kQ;
  int64_t gi = 0;  // producer: (chunk, K slice) stages issued

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accfull[b], 1);
      mbar_init(&accempty[b], 128);
    }
    mbar_init(&fin, 1);
    abort_word = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmY);
  }
  if (warp == 0) tmem_alloc(&tmem_base, 128);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 4) {
    // ---- producer: X and Y tiles of every (chunk, K slice) this CTA owns
    if (lane == 0) {
      bool go = true;
      for (int64_t c = blockIdx.x; go && c < nchunks; c += gridDim.x) {
        const int32_t r = (int32_t)(c * kC);
        for (int q = 0; q < nq; ++q, ++gi) {
          const int s = (int)(gi % kStages);
          const uint32_t ph = (uint32_t)((gi / kStages) & 1);
          if (!wait(&empty[s], ph ^ 1u)) {
            go = false;  // no further copies
            break;
          }
          unsigned char* st = sm + s * kStageBytes;
          mbar_expect_tx(&full[s], kStageBytes);
          for (int b = 0; b < kQ / 64; ++b) {
            tma_load_2d(st + b * 8192, &tmX, q * kQ + b * 64, r, &full[s]);
            tma_load_2d(st + kHalf + b * 8192, &tmY, q * kQ + b * 64, r, &full[s]);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---- MMA issuer: X Y^T, accumulated over the K slices
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16(64, 64, false, false);
      int64_t gi = 0;
      int k = 0;
      for (int64_t c = blockIdx.x; c < nchunks && !wait.aborted(); c += gridDim.x, ++k) {
        const int b = k & 1;
        if (!wait(&accempty[b], (uint32_t)(((k >> 1) & 1) ^ 1))) break;
        tc_fence_after();
        for (int q = 0; q < nq; ++q, ++gi) {
          const int s = (int)(gi % kStages);
          if (!wait(&full[s], (uint32_t)((gi / kStages) & 1))) break;
          tc_fence_after();
          const uint32_t a0 = smem_u32(sm + s * kStageBytes), b0 = a0 + kHalf;
#pragma unroll
          for (int m = 0; m < kQ / 16; ++m) {
            const uint32_t koff = (uint32_t)((m >> 2) * 8192 + (m & 3) * 32);
            umma_bf16(tmem + b * 64, sdesc_sw128(a0 + koff, 16, 1024),
                      sdesc_sw128(b0 + koff, 16, 1024), id, (q | m) ? 1u : 0u);
          }
          umma_commit(&empty[s]);
        }
        umma_commit(&accfull[b]);
      }
      if (wait.aborted()) {
        // no MMA may still write tensor memory when it is freed
        umma_commit(&fin);
        (void)mbar_wait(&fin, 0u);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue (warps 0-3): mask s <= t, round, store row t
    int k = 0;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++k) {
      const int b = k & 1;
      if (!wait(&accfull[b], (uint32_t)((k >> 1) & 1))) break;
      tc_fence_after();
      float a[64];
      tmem_ld32(tmem + lane_off + b * 64, a);
      tmem_ld32(tmem + lane_off + b * 64 + 32, a + 32);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&accempty[b]);
      if (lane < 16) {
        const int t = warp * 16 + lane;
        uint4* dst = reinterpret_cast<uint4*>(P + (size_t)(c * kC + t) * kC);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int s0 = c8 * 8 + 2 * u;
            w4[u] = pack_bf16(s0 <= t ? a[s0] : 0.f, s0 + 1 <= t ? a[s0 + 1] : 0.f);
          }
          dst[c8] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 128);
  // after the CTA's last barrier every thread has finished: if any wait gave up,
  // copies still in flight land before the CTA exits (stage s has been issued
  // ceil((gi - s) / kStages) times; bounded waits)
  if (warp == 4 && lane == 0 && wait.aborted())
    for (int s = 0; s < kStages; ++s) {
      const int64_t n = gi > s ? (gi - s + kStages - 1) / kStages : 0;
      drain_phase(&full[s], (uint32_t)n);
    }
}

}  // namespace

bool tc_dA_supported(const Dims& d) { return d.bf16 && d.C == kC && d.dv % 64 == 0; }
bool tc_A_supported(const Dims& d) { return d.bf16 && d.C == kC && d.dk % 64 == 0; }

namespace {
cudaError_t launch_masked(const Dims& d, const void* X, const void* Y, int K, void* P,
                          cudaStream_t st) {
  CUtensorMap tx, ty;
  const uint64_t rows = (uint64_t)(d.B * d.H * d.T);
  if (!make_tmap_bf16(&tx, X, rows, K, kC) || !make_tmap_bf16(&ty, Y, rows, K, kC))
    return cudaErrorInvalidValue;
  const int smem = kStages * kStageBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(tc_masked_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const int64_t nchunks = (int64_t)rows / kC;
  const unsigned grid = (unsigned)(nchunks < sms ? nchunks : sms);
  prof_start(st);
  tc_masked_kernel<<<grid, kThreads, smem, st>>>(tx, ty, (__nv_bfloat16*)P, nchunks, K);
  return cudaGetLastError();
}
}  // namespace

cudaError_t tc_dA(const Dims& d, const void* d_o, const void* v, void* P, cudaStream_t st) {
  cudaError_t e = launch_masked(d, d_o, v, (int)d.dv, P, st);
  prof_mark("tc_dA", st);
  return e;
}

cudaError_t tc_A(const Dims& d, const void* Qt, const void* Kt, void* P, cudaStream_t st) {
  cudaError_t e = launch_masked(d, Qt, Kt, (int)d.dk, P, st);
  prof_mark("tc_A", st);
  return e;
}

// Reads and clears this file's bounded-wait flag (nonzero: a wait gave up).
int tc_scores_take_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_scores_status, sizeof(v)) != cudaSuccess) return -1;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_scores_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace zeco
