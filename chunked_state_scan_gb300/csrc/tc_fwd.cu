// tc_fwd.cu -- pass 2 of the forward on tcgen05 tensor cores.
//
// Every segment re-runs its chunks from its incoming global state S_in[p] and
// writes its outputs: intra-chunk decay-masked attention ("diagonal
// attention") plus the inter-chunk state term, with the chunk state carried
// on chip (ZeCO two-pass operator, second pass over Q, K, V: Pith review of
// ZeCO, referee major comment 3 on Algorithm 1; the chunk loop is sequential,
// minor comment 5 on Algorithm 3).  Per chunk of C = 64 tokens, with b the
// inclusive cumulative log-decay from the chunk start (per d_k row):
//
//   Q~ = q .* e^{b},   K~ = k .* e^{-b}                   (Pith review, minor comment 4:
//                                                          the K/Lambda, K.Gamma pair)
//   A  = Q~ K~^T,  masked to s <= t                        (intra-chunk scores)
//   o  = Q~ S + A V                                        (S = state before the chunk)
//   S <- e^{b_last} .* (S + K~^T V)                        (state after the chunk)
//
// One CTA owns (b, h, segment, 128 d_v columns) and keeps S^T (lanes = d_v
// column j, TMEM columns = d_k row i) in fp32 in tensor memory, plus a bf16
// copy of S^T that is the A operand (read from TMEM) of o^T = S^T Q~^T.
// Q~, K~, e^{b_last} (tc_decay.cu), the masked scores A (tc_scores.cu) and
// the V tile arrive by TMA one chunk ahead (two buffers each; later chunks are
// prefetched into L2), so a chunk is one group of MMAs plus the
// state pass; the output accumulator is double-buffered so that warps 0-7
// write chunk n-1 while the tensor cores run chunk n (through a shared-memory
// stage and one TMA store per chunk).  Thread 256 issues the
// MMAs and thread 288 the copies, away from the epilogue warps.
//
// The same kernel, run backwards over the chunks (BWD = true), computes dv
// from the adjoint state dS of the segment end (D[p+1], from the reverse
// segment scan): per chunk, in reverse,
//
//   dS <- e^{b_last} .* dS                     (adjoint of the state after the chunk,
//                                               carried to the chunk's tokens)
//   dv = K~ dS + (A masked)^T do               (K~ (e^{b_last} dS) = K^ dS of the pages)
//   dS <- dS + Q~^T do                         (adjoint of the state before the chunk)
//
// with q/k roles swapped on the output side and do in place of v.
//
// TMEM columns: [0, DK) S^T fp32 | [256, 256 + DK/2) S^T bf16 | [384, 448) and
// [448, 512) o^T (dv^T when BWD), chunk parity.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);
bool make_tmap_bf16_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_cols, uint32_t box_rows);

namespace {

using namespace tc;

constexpr int kC = 64;        // chunk length
constexpr int kNV = 128;      // d_v columns per CTA
constexpr int kThreads = 512;  // 16 warps
constexpr uint32_t kColS16 = 256, kColO = 384;
constexpr int kMmaTid = 256, kTmaTid = 288;
// backward: the state pass after chunk n scales by the next chunk's e^{b_last},
// so those rows come through a ring loaded two chunks ahead
constexpr int kESlots = 3;
// chunks ahead whose operands are prefetched into L2 (the shared memory holds
// the current and the next chunk)
constexpr int kPf = 2;

__device__ int g_fwd_status = 0;

template <int DK>
struct FwdSmem {
  static constexpr int kTile = DK * kC * 2;  // Q~ / K~ tile bytes
  static constexpr int kP = 2 * kTile;       // masked scores [64 t][64 s] bf16
  static constexpr int kEx = kP + kC * kC * 2;  // forward: the chunk's e^{b_last} [DK] fp32
  static constexpr int kXBuf = (kEx + DK * 4 + 1023) / 1024 * 1024;
  static constexpr int kX = 0;               // 2 buffers (chunk parity)
  static constexpr int kV = 2 * kXBuf;       // V / do tiles, 2 buffers (chunk parity)
  static constexpr int kVBuf = kNV * kC * 2;
  static constexpr int kE = kV + 2 * kVBuf;  // backward: e^{b_last} [DK] fp32, a ring of kESlots
  // the output tile [64 t][128 j] bf16, staged for its TMA store
  static constexpr int kO = (kE + kESlots * DK * 4 + 1023) / 1024 * 1024;
  static constexpr int kBytes = kO + kC * kNV * 2;
};

// A warp's W consecutive fp32 columns of its 32 lanes (W = 32 or 16), and their
// bf16 pairs packed into W / 2 columns
template <int W>
__device__ __forceinline__ void st_cols(uint32_t taddr, const float* r) {
  if constexpr (W == 32)
    tmem_st32(taddr, r);
  else
    tmem_st16(taddr, reinterpret_cast<const uint32_t*>(r));
}
template <int W>
__device__ __forceinline__ void st_half(uint32_t taddr, const float* r) {
  uint32_t h[W / 2];
#pragma unroll
  for (int u = 0; u < W / 2; ++u) h[u] = pack_bf16(r[2 * u], r[2 * u + 1]);
  if constexpr (W == 32)
    tmem_st16(taddr, h);
  else
    tmem_st8(taddr, h);
}

template <int DK, bool BWD>
__global__ void __launch_bounds__(kThreads, 1)
tc_sweep_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmP,
                const __grid_constant__ CUtensorMap tmO, const float* __restrict__ Eb,
                const float* __restrict__ S_src, int64_t T, int dv, int P, int64_t L,
                int p_begin, int p_count) {
  using SM = FwdSmem<DK>;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = align1024(smraw);
  unsigned char* sV = sm + SM::kV;
  __shared__ uint64_t bar_x[2], bar_v[2], bar_e[kESlots], bar_u, bar_g, bar_fin;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_word;  // set when a bounded wait of this CTA gives up
  // After a wait of this CTA has given up, the abort word makes every later wait
  // of the CTA give up within 64 polls and the copy thread issues no further
  // copies: the chunk loop runs to its end without waiting, and the CTA drains
  // what it has in flight before exit.
  const Waits wait{smem_u32(&abort_word), &g_fwd_status};
  auto wt = [&](uint64_t* bar, uint32_t parity) { (void)wait(bar, parity); };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = warp & 3;       // TMEM lane group of this warp
  const int cq = warp >> 2;      // which quarter of the d_k columns this warp's state pass handles
  const int half = (warp >> 2) & 1;  // epilogue: which half of the 64 tokens (warps 0..7)
  // segments [p_begin, p_begin + p_count) of every (b, h)
  // block x = ((b h) * p_count + segment - p_begin) * (d_v / kNV) + d_v tile
  // (a last partial tile of d_v columns starts from a zero state, reads zeros
  // past the end of V and stores only the columns that exist)
  const int nx = (dv + kNV - 1) / kNV;
  const int bx = (int)(blockIdx.x % nx);
  const int64_t by = (int64_t)(blockIdx.x / nx);
  const int64_t bh = by / p_count;
  const int p = p_begin + (int)(by % p_count);
  const int j0 = bx * kNV;
  const int64_t row0 = bh * T + (int64_t)p * L;
  const int nc = (int)(L / kC);

  if (tid == 0) {
    mbar_init(&bar_x[0], 1);
    mbar_init(&bar_x[1], 1);
    mbar_init(&bar_v[0], 1);
    mbar_init(&bar_v[1], 1);
    for (int k = 0; k < kESlots; ++k) mbar_init(&bar_e[k], 1);
    mbar_init(&bar_u, 1);
    mbar_init(&bar_g, 1);
    mbar_init(&bar_fin, 1);
    abort_word = 0;
    fence_mbar_init();
  }
  if (tid == kTmaTid) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmP);
    prefetch_tmap(&tmO);
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_off = (uint32_t)(lg * 32) << 16;

  // chunks whose tiles (x and v) and e^{b_last} rows the copy thread has
  // requested: chunk c of the sweep goes to buffer c % 2 and ring slot c % kESlots,
  // so these totals give the phases issued on every copy barrier (after an abort
  // the copies still in flight are waited for before the CTA exits)
  uint32_t n_xv = 0, n_e = 0;
  // Q~, K~ and masked-score tiles (forward: and the e^{b_last} row) of chunk n
  // into buffer `buf`
  auto issue_x = [&](int n, int buf) {
    ++n_xv;
    const int32_t r = (int32_t)(row0 + (int64_t)n * kC);
    unsigned char* xb = sm + SM::kX + buf * SM::kXBuf;
    mbar_expect_tx(&bar_x[buf], 2 * SM::kTile + kC * kC * 2 + (BWD ? 0 : DK * 4));
    for (int b = 0; b < DK / 64; ++b) {
      tma_load_2d(xb + b * 8192, &tmQ, b * 64, r, &bar_x[buf]);
      tma_load_2d(xb + SM::kTile + b * 8192, &tmK, b * 64, r, &bar_x[buf]);
    }
    tma_load_2d(xb + SM::kP, &tmP, 0, r, &bar_x[buf]);
    if (!BWD) bulk_load(xb + SM::kEx, Eb + (size_t)(r / kC) * DK, DK * 4, &bar_x[buf]);
  };
  // e^{b_last} of the chunk processed at iteration `it` into ring slot it % kESlots
  auto issue_e = [&](int it) {
    const int n = BWD ? nc - 1 - it : it;
    const int k = it % kESlots;
    const int32_t r = (int32_t)(row0 + (int64_t)n * kC);
    ++n_e;
    mbar_expect_tx(&bar_e[k], DK * 4);
    bulk_load(sm + SM::kE + k * DK * 4, Eb + (size_t)(r / kC) * DK, DK * 4, &bar_e[k]);
  };
  auto e_slot = [&](int it) -> const float* {  // waits for, and returns, iteration it's row
    const int k = it % kESlots;
    wt(&bar_e[k], (uint32_t)((it / kESlots) & 1));
    return reinterpret_cast<const float*>(sm + SM::kE + k * DK * 4);
  };
  auto issue_v = [&](int n, int buf) {
    const int32_t r = (int32_t)(row0 + (int64_t)n * kC);
    unsigned char* vb = sV + buf * SM::kVBuf;
    mbar_expect_tx(&bar_v[buf], kNV * kC * 2);
    for (int b = 0; b < kNV / 64; ++b)
      tma_load_2d(vb + b * 8192, &tmV, j0 + b * 64, r, &bar_v[buf]);
  };
  // L2 prefetch of chunk n's operands (the tiles shared by the d_v tiles of a
  // segment, by the first of them only)
  auto prefetch = [&](int n) {
    const int32_t r = (int32_t)(row0 + (int64_t)n * kC);
    if (bx == 0) {
      for (int b = 0; b < DK / 64; ++b) {
        tma_prefetch_2d(&tmQ, b * 64, r);
        tma_prefetch_2d(&tmK, b * 64, r);
      }
      tma_prefetch_2d(&tmP, 0, r);
      bulk_prefetch(Eb + (size_t)(r / kC) * DK, DK * 4);
    }
    for (int b = 0; b < kNV / 64; ++b)
      if (j0 + b * 64 < dv) tma_prefetch_2d(&tmV, j0 + b * 64, r);
  };
  if (tid == kTmaTid) {
    issue_x(BWD ? nc - 1 : 0, 0);
    issue_v(BWD ? nc - 1 : 0, 0);
    if (BWD)
      for (int it = 0; it < kESlots - 1 && it < nc; ++it) issue_e(it);
    for (int it = 1; it < kPf && it < nc; ++it) prefetch(BWD ? nc - 1 - it : it);
  }

  // ---- initial state: S^T fp32 (and, forward, its bf16 copy) from the state
  //      entering the segment (forward: S_in[p]) or the adjoint at its end
  //      (backward: D[p+1]).
  constexpr int kQ = DK / 4;            // TMEM columns of one warp's quarter
  constexpr int kW = kQ < 32 ? kQ : 32;  // columns per tensor-memory load / store
  {
    const int jl = j0 + lg * 32 + lane;  // this thread's d_v column
    const bool live = jl < dv;
    const float* Sp =
        S_src + ((size_t)bh * (P + 1) + p + (BWD ? 1 : 0)) * DK * dv + (live ? jl : 0);
    for (int c = cq * kQ; c < (cq + 1) * kQ; c += kW) {
      float r[kW];
#pragma unroll
      for (int u = 0; u < kW; ++u) r[u] = live ? Sp[(size_t)(c + u) * dv] : 0.f;
      st_cols<kW>(tmem + lane_off + c, r);
      if (!BWD) st_half<kW>(tmem + lane_off + kColS16 + c / 2, r);
    }
    tmem_st_wait();
  }

  // The state pass in two parts.  Part 1: S^T (fp32) <- e^{b_last} .* S^T (column
  // i scaled by sE[i]), the scaled values kept in r; it needs only the chunk's
  // state update.  Part 2: the bf16 copy of the scaled state (the A operand of
  // the next chunk's output MMAs); it waits until this chunk's output MMAs have
  // read the old copy.
  auto scale_part = [&](const float* sE, float* r) {
    const int c0 = cq * kQ;
    if constexpr (kW == 32) {
#pragma unroll
      for (int c = 0; c < kQ; c += 32) tmem_ld32(tmem + lane_off + c0 + c, r + c);
      tmem_ld_wait();
    } else {
      tmem_ld16(tmem + lane_off + c0, r);
      tmem_ld_wait16(r);
    }
    const float4* e4 = reinterpret_cast<const float4*>(sE + c0);
#pragma unroll
    for (int u = 0; u < kQ / 4; ++u) {
      const float4 e = e4[u];
      r[4 * u] *= e.x;
      r[4 * u + 1] *= e.y;
      r[4 * u + 2] *= e.z;
      r[4 * u + 3] *= e.w;
    }
#pragma unroll
    for (int c = 0; c < kQ; c += kW) st_cols<kW>(tmem + lane_off + c0 + c, r + c);
  };
  auto copy_part = [&](const float* r) {
    const int c0 = cq * kQ;
#pragma unroll
    for (int c = 0; c < kQ; c += kW) st_half<kW>(tmem + lane_off + kColS16 + (c0 + c) / 2, r + c);
    tmem_st_wait();
  };

  // o^T of chunk n (TMEM buffer ob) -> o (warps 0-7: lane group lg, token half), through
  // the [64 t][128 j] bf16 stage and one TMA store issued by thread 0
  auto epi_bar = []() { asm volatile("bar.sync 1, 256;" ::: "memory"); };
  auto epilogue = [&](int n, int ob) {
    float r[32];
    tmem_ld32(tmem + lane_off + kColO + ob * 64 + half * 32, r);
    tmem_ld_wait();
    if (tid == 0) bulk_wait_read_all();  // the previous chunk's store has read the stage
    epi_bar();
    __nv_bfloat16* so =
        reinterpret_cast<__nv_bfloat16*>(sm + SM::kO) + half * 32 * kNV + lg * 32 + lane;
#pragma unroll
    for (int u = 0; u < 32; ++u) so[u * kNV] = __float2bfloat16_rn(r[u]);
    fence_async_smem();
    epi_bar();
    if (tid == 0) {
      tma_store_2d(&tmO, sm + SM::kO, j0, (int32_t)(row0 + (int64_t)n * kC));
      bulk_commit();
    }
  };

  // backward: the adjoint entering the first chunk (the segment's last) is
  // scaled by that chunk's e^{b_last} before the chunk's products
  if (BWD) {
    float r[kQ];
    scale_part(e_slot(0), r);
    copy_part(r);
  }
  tc_fence_before();
  __syncthreads();

  for (int it = 0; it < nc; ++it) {
    const int n = BWD ? (nc - 1 - it) : it;  // chunk index in the segment
    const uint32_t par = (uint32_t)(it & 1);
    const int xbuf = it & 1;
    unsigned char* sQ = sm + SM::kX + xbuf * SM::kXBuf;
    unsigned char* sK = sQ + SM::kTile;
    unsigned char* sP = sQ + SM::kP;
    wt(&bar_x[xbuf], (uint32_t)((it >> 1) & 1));
    // the next chunk's tiles go to the other buffers (their last readers, the MMAs
    // and the state pass of the previous chunk, completed before the block barrier
    // that ended the previous iteration); none once a wait has given up
    if (tid == kTmaTid && it + 1 < nc && !wait.aborted()) {
      issue_x(BWD ? n - 1 : n + 1, xbuf ^ 1);
      issue_v(BWD ? n - 1 : n + 1, xbuf ^ 1);
      // (slot (it + 2) % 3 was last read by the state pass of iteration it - 1)
      if (BWD && it + kESlots - 1 < nc) issue_e(it + kESlots - 1);
      if (kPf > 1 && it + kPf < nc) prefetch(BWD ? n - kPf : n + kPf);
    }
    // ------------------------------------------------ the chunk's MMAs
    if (tid == kMmaTid) {
      tc_fence_after();
      const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK), p0 = smem_u32(sP);
      const uint32_t v0 = smem_u32(sV + xbuf * SM::kVBuf);
      const uint32_t oc = tmem + kColO + (uint32_t)xbuf * 64;
      wt(&bar_v[xbuf], (uint32_t)((it >> 1) & 1));
      tc_fence_after();
      // the state update first: its completion releases part 1 of the state pass
      // forward:  S^T  += V^T  K~   (M = 128 columns j, N = DK rows i, K = 64 tokens s)
      // backward: dS^T += do^T Q~   (M = 128 columns j, N = DK rows i, K = 64 tokens t)
      const uint32_t u0 = BWD ? q0 : k0;
      constexpr uint32_t idS = idesc_bf16(128, DK, true, true);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t vd = sdesc_sw128(v0 + kk * 2048, 8192, 1024);
        const uint64_t ud = sdesc_sw128(u0 + kk * 2048, 8192, 1024);
        umma_bf16(tmem, vd, ud, idS, 1u);
      }
      umma_commit(&bar_u);
      // forward:  o^T  = S^T  Q~^T   (M = 128 columns j, N = 64 tokens t, K = DK; A from TMEM)
      // backward: dv^T = dS^T K~^T   (M = 128 columns j, N = 64 tokens s, K = DK; A from TMEM)
      // (A = the bf16 copy of the state before this chunk's update)
      constexpr uint32_t idO = idesc_bf16(128, 64, false, false);
      const uint32_t x0 = BWD ? k0 : q0;
#pragma unroll
      for (int kb = 0; kb < DK / 64; ++kb)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t xd = sdesc_sw128(x0 + kb * 8192 + kk * 32, 16, 1024);
          umma_bf16_ta(oc, tmem + kColS16 + kb * 32 + kk * 8, xd, idO, (kb | kk) ? 1u : 0u);
        }
      // forward:  o^T  += V^T  A^T  (B = A, K = s contiguous: K-major)
      // backward: dv^T += do^T A    (B = A, K = t rows, N = s contiguous: MN-major)
      constexpr uint32_t idO2 = idesc_bf16(128, 64, true, BWD);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t vd = sdesc_sw128(v0 + kk * 2048, 8192, 1024);
        const uint64_t pd = BWD ? sdesc_sw128(p0 + kk * 2048, 8192, 1024)
                                : sdesc_sw128(p0 + kk * 32, 16, 1024);
        umma_bf16(oc, vd, pd, idO2, 1u);
      }
      umma_commit(&bar_g);
    }
    __syncwarp();
    // ------------------------------------------------ the previous chunk's output
    if (warp < 8 && it > 0) epilogue(BWD ? n + 1 : n - 1, xbuf ^ 1);
    // ------------------------------------------------ the state pass for the next chunk
    //   forward:  S  <- e^{b_last}(this chunk) .* S
    //   backward: dS <- e^{b_last}(next chunk) .* dS  (the adjoint carried to its tokens)
    const bool more = it + 1 < nc;
    float r[kQ];
    if (more) {
      wt(&bar_u, par);
      tc_fence_after();
      scale_part(BWD ? e_slot(it + 1) : reinterpret_cast<const float*>(sQ + SM::kEx), r);
    }
    wt(&bar_g, par);
    tc_fence_after();
    if (more) copy_part(r);
    tc_fence_before();
    __syncthreads();
  }
  if (!wait.aborted()) {
    if (warp < 8) epilogue(BWD ? 0 : nc - 1, (nc - 1) & 1);
  } else {
    // a wait gave up: no MMA may still write tensor memory and no copy may still
    // write shared memory when the CTA exits (both waits bounded again)
    if (tid == kMmaTid) {
      umma_commit(&bar_fin);
      (void)mbar_wait(&bar_fin, 0u);
    }
    if (tid == kTmaTid) {
      for (uint32_t b = 0; b < 2; ++b) {
        const uint32_t ph = n_xv > b ? (n_xv - b + 1) / 2 : 0;
        drain_phase(&bar_x[b], ph);
        drain_phase(&bar_v[b], ph);
      }
      for (uint32_t k = 0; k < (uint32_t)kESlots; ++k)
        drain_phase(&bar_e[k], n_e > k ? (n_e - k + kESlots - 1) / kESlots : 0);
    }
  }
  if (tid == 0) bulk_wait_all();  // the output stores have read the stage and completed
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <int DK, bool BWD>
cudaError_t launch_sweep(const Dims& d, const void* Qt, const void* Kt, const void* v,
                         const void* A, const float* Eb, const float* S_src, void* o,
                         cudaStream_t st, int p_begin, int p_count) {
  CUtensorMap tq, tk, tv, tp, to;
  const uint64_t rows = (uint64_t)(d.B * d.H * d.T);
  if (!make_tmap_bf16(&tq, Qt, rows, DK, kC) || !make_tmap_bf16(&tk, Kt, rows, DK, kC) ||
      !make_tmap_bf16(&tv, v, rows, d.dv, kC) || !make_tmap_bf16(&tp, A, rows, kC, kC) ||
      !make_tmap_bf16_plain(&to, o, rows, d.dv, kNV, kC))
    return cudaErrorInvalidValue;
  const int smem = FwdSmem<DK>::kBytes + 1024;
  auto kern = tc_sweep_kernel<DK, BWD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(d.B * d.H * p_count * ((d.dv + kNV - 1) / kNV));
  prof_start(st);
  kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, tp, to, Eb, S_src, d.T,
                                     (int)d.dv, d.P, d.L, p_begin, p_count);
  return cudaGetLastError();
}

}  // namespace

bool tc_fwd_supported(const Dims& d) {
  return d.bf16 && (d.dk == 64 || d.dk == 128 || d.dk == 256) && d.dv % 64 == 0 &&
         d.C == kC && d.L % kC == 0;
}

cudaError_t tc_fwd_out(const Dims& d, const void* Qt, const void* Kt, const void* v,
                       const void* A, const float* Eb, const float* S_in, void* o,
                       cudaStream_t st, int p_begin, int p_count) {
  if (p_count < 0) p_count = d.P - p_begin;
  cudaError_t e =
      d.dk == 256   ? launch_sweep<256, false>(d, Qt, Kt, v, A, Eb, S_in, o, st, p_begin, p_count)
      : d.dk == 128 ? launch_sweep<128, false>(d, Qt, Kt, v, A, Eb, S_in, o, st, p_begin, p_count)
                    : launch_sweep<64, false>(d, Qt, Kt, v, A, Eb, S_in, o, st, p_begin, p_count);
  prof_mark("tc_fwd_out", st);
  return e;
}

cudaError_t tc_bwd_dv(const Dims& d, const void* Qt, const void* Kt, const void* d_o,
                      const void* A, const float* Eb, const float* D, void* dv,
                      cudaStream_t st) {
  cudaError_t e = d.dk == 256   ? launch_sweep<256, true>(d, Qt, Kt, d_o, A, Eb, D, dv, st, 0, d.P)
                  : d.dk == 128 ? launch_sweep<128, true>(d, Qt, Kt, d_o, A, Eb, D, dv, st, 0, d.P)
                                : launch_sweep<64, true>(d, Qt, Kt, d_o, A, Eb, D, dv, st, 0, d.P);
  prof_mark("tc_bwd_dv", st);
  return e;
}

// Reads and clears this file's bounded-wait flag (nonzero: a wait gave up).
int tc_fwd_take_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fwd_status, sizeof(v)) != cudaSuccess) return -1;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace zeco
