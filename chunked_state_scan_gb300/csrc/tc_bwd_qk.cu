// tc_bwd_qk.cu -- dq, dk and dlog_alpha of the backward on tcgen05 tensor cores.
//
// dq and dk contract over all d_v columns of the state, so the work is split
// by d_k rows: a pair of CTAs (a thread-block cluster of 2) owns a block of 64
// d_k rows i of one (b, h, segment); CTA r of the pair holds d_v columns
// [256 r, 256 r + 256).  Two launches sweep the segment's chunks:
//
//   forward sweep, state S (from S_in[p], the global state held since the
//   forward pass: Pith review of ZeCO, assumptions: Appendix A.4):
//     dA = do v^T (masked s <= t)
//     dq = e^{b} .* ( do S^T + dA K~ )          K~ = k .* e^{-b}
//     S <- e^{b_last} .* (S + K~^T v)
//   reverse sweep, adjoint dS (from D[p+1], the reverse segment scan):
//     dS <- e^{b_last} .* dS
//     dk = e^{-b} .* ( v dS^T + dA^T Q~ )       Q~ = q .* e^{b}
//     dS <- dS + Q~^T do
//     dlog_alpha_t = c_p + sum_{u >= t in segment} (q_u dq_u - k_u dk_u)
//
// (b: inclusive cumulative log-decay from the chunk start; c_p comes from the
// reverse segment scan.)  Each CTA forms partial dq^T / dk^T over its half of
// d_v (both products are linear in the d_v contraction, dA included); the pair
// adds the two halves through distributed shared memory and each CTA finishes
// 32 of the 64 rows.
//
// Q~, K~ (bf16) and e^{b_last} come from the decay pass (tc_decay.cu); the
// epilogue rebuilds e^{+-b_t} of its own elements from log_alpha.
//
// Precision of dlog_alpha.  Its suffix sum runs over the whole segment, so
// errors in the terms add up like a random walk.  Two measures keep them
// small: (1) the state copy used by the tensor cores is split into two bf16
// parts (hi + lo), so the state products are accurate to ~2^-17; (2) the terms
// use the rounded operands that the state itself was built from
// (the stored bf16 Q~ and K~ times the raw accumulators), so that the
// identity's telescoping holds for the rounded model instead of breaking on
// the rounding.
//
// The masked intra-chunk score gradient dA = do v^T comes precomputed in bf16
// (tc_scores.cu); CTA rank 0 of the pair adds its term.
//
// Tensor-memory layout.  A CTA keeps its 64 x 256 block of the state (or the
// adjoint) S[i, j] in fp32 twice, in lanes i and 64 + i (columns j): the
// update S += K~^T v is one M = 128, N = 256 MMA per 16 tokens whose A operand
// reads the [t][i] tile twice (both 64-row blocks at the same address).  Lanes
// 0-63 turn their copy into the bf16 high part of S and lanes 64-127 into the
// low part, which together are the A operand (rows = lanes, K = j in bf16
// pairs) of dq^T = S do^T: one M = 128 MMA per 16 columns j gives the high-part
// product in rows 0-63 and the low-part product in rows 64-127 of the
// accumulator.  The dA term joins rows 0-63 (its A operand's second block is a
// zero tile).  The two parts of each row go to separate partial-sum buffers
// that the epilogue adds.
//
// Warp roles (384 threads): thread 0 issues the copies and the MMAs; warps 0-7
// (warps w and w + 4 share lane quarter w % 4, each half of the columns) rescale
// the state, rebuild its hi/lo copy and send the partial sums; warps 8-11 run
// the epilogue of the previous chunk and read this chunk's epilogue factors.
//
// TMEM columns: [0, 256) state fp32 (two copies) | [256, 384) hi/lo copy |
// [384, 448) dq^T or dk^T (rows 0-63 hi part + dA term, 64-127 lo part).
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);
bool make_tmap_f32_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_cols, uint32_t box_rows);

namespace {

using namespace tc;

constexpr int kC = 64;
constexpr int kKB = 64;    // d_k rows per CTA pair
constexpr int kDV = 512;   // d_v
constexpr int kDVH = 256;  // d_v columns per CTA
constexpr int kThreads = 384;
constexpr uint32_t kColS = 0, kColHL = 256, kColAcc = 384;

// shared memory (bytes, 1024-aligned regions)
constexpr int kOffDO = 0;                        // do tile [64 t][256 j] (4 blocks of 64 j)
constexpr int kOffV = kOffDO + kC * kDVH * 2;    // v tile
constexpr int kXTile = kC * kKB * 2;             // one [64 t][64 i] bf16 tile
// Q~, K~, log_alpha tiles + q.dq rows [64 t][32 i] fp32 + e^{b_last} [64] fp32
constexpr int kXBuf = 3 * kXTile + 32 * kC * 4 + 1024;
constexpr int kOffX = kOffV + kC * kDVH * 2;     // 2 buffers of kXBuf (chunk parity)
constexpr int kOffP = kOffX + 2 * kXBuf;         // masked dA [64 t][64 s] bf16 (with do, v)
constexpr int kRS = kC + 4;                      // row stride of the partial sums (floats)
constexpr int kPart = 32 * kRS * 4;              // one [32 rows][kRS] fp32 partial-sum buffer
// partial sums for my 32 rows: the peer's high and low parts, then my own
constexpr int kOffR = kOffP + kC * kC * 2;       // peer: hi at +0, lo at +kPart
// own partials, double-buffered by chunk parity (written in a chunk's iteration,
// read by its epilogue in the next one): [parity][hi, lo]
constexpr int kOffOwn = kOffR + 2 * kPart;
constexpr int kOffZero = kOffOwn + 4 * kPart;    // zero tile [64][64] bf16 (dA term's A rows 64-127)
constexpr int kOffGq = kOffZero + kC * kC * 2;   // sums of log_alpha per 16 tokens [4][32]
constexpr int kOffQS = kOffGq + 1024;            // reverse: sums of dg terms per 16 tokens [4][32]
constexpr int kOffRun = kOffQS + 1024;           // reverse: dg suffix carried per row [32]
constexpr int kSmem = kOffRun + 128;

__device__ int g_qk_status = 0;

template <bool REV>
__global__ void __launch_bounds__(kThreads, 1)
tc_bwd_qk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmG, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmDO, const __grid_constant__ CUtensorMap tmQD,
                 const __grid_constant__ CUtensorMap tmP, const float* __restrict__ Eb,
                 const float* __restrict__ S_src,
                 const float* __restrict__ carry, __nv_bfloat16* __restrict__ out,
                 __nv_bfloat16* __restrict__ dg, float* __restrict__ qdq, int64_t T, int dk,
                 int P, int64_t L) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = (unsigned char*)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  unsigned char* sDO = sm + kOffDO;
  unsigned char* sV = sm + kOffV;
  unsigned char* sP = sm + kOffP;
  float* sR = reinterpret_cast<float*>(sm + kOffR);
  float* sOwn = reinterpret_cast<float*>(sm + kOffOwn);
  float* sGq = reinterpret_cast<float*>(sm + kOffGq);
  float* sQS = reinterpret_cast<float*>(sm + kOffQS);
  float* sRun = reinterpret_cast<float*>(sm + kOffRun);
  // bar_full: the peer's partial for my rows has landed in sR (complete_tx from
  // the peer's st.async); bar_empty: the peer has read the partial I sent it.
  // bar_a: the state update of the chunk is done, so the state may be rescaled
  // while the dq^T / dk^T MMAs run.
  __shared__ uint64_t bar_x[2], bar_dv, bar_a, bar_g1, bar_full, bar_empty;
  __shared__ uint32_t tmem_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = warp & 3;                   // TMEM lane quarter of this warp
  const uint32_t rank = cluster_ctarank();   // which half of d_v
  const int64_t bh = blockIdx.y / P;
  const int p = blockIdx.y % P;
  const int i0 = (blockIdx.x >> 1) * kKB;
  const int jb = (int)rank * kDVH;
  const int64_t row0 = bh * T + (int64_t)p * L;
  const int nc = (int)(L / kC);
  // state warps 0-7: lane `lane` of quarter lg is TMEM row r = 32 lg + lane, the
  // high part (r < 64) or low part (r >= 64) of d_k row ii = r % 64 of the block;
  // warp w handles columns [128 ch, 128 ch + 128) of the state with ch = w / 4
  const int r_tm = 32 * lg + lane;
  const int ii = r_tm & 63;                              // d_k row within the block
  const int part = r_tm >> 6;                            // 0: high part, 1: low part
  const int ch = (warp >> 2) & 1;
  const bool owned = (uint32_t)(ii >> 5) == rank;       // finished by this CTA

  if (tid == 0) {
    mbar_init(&bar_x[0], 1);
    mbar_init(&bar_x[1], 1);
    mbar_init(&bar_dv, 1);
    mbar_init(&bar_a, 1);
    mbar_init(&bar_g1, 1);
    mbar_init(&bar_full, 1);
    mbar_init(&bar_empty, 1);
    fence_mbar_init();
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmG);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmDO);
    prefetch_tmap(&tmP);
    if (REV) prefetch_tmap(&tmQD);
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  for (int u = tid; u < kC * kC * 2 / 16; u += kThreads)
    reinterpret_cast<uint4*>(sm + kOffZero)[u] = make_uint4(0u, 0u, 0u, 0u);
  fence_async_smem();  // the zero tile is read by the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive or st.async
  const uint32_t tmem = tmem_base;
  const uint32_t lane_off = (uint32_t)(lg * 32) << 16;

  auto chunk_row = [&](int n) { return (int32_t)(row0 + (int64_t)n * kC); };
  // Q~, K~, log_alpha tiles of chunk n, its e^{b_last} for rows i0.. and, reverse,
  // this CTA's q.dq rows, into buffer `buf`
  auto issue_x = [&](int n, int buf) {
    const int32_t r = chunk_row(n);
    unsigned char* xb = sm + kOffX + buf * kXBuf;
    mbar_expect_tx(&bar_x[buf], 3 * kXTile + kKB * 4 + (REV ? 32 * kC * 4 : 0));
    tma_load_2d(xb, &tmQ, i0, r, &bar_x[buf]);
    tma_load_2d(xb + kXTile, &tmK, i0, r, &bar_x[buf]);
    tma_load_2d(xb + 2 * kXTile, &tmG, i0, r, &bar_x[buf]);
    bulk_load(xb + 3 * kXTile + 32 * kC * 4, Eb + (size_t)(r / kC) * dk + i0, kKB * 4,
              &bar_x[buf]);
    if (REV) tma_load_2d(xb + 3 * kXTile, &tmQD, i0 + 32 * (int)rank, r, &bar_x[buf]);
  };
  // do, v halves and the masked dA of chunk n
  auto issue_dv = [&](int n) {
    const int32_t r = chunk_row(n);
    mbar_expect_tx(&bar_dv, 2 * kC * kDVH * 2 + kC * kC * 2);
    for (int b = 0; b < kDVH / 64; ++b) {
      tma_load_2d(sDO + b * 8192, &tmDO, jb + b * 64, r, &bar_dv);
      tma_load_2d(sV + b * 8192, &tmV, jb + b * 64, r, &bar_dv);
    }
    tma_load_2d(sP, &tmP, 0, r, &bar_dv);
  };
  if (tid == 0) {
    issue_x(REV ? nc - 1 : 0, 0);
    issue_dv(REV ? nc - 1 : 0);
  }

  // ---- state helpers (warps 0-7): this thread's TMEM row r_tm, the columns
  //      [128 ch, 128 ch + 128) of the state
  const uint32_t srow = tmem + lane_off + kColS + 128 * (uint32_t)ch;
  // S <- e^{b_last} .* S (row ii scaled by sE[ii]); 64 columns per load batch
  auto scale_state = [&](const float* sE) {
    const float e = sE[ii];
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float r[64];
      tmem_ld32(srow + 64 * h, r);
      tmem_ld32(srow + 64 * h + 32, r + 32);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < 64; ++u) r[u] *= e;
      tmem_st32(srow + 64 * h, r);
      tmem_st32(srow + 64 * h + 32, r + 32);
    }
    tmem_st_wait();
  };
  // this thread's part (high: bf16(S); low: bf16(S - high)) of the bf16 copy
  auto make_copy = [&]() {
    const uint32_t crow = tmem + lane_off + kColHL + 64 * (uint32_t)ch;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float r[64];
      tmem_ld32(srow + 64 * h, r);
      tmem_ld32(srow + 64 * h + 32, r + 32);
      tmem_ld_wait();
      uint32_t w32[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(r[2 * u], r[2 * u + 1]);
        const float2 hf = __bfloat1622float2(h2);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(r[2 * u] - hf.x, r[2 * u + 1] - hf.y);
        w32[u] = part ? *reinterpret_cast<const uint32_t*>(&l2)
                      : *reinterpret_cast<const uint32_t*>(&h2);
      }
      tmem_st16(crow + 32 * h, w32);
      tmem_st16(crow + 32 * h + 16, w32 + 16);
    }
    tmem_st_wait();
  };

  // ---- initial state: rows i0..i0+63, this CTA's columns (both copies)
  if (warp < 8) {
    const float* Sp = S_src + (((size_t)bh * (P + 1) + p + (REV ? 1 : 0)) * dk + i0 + ii) * kDV +
                      jb + 128 * ch;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float r[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 x = reinterpret_cast<const float4*>(Sp + 32 * c)[u];
        r[4 * u] = x.x;
        r[4 * u + 1] = x.y;
        r[4 * u + 2] = x.z;
        r[4 * u + 3] = x.w;
      }
      tmem_st32(srow + 32 * c, r);
    }
    tmem_st_wait();
    if (REV) {
      // the first chunk's adjoint is scaled by its e^{b_last} before its MMAs
      if (!mbar_wait(&bar_x[0], 0u)) atomicExch(&g_qk_status, 1);
      scale_state(reinterpret_cast<const float*>(sm + kOffX + 3 * kXTile + 32 * kC * 4));
    }
    make_copy();
  }

  // element (t, column c) of a [64 t][64 i] tile
  auto tile_at = [&](unsigned char* base, int t, int c) -> __nv_bfloat16* {
    return reinterpret_cast<__nv_bfloat16*>(base + sw128((uint32_t)t, (uint32_t)((c & 63) >> 3)) +
                                            (uint32_t)(c & 7) * 2u);
  };
  // Epilogue workers (warps 8-11): owned row er (d_k row ec of the block) x the
  // 16 tokens 16 eq .. 16 eq + 15.
  const int er = tid & 31, eq = (warp - 8) & 3;
  const int ec = 32 * (int)rank + er;
  const bool epi = warp >= 8;

  if (REV && tid < 32) sRun[tid] = carry[((size_t)bh * P + p) * dk + i0 + 32 * (int)rank + tid];
  const uint32_t peer = rank ^ 1u;
  const uint32_t peer_full = map_to_rank(smem_u32(&bar_full), peer);
  const uint32_t peer_empty = map_to_rank(smem_u32(&bar_empty), peer);
  if (tid == 256) mbar_expect_tx(&bar_full, 2 * 32 * kC * 4);  // phase 0: the first partial

  // Per-element factors of a chunk's epilogue, read from the chunk's tiles in its
  // own iteration and kept in registers until the epilogue runs in the next one
  // (so the tile buffers are free for the next prefetch): ef = e^{b_t} (forward)
  // or e^{-b_t} (reverse), xr = the stored rounded Q~ (forward) or K~ (reverse),
  // qd = q.dq (reverse).  b_t sums log_alpha over the earlier 16-token quarters
  // of the chunk plus the running sum within this one.
  float ef[16], xr[16], qd[16];
  auto epi_sync = []() { asm volatile("bar.sync 1, 128;" ::: "memory"); };
  auto prefetch = [&](const unsigned char* sQ, const unsigned char* sK,
                      const unsigned char* sG, const float* sQD) {
    float gl[16];
    float gs = 0.f;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      gl[u] = __bfloat162float(*tile_at(const_cast<unsigned char*>(sG), 16 * eq + u, ec));
      gs += gl[u];
    }
    sGq[eq * 32 + er] = gs;
    epi_sync();
    float b = 0.f;
    for (int q2 = 0; q2 < eq; ++q2) b += sGq[q2 * 32 + er];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      b += gl[u];
      ef[u] = __expf(REV ? -b : b);
      xr[u] = __bfloat162float(*tile_at(const_cast<unsigned char*>(REV ? sK : sQ), 16 * eq + u, ec));
      if (REV) qd[u] = sQD[(16 * eq + u) * 32 + er];
    }
  };
  // outputs of chunk n from the four partial sums (peer's and own, high and low
  // parts)
  auto epilogue = [&](int n, int it) {
    const float* own = sOwn + (it & 1) * (2 * kPart / 4);
    const float4* rh = reinterpret_cast<const float4*>(sR + er * kRS + 16 * eq);
    const float4* rl = reinterpret_cast<const float4*>(sR + kPart / 4 + er * kRS + 16 * eq);
    const float4* oh = reinterpret_cast<const float4*>(own + er * kRS + 16 * eq);
    const float4* ol = reinterpret_cast<const float4*>(own + kPart / 4 + er * kRS + 16 * eq);
    float acc[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 a4 = rh[c], b4 = rl[c], c4 = oh[c], d4 = ol[c];
      acc[4 * c] = (a4.x + c4.x) + (b4.x + d4.x);
      acc[4 * c + 1] = (a4.y + c4.y) + (b4.y + d4.y);
      acc[4 * c + 2] = (a4.z + c4.z) + (b4.z + d4.z);
      acc[4 * c + 3] = (a4.w + c4.w) + (b4.w + d4.w);
    }
    const size_t base = (size_t)(chunk_row(n) + 16 * eq) * dk + i0 + ec;
    if (!REV) {
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        out[base + (size_t)u * dk] = __float2bfloat16_rn(acc[u] * ef[u]);
        // the stored rounded Q~ times the raw accumulator (= q_eff dq)
        qdq[base + (size_t)u * dk] = xr[u] * acc[u];
      }
    } else {
      float term[16];
      float s = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        out[base + (size_t)u * dk] = __float2bfloat16_rn(acc[u] * ef[u]);
        // the stored rounded K~ times the raw accumulator (= k_eff dk)
        term[u] = qd[u] - xr[u] * acc[u];
        s += term[u];
      }
      sQS[eq * 32 + er] = s;
      epi_sync();
      float runq = sRun[er];
      for (int q2 = 3; q2 > eq; --q2) runq += sQS[q2 * 32 + er];
#pragma unroll
      for (int u = 15; u >= 0; --u) {
        runq += term[u];
        dg[base + (size_t)u * dk] = __float2bfloat16_rn(runq);
      }
      epi_sync();
      if (eq == 0) sRun[er] = runq;  // suffix through the whole chunk
    }
  };
  // epilogue of chunk n = the it-th processed (warps 8-11): wait for the peer's
  // partial, then release sR back to the peer and arm bar_full for the next one
  auto finish = [&](int n, int it) {
    if (!mbar_wait(&bar_full, (uint32_t)(it & 1))) atomicExch(&g_qk_status, 1);
    epilogue(n, it);
    epi_sync();  // every epilogue thread has read sR
    if (tid == 256 && it + 1 < nc) {
      mbar_arrive_remote(peer_empty);
      mbar_expect_tx(&bar_full, 2 * 32 * kC * 4);
    }
  };

  // Per chunk: thread 0 issues the state update (one M = 128, N = 256 MMA per 16
  // tokens, both copies) and commits bar_a, then dq^T / dk^T from the hi/lo copy
  // (16 M = 128 MMAs, A in tensor memory) and, rank 0, the dA term, and commits
  // bar_g1.  Warps 0-7 rescale the state once bar_a completes (forward: by this
  // chunk's e^{b_last}; reverse: by the next chunk's), send this chunk's partial
  // sums after bar_g1 and rebuild the hi/lo copy; warps 8-11 run the previous
  // chunk's epilogue and read this chunk's epilogue factors meanwhile.
  for (int it = 0; it < nc; ++it) {
    const int n = REV ? (nc - 1 - it) : it;
    const int nn = REV ? n - 1 : n + 1;  // the next chunk processed
    const bool more = it + 1 < nc;
    const uint32_t par = (uint32_t)(it & 1);
    const int xbuf = it & 1;
    unsigned char* sQ = sm + kOffX + xbuf * kXBuf;
    unsigned char* sK = sQ + kXTile;
    unsigned char* sG = sQ + 2 * kXTile;
    const float* sQD = reinterpret_cast<const float*>(sQ + 3 * kXTile);
    const float* sE = sQD + 32 * kC;  // e^{b_last} of rows i0..i0+63
    const float* sEn =                // the next chunk's, in the other buffer
        reinterpret_cast<const float*>(sm + kOffX + (xbuf ^ 1) * kXBuf + 3 * kXTile + 32 * kC * 4);
    // the next chunk's tiles go to the other buffer (freed at the end of the last iteration)
    if (tid == 0 && more) issue_x(nn, xbuf ^ 1);
    if (!mbar_wait(&bar_x[xbuf], (uint32_t)((it >> 1) & 1))) atomicExch(&g_qk_status, 1);
    tc_fence_before();
    __syncthreads();
    // ---- the chunk's MMAs
    if (tid == 0) {
      if (!mbar_wait(&bar_dv, par)) atomicExch(&g_qk_status, 1);
      tc_fence_after();
      const uint32_t o0 = smem_u32(sDO), v0 = smem_u32(sV);
      const uint32_t x0 = smem_u32(REV ? sQ : sK);
      // forward: S += K~^T v    reverse: dS += Q~^T do   (M = 128: rows 0-63 and 64-127
      // both read the [t][i] tile (block stride 0), N = 256 j, K = 64 t; B = the
      // [t][j] tile read MN-major)
      constexpr uint32_t idU = idesc_bf16(128, 256, true, true);
      const uint32_t u0 = REV ? o0 : v0;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        umma_bf16(tmem + kColS, sdesc_sw128(x0 + kk * 2048, 0, 1024),
                  sdesc_sw128(u0 + kk * 2048, 8192, 1024), idU, 1u);
      umma_commit(&bar_a);
      // forward: dq^T = S do^T    reverse: dk^T = (e^{b_last} dS) v^T, hi and lo parts
      // (M = 128 hi/lo rows, A = the copy in tensor memory; N = 64, K = 256 j)
      constexpr uint32_t idT = idesc_bf16(128, 64, false, false);
      const uint32_t z0 = REV ? v0 : o0;
#pragma unroll 4
      for (int m = 0; m < kDVH / 16; ++m) {
        const uint32_t koff = (uint32_t)((m >> 2) * 8192 + (m & 3) * 32);
        umma_bf16_ta(tmem + kColAcc, tmem + kColHL + m * 8, sdesc_sw128(z0 + koff, 16, 1024),
                     idT, m ? 1u : 0u);
      }
      // rank 0: forward K~^T dA^T ; reverse Q~^T dA into rows 0-63 (M = 128: the A
      // operand's second 64-row block is the zero tile; N = 64, K = 64)
      if (rank == 0) {
        const uint32_t p0 = smem_u32(sP);
        const uint32_t zoff = smem_u32(sm + kOffZero) - x0;  // block stride to the zero tile
        constexpr uint32_t id2 = idesc_bf16(128, 64, true, REV);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t xd = sdesc_sw128(x0 + kk * 2048, zoff, 1024);
          const uint64_t pd = REV ? sdesc_sw128(p0 + kk * 2048, 8192, 1024)
                                  : sdesc_sw128(p0 + kk * 32, 16, 1024);
          umma_bf16(tmem + kColAcc, xd, pd, id2, 1u);
        }
      }
      umma_commit(&bar_g1);
    }
    if (!epi) {
      // ---- warps 0-7: rescale the state while dq^T / dk^T run
      if (!mbar_wait(&bar_a, par)) atomicExch(&g_qk_status, 1);
      tc_fence_after();
      if (more) {
        if (!REV) {
          scale_state(sE);
        } else {
          if (!mbar_wait(&bar_x[xbuf ^ 1], (uint32_t)(((it + 1) >> 1) & 1)))
            atomicExch(&g_qk_status, 1);
          scale_state(sEn);
        }
      }
      if (!mbar_wait(&bar_g1, par)) atomicExch(&g_qk_status, 1);
      tc_fence_after();
      if (tid == 0 && more) issue_dv(nn);  // do, v, dA buffers are free
      // ---- partial sums of this chunk, this thread's part of row ii, tokens
      //      [32 ch, 32 ch + 32): the peer's rows into the peer's buffers
      //      (st.async, completing on the peer's bar_full), mine into sOwn
      {
        float a[32];
        tmem_ld32(tmem + lane_off + kColAcc + 32 * ch, a);
        tmem_ld_wait();
        const int off = part * (kPart / 4) + (ii & 31) * kRS + 32 * ch;
        if (owned) {
          float4* dst = reinterpret_cast<float4*>(sOwn + (it & 1) * (2 * kPart / 4) + off);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            dst[c] = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
        } else {
          // the peer has read the partial of the previous chunk
          if (!mbar_wait(&bar_empty, par ^ 1u)) atomicExch(&g_qk_status, 1);
          const uint32_t dst = map_to_rank(smem_u32(sR + off), peer);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_async_v4(dst + c * 16, a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3],
                        peer_full);
        }
      }
      // ---- the next chunk's hi/lo copy
      if (more) make_copy();
    } else {
      // ---- warps 8-11: the previous chunk's epilogue, then this chunk's factors
      if (it > 0) finish(REV ? n + 1 : n - 1, it - 1);
      prefetch(sQ, sK, sG, sQD);
      if (!mbar_wait(&bar_g1, par)) atomicExch(&g_qk_status, 1);
    }
    tc_fence_before();
    __syncthreads();
  }
  if (epi) finish(REV ? 0 : nc - 1, nc - 1);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no st.async or remote arrive is still in flight to either CTA
  if (warp == 0) tmem_dealloc(tmem, 512);
}

template <bool REV>
cudaError_t launch_qk(const Dims& d, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tg, const CUtensorMap& tv, const CUtensorMap& tdo,
                      const CUtensorMap& tqd, const CUtensorMap& tp, const float* Eb,
                      const float* S_src, const float* carry, void* out, void* dg, float* qdq,
                      cudaStream_t st) {
  auto kern = tc_bwd_qk_kernel<REV>;
  const int smem = kSmem + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * d.dk / kKB), (unsigned)(d.B * d.H * d.P), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tg, tv, tdo, tqd, tp, Eb, S_src, carry,
                            (__nv_bfloat16*)out,
                            (__nv_bfloat16*)dg, qdq, d.T, (int)d.dk, d.P, d.L);
}

}  // namespace

bool tc_bwd_qk_supported(const Dims& d) {
  return d.bf16 && d.dk % kKB == 0 && d.dv == kDV && d.C == kC && d.L % kC == 0;
}

cudaError_t tc_bwd_qk(const Dims& d, const void* Qt, const void* Kt, const void* v,
                      const void* g, const float* Eb, const void* dA, const float* S_in,
                      const void* d_o, void* dq, void* dk, void* dg, float* D, float* carry,
                      float* qdq, cudaStream_t st) {
  CUtensorMap tq, tk, tg, tv, tdo, tqd, tp;
  const uint64_t rows = (uint64_t)(d.B * d.H * d.T);
  if (!make_tmap_bf16(&tq, Qt, rows, d.dk, kC) || !make_tmap_bf16(&tk, Kt, rows, d.dk, kC) ||
      !make_tmap_bf16(&tg, g, rows, d.dk, kC) || !make_tmap_bf16(&tv, v, rows, d.dv, kC) ||
      !make_tmap_bf16(&tdo, d_o, rows, d.dv, kC) || !make_tmap_bf16(&tp, dA, rows, kC, kC) ||
      !make_tmap_f32_plain(&tqd, qdq, rows, d.dk, 32, kC))
    return cudaErrorInvalidValue;
  cudaError_t e =
      launch_qk<false>(d, tq, tk, tg, tv, tdo, tqd, tp, Eb, S_in, carry, dq, dg, qdq, st);
  prof_mark("tc_bwd_dq", st);
  if (e != cudaSuccess) return e;
  e = launch_qk<true>(d, tq, tk, tg, tv, tdo, tqd, tp, Eb, D, carry, dk, dg, qdq, st);
  prof_mark("tc_bwd_dk", st);
  return e;
}

// Reads and clears this file's bounded-wait flag (nonzero: a wait gave up).
int tc_bwd_qk_take_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_qk_status, sizeof(v)) != cudaSuccess) return -1;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_qk_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace zeco
