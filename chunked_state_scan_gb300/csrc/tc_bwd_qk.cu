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
// TMEM columns: [0, 128) state (d_v group g of this CTA at 64 g) | [192, 256)
// dq^T or dk^T (M = 64 layout, lane = d_k row).
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
constexpr int kThreads = 256;
constexpr uint32_t kColAcc = 192;

// shared memory (bytes, 1024-aligned regions)
constexpr int kOffDO = 0;                        // do tile [64 t][256 j] (4 blocks of 64 j)
constexpr int kOffV = kOffDO + kC * kDVH * 2;    // v tile
constexpr int kOffHi = kOffV + kC * kDVH * 2;    // state copy, high part [256 j][64 i]
constexpr int kOffLo = kOffHi + kDVH * kKB * 2;  // state copy, low part
constexpr int kXTile = kC * kKB * 2;             // one [64 t][64 i] bf16 tile
// Q~, K~, log_alpha tiles + q.dq rows [64 t][32 i] fp32 + e^{b_last} [64] fp32
constexpr int kXBuf = 3 * kXTile + 32 * kC * 4 + 1024;
constexpr int kOffX = kOffLo + kDVH * kKB * 2;   // 2 buffers of kXBuf (chunk parity)
constexpr int kOffP = kOffX + 2 * kXBuf;         // masked dA [64 t][64 s] bf16 (with do, v)
constexpr int kRS = kC + 4;                      // row stride of the partial sums (floats)
constexpr int kOffR = kOffP + kC * kC * 2;       // peer's partial for my rows [32][kRS] fp32
constexpr int kOffOwn = kOffR + 32 * kRS * 4;    // my own partial for my rows [32][kRS] fp32
constexpr int kOffGq = kOffOwn + 32 * kRS * 4;   // sums of log_alpha per 8 tokens [8][32]
constexpr int kOffQS = kOffGq + 1024;            // reverse: sums of dg terms per 8 tokens [8][32]
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
  unsigned char* sHi = sm + kOffHi;
  unsigned char* sLo = sm + kOffLo;
  unsigned char* sP = sm + kOffP;
  float* sR = reinterpret_cast<float*>(sm + kOffR);
  float* sOwn = reinterpret_cast<float*>(sm + kOffOwn);
  float* sGq = reinterpret_cast<float*>(sm + kOffGq);
  float* sQS = reinterpret_cast<float*>(sm + kOffQS);
  float* sRun = reinterpret_cast<float*>(sm + kOffRun);
  // bar_full: the peer's partial for my rows has landed in sR (complete_tx from
  // the peer's st.async); bar_empty: the peer has read the partial I sent it.
  __shared__ uint64_t bar_x[2], bar_dv, bar_g1, bar_full, bar_empty;
  __shared__ uint32_t tmem_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lg = warp & 3, grp = warp >> 2;  // TMEM lane group; this warp's d_v group
  const uint32_t rank = cluster_ctarank();   // which half of d_v
  const int64_t bh = blockIdx.y / P;
  const int p = blockIdx.y % P;
  const int i0 = (blockIdx.x >> 1) * kKB;
  const int jb = (int)rank * kDVH;
  const int64_t row0 = bh * T + (int64_t)p * L;
  const int nc = (int)(L / kC);
  // the M = 64 TMEM layout: warp w < 4, lane l < 16 holds row 16 w + l
  const bool rowt = warp < 4 && lane < 16;
  const int ii = warp * 16 + lane;                      // d_k row within the block
  const bool owned = rowt && (uint32_t)(ii >> 5) == rank;  // finished by this CTA

  if (tid == 0) {
    mbar_init(&bar_x[0], 1);
    mbar_init(&bar_x[1], 1);
    mbar_init(&bar_dv, 1);
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
  if (warp == 0) tmem_alloc(&tmem_base, 256);
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

  // bf16 hi/lo copy of this warp's state group (lanes = local d_v column j)
  auto write_copy = [&](const float* r) {
    const uint32_t j = (uint32_t)(grp * 128 + lg * 32 + lane);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float a = r[8 * c + 2 * u], b = r[8 * c + 2 * u + 1];
        const __nv_bfloat16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
        __nv_bfloat162 h2, l2;
        h2.x = ha;
        h2.y = hb;
        l2 = __floats2bfloat162_rn(a - __bfloat162float(ha), b - __bfloat162float(hb));
        hw[u] = *reinterpret_cast<uint32_t*>(&h2);
        lw[u] = *reinterpret_cast<uint32_t*>(&l2);
      }
      const uint32_t off = sw128(j, (uint32_t)c);
      *reinterpret_cast<uint4*>(sHi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
      *reinterpret_cast<uint4*>(sLo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    }
  };

  // ---- initial state: rows i0..i0+63, this CTA's columns
  {
    const float* Sp = S_src + (((size_t)bh * (P + 1) + p + (REV ? 1 : 0)) * dk + i0) * kDV + jb +
                      grp * 128 + lg * 32 + lane;
    float r[64];
#pragma unroll
    for (int u = 0; u < 64; ++u) r[u] = Sp[(size_t)u * kDV];
    tmem_st32(tmem + lane_off + grp * 64, r);
    tmem_st32(tmem + lane_off + grp * 64 + 32, r + 32);
    if (!REV) write_copy(r);
    tmem_st_wait();
  }

  // state <- e^{b_last} .* state (column i scaled by sE[i]) and its hi/lo copy
  auto state_pass = [&](const float* sE) {
    float r[64];
    tmem_ld32(tmem + lane_off + grp * 64, r);
    tmem_ld32(tmem + lane_off + grp * 64 + 32, r + 32);
    tmem_ld_wait();
#pragma unroll
    for (int u = 0; u < 64; ++u) r[u] *= sE[u];
    tmem_st32(tmem + lane_off + grp * 64, r);
    tmem_st32(tmem + lane_off + grp * 64 + 32, r + 32);
    write_copy(r);
    tmem_st_wait();
  };

  // element (t, column c) of a [64 t][64 i] tile
  auto tile_at = [&](unsigned char* base, int t, int c) -> __nv_bfloat16* {
    return reinterpret_cast<__nv_bfloat16*>(base + sw128((uint32_t)t, (uint32_t)((c & 63) >> 3)) +
                                            (uint32_t)(c & 7) * 2u);
  };
  // Warp roles within a chunk: thread 0 issues the TMA copies and the MMAs;
  // warps 0-3 read the dA and partial-sum accumulators (the M = 64 layout puts
  // rows in their lanes) and mask dA; all 8 warps run the state pass; warps 4-7
  // run the previous chunk's epilogue and this chunk's epilogue prefetch while
  // the tensor cores execute MMA group 1.
  // Epilogue workers (warps 4-7): owned row er (d_k row ec of the block) x the
  // 16 tokens 16 eq .. 16 eq + 15.
  const int er = tid & 31, eq = (warp - 4) & 3;
  const int ec = 32 * (int)rank + er;
  const bool epi = warp >= 4;

  if (REV && tid < 32) sRun[tid] = carry[((size_t)bh * P + p) * dk + i0 + 32 * (int)rank + tid];
  const uint32_t peer = rank ^ 1u;
  const uint32_t peer_full = map_to_rank(smem_u32(&bar_full), peer);
  const uint32_t peer_empty = map_to_rank(smem_u32(&bar_empty), peer);
  if (tid == 128) mbar_expect_tx(&bar_full, 32 * kC * 4);  // phase 0: the first partial

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
  // outputs of chunk n from the two partial sums (peer's + own)
  auto epilogue = [&](int n) {
    const float4* rp = reinterpret_cast<const float4*>(sR + er * kRS + 16 * eq);
    const float4* op = reinterpret_cast<const float4*>(sOwn + er * kRS + 16 * eq);
    float acc[16];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 r4 = rp[c], o4 = op[c];
      acc[4 * c] = r4.x + o4.x;
      acc[4 * c + 1] = r4.y + o4.y;
      acc[4 * c + 2] = r4.z + o4.z;
      acc[4 * c + 3] = r4.w + o4.w;
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
  // epilogue of chunk n = the it-th processed (warps 4-7): wait for the peer's
  // partial, then release sR back to the peer and arm bar_full for the next one
  auto finish = [&](int n, int it) {
    if (!mbar_wait(&bar_full, (uint32_t)(it & 1))) atomicExch(&g_qk_status, 1);
    epilogue(n);
    epi_sync();  // every epilogue thread has read sR
    if (tid == 128 && it + 1 < nc) {
      mbar_arrive_remote(peer_empty);
      mbar_expect_tx(&bar_full, 32 * kC * 4);
    }
  };

  for (int it = 0; it < nc; ++it) {
    const int n = REV ? (nc - 1 - it) : it;
    const uint32_t par = (uint32_t)(it & 1);
    const int xbuf = it & 1;
    unsigned char* sQ = sm + kOffX + xbuf * kXBuf;
    unsigned char* sK = sQ + kXTile;
    unsigned char* sG = sQ + 2 * kXTile;
    const float* sQD = reinterpret_cast<const float*>(sQ + 3 * kXTile);
    const float* sE = sQD + 32 * kC;  // e^{b_last} of rows i0..i0+63
    // the next chunk's tiles go to the other buffer (freed at the end of the last iteration)
    if (tid == 0 && it + 1 < nc) issue_x(REV ? n - 1 : n + 1, xbuf ^ 1);
    if (!mbar_wait(&bar_x[xbuf], (uint32_t)((it >> 1) & 1))) atomicExch(&g_qk_status, 1);
    if (REV) state_pass(sE);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- MMA group 1
    if (tid == 0) {
      if (!mbar_wait(&bar_dv, par)) atomicExch(&g_qk_status, 1);
      tc_fence_after();
      const uint32_t o0 = smem_u32(sDO), v0 = smem_u32(sV), h0 = smem_u32(sHi),
                     l0 = smem_u32(sLo);
      const uint32_t x0 = smem_u32(REV ? sQ : sK);
      constexpr uint32_t idT = idesc_bf16(64, 64, true, false);    // copy (x) do or v
#pragma unroll 4
      for (int m = 0; m < kDVH / 16; ++m) {  // K = this CTA's d_v half, 16 per step
        const uint32_t koff = (uint32_t)((m >> 2) * 8192 + (m & 3) * 32);
        const uint64_t yd = sdesc_sw128((REV ? v0 : o0) + koff, 16, 1024);
        const uint64_t hd = sdesc_sw128(h0 + m * 2048, 8192, 1024);
        const uint64_t ld = sdesc_sw128(l0 + m * 2048, 8192, 1024);
        // forward: dq^T = S do^T     reverse: dk^T = (e^{b_last} dS) v^T   (M = 64 i, N = 64)
        umma_bf16(tmem + kColAcc, hd, yd, idT, m ? 1u : 0u);
        umma_bf16(tmem + kColAcc, ld, yd, idT, 1u);
      }
      // rank 0: forward dq^T += K~^T dA^T ; reverse dk^T += Q~^T dA   (M = 64 i, N = 64, K = 64)
      if (rank == 0) {
        const uint32_t p0 = smem_u32(sP);
        constexpr uint32_t id2 = idesc_bf16(64, 64, true, REV);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t xd = sdesc_sw128(x0 + kk * 2048, 8192, 1024);
          const uint64_t pd = REV ? sdesc_sw128(p0 + kk * 2048, 8192, 1024)
                                  : sdesc_sw128(p0 + kk * 32, 16, 1024);
          umma_bf16(tmem + kColAcc, xd, pd, id2, 1u);
        }
      }
      // forward: S^T_g += v_g^T K~    reverse: dS^T_g += do_g^T Q~   (M = 128 j, N = 64 i, K = 64)
      constexpr uint32_t idS = idesc_bf16(128, 64, true, true);
      const uint32_t y0 = REV ? o0 : v0;
#pragma unroll
      for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t yd = sdesc_sw128(y0 + g * 16384 + kk * 2048, 8192, 1024);
          const uint64_t xd = sdesc_sw128(x0 + kk * 2048, 8192, 1024);
          umma_bf16(tmem + g * 64, yd, xd, idS, 1u);
        }
      umma_commit(&bar_g1);
    }
    // ---- warps 4-7, while the tensor cores run group 1: the previous chunk's
    //      epilogue, then this chunk's epilogue factors
    if (epi) {
      if (it > 0) finish(REV ? n + 1 : n - 1, it - 1);
      prefetch(sQ, sK, sG, sQD);
    }
    if (!mbar_wait(&bar_g1, par)) atomicExch(&g_qk_status, 1);
    tc_fence_after();
    if (tid == 0 && it + 1 < nc) issue_dv(REV ? n - 1 : n + 1);  // do, v, dA buffers are free
    if (!REV) state_pass(sE);  // forward: post-scale and copy for the next chunk
    // ---- partial sums of this chunk: the peer's rows into the peer's sR
    //      (st.async, completing on the peer's bar_full), mine into sOwn
    if (warp < 4) {
      float a[64];
      tmem_ld32(tmem + lane_off + kColAcc, a);
      tmem_ld32(tmem + lane_off + kColAcc + 32, a + 32);
      tmem_ld_wait();
      if (rowt) {
        if (owned) {
          float4* dst = reinterpret_cast<float4*>(sOwn + (ii & 31) * kRS);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            dst[c] = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
        } else {
          // the peer has read the partial of the previous chunk
          if (!mbar_wait(&bar_empty, par ^ 1u)) atomicExch(&g_qk_status, 1);
          const uint32_t dst = map_to_rank(smem_u32(sR + (ii & 31) * kRS), peer);
#pragma unroll
          for (int c = 0; c < 16; ++c)
            st_async_v4(dst + c * 16, a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3],
                        peer_full);
        }
      }
    }
    fence_async_smem();  // forward: the state copy, read by the next group 1
    tc_fence_before();
    __syncthreads();
  }
  if (epi) finish(REV ? 0 : nc - 1, nc - 1);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no st.async or remote arrive is still in flight to either CTA
  if (warp == 0) tmem_dealloc(tmem, 256);
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

}  // namespace zeco
