// tc_bwd_qk.cu -- dq, dk and dlog_alpha of the backward on tcgen05 tensor cores.
//
// dq and dk contract over all d_v columns of the state.  A cluster of four CTAs
// owns a block of 128 d_k rows i of one (b, h, segment); CTA r of the cluster
// holds the d_v columns [128 r, 128 r + 128).  For d_v < 512 (a multiple of 64)
// the columns beyond d_v hold a zero state and receive zero v / do tiles (the
// copies of boxes past the end of a tensor read zeros), so their partial sums
// are zero and the results are those of the d_v columns that exist.  Likewise a
// d_k that is not a multiple of 128 (d_k = 64, 192) pads its last block with
// zero rows, which are not stored.
// Two launches sweep the segment's chunks:
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
// reverse segment scan.)  Each CTA forms a partial dq^T / dk^T [128 i][64 t] over
// its quarter of d_v (both products are linear in the d_v contraction, the dA
// term included: CTA r adds the 16 intra-chunk positions s in [16 r, 16 r + 16));
// the four quarters meet in distributed shared memory, and CTA r finishes the 32
// rows [32 r, 32 r + 32) of the block.
//
// Q~, K~ (bf16) and e^{b_last} come from the decay pass (tc_decay.cu; the
// forward keeps them for the backward); the masked dA = do v^T from the score
// pass (tc_scores.cu); the epilogue rebuilds e^{+-b_t} of its own elements from
// log_alpha.  The state warps read their rows' e^{b_last} straight from global
// memory a chunk ahead, so the serial state chain never waits on an operand
// copy.  The partial sums travel in token-quad-major slots: each st.async of a
// warp writes 512 contiguous bytes.
//
// Precision of dlog_alpha.  Its suffix sum runs over the whole segment, so
// errors in the terms add up like a random walk.  Two measures keep them
// small: (1) the state copy used by the tensor cores is split into two bf16
// parts (hi + lo, both multiplied into the same fp32 accumulator), so the state
// products are accurate to ~2^-17; (2) the terms use the rounded operands that
// the state itself was built from (the stored bf16 Q~ and K~ times the raw
// accumulators), so that the identity's telescoping holds for the rounded model
// instead of breaking on the rounding.  The no-decay form has no dlog_alpha:
// it writes and multiplies only the high part (9 MMAs per chunk instead of 17).
//
// Tensor memory (512 columns): the CTA's state block S[i][j] in fp32 (lane i,
// column j) | two bf16 hi/lo copies of it (lane i; 64 columns of packed pairs
// of the high parts, then 64 of the low parts), one per chunk parity | two
// [128 i][64 t] accumulators, one per chunk parity.
//
// Per chunk the serial chain is short: the MMA warp adds K~^T v (or Q~^T do) to
// the state (four M = 128, N = 128 MMAs) and commits; the state warps rescale
// the state and write the next chunk's hi/lo copy in one pass over it and hand
// it back.  The dq^T / dk^T MMAs of the chunk (one dA-term MMA and 16 MMAs with
// A in tensor memory) run meanwhile, into the accumulator of the chunk's
// parity; copies run two chunks ahead; the exchange and epilogue of a chunk
// overlap the next chunks.
//
// Warp roles (704 threads): warps 0-7 state (warps w and w + 4 share TMEM lane
// quarter w % 4, each half of the columns); warps 8-11 exchange (lane quarter
// w - 8 of the accumulator goes to CTA w - 8); warps 12-19 epilogue in two
// groups of four that take alternate chunks (receive buffer, factor stage and
// named barriers by chunk parity), each warp 16 tokens of this CTA's 32 rows,
// so that one chunk's epilogue may take up to two chunk periods; warp 20
// copies the MMA operands; warp 21 issues the MMAs.  A group's first thread
// copies the group's epilogue factors two chunks ahead, hands each receive
// buffer back once the group has read it (locally and to the other three
// CTAs; relaxed arrives, as the reads they release were performed before the
// group's barrier, while a release arrive would wait for memory operations in
// flight), and stores the chunk's outputs (dq or dk, and q.dq or dlog_alpha)
// by TMA from the factor stage, where the group's threads write each output
// over the factor they read at the same position.  The reverse sweep's
// dlog_alpha suffix passes from group to group through shared memory and an
// mbarrier.  The partials are received double-buffered, so that the four CTAs
// of a cluster need not move in lockstep.
//
// Decay forms.  The scalar-decay form copies the chunk's 64 log-decays (one per
// token) instead of a [64 t][32 i] tile, and its reverse sweep sums each
// token's dlog_alpha over this CTA's 32 rows in the warp (a shuffle tree) and
// stores the fp32 partial of the rows [32 c, 32 c + 32), c = i0 / 32 + rank,
// at dlog_alpha_part[c][t]; a small kernel adds the d_k / 32 partials of a
// token (decay_forms.cu).  The no-decay form (b = 0) copies no log-decay and
// neither writes q.dq nor computes dlog_alpha.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows);
bool make_tmap_bf16_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_cols, uint32_t box_rows);
bool make_tmap_f32_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_cols, uint32_t box_rows);

namespace {

using namespace tc;

constexpr int kC = 64;       // tokens per chunk
constexpr int kKB = 128;     // d_k rows per cluster
constexpr int kDVMax = 512;  // d_v covered by the four CTAs of a cluster
constexpr int kNB = 128;     // d_v columns per CTA
constexpr int kRanks = 4;    // CTAs per cluster
constexpr int kOwn = 32;     // rows finished per CTA
constexpr int kThreads = 704;
constexpr int kWarpEx = 8, kWarpEpi = 12, kWarpLoad = 20, kWarpMma = 21;
constexpr uint32_t kColS = 0, kColHL = 128, kColAcc = 384;

// shared memory (bytes; tiles 1024-aligned)
constexpr int kTile = kC * 64 * 2;            // one [64 t][64] bf16 tile, 128-byte swizzle
// MMA stage: X = K~ (fwd) / Q~ (rev) [64 t][128 i]; U = v / do [64 t][128 j] (B of
// the state update); Z = do / v [64 t][128 j] (B of dq^T / dk^T); P = masked dA
// [64][64].  (The state warps read e^{b_last} of their rows straight from global
// memory a chunk ahead, so the state chain never waits on a stage.)
constexpr int kMsX = 0, kMsU = 2 * kTile, kMsZ = 4 * kTile, kMsP = 6 * kTile;
constexpr int kMsStage = 7 * kTile;
constexpr int kMsStages = 2;
// epilogue stage (this CTA's 32 rows, no swizzle), one per epilogue group:
// Y = Q~ (fwd) / K~ (rev) and G = log_alpha [64 t][32 i] bf16, QD = q.dq
// [64 t][32 i] fp32 (loaded by the reverse sweep).  The outputs are staged in
// place for their TMA stores: dq / dk over Y, q.dq (fwd) over QD, dlog_alpha
// (rev) over G -- each thread overwrites only the elements it has read.
constexpr int kEpY = 0, kEpG = kC * kOwn * 2, kEpQD = 2 * kC * kOwn * 2;
constexpr int kEpStage = kEpQD + kC * kOwn * 4;
constexpr int kEpStages = 2;
// one sender's partial for this CTA's 32 rows, token-quad major: element (row,
// t) at ((t / 4) * 32 + row) * 4 + t % 4, so that a warp's 16-byte store of four
// tokens of its 32 rows covers 512 contiguous bytes and the epilogue's 16-byte
// reads are conflict-free
constexpr int kSlot = kOwn * kC;  // floats
constexpr int kOffMs = 0;
constexpr int kOffEp = kOffMs + kMsStages * kMsStage;
constexpr int kOffRcv = kOffEp + kEpStages * kEpStage;   // [2 buffers][4 slots by sender]
constexpr int kOffGq = kOffRcv + 2 * kRanks * kSlot * 4;  // per group: log_alpha sums [4][32]
constexpr int kOffQS = kOffGq + 2 * 4 * kOwn * 4;        // per group: dg-term sums [4][32]
constexpr int kOffRun = kOffQS + 2 * 4 * kOwn * 4;       // reverse: dg carry into a chunk [2][32]
constexpr int kSmem = kOffRun + 2 * kOwn * 4;
static_assert(kMsStage % 1024 == 0 && kEpStage % 1024 == 0, "stage alignment");
static_assert(kSmem + 1024 <= 227 * 1024, "shared memory");

__device__ int g_qk_status = 0;

template <bool REV, int FORM>
__global__ void __launch_bounds__(kThreads, 1)
tc_bwd_qk_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmU,
                 const __grid_constant__ CUtensorMap tmZ, const __grid_constant__ CUtensorMap tmP,
                 const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmG,
                 const __grid_constant__ CUtensorMap tmQD, const __grid_constant__ CUtensorMap tmOut,
                 const __grid_constant__ CUtensorMap tmAux, const float* __restrict__ Eb,
                 const float* __restrict__ S_src, const float* __restrict__ carry,
                 float* __restrict__ dg_part, int64_t T, int64_t nrows, int dk, int dv, int P,
                 int64_t L) {
  constexpr bool kDiag = FORM == ZECO_DECAY_DIAG, kScalar = FORM == ZECO_DECAY_SCALAR;
  constexpr bool kDecay = FORM != ZECO_DECAY_NONE;
  // the low bf16 part of the state copy serves dlog_alpha's long suffix sums; the
  // no-decay form has none, and its dq / dk need only the high part
  constexpr int kParts = kDecay ? 2 : 1;
  // the second output of the sweep, stored by TMA: q.dq (forward, both decaying
  // forms), dlog_alpha (reverse, diagonal form)
  constexpr bool kAux = REV ? kDiag : kDecay;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = align1024(smraw);
  float* sRcv = reinterpret_cast<float*>(sm + kOffRcv);
  float* sGq = reinterpret_cast<float*>(sm + kOffGq);
  float* sQS = reinterpret_cast<float*>(sm + kOffQS);
  float* sRun = reinterpret_cast<float*>(sm + kOffRun);
  // ms_full / ms_empty: MMA-operand stages; ep_full: epilogue stages; u_done:
  // the state update of a chunk has completed; s_ready: the state warps have
  // rescaled the state and written the next hi/lo copy; q_done / acc_free: a
  // chunk's accumulator is complete / has been read; rcv_full[rb]: all four
  // partials of a chunk for this CTA's rows are in receive buffer rb;
  // consumed[rb]: this CTA's epilogue has read its receive buffer rb;
  // empty_from[q][rb]: CTA q has read its receive buffer rb (so this CTA's slot
  // there may be rewritten); carry_full[g]: (reverse) the other epilogue group
  // has left the dlog_alpha suffix of its chunk in sRun for group g; fin: every
  // MMA of this CTA has completed.
  __shared__ uint64_t ms_full[kMsStages], ms_empty[kMsStages], ep_full[kEpStages], u_done,
      s_ready, q_done[2], acc_free[2], rcv_full[2], consumed[2], empty_from[kRanks][2],
      carry_full[2], fin;
  __shared__ uint32_t tmem_base;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();   // which quarter of d_v; rows finished
  // block x = (b h p) * (kRanks d_k / kKB) + kRanks * d_k block + rank: a cluster is
  // kRanks consecutive blocks of one (b, h, segment, d_k block)
  // (a last partial block of d_k rows holds zeros past d_k: zero state rows and
  // operand columns, no stores)
  const int nx = kRanks * ((dk + kKB - 1) / kKB);
  const int64_t bhp = (int64_t)(blockIdx.x / nx);
  const int64_t bh = bhp / P;
  const int p = (int)(bhp % P);
  const int i0 = (int)((blockIdx.x % nx) / kRanks) * kKB;
  const int j0 = (int)rank * kNB;
  const int64_t row0 = bh * T + (int64_t)p * L;
  const int nc = (int)(L / kC);
  bool ok = true;  // false after a bounded wait gave up: no further waits or copies
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (ok && !mbar_wait(bar, parity)) {
      ok = false;
      atomicExch(&g_qk_status, 1);
    }
  };

  if (tid == 0) {
    for (int s = 0; s < kMsStages; ++s) {
      mbar_init(&ms_full[s], 1);
      mbar_init(&ms_empty[s], 1);  // the MMA commit
    }
    for (int s = 0; s < kEpStages; ++s) mbar_init(&ep_full[s], 1);
    mbar_init(&u_done, 1);
    mbar_init(&s_ready, 8);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&q_done[b], 1);
      mbar_init(&acc_free[b], 4);
    }
    for (int rb = 0; rb < 2; ++rb) {
      mbar_init(&rcv_full[rb], 32);  // the own-quarter warp's lanes (+ the peers' bytes)
      mbar_init(&consumed[rb], 1);
      for (int q = 0; q < kRanks; ++q) mbar_init(&empty_from[q][rb], 1);
      mbar_init(&carry_full[rb], 32);  // the first warp of the other group
    }
    mbar_init(&fin, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(&tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // all barriers of the cluster exist before any remote arrive or st.async
  const uint32_t tmem = tmem_base;
  auto chunk_row = [&](int n) { return (int32_t)(row0 + (int64_t)n * kC); };
  auto chunk_of = [&](int it) { return REV ? nc - 1 - it : it; };

  if (warp == kWarpLoad) {
    // ---- MMA operands of chunk `it`, two chunks ahead of the MMAs
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmU);
      prefetch_tmap(&tmZ);
      prefetch_tmap(&tmP);
      int issued = 0;
      for (int it = 0; it < nc; ++it) {
        const int s = it % kMsStages;
        if (it >= kMsStages) wait(&ms_empty[s], (uint32_t)((it / kMsStages - 1) & 1));
        if (!ok) break;
        unsigned char* stg = sm + kOffMs + s * kMsStage;
        const int32_t r = chunk_row(chunk_of(it));
        mbar_expect_tx(&ms_full[s], 7 * kTile);
        for (int b = 0; b < 2; ++b) {
          tma_load_2d(stg + kMsX + b * kTile, &tmX, i0 + 64 * b, r, &ms_full[s]);
          tma_load_2d(stg + kMsU + b * kTile, &tmU, j0 + 64 * b, r, &ms_full[s]);
          tma_load_2d(stg + kMsZ + b * kTile, &tmZ, j0 + 64 * b, r, &ms_full[s]);
        }
        tma_load_2d(stg + kMsP, &tmP, 0, r, &ms_full[s]);
        issued = it + 1;
      }
      // the last copy into each stage has landed (normally seen long ago)
      for (int it = issued > kMsStages ? issued - kMsStages : 0; it < issued; ++it)
        if (!mbar_wait(&ms_full[it % kMsStages], (uint32_t)((it / kMsStages) & 1)))
          atomicExch(&g_qk_status, 1);
    }
  } else if (warp == kWarpMma) {
    // ---- MMAs of chunk `it`: the state update, then the chunk's dq^T / dk^T
    if (lane == 0) {
      // S[i][j] += sum_t X[t][i] U[t][j]: M = 128 i, N = 128 j, K = 16 t per MMA
      constexpr uint32_t idU = idesc_bf16(kKB, kNB, true, true);
      // dA term: M = 128 i, N = 64 t, K = 16 positions s (forward: B = dA[t][s],
      // K-major; reverse: B = dA[s][t], MN-major)
      constexpr uint32_t idP = idesc_bf16(kKB, kC, true, REV);
      // state term: A = hi or lo copy [128 i][16 j] in tensor memory, B = Z[t][j]
      constexpr uint32_t idT = idesc_bf16(kKB, kC, false, false);
      for (int it = 0; it < nc; ++it) {
        const int s = it % kMsStages, b = it & 1;
        // the operands first (normally long landed), then the state warps' hand-off
        wait(&ms_full[s], (uint32_t)((it / kMsStages) & 1));
        wait(&s_ready, (uint32_t)(it & 1));  // state rescaled, hi/lo copy b written
        if (!ok) break;
        tc_fence_after();
        const uint32_t stg = smem_u32(sm + kOffMs + s * kMsStage);
        const uint32_t x0 = stg + kMsX, u0 = stg + kMsU, z0 = stg + kMsZ, p0 = stg + kMsP;
#pragma unroll
        for (int kk = 0; kk < kC / 16; ++kk)
          umma_bf16(tmem + kColS, sdesc_sw128(x0 + kk * 2048, kTile, 1024),
                    sdesc_sw128(u0 + kk * 2048, kTile, 1024), idU, 1u);
        umma_commit(&u_done);
        if (it >= 2) {
          wait(&acc_free[b], (uint32_t)(((it >> 1) - 1) & 1));  // chunk it-2 read out
          if (!ok) break;
          tc_fence_after();
        }
        const uint32_t acc = tmem + kColAcc + 64 * b;
        const uint64_t pd = REV ? sdesc_sw128(p0 + rank * 2048, kTile, 1024)
                                : sdesc_sw128(p0 + rank * 32, 16, 1024);
        umma_bf16(acc, sdesc_sw128(x0 + rank * 2048, kTile, 1024), pd, idP, 0u);
        const uint32_t hl = tmem + kColHL + 128 * b;
#pragma unroll
        for (int part = 0; part < kParts; ++part)
#pragma unroll
          for (int m = 0; m < kNB / 16; ++m)
            umma_bf16_ta(acc, hl + 64 * part + 8 * m,
                         sdesc_sw128(z0 + (m >> 2) * kTile + (m & 3) * 32, 16, 1024), idT, 1u);
        umma_commit(&q_done[b]);
        if (it + kMsStages < nc) umma_commit(&ms_empty[s]);
      }
      umma_commit(&fin);
      if (!mbar_wait(&fin, 0u)) atomicExch(&g_qk_status, 1);
    }
  } else if (warp < 8) {
    // ---- state warps: TMEM lane quarter lg (rows 32 lg ..), columns [64 h, 64 h + 64)
    const int lg = warp & 3, h = warp >> 2;
    const int row = 32 * lg + lane;
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const uint32_t sS = tmem + lane_off + kColS + 64 * h;
    {
      // (the columns past d_v and the rows past d_k start from zero: d_v and d_k
      // are multiples of 64)
      const bool live = j0 + 64 * h < dv && i0 + row < dk;
      const float* Sp =
          live ? S_src + (((size_t)bh * (P + 1) + p + (REV ? 1 : 0)) * dk + i0 + row) * dv +
                     j0 + 64 * h
               : S_src;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float r[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float4 x4 = live ? reinterpret_cast<const float4*>(Sp + 32 * c)[u]
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
          r[4 * u] = x4.x;
          r[4 * u + 1] = x4.y;
          r[4 * u + 2] = x4.z;
          r[4 * u + 3] = x4.w;
        }
        tmem_st32(sS + 32 * c, r);
      }
      tmem_st_wait();
    }
    // rescale this thread's 64 state entries by e (if `scale`) and write their
    // high and low bf16 parts into copy hb, a quarter of 16 columns at a time, the
    // next quarter's load in flight while this one is converted
    auto pass = [&](float e, bool scale, int hb) {
      const uint32_t hl = tmem + lane_off + kColHL + 128 * hb + 32 * h;
      float rq[2][16];
      tmem_ld16(sS, rq[0]);
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        float* r = rq[qd & 1];
        tmem_ld_wait16(r);
        if (qd + 1 < 4) tmem_ld16(sS + 16 * (qd + 1), rq[(qd + 1) & 1]);
        if (scale) {
#pragma unroll
          for (int u = 0; u < 16; ++u) r[u] *= e;
          tmem_st16(sS + 16 * qd, reinterpret_cast<const uint32_t*>(r));
        }
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float x0 = r[2 * u], x1 = r[2 * u + 1];
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
          const float2 hf = __bfloat1622float2(h2);
          const __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
          hi[u] = *reinterpret_cast<const uint32_t*>(&h2);
          lo[u] = *reinterpret_cast<const uint32_t*>(&l2);
        }
        tmem_st8(hl + 8 * qd, hi);
        if (kParts == 2) tmem_st8(hl + 64 + 8 * qd, lo);
      }
      tmem_st_wait();
    };
    // e^{b_last} of row `row` for the chunk processed at iteration ie (1 past the end)
    auto e_of = [&](int ie) -> float {
      if (ie >= nc || i0 + row >= dk) return 1.f;
      return __ldg(Eb + (size_t)(chunk_row(chunk_of(ie)) / kC) * dk + i0 + row);
    };
    auto ready = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_ready);
    };
    // the first chunk's copy (reverse: of the adjoint rescaled by that chunk's e^{b_last})
    pass(REV ? e_of(0) : 1.f, REV, 0);
    ready();
    // forward: S_{n+1} = e^{b_last,n} (S_n + K~^T v); reverse: the next chunk's
    // factor.  Each is loaded one iteration before it is used.
    float e = e_of(REV ? 1 : 0);
    for (int it = 0; it + 1 < nc; ++it) {
      const float e_next = e_of(REV ? it + 2 : it + 1);
      wait(&u_done, (uint32_t)(it & 1));
      __syncwarp();
      tc_fence_after();
      pass(e, true, (it + 1) & 1);
      ready();
      e = e_next;
    }
  } else if (warp < kWarpEpi) {
    // ---- exchange: lane quarter eq of the accumulator (rows 32 eq ..) to CTA eq,
    //      into its receive buffer of the chunk's parity, slot `rank`
    const int eq = warp - kWarpEx;
    const uint32_t lane_off = (uint32_t)(eq * 32) << 16;
#pragma unroll 1
    for (int it = 0; it < nc; ++it) {
      const int b = it & 1;
      wait(&q_done[b], (uint32_t)((it >> 1) & 1));
      __syncwarp();
      tc_fence_after();
      float a[64];
      tmem_ld32(tmem + lane_off + kColAcc + 64 * b, a);
      tmem_ld32(tmem + lane_off + kColAcc + 64 * b + 32, a + 32);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0 && it + 2 < nc) mbar_arrive(&acc_free[b]);
      // CTA eq (this CTA for the own quarter) has read chunk it-2 out of buffer b
      if (it >= 2)
        wait((uint32_t)eq == rank ? &consumed[b] : &empty_from[eq][b],
             (uint32_t)(((it >> 1) - 1) & 1));
      float* slot = sRcv + (b * kRanks + (int)rank) * kSlot;
      if ((uint32_t)eq == rank) {
        float4* d4 = reinterpret_cast<float4*>(slot);
#pragma unroll
        for (int c = 0; c < kC / 4; ++c)
          d4[c * 32 + lane] = make_float4(a[4 * c], a[4 * c + 1], a[4 * c + 2], a[4 * c + 3]);
      } else if (ok) {
        const uint32_t dst = map_to_rank(smem_u32(slot), (uint32_t)eq) + 16u * (uint32_t)lane;
        const uint32_t full = map_to_rank(smem_u32(&rcv_full[b]), (uint32_t)eq);
#pragma unroll
        for (int c = 0; c < kC / 4; ++c)
          st_async_v4(dst + 512u * (uint32_t)c, a[4 * c], a[4 * c + 1], a[4 * c + 2],
                      a[4 * c + 3], full);
      }
      if ((uint32_t)eq == rank) {
        if (lane == 0)
          mbar_expect_tx(&rcv_full[b], (kRanks - 1) * kOwn * kC * 4);
        else
          mbar_arrive(&rcv_full[b]);
      }
    }
  } else if (warp < kWarpLoad) {
    // ---- epilogue, two groups of four warps: group g takes the chunks of parity
    //      g (receive buffer g, factor stage g), so that each group has two chunk
    //      periods per chunk; warp eq of a group takes this CTA's 32 rows x tokens
    //      [16 eq, 16 eq + 16)
    const int g = (warp - kWarpEpi) >> 2, eq = (warp - kWarpEpi) & 3, er = lane;
    const int ec = kOwn * (int)rank + er;  // d_k row within the block finished here
    const bool leader = eq == 0 && lane == 0;
    const uint32_t bar_read = 1 + 2 * g, bar_sync = 2 + 2 * g;
    auto grp_bar = [](uint32_t id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); };
    float* gq = sGq + g * 4 * kOwn;
    float* qs = sQS + g * 4 * kOwn;
    unsigned char* ep = sm + kOffEp + g * kEpStage;
    __nv_bfloat16* epY = reinterpret_cast<__nv_bfloat16*>(ep + kEpY);
    __nv_bfloat16* epG = reinterpret_cast<__nv_bfloat16*>(ep + kEpG);
    float* epQD = reinterpret_cast<float*>(ep + kEpQD);
    // the epilogue factors of chunk `it` into this group's stage (leader)
    auto issue_ep = [&](int it) {
      const int32_t r = chunk_row(chunk_of(it));
      const int x = i0 + kOwn * (int)rank;
      constexpr uint32_t kGBytes = kDiag ? kC * kOwn * 2 : kScalar ? kC * 2 : 0;
      mbar_expect_tx(&ep_full[g], kC * kOwn * 2 + kGBytes + (REV && kDecay ? kC * kOwn * 4 : 0));
      tma_load_2d(ep + kEpY, &tmY, x, r, &ep_full[g]);
      // scalar form: the map views log_alpha as rows of one chunk's 64 tokens
      if (kDiag) tma_load_2d(ep + kEpG, &tmG, x, r, &ep_full[g]);
      if (kScalar) tma_load_2d(ep + kEpG, &tmG, 0, r / kC, &ep_full[g]);
      if (REV && kDecay) tma_load_2d(ep + kEpQD, &tmQD, x, r, &ep_full[g]);
    };
    int last = -1;  // leader: the last chunk whose factors were requested
    if (leader) {
      prefetch_tmap(&tmY);
      if (kDecay) prefetch_tmap(&tmG);
      if (REV && kDecay) prefetch_tmap(&tmQD);
      prefetch_tmap(&tmOut);
      if (kAux) prefetch_tmap(&tmAux);
      if (g < nc) {
        issue_ep(g);
        last = g;
      }
    }
    if (REV && kDecay && g == 0 && eq == 0)
      sRun[er] = i0 + ec < dk ? carry[((size_t)bh * P + p) * dk + i0 + ec] : 0.f;
#pragma unroll 1
    for (int it = g; it < nc; it += 2) {
      const int n = chunk_of(it);
      const uint32_t ph = (uint32_t)((it >> 1) & 1);
      // ---- the four partials of my rows, summed in rank order
      wait(&rcv_full[g], ph);
      float acc[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) acc[u] = 0.f;
#pragma unroll
      for (int q = 0; q < kRanks; ++q) {
        const float4* src = reinterpret_cast<const float4*>(sRcv + (g * kRanks + q) * kSlot);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float4 v4 = src[(4 * eq + c) * 32 + er];
          acc[4 * c] += v4.x;
          acc[4 * c + 1] += v4.y;
          acc[4 * c + 2] += v4.z;
          acc[4 * c + 3] += v4.w;
        }
      }
      // every thread of the group has read receive buffer g: hand it back to this
      // CTA's own-quarter sender and to the three other CTAs.  Relaxed arrives:
      // the reads were performed before the barrier, and a release arrive would
      // wait for memory operations in flight (thousands of cycles per chunk).
      grp_bar(bar_read);
      if (leader && it + 2 < nc && ok) {
        mbar_arrive_relaxed(&consumed[g]);
        const uint32_t mine = smem_u32(&empty_from[rank][g]);
        for (uint32_t q = 0; q < (uint32_t)kRanks; ++q)
          if (q != rank) mbar_arrive_remote_relaxed(map_to_rank(mine, q));
      }
      // ---- factors: e^{+-b_t} from log_alpha, the stored rounded Q~ (fwd) or
      //      K~ (rev), q.dq (rev)
      wait(&ep_full[g], ph);
      const int sb = 16 * eq * kOwn + er;  // stage element of (token 16 eq, row er)
      float gl[16], xa[16], term[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        gl[u] = kDiag     ? __bfloat162float(epG[sb + u * kOwn])
                : kScalar ? __bfloat162float(epG[16 * eq + u])
                          : 0.f;
        // the stored rounded Q~ (fwd) / K~ (rev) times the raw accumulator
        // (= q_eff dq / k_eff dk)
        xa[u] = __bfloat162float(epY[sb + u * kOwn]) * acc[u];
        if (REV && kDecay) term[u] = epQD[sb + u * kOwn] - xa[u];
      }
      float gs = 0.f, ssum = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        gs += gl[u];
        if (!REV && kDecay)
          epQD[sb + u * kOwn] = xa[u];  // q.dq, staged for its store
        else if (REV && kDecay)
          ssum += term[u];
      }
      gq[eq * 32 + er] = gs;
      if (REV && kDecay) qs[eq * 32 + er] = ssum;
      grp_bar(bar_sync);
      float bsum = 0.f;  // log-decay of the earlier 16-token quarters of the chunk
      for (int q2 = 0; q2 < eq; ++q2) bsum += gq[q2 * 32 + er];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        bsum += gl[u];
        const float x = kDecay ? acc[u] * __expf(REV ? -bsum : bsum) : acc[u];
        epY[sb + u * kOwn] = __float2bfloat16_rn(x);
      }
      if (REV && kDecay) {
        // this chunk's total, and the part of it after this warp's 16 tokens
        float tot = 0.f, after = 0.f;
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
          const float v = qs[q2 * 32 + er];
          tot += v;
          if (q2 > eq) after += v;
        }
        // the suffix of the chunks after this one (left by the other group in slot
        // g); once the whole group has read it, the carry into the next chunk goes
        // on at once -- the serial chain between the groups is one add per chunk
        if (it > 0) wait(&carry_full[g], (uint32_t)(((it - 1) >> 1) & 1));
        const float cin = sRun[g * kOwn + er];
        grp_bar(bar_read);
        if (eq == 0) {
          sRun[(g ^ 1) * kOwn + er] = cin + tot;
          if (it + 1 < nc) mbar_arrive(&carry_full[g ^ 1]);
        }
        float runq = cin + after;
        if (kDiag) {
#pragma unroll
          for (int u = 15; u >= 0; --u) {
            runq += term[u];
            epG[sb + u * kOwn] = __float2bfloat16_rn(runq);
          }
        } else {
          // scalar form: the sum over this CTA's 32 rows (the warp's lanes) of
          // each of the warp's 16 tokens.  A halving tree: at offset o a lane
          // keeps the upper or lower half of its values (by bit o of its lane)
          // and adds its partner's copy of that half, so that after offsets
          // 16, 8, 4, 2 lane l holds token l / 2, and offset 1 adds the pair.
          float v[16];
#pragma unroll
          for (int u = 15; u >= 0; --u) {
            runq += term[u];
            v[u] = runq;
          }
#pragma unroll
          for (int o = 16, n2 = 8; o >= 2; o >>= 1, n2 >>= 1) {
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int u = 0; u < n2; ++u) {
              const float send = up ? v[u] : v[u + n2];
              const float keep = up ? v[u + n2] : v[u];
              v[u] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
          }
          v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
          if ((lane & 1) == 0 && i0 + kOwn * (int)rank < dk) {
            const int c = (i0 + kOwn * (int)rank) / kOwn;
            dg_part[(size_t)c * nrows + chunk_row(n) + 16 * eq + (lane >> 1)] = v[0];
          }
        }
      }
      // the chunk's outputs leave by TMA from the stage
      fence_async_smem();
      grp_bar(bar_sync);
      if (leader) {
        const int32_t r = chunk_row(n), x = i0 + kOwn * (int)rank;
        if (x < dk) {  // (rows past d_k are not stored)
          tma_store_2d(&tmOut, ep + kEpY, x, r);
          if (kAux) tma_store_2d(&tmAux, ep + (REV ? kEpG : kEpQD), x, r);
        }
        bulk_commit();
        if (it + 2 < nc && ok) {
          bulk_wait_read_all();  // the stores have read the stage: refill it
          issue_ep(it + 2);
          last = it + 2;
        }
      }
    }
    if (leader) {
      bulk_wait_all();
      // the last factor copy has landed (normally seen already)
      if (last >= 0 && !mbar_wait(&ep_full[g], (uint32_t)((last >> 1) & 1)))
        atomicExch(&g_qk_status, 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no st.async or remote arrive is still in flight to any CTA of the cluster
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <bool REV, int FORM>
cudaError_t launch_qk(const Dims& d, const CUtensorMap& tx, const CUtensorMap& tu,
                      const CUtensorMap& tz, const CUtensorMap& tp, const CUtensorMap& ty,
                      const CUtensorMap& tg, const CUtensorMap& tqd, const CUtensorMap& tout,
                      const CUtensorMap& taux, const float* Eb, const float* S_src,
                      const float* carry, float* dg_part, cudaStream_t st) {
  auto kern = tc_bwd_qk_kernel<REV, FORM>;
  const int smem = kSmem + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(d.B * d.H * d.P * (kRanks * ((d.dk + kKB - 1) / kKB))), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRanks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_start(st);
  return cudaLaunchKernelEx(&cfg, kern, tx, tu, tz, tp, ty, tg, tqd, tout, taux, Eb, S_src,
                            carry, dg_part, d.T, d.B * d.H * d.T, (int)d.dk, (int)d.dv, d.P,
                            d.L);
}

// the tensor maps of the two sweeps (tc_bwd_qk)
enum { kMapQs, kMapKs, kMapV, kMapDo, kMapDA, kMapQp, kMapKp, kMapG, kMapQD, kMapDq, kMapDk,
       kMapDg, kMaps };

template <int FORM>
cudaError_t launch_sweeps(const Dims& d, const CUtensorMap* m, const float* Eb,
                          const float* S_in, const float* D, const float* carry, float* dg_part,
                          cudaStream_t st) {
  cudaError_t e = launch_qk<false, FORM>(d, m[kMapKs], m[kMapV], m[kMapDo], m[kMapDA], m[kMapQp],
                                         m[kMapG], m[kMapQD], m[kMapDq], m[kMapQD], Eb, S_in,
                                         carry, dg_part, st);
  prof_mark("tc_bwd_dq", st);
  if (e != cudaSuccess) return e;
  e = launch_qk<true, FORM>(d, m[kMapQs], m[kMapDo], m[kMapV], m[kMapDA], m[kMapKp], m[kMapG],
                            m[kMapQD], m[kMapDk], m[kMapDg], Eb, D, carry, dg_part, st);
  prof_mark("tc_bwd_dk", st);
  return e;
}

}  // namespace

bool tc_bwd_qk_supported(const Dims& d) {
  return d.bf16 && d.dk % 64 == 0 && d.dv % 64 == 0 && d.dv <= kDVMax && d.C == kC &&
         d.L % kC == 0;
}

cudaError_t tc_bwd_qk(const Dims& d, const void* Qt, const void* Kt, const void* v,
                      const void* g, const float* Eb, const void* dA, const float* S_in,
                      const void* d_o, void* dq, void* dk, void* dg, float* D, float* carry,
                      float* qdq, cudaStream_t st) {
  // swizzled [64 t][64] tiles for the MMAs; plain [64 t][32 i] tiles for the
  // epilogue.  The log-decay and its gradient by form: diagonal [rows][d_k] bf16
  // both; scalar g [rows] bf16 (read as [rows / 64][64]) and dg the fp32
  // partials [d_k / 32][rows]; none: neither is read or written (their maps
  // repeat another one's).
  CUtensorMap m[kMaps];
  const uint64_t rows = (uint64_t)(d.B * d.H * d.T);
  bool ok = make_tmap_bf16(&m[kMapQs], Qt, rows, d.dk, kC) &&
            make_tmap_bf16(&m[kMapKs], Kt, rows, d.dk, kC) &&
            make_tmap_bf16(&m[kMapV], v, rows, d.dv, kC) &&
            make_tmap_bf16(&m[kMapDo], d_o, rows, d.dv, kC) &&
            make_tmap_bf16(&m[kMapDA], dA, rows, kC, kC) &&
            make_tmap_bf16_plain(&m[kMapQp], Qt, rows, d.dk, kOwn, kC) &&
            make_tmap_bf16_plain(&m[kMapKp], Kt, rows, d.dk, kOwn, kC) &&
            make_tmap_f32_plain(&m[kMapQD], qdq, rows, d.dk, kOwn, kC) &&
            make_tmap_bf16_plain(&m[kMapDq], dq, rows, d.dk, kOwn, kC) &&
            make_tmap_bf16_plain(&m[kMapDk], dk, rows, d.dk, kOwn, kC);
  if (ok && d.decay == ZECO_DECAY_DIAG)
    ok = make_tmap_bf16_plain(&m[kMapG], g, rows, d.dk, kOwn, kC) &&
         make_tmap_bf16_plain(&m[kMapDg], dg, rows, d.dk, kOwn, kC);
  else if (ok && d.decay == ZECO_DECAY_SCALAR)
    ok = make_tmap_bf16_plain(&m[kMapG], g, rows / kC, kC, kC, 1);
  if (!ok) return cudaErrorInvalidValue;
  if (d.decay != ZECO_DECAY_DIAG) m[kMapDg] = m[kMapDk];
  if (d.decay == ZECO_DECAY_NONE) m[kMapG] = m[kMapQp];
  float* part = d.decay == ZECO_DECAY_SCALAR ? (float*)dg : nullptr;
  if (d.decay == ZECO_DECAY_SCALAR)
    return launch_sweeps<ZECO_DECAY_SCALAR>(d, m, Eb, S_in, D, carry, part, st);
  if (d.decay == ZECO_DECAY_NONE)
    return launch_sweeps<ZECO_DECAY_NONE>(d, m, Eb, S_in, D, carry, part, st);
  return launch_sweeps<ZECO_DECAY_DIAG>(d, m, Eb, S_in, D, carry, part, st);
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
