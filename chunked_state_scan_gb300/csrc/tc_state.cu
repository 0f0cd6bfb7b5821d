// tc_state.cu -- segment-state contraction on tcgen05 tensor cores.
//
// Pass 1 of the forward (local state of every segment from a zero state;
// ZeCO two-pass operator, Pith review of ZeCO, referee major comment 3 on
// Algorithm 1, and the Appendix A.1 decomposition) and the backward's
// pre-pass (the adjoint state each segment sends backward, the dKV pass of
// Linear Attention Sequence Parallelism) are the same weighted contraction
// over the L tokens of a segment:
//
//   out[i, j] = sum_{t in segment} w_t[i] * x_t[i] * y_t[j]
//
//   forward  (REV): x = k, y = v,  w_t = exp(sum_{r > t} g_r)   (decay t -> segment end)
//   backward (FWD): x = q, y = do, w_t = exp(sum_{r <= t} g_r)  (decay segment start -> t)
//
// Both weights are <= 1, so no chunk-level rescaling of the accumulator is
// needed: the running log-decay is carried by the thread that owns row i,
// walking the segment backwards (REV) or forwards (FWD).  The forward also
// writes gamma_p[i] = exp(sum_{t in segment} g_t[i]).
//
// Tiling: one CTA = 128 d_k rows (M) x NT d_v columns (N, 256 or 128) of one
// (b, h, segment); K = 64 tokens per stage, 3 stages (4 with the decay pass's
// operands, one CTA per SM).  A last tile of d_k = 64 or 192 rows, or of d_v not
// a multiple of NT, is partial.  A = (w .* x)^T is
// written by the threads straight into the 128B-swizzled MN-major operand
// layout (row i contiguous over tokens' rows); B = y arrives by TMA in the
// same layout.  The accumulator lives in TMEM (NT fp32 columns); one thread
// issues the MMAs.
#include <cuda.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

namespace zeco {
namespace {

using namespace tc;

constexpr int kStages = 3;
// PRE: stages of the copy ring of one CTA per SM (each ~49 KB at 256 d_v columns)
constexpr int kStagesPre = 4;
constexpr int kTok = 64;                // tokens per stage (MMA K)
constexpr int kM = 128;                 // d_k rows per CTA
constexpr int kXBytes = kTok * kM * 2;  // 16 KB: x tile, overwritten in place by A = (w .* x)
constexpr int kGBytes = kTok * kM * 2;  // 16 KB: log_alpha tile

__device__ int g_tc_status = 0;  // set when a bounded wait gives up

constexpr int kStateThreads = 512;  // compute threads: 128 rows x 4 token quarters
// plus one producer warp that issues the copies (waiting for a stage's previous
// MMAs without holding up the compute threads)
constexpr int kStateBlock = kStateThreads + 32;

// PRE: x is the decay pass's K~ = k e^{-b} (REV) or Q~ = q e^{b} (forward), and
// the weight of a token of chunk n factors into one value per row and chunk:
//   REV:  e^{G_end - G_t} = e^{-b_t} * prod_{m >= n} e^{b_last,m}
//   fwd:  e^{G_t}         = e^{b_t}  * prod_{m <  n} e^{b_last,m}
// (G: cumulative log-decay from the segment start, b: from the chunk start), so a
// stage loads the chunk's e^{b_last} row instead of the log_alpha tile and scales
// the tile by a running product, with no exponential per element.
template <int NT, bool REV, bool PRE>
__global__ void __launch_bounds__(kStateBlock, 1)
tc_seg_state_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmY, const float* __restrict__ Eb,
                    float* __restrict__ out, float* __restrict__ gamma, int64_t T, int dk, int dv,
                    int P, int64_t L, int slot_off) {
  constexpr int kBBytes = kTok * NT * 2;
  // PRE: the log_alpha slot holds only the e^{b_last} row; one CTA per SM with four
  // stages of ~49 KB (two CTAs of two stages each keep as many copies in flight, but
  // their 1,024 CTAs at the 1M-token shape make 3.4 waves of 304 instead of 6.7 of
  // 152: 1.24 -> 1.17 ms for pass 1)
  constexpr int SG = PRE ? kStagesPre : kStages;
  constexpr int GB = PRE ? 1024 : kGBytes;
  constexpr int kStageBytes = kXBytes + GB + kBBytes;
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* sm = align1024(smraw);
  __shared__ uint64_t tma_bar[SG], mma_bar[SG], fin_bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;  // set when a bounded wait of this CTA gives up
  // After a wait of this CTA has given up, the abort word makes every later wait
  // of the CTA give up within 64 polls and the producer issues no further copies:
  // the stage loop runs to its end without waiting and the CTA drains what it has
  // in flight before exit.
  const Waits wait{smem_u32(&abort_flag), &g_tc_status};
  auto wt = [&](uint64_t* bar, uint32_t parity) { return wait(bar, parity); };
  __shared__ float Gq[4][kM];  // per-quarter sums of log_alpha of the current stage

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & (kM - 1), qd = tid >> 7;  // row within the tile, token quarter
  // block x = ((b h p) * (d_k / kM) + d_k tile) * (d_v / NT) + d_v tile: the CTAs of
  // one segment are launched together and share its operand tiles in L2
  // (a last partial tile of d_k rows or d_v columns reads zeros past the end of
  // its operands and stores only the rows and columns that exist)
  const int nx = (dv + NT - 1) / NT, ny = (dk + kM - 1) / kM;
  const int bx = (int)(blockIdx.x % nx), by = (int)((blockIdx.x / nx) % ny);
  const int64_t bhp = (int64_t)(blockIdx.x / nx) / ny;
  const int64_t bh = bhp / P;
  const int p = (int)(bhp % P);
  const int i0 = by * kM, j0 = bx * NT;
  const int i = i0 + row;
  const int nE = dk - i0 < kM ? dk - i0 : kM;  // rows of this tile that exist
  const int64_t row0 = bh * T + (int64_t)p * L;  // first token row of the segment
  const int nblk = (int)(L / kTok);

  if (tid == 0) {
    for (int s = 0; s < SG; ++s) {
      mbar_init(&tma_bar[s], 1);
      mbar_init(&mma_bar[s], 1);
    }
    mbar_init(&fin_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmX);
    if (!PRE) prefetch_tmap(&tmG);
    prefetch_tmap(&tmY);
  }
  if (warp == 0) tmem_alloc(&tmem_base, NT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  auto blk_row = [&](int it) -> int32_t {  // first token row of the it-th stage
    const int b = REV ? (nblk - 1 - it) : it;
    return (int32_t)(row0 + (int64_t)b * kTok);
  };
  auto issue_tma = [&](int it) {
    const int s = it % SG;
    unsigned char* base = sm + s * kStageBytes;
    const int32_t r = blk_row(it);
    mbar_expect_tx(&tma_bar[s], PRE ? kXBytes + nE * 4 + kBBytes : kStageBytes);
    for (int mb = 0; mb < kM / 64; ++mb) {
      tma_load_2d(base + mb * 8192, &tmX, i0 + mb * 64, r, &tma_bar[s]);
      if (!PRE) tma_load_2d(base + kXBytes + mb * 8192, &tmG, i0 + mb * 64, r, &tma_bar[s]);
    }
    if (PRE) bulk_load(base + kXBytes, Eb + (size_t)(r / kTok) * dk + i0, nE * 4, &tma_bar[s]);
    for (int nb = 0; nb < NT / 64; ++nb)
      tma_load_2d(base + kXBytes + GB + nb * 8192, &tmY, j0 + nb * 64, r, &tma_bar[s]);
  };

  // the compute threads' barrier (the producer warp does not take part)
  auto cbar = []() { asm volatile("bar.sync 1, %0;" ::"n"(kStateThreads) : "memory"); };
  if (warp == kStateThreads / 32) {
    // ---- producer: stage it once the MMAs that last read its buffers are done
    int issued = 0;
    if (lane == 0) {
      for (int it = 0; it < nblk; ++it) {
        const int jn = it - SG;
        if (jn >= 0 && !wt(&mma_bar[it % SG], (jn / SG) & 1)) break;
        if (wait.aborted()) break;  // another thread's wait gave up: no further copies
        issue_tma(it);
        issued = it + 1;
      }
    }
    tc_fence_before();
    __syncthreads();
    // after the CTA's last barrier every thread has finished: if any wait gave
    // up, copies still in flight land before the CTA exits (bounded waits)
    if (lane == 0 && wait.aborted())
      for (int s = 0; s < SG; ++s)
        drain_phase(&tma_bar[s], (uint32_t)(issued > s ? (issued - s + SG - 1) / SG : 0));
    return;
  }
  float run = 0.f;  // log-decay of row i summed over the stages already done
  // PRE: this thread's 8 rows (p_r8 ..) of the tile and the products of e^{b_last}
  // over the chunks already done for each
  const int p_r8 = 64 * ((tid >> 3) & 1) + 8 * (tid & 7);
  float run8[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) run8[u] = 1.f;
  // row i of the tiles lives in MN block row/64, 16-byte chunk (row%64)/8, element row%8
  const uint32_t a_blk = (uint32_t)(row >> 6) * 8192u;
  const uint32_t a_chunk = (uint32_t)((row & 63) >> 3);
  const uint32_t a_sub = (uint32_t)(row & 7) * 2u;

  for (int it = 0; it < nblk; ++it) {
    const int s = it % SG;
    unsigned char* xbuf = sm + s * kStageBytes;
    wt(&tma_bar[s], (it / SG) & 1);
    if (PRE) {
      // every 16-byte group of 8 rows of the tile scaled in place (2 per thread, the
      // same 8 rows in every stage): this stage's factor of each of those rows from
      // the running products this thread carries (rows past d_k are zeros and stay
      // so; their factors were not loaded)
      if (p_r8 < nE) {
        const float4* e4 = reinterpret_cast<const float4*>(xbuf + kXBytes + 4 * p_r8);
        const float4 ea = e4[0], eb = e4[1];
        const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
        float f[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (REV) run8[u] *= ev[u];
          f[u] = run8[u];
          if (!REV) run8[u] *= ev[u];
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = tid + h * kStateThreads;  // 64 tokens x 2 row blocks x 8 groups
          const int t = c >> 4, mb = (c >> 3) & 1, c8 = c & 7;
          uint4* ptr = reinterpret_cast<uint4*>(xbuf + mb * 8192 + sw128((uint32_t)t, (uint32_t)c8));
          uint4 wv = *ptr;
          __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&wv);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 x2 = __bfloat1622float2(h2[u]);
            h2[u] = __floats2bfloat162_rn(x2.x * f[2 * u], x2.y * f[2 * u + 1]);
          }
          *ptr = wv;
        }
      }
    } else
    // A = (w .* x) written over x; this thread: row i, tokens 16 qd .. 16 qd + 15
    {
      float gl[16];
      float gsum = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t off = a_blk + sw128((uint32_t)(16 * qd + u), a_chunk) + a_sub;
        gl[u] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(xbuf + kXBytes + off));
        gsum += gl[u];
      }
      Gq[qd][row] = gsum;
      cbar();
      float off_q = run;  // log-decay from the processed stages plus the other quarters
      float stage = 0.f;
#pragma unroll
      for (int q2 = 0; q2 < 4; ++q2) {
        const float gq = Gq[q2][row];
        stage += gq;
        if (REV ? (q2 > qd) : (q2 < qd)) off_q += gq;
      }
      if (REV) {
        // w_t = exp(sum of g over the later tokens of the segment)
        float loc = off_q;
#pragma unroll
        for (int u = 15; u >= 0; --u) {
          const uint32_t off = a_blk + sw128((uint32_t)(16 * qd + u), a_chunk) + a_sub;
          __nv_bfloat16* xe = reinterpret_cast<__nv_bfloat16*>(xbuf + off);
          *xe = __float2bfloat16_rn(__bfloat162float(*xe) * __expf(loc));
          loc += gl[u];
        }
      } else {
        // w_t = exp(sum of g from the segment start through t)
        float loc = off_q;
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          loc += gl[u];
          const uint32_t off = a_blk + sw128((uint32_t)(16 * qd + u), a_chunk) + a_sub;
          __nv_bfloat16* xe = reinterpret_cast<__nv_bfloat16*>(xbuf + off);
          *xe = __float2bfloat16_rn(__bfloat162float(*xe) * __expf(loc));
        }
      }
      run += stage;
    }
    fence_async_smem();
    cbar();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t a0 = smem_u32(xbuf), b0 = a0 + kXBytes + GB;
      constexpr uint32_t id = idesc_bf16(kM, NT, true, true);
#pragma unroll
      for (int kk = 0; kk < kTok / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(a0 + kk * 2048, 8192, 1024);
        const uint64_t bd = sdesc_sw128(b0 + kk * 2048, 8192, 1024);
        umma_bf16(tmem, ad, bd, id, (it > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit(&mma_bar[s]);
    }
  }
  cbar();
  const bool ok = !wait.aborted();
  // PRE: gamma_p of every row is the product over all the segment's chunks
  if (PRE && REV && ok && gamma && bx == 0 && tid < 16 && p_r8 < nE)
#pragma unroll
    for (int u = 0; u < 8; ++u) gamma[((size_t)bh * P + p) * dk + i0 + p_r8 + u] = run8[u];
  if (ok && warp < 4 && warp * 32 < nE) {
    const int last = nblk - 1;
    wt(&mma_bar[last % SG], (last / SG) & 1);
    tc_fence_after();
    float* orow = out + (((size_t)bh * (P + 1) + p + slot_off) * dk + i) * dv + j0;
#pragma unroll 1
    for (int c = 0; c < NT && j0 + c < dv; c += 32) {
      float r[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c, r);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(orow + c);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        dst[u] = make_float4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
    }
    if (!PRE && REV && gamma && bx == 0) gamma[((size_t)bh * P + p) * dk + i] = __expf(run);
    (void)lane;
  }
  if (tid == 0 && wait.aborted()) {
    // a wait gave up: no MMA may still write tensor memory when it is freed
    // (bounded wait)
    umma_commit(&fin_bar);
    (void)mbar_wait(&fin_bar, 0u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, NT);
}

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry
// point query, so the library does not link the driver library itself (it
// loads on machines without a GPU driver; the lookup fails there, and so do
// the launches, with an error code).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

// 2D bf16 tensor map over a [rows, cols] row-major matrix with a box of
// 64 columns x box_rows rows and 128-byte swizzle.
bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstr[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  EncodeTiledFn enc = encode_tiled();
  return enc && enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 tensor map, box_cols x box_rows, no swizzle (rows of box_cols * 4 bytes).
bool make_tmap_f32_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                         uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstr[1] = {(cuuint64_t)cols * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  EncodeTiledFn enc = encode_tiled();
  return enc && enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
                                gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D bf16 tensor map, box_cols x box_rows, no swizzle (rows of box_cols * 2 bytes).
bool make_tmap_bf16_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                          uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t gdim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t gstr[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  EncodeTiledFn enc = encode_tiled();
  return enc && enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
                                gdim, gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NT, bool REV, bool PRE>
static cudaError_t launch_state(const Dims& d, const void* x, const void* y, const void* g,
                                const float* Eb, float* out, float* gamma, int slot_off,
                                cudaStream_t st) {
  CUtensorMap tx, tg, ty;
  const uint64_t rows = (uint64_t)(d.B * d.H * d.T);
  if (!make_tmap_bf16(&tx, x, rows, (uint64_t)d.dk, kTok) ||
      !make_tmap_bf16(&tg, PRE ? x : g, rows, (uint64_t)d.dk, kTok) ||
      !make_tmap_bf16(&ty, y, rows, (uint64_t)d.dv, kTok))
    return cudaErrorInvalidValue;
  const int smem = (PRE ? kStagesPre : kStages) * (kXBytes + (PRE ? 1024 : kGBytes) + kTok * NT * 2) + 1024;
  auto kern = tc_seg_state_kernel<NT, REV, PRE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid =
      (unsigned)(d.B * d.H * d.P * ((d.dk + kM - 1) / kM) * ((d.dv + NT - 1) / NT));
  prof_start(st);
  kern<<<grid, kStateBlock, smem, st>>>(tx, tg, ty, Eb, out, gamma, d.T, (int)d.dk,
                                          (int)d.dv, d.P, d.L, slot_off);
  return cudaGetLastError();
}

template <bool REV>
static cudaError_t launch_state_any(const Dims& d, const void* x, const void* y, const void* g,
                                    const float* Eb, float* out, float* gamma, int slot_off,
                                    cudaStream_t st) {
  if (Eb)
    return d.dv % 256 == 0 ? launch_state<256, REV, true>(d, x, y, g, Eb, out, gamma, slot_off, st)
                           : launch_state<128, REV, true>(d, x, y, g, Eb, out, gamma, slot_off, st);
  return d.dv % 256 == 0 ? launch_state<256, REV, false>(d, x, y, g, Eb, out, gamma, slot_off, st)
                         : launch_state<128, REV, false>(d, x, y, g, Eb, out, gamma, slot_off, st);
}

bool tc_state_supported(const Dims& d) {
  return d.bf16 && d.dk % 64 == 0 && d.dv % 64 == 0 && d.L % kTok == 0;
}

cudaError_t tc_chunk_state(const Dims& d, const void* k, const void* v, const void* g,
                           const void* Kt, const float* Eb, float* S_in, float* gamma,
                           cudaStream_t st) {
  cudaError_t e = Eb ? launch_state_any<true>(d, Kt, v, g, Eb, S_in, gamma, 1, st)
                     : launch_state_any<true>(d, k, v, g, nullptr, S_in, gamma, 1, st);
  prof_mark("tc_chunk_state", st);
  return e;
}

cudaError_t tc_dstate_local(const Dims& d, const void* q, const void* d_o, const void* g,
                            const void* Qt, const float* Eb, float* D, cudaStream_t st) {
  cudaError_t e = Eb ? launch_state_any<false>(d, Qt, d_o, g, Eb, D, nullptr, 0, st)
                     : launch_state_any<false>(d, q, d_o, g, nullptr, D, nullptr, 0, st);
  prof_mark("tc_dstate_local", st);
  return e;
}

// Reads and clears this file's bounded-wait flag (nonzero: a wait gave up).
int tc_state_take_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(v)) != cudaSuccess) return -1;
  if (v != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(zero));
  }
  return v;
}

}  // namespace zeco
