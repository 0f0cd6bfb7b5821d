// tc_decay.cu -- the decay-weighted operands of the chunked form, computed once
// per call and shared by every tensor-core sweep.
//
// Per chunk of C = 64 tokens and d_k column i, with b_t the inclusive
// cumulative log-decay from the chunk start (Gated Linear Attention, chunkwise
// form: Pith review of ZeCO, minor comment 4, the K/Lambda, K.Gamma pair):
//
//   Q~_t = bf16(q_t .* e^{b_t}),   K~_t = bf16(k_t .* e^{-b_t}),   E_c = e^{b_last} (fp32)
//
// The sweeps use these rounded operands for the state recurrence and the
// intra-chunk scores, so every kernel that builds or consumes a state works
// from the same bf16 values.  The pass is bound by HBM: each thread owns 8
// columns of one chunk and walks its 64 tokens with 16-byte loads and stores
// (a warp reads whole 512-byte rows when d_k = 256; d_k = 64, 128 or 256).
//
// The scalar-decay form reads its one log-decay per token ([B,H,T]; every
// thread of a chunk reads the same value), the no-decay form reads none: b = 0,
// Q~ = q, K~ = k, e^{b_last} = 1.
#include "common.cuh"
#include "launch.h"

namespace zeco {
namespace {

constexpr int kC = 64;

__device__ __forceinline__ void unpack8(const uint4& w, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __bfloat1622float2(h[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 w;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
  return w;
}

template <int DK, int FORM>
__global__ void __launch_bounds__(256)
decay_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
             const __nv_bfloat16* __restrict__ g, __nv_bfloat16* __restrict__ Qt,
             __nv_bfloat16* __restrict__ Kt, float* __restrict__ Eb, int64_t nchunks) {
  constexpr int kTPC = DK / 8;  // threads per chunk
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t chunk = gt / kTPC;
  const int cg = (int)(gt % kTPC);
  if (chunk >= nchunks) return;
  const size_t base = (size_t)chunk * kC * DK + (size_t)cg * 8;
  float b[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) b[e] = 0.f;
#pragma unroll 8
  for (int u = 0; u < kC; ++u) {
    const size_t o = base + (size_t)u * DK;
    const uint4 qw = __ldg(reinterpret_cast<const uint4*>(q + o));
    const uint4 kw = __ldg(reinterpret_cast<const uint4*>(k + o));
    float gf[8], qf[8], kf[8];
    if (FORM == ZECO_DECAY_DIAG) {
      unpack8(__ldg(reinterpret_cast<const uint4*>(g + o)), gf);
    } else {
      const float gs = FORM == ZECO_DECAY_SCALAR ? __bfloat162float(g[chunk * kC + u]) : 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) gf[e] = gs;
    }
    unpack8(qw, qf);
    unpack8(kw, kf);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      b[e] += gf[e];
      qf[e] *= __expf(b[e]);
      kf[e] *= __expf(-b[e]);
    }
    *reinterpret_cast<uint4*>(Qt + o) = pack8(qf);
    *reinterpret_cast<uint4*>(Kt + o) = pack8(kf);
  }
  float4* ep = reinterpret_cast<float4*>(Eb + (size_t)chunk * DK + (size_t)cg * 8);
  ep[0] = make_float4(__expf(b[0]), __expf(b[1]), __expf(b[2]), __expf(b[3]));
  ep[1] = make_float4(__expf(b[4]), __expf(b[5]), __expf(b[6]), __expf(b[7]));
}

}  // namespace

template <int DK>
static void launch_decay(const Dims& d, const __nv_bfloat16* q, const __nv_bfloat16* k,
                         const __nv_bfloat16* g, __nv_bfloat16* Qt, __nv_bfloat16* Kt, float* Eb,
                         int64_t nchunks, unsigned blocks, cudaStream_t st) {
  if (d.decay == ZECO_DECAY_SCALAR)
    decay_kernel<DK, ZECO_DECAY_SCALAR><<<blocks, 256, 0, st>>>(q, k, g, Qt, Kt, Eb, nchunks);
  else if (d.decay == ZECO_DECAY_NONE)
    decay_kernel<DK, ZECO_DECAY_NONE><<<blocks, 256, 0, st>>>(q, k, g, Qt, Kt, Eb, nchunks);
  else
    decay_kernel<DK, ZECO_DECAY_DIAG><<<blocks, 256, 0, st>>>(q, k, g, Qt, Kt, Eb, nchunks);
}

cudaError_t tc_decay(const Dims& d, const void* q, const void* k, const void* g, void* Qt,
                     void* Kt, float* Eb, cudaStream_t st) {
  const int64_t nchunks = d.B * d.H * d.T / kC;
  const int64_t threads = nchunks * (d.dk / 8);
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  auto qb = (const __nv_bfloat16*)q;
  auto kb = (const __nv_bfloat16*)k;
  auto gb = (const __nv_bfloat16*)g;
  auto Qb = (__nv_bfloat16*)Qt;
  auto Kb = (__nv_bfloat16*)Kt;
  if (d.dk != 64 && d.dk != 128 && d.dk != 256) return cudaErrorInvalidValue;
  prof_start(st);
  if (d.dk == 256)
    launch_decay<256>(d, qb, kb, gb, Qb, Kb, Eb, nchunks, blocks, st);
  else if (d.dk == 128)
    launch_decay<128>(d, qb, kb, gb, Qb, Kb, Eb, nchunks, blocks, st);
  else
    launch_decay<64>(d, qb, kb, gb, Qb, Kb, Eb, nchunks, blocks, st);
  prof_mark("tc_decay", st);
  return cudaGetLastError();
}

}  // namespace zeco
