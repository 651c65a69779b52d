// gemv_rows.cu -- GEMV on the CUDA cores for one activation row (M = 1) when K
// is beyond the pipelined M = 1 kernel's range (gemv_m1.cu); the kernel is
// written for M rows and instantiated for M = 1.
//
// Same operation as gemv_m1.cu (INT4 group-128 weights x FP16 activations,
// FP32 accumulation; "Costruire un runtime di inference LLM da zero",
// "Tre bug che insegnano"): every packed weight is read from HBM once and
// multiplied by all M activation rows.
//
// Mapping: a CTA of 8 warps owns a block of R rows.  The 8 warps split K:
// warp w, lane l walks the 16-k units u = 32 w + l + 256 i (two packed words
// per row per unit, so each load instruction covers 256 contiguous bytes of a
// row), keeping kDepth units of loads in flight.  The unit's activations for
// all M rows come from global memory through L1 (a few tens of KB shared by
// every CTA).  Nibbles are unpacked to exact fp16 q (ptx.cuh), multiplied in
// f16 x f16 -> f32 FMAs and scaled per unit.  The R x M sums are reduced in a
// fixed order (warp butterflies, then the 8 warps through shared memory), so
// results are deterministic.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kRowsWarps = 8;
constexpr int kRowsThreads = kRowsWarps * 32;

// R rows per CTA, D units of loads in flight per lane (R x D x 8 bytes of
// loads in flight per lane, 32 registers of ring either way).  Large K gives
// each lane several units per row, so fewer rows and a deeper ring; small K
// (a few units per row, about one per lane) gives each lane more rows.
template <int M, bool kSmallK>
struct RowsCfg {
  static constexpr int R = kSmallK ? (M <= 3 ? 8 : 4) : (M <= 4 ? 4 : 2);
  static constexpr int D = kSmallK ? (M <= 1 ? 2 : (M <= 3 ? 1 : 2)) : (M <= 4 ? 4 : 8);
};

template <int M, bool kSmallK>
__global__ void __launch_bounds__(kRowsThreads, 2) gemv_rows_kernel(const GemvArgs a) {
  constexpr int R = RowsCfg<M, kSmallK>::R;
  constexpr int kDepth = RowsCfg<M, kSmallK>::D;
  __shared__ float red[kRowsWarps][R * M];
  pdl_launch_dependents();
  pdl_wait();  // x may be the previous kernel's output
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t N = a.N;
  const int K = a.K;
  const int units = K / 16;  // 16-k units per row
  const int wpr = K / 8;     // words per row
  const int gpr = K / 128;   // groups per row
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * R;

  // rows past N re-read row N-1 (in bounds) and are never stored
  const uint32_t* wrow[R];
  const uint16_t* srow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int64_t row = (r0 + r < N) ? r0 + r : N - 1;
    wrow[r] = a.qweight + row * wpr;
    srow[r] = a.scales + row * gpr;
  }
  float acc[R][M];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

  const int u0 = warp * 32 + lane;
  constexpr int kStride = kRowsThreads;  // units between consecutive iterations of a lane
  uint2 ring[kDepth][R];
#pragma unroll
  for (int d = 0; d < kDepth; ++d) {
    const int u = u0 + d * kStride;
    if (u < units) {
#pragma unroll
      for (int r = 0; r < R; ++r) ring[d][r] = ld_stream_u2(wrow[r] + 2 * u);
    }
  }
  for (int ub = u0; ub < units; ub += kDepth * kStride) {
#pragma unroll
    for (int d = 0; d < kDepth; ++d) {
      const int u = ub + d * kStride;
      if (u < units) {
        uint2 w[R];
#pragma unroll
        for (int r = 0; r < R; ++r) w[r] = ring[d][r];
        const int un = u + kDepth * kStride;
        if (un < units) {
#pragma unroll
          for (int r = 0; r < R; ++r) ring[d][r] = ld_stream_u2(wrow[r] + 2 * un);
        }
        const int g = u >> 3;  // 8 units per group
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) sc[r] = __half2float(__ushort_as_half(ld_nc_u16(srow[r] + g)));
        XPairs xp[M][2];
        // checked build: the unit's activations inside every row of x
        if (!W4A16_IN(a.status, 16 * u + 16 <= K && (M - 1) * a.ldx + K <= static_cast<int64_t>(M) * a.ldx)) continue;
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint16_t* xr = a.x + m * a.ldx + 16 * u;
          xp[m][0] = pair_activations(__ldg(reinterpret_cast<const uint4*>(xr)));
          xp[m][1] = pair_activations(__ldg(reinterpret_cast<const uint4*>(xr + 8)));
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const Unpacked q0 = unpack_exact(w[r].x);
          const Unpacked q1 = unpack_exact(w[r].y);
#pragma unroll
          for (int m = 0; m < M; ++m) {
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
            fma_f32_f16x2(s0, s1, q0.h0, xp[m][0].p0);
            fma_f32_f16x2(s2, s3, q0.h1, xp[m][0].p1);
            fma_f32_f16x2(s0, s1, q0.h2, xp[m][0].p2);
            fma_f32_f16x2(s2, s3, q0.h3, xp[m][0].p3);
            fma_f32_f16x2(s0, s1, q1.h0, xp[m][1].p0);
            fma_f32_f16x2(s2, s3, q1.h1, xp[m][1].p1);
            fma_f32_f16x2(s0, s1, q1.h2, xp[m][1].p2);
            fma_f32_f16x2(s2, s3, q1.h3, xp[m][1].p3);
            acc[r][m] = fmaf(sc[r], (s0 + s1) + (s2 + s3), acc[r][m]);
          }
        }
      }
    }
  }
  // warp butterflies, then the 8 warps in order through shared memory
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < M; ++m) {
      float v = acc[r][m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) red[warp][r * M + m] = v;
    }
  __syncthreads();
  if (threadIdx.x < R * M) {
    const int r = threadIdx.x / M;
    const int m = threadIdx.x % M;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kRowsWarps; ++w) v += red[w][threadIdx.x];
    if (r0 + r < N && W4A16_IN(a.status, m < a.M)) store_out(a, m, r0 + r, v);
  }
}

template <int M, bool kSmallK>
cudaError_t launch_rows_mk(const GemvArgs& a, cudaStream_t st) {
  constexpr int R = RowsCfg<M, kSmallK>::R;
  const int64_t grid = (static_cast<int64_t>(a.N) + R - 1) / R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kRowsThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_rows_kernel<M, kSmallK>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Small K: at most two 16-k units per lane of the 8 warps (K <= 8192).
template <int M>
cudaError_t launch_rows_m(const GemvArgs& a, cudaStream_t st) {
  return a.K <= 2 * 16 * kRowsThreads ? launch_rows_mk<M, true>(a, st) : launch_rows_mk<M, false>(a, st);
}

}  // namespace

cudaError_t launch_gemv_rows(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  (void)d;
  if (a.M != 1) return cudaErrorInvalidValue;
  return launch_rows_m<1>(a, st);
}

}  // namespace w4a16
