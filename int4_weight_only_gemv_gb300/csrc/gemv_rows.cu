// gemv_rows.cu -- small-batch GEMV on the CUDA cores, M = 1..7 activation rows.
//
// Same operation as gemv_m1.cu (INT4 group-128 weights x FP16 activations,
// FP32 accumulation; "Costruire un runtime di inference LLM da zero",
// "Tre bug che insegnano"), for small-batch decode: every packed weight is
// read from HBM once and multiplied by all M activation rows.
//
// Mapping: each warp owns a block of R rows; lane l walks 16-k units
// u = l, l + 32, ... of those rows (two packed words per row per unit, loaded
// with coalesced 8-byte streaming loads, the next unit's loads issued before
// the current one is computed).  The unit's activations for all M rows come
// from global memory through L1 (x is a few tens of KB and shared by every
// warp).  Nibbles are unpacked to exact fp16 q (ptx.cuh), multiplied in
// f16 x f16 -> f32 FMAs and scaled per unit.  The R x M sums are reduced over
// the warp with shuffles in a fixed order, so results are deterministic.
// This kernel also serves M = 1 when K is beyond the pipelined kernel's range.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kRowsThreads = 256;

template <int M>
struct RowsCfg {
  static constexpr int R = M <= 2 ? 4 : 2;  // rows per warp block
};

template <int M>
__global__ void __launch_bounds__(kRowsThreads) gemv_rows_kernel(const GemvArgs a) {
  constexpr int R = RowsCfg<M>::R;
  pdl_launch_dependents();
  pdl_wait();  // x may be the previous kernel's output
  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * kRowsThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kRowsThreads) >> 5;
  const int64_t N = a.N;
  const int K = a.K;
  const int units = K / 16;       // 16-k units per row
  const int wpr = K / 8;          // words per row
  const int gpr = K / 128;        // groups per row
  const int64_t nblocks = (N + R - 1) / R;

  for (int64_t blk = warp_global; blk < nblocks; blk += nwarps) {
    const int64_t r0 = blk * R;
    float acc[R][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    // rows past N re-read row N-1 (in bounds) and are never stored
    int64_t rows[R];
#pragma unroll
    for (int r = 0; r < R; ++r) rows[r] = (r0 + r < N) ? r0 + r : N - 1;

    uint2 wcur[R];
    int u = lane;
    if (u < units) {
#pragma unroll
      for (int r = 0; r < R; ++r) wcur[r] = ld_stream_u2(a.qweight + rows[r] * wpr + 2 * u);
    }
    for (; u < units; u += 32) {
      uint2 wnext[R];
      const int un = u + 32;
      if (un < units) {
#pragma unroll
        for (int r = 0; r < R; ++r) wnext[r] = ld_stream_u2(a.qweight + rows[r] * wpr + 2 * un);
      }
      const int g = u >> 3;  // 8 units per group
      float sc[R];
#pragma unroll
      for (int r = 0; r < R; ++r)
        sc[r] = __half2float(__ushort_as_half(ld_nc_u16(a.scales + rows[r] * gpr + g)));

      // activations of this unit for every m, paired to match the unpack
      XPairs xp[M][2];
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint16_t* xr = a.x + m * a.ldx + 16 * u;
        xp[m][0] = pair_activations(__ldg(reinterpret_cast<const uint4*>(xr)));
        xp[m][1] = pair_activations(__ldg(reinterpret_cast<const uint4*>(xr + 8)));
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const Unpacked q0 = unpack_exact(wcur[r].x);
        const Unpacked q1 = unpack_exact(wcur[r].y);
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
      if (un < units) {
#pragma unroll
        for (int r = 0; r < R; ++r) wcur[r] = wnext[r];
      }
    }
    // warp reduction, fixed butterfly order
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = acc[r][m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        acc[r][m] = v;
      }
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r0 + r < N)
#pragma unroll
          for (int m = 0; m < M; ++m)
            *out_ptr(a, m, r0 + r) = __half_as_ushort(__float2half_rn(acc[r][m]));
    }
  }
}

template <int M>
cudaError_t launch_rows_m(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  constexpr int R = RowsCfg<M>::R;
  const int64_t nblocks = (static_cast<int64_t>(a.N) + R - 1) / R;
  const int64_t warps_per_cta = kRowsThreads / 32;
  int64_t grid = (nblocks + warps_per_cta - 1) / warps_per_cta;
  const int64_t cap = static_cast<int64_t>(d.sms) * 8;
  if (grid > cap) grid = cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kRowsThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_rows_kernel<M>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_rows(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  switch (a.M) {
    case 1: return launch_rows_m<1>(a, d, st);
    case 2: return launch_rows_m<2>(a, d, st);
    case 3: return launch_rows_m<3>(a, d, st);
    case 4: return launch_rows_m<4>(a, d, st);
    case 5: return launch_rows_m<5>(a, d, st);
    case 6: return launch_rows_m<6>(a, d, st);
    case 7: return launch_rows_m<7>(a, d, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace w4a16
