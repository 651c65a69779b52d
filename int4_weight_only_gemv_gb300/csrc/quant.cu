// quant.cu -- the load-time encoder (fp32 W -> packed INT4 + fp16 scales) and
// the debug dequantiser (packed -> fp16 W_hat).
//
// Format: INT4, symmetric, group-wise with group 128 along K, one FP16 scale
// per group ("Costruire un runtime di inference LLM da zero", datastack.it,
// "Tre bug che insegnano", last paragraph).  Per (row, group):
//   s = fp16_RN(fp32(max|w| / 7)),  q = clamp(round_half_away(w / s), -8, 7)
// packed eight nibbles per uint32, nibble i of word j = k 8j + i.
//
// The rounding decision is the one of the exact real quotient w / s, found
// without a division that could land on the wrong side of a half-integer:
// an fp32 quotient gives a candidate c, then c is corrected with exact fp32
// comparisons of |w| against (c +- 1/2) s (those products have at most 15
// significant bits, so they are exact).
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kQuantThreads = 256;

// round_half_away(a / s) for a >= 0, s > 0, exact.
__device__ __forceinline__ int round_quotient(float a, float s) {
  float c = floorf(__fdiv_rn(a, s) + 0.5f);
  if (a >= (c + 0.5f) * s) {
    c += 1.f;
  } else if (c > 0.f && a < (c - 0.5f) * s) {
    c -= 1.f;
  }
  return static_cast<int>(c);
}

// One thread per packed word (8 consecutive k of one row); the 16 threads of
// a group of 128 reduce max|w| with shuffles.
__global__ void __launch_bounds__(kQuantThreads) quantize_kernel(const float* __restrict__ w,
                                                                 uint32_t* __restrict__ qweight,
                                                                 uint16_t* __restrict__ scales,
                                                                 int64_t words, int K,
                                                                 uint32_t* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x;
  // words is a multiple of 16 (K % 128 == 0), so a group never straddles the
  // bound and whole 16-lane groups are either in or out
  const bool in = i < words;
  float v[8];
  if (in) {
    const float4 a = *reinterpret_cast<const float4*>(w + 8 * i);
    const float4 b = *reinterpret_cast<const float4*>(w + 8 * i + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
  }
  float amax = 0.f;
  bool finite = true;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    finite = finite && isfinite(v[j]);
    amax = fmaxf(amax, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    finite = __shfl_xor_sync(0xffffffffu, static_cast<int>(finite), o) && finite;
  }
  if (!in) return;
  const __half sh = __float2half_rn(__fdiv_rn(amax, 7.f));
  const float s = __half2float(sh);
  uint32_t word = 0;
  bool bad = false;
  if (!finite) {
    bad = true;
    if ((threadIdx.x & 15) == 0) atomicOr(status, W4A16_DEV_NONFINITE);
  } else if (__hisinf(sh)) {
    bad = true;
    if ((threadIdx.x & 15) == 0) atomicOr(status, W4A16_DEV_SCALE_OVERFLOW);
  } else if (s > 0.f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int q = round_quotient(fabsf(v[j]), s);
      if (v[j] < 0.f) q = -q;
      q = q > 7 ? 7 : (q < -8 ? -8 : q);
      word |= (static_cast<uint32_t>(q) & 0xFu) << (4 * j);
    }
  }
  qweight[i] = word;
  if ((threadIdx.x & 15) == 0) {
    const int64_t row = (8 * i) / K;
    const int64_t g = ((8 * i) % K) / 128;
    scales[row * (K / 128) + g] = bad ? 0 : __half_as_ushort(sh);
  }
}

// One thread per packed word: eight fp16 outputs, w_hat = fp16_RN(q * s); the
// product is exact in fp32, so this is the single rounding of the definition.
__global__ void __launch_bounds__(kQuantThreads) dequant_kernel(const uint32_t* __restrict__ qweight,
                                                                const uint16_t* __restrict__ scales,
                                                                uint16_t* __restrict__ w_out,
                                                                int64_t words, int K) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x;
  if (i >= words) return;
  const uint32_t word = qweight[i];
  const int64_t row = (8 * i) / K;
  const int64_t g = ((8 * i) % K) / 128;
  const float s = __half2float(__ushort_as_half(scales[row * (K / 128) + g]));
  uint32_t out[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int n0 = static_cast<int>((word >> (8 * j)) & 0xF);
    const int n1 = static_cast<int>((word >> (8 * j + 4)) & 0xF);
    const int q0 = n0 >= 8 ? n0 - 16 : n0;
    const int q1 = n1 >= 8 ? n1 - 16 : n1;
    const uint32_t h0 = __half_as_ushort(__float2half_rn(static_cast<float>(q0) * s));
    const uint32_t h1 = __half_as_ushort(__float2half_rn(static_cast<float>(q1) * s));
    out[j] = h0 | (h1 << 16);
  }
  *reinterpret_cast<uint4*>(w_out + 8 * i) = make_uint4(out[0], out[1], out[2], out[3]);
}

}  // namespace

cudaError_t launch_quantize(const float* w, uint32_t* qweight, uint16_t* scales, int N, int K,
                            uint32_t* status, cudaStream_t st) {
  const int64_t words = static_cast<int64_t>(N) * (K / 8);
  const int64_t blocks = (words + kQuantThreads - 1) / kQuantThreads;
  quantize_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, st>>>(w, qweight, scales, words,
                                                                           K, status);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* qweight, const uint16_t* scales, uint16_t* w_out,
                           int N, int K, cudaStream_t st) {
  const int64_t words = static_cast<int64_t>(N) * (K / 8);
  const int64_t blocks = (words + kQuantThreads - 1) / kQuantThreads;
  dequant_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, st>>>(qweight, scales, w_out,
                                                                          words, K);
  return cudaGetLastError();
}

}  // namespace w4a16

namespace w4a16 {
namespace {

// Self-test of the bounded wait used by the pipelined kernels: one thread
// waits on an mbarrier that nothing ever arrives on.  The wait gives up after
// limit_ns, records W4A16_DEV_PIPE_TIMEOUT and the kernel returns normally.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, uint32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  fence_barrier_init();
  if (!mbar_wait_bounded(b, 0, limit_ns)) atomicOr(status, W4A16_DEV_PIPE_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, uint32_t* status, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 1, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace w4a16

namespace w4a16 {
namespace {

// The SwiGLU step of a decoder layer's feed-forward (the page on hipfire,
// "Overview of hipfire-arch-qwen2", "Key Technical Specifications": SwiGLU
// FFN): h = fp16_RN(silu(g) u) with silu(g) = g / (1 + e^-g) in FP32 (fast
// exponential and division, as the M = 1 task lists' epilogue), one thread
// per element.  Runs between the [gate; up] and down GEMVs of a layer
// sequence outside the M = 1 task lists.
__global__ void swiglu_kernel(const uint16_t* __restrict__ g, const uint16_t* __restrict__ u, int64_t ld,
                              uint16_t* __restrict__ h, int M, int n) {
  pdl_launch_dependents();
  pdl_wait();  // g and u are the previous kernel's output
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(M) * n) return;
  const int64_t m = i / n, j = i % n;
  const float gv = __half2float(__ushort_as_half(g[m * ld + j]));
  const float uv = __half2float(__ushort_as_half(u[m * ld + j]));
  h[i] = __half_as_ushort(__float2half_rn(__fdividef(gv, 1.f + __expf(-gv)) * uv));
}

}  // namespace

cudaError_t launch_swiglu(const uint16_t* g, const uint16_t* u, int64_t ld, uint16_t* h, int M, int n,
                          bool pdl, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(M) * n;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((total + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, swiglu_kernel, g, u, ld, h, M, n);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace w4a16
