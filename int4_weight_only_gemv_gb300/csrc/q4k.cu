// q4k.cu -- GGUF Q4_K super-blocks: the reference dequantisation and the
// M = 1 GEMV straight from the stored blocks.
//
// The format is the one the page "VTE" dequantises byte for byte in llama.cpp's
// layout and the hipEngine page serves from GGUF Q4_K_M files: per 256
// weights of a row one 144-byte block holding d and dmin (fp16), eight 6-bit
// scales sc_j and minima m_j packed into 12 bytes, and 256 unsigned 4-bit
// codes q (in each 32-byte chunk c: low nibbles are sub-block 2c, high nibbles
// sub-block 2c + 1).  The weight is w = d sc_j q - dmin m_j.
//
// The blocks are read as stored: 144 bytes is a multiple of 16, so every
// block starts 16-byte aligned and no load-time repack is needed.
//
// q4k_gemv_kernel (M = 1): one warp per row, lane l taking the 64-weight units
// u = l, l + 32, ... (unit u = chunk u % 4 of block u / 4: 32 code bytes plus
// the block's 16-byte header), so a warp reads 8 consecutive blocks per step,
// two steps' loads in flight.  Each CTA first copies x into shared memory
// (padded per unit against bank conflicts); the grid is persistent (four
// CTAs per SM looping over groups of 8 rows), so x is copied once per CTA.
// Codes become fp16 1024 + q with one LOP3 per two (mask, OR 0x6400) and meet
// the activations in f16 x f16 -> f32 FMAs; per sub-block j the sum
// D_j = sum (1024 + q) x is turned into d sc_j (D_j - 1024 S_j) - dmin m_j S_j
// with S_j = sum_{k in j} x_k, which each CTA computes once into shared memory.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kQkBlock = 256;   // weights per block
constexpr int kQkBytes = 144;   // bytes per block
constexpr int kQkWarps = 8;     // rows per CTA
constexpr int kQkThreads = 32 * kQkWarps;

// Two halves a (low) and b (high) of a word pair.
__device__ __forceinline__ uint32_t pair_halves(uint32_t lo_word, uint32_t hi_word, uint32_t sel) {
  return __byte_perm(lo_word, hi_word, sel);
}

// Reference dequantisation: thread t handles code bytes 4 i .. 4 i + 3 of
// chunk c of one block (8 weights), w = (d sc) q - dmin m in three FP32
// roundings (no fused multiply-add).
__global__ void q4k_dequant_kernel(const uint8_t* __restrict__ blocks, float* __restrict__ w, int64_t nblocks) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= nblocks * 32) return;
  const int64_t blk = t / 32;
  const int c = static_cast<int>(t % 32) / 8;   // chunk 0..3
  const int i = static_cast<int>(t % 8) * 4;    // first code byte in the chunk
  const uint8_t* p = blocks + blk * kQkBytes;
  const uint4 h = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t sb[3] = {h.y, h.z, h.w};
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16)));
  int sc0, m0, sc1, m1;
  q4k_scale_min(sb, 2 * c, sc0, m0);
  q4k_scale_min(sb, 2 * c + 1, sc1, m1);
  const float d0 = __fmul_rn(d, static_cast<float>(sc0)), n0 = __fmul_rn(dmin, static_cast<float>(m0));
  const float d1 = __fmul_rn(d, static_cast<float>(sc1)), n1 = __fmul_rn(dmin, static_cast<float>(m1));
  const uint32_t q = __ldg(reinterpret_cast<const uint32_t*>(p + 16 + 32 * c + i));
  float lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    lo[k] = __fsub_rn(__fmul_rn(d0, static_cast<float>((q >> (8 * k)) & 15u)), n0);
    hi[k] = __fsub_rn(__fmul_rn(d1, static_cast<float>((q >> (8 * k + 4)) & 15u)), n1);
  }
  float* out = w + blk * kQkBlock + 64 * c + i;
  *reinterpret_cast<float4*>(out) = make_float4(lo[0], lo[1], lo[2], lo[3]);
  *reinterpret_cast<float4*>(out + 32) = make_float4(hi[0], hi[1], hi[2], hi[3]);
}

// Activations in shared memory: 64 per unit plus 4 halves of padding, so the
// lanes of a warp (one unit each, 136 bytes apart) read 8-byte pairs without
// bank conflicts.
constexpr int kQkXPitch = 68;  // halves per unit in shared memory

// One unit (64 weights: chunk c of a block) of one lane: the dot products of
// its two sub-blocks' biased codes with the activations, scaled and
// corrected.  h: the block's 16-byte header; q[8]: the chunk's code words;
// xs: shared address of the unit's activations; s0, s1: the sub-block sums.
__device__ __forceinline__ float q4k_unit(const uint4 h, const uint32_t (&q)[8], uint32_t xs, int c, float s0,
                                          float s1) {
  float dlo0 = 0.f, dlo1 = 0.f, dhi0 = 0.f, dhi1 = 0.f;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    uint32_t xl0, xl1, xh0, xh1;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(xl0), "=r"(xl1) : "r"(xs + 8 * t));
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(xh0), "=r"(xh1) : "r"(xs + 64 + 8 * t));
    const uint32_t v = q[t];
    // {1024 + q(k), 1024 + q(k + 2)} pairs against {x(k), x(k + 2)}
    // (the mask and the OR as one explicit LOP3: the two never share a bit)
    const uint32_t l02 = lop3_and_xor(v, 0x000F000Fu, 0x64006400u);
    const uint32_t l13 = lop3_and_xor(v >> 8, 0x000F000Fu, 0x64006400u);
    const uint32_t h02 = lop3_and_xor(v >> 4, 0x000F000Fu, 0x64006400u);
    const uint32_t h13 = lop3_and_xor(v >> 12, 0x000F000Fu, 0x64006400u);
    fma_f32_f16x2(dlo0, dlo1, l02, pair_halves(xl0, xl1, 0x5410u));
    fma_f32_f16x2(dlo0, dlo1, l13, pair_halves(xl0, xl1, 0x7632u));
    fma_f32_f16x2(dhi0, dhi1, h02, pair_halves(xh0, xh1, 0x5410u));
    fma_f32_f16x2(dhi0, dhi1, h13, pair_halves(xh0, xh1, 0x7632u));
  }
  const uint32_t sb[3] = {h.y, h.z, h.w};
  const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(h.x >> 16)));
  int sc0, m0, sc1, m1;
  q4k_scale_min(sb, 2 * c, sc0, m0);
  q4k_scale_min(sb, 2 * c + 1, sc1, m1);
  float r = d * static_cast<float>(sc0) * fmaf(-1024.f, s0, dlo0 + dlo1);
  r = fmaf(d * static_cast<float>(sc1), fmaf(-1024.f, s1, dhi0 + dhi1), r);
  return fmaf(-dmin, fmaf(static_cast<float>(m0), s0, static_cast<float>(m1) * s1), r);
}

__global__ void __launch_bounds__(kQkThreads) q4k_gemv_kernel(const uint8_t* __restrict__ blocks,
                                                             const uint16_t* __restrict__ x, uint16_t* y, int N,
                                                             int K) {
  // shared: S[K / 32] sub-block sums of x, then x itself (kQkXPitch per unit)
  extern __shared__ __align__(16) float S[];
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nblk = K / kQkBlock;
  const int U = 4 * nblk;  // units per row
  uint16_t* xsh = reinterpret_cast<uint16_t*>(S + K / 32);
  const uint32_t xs0 = smem_addr(xsh);
  pdl_wait();  // x may be the previous kernel's output
  // x into shared memory, 16 bytes per thread and step (8 per unit: pitch)
  for (int i = threadIdx.x; i < K / 8; i += kQkThreads) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
    const int u = i >> 3, part = i & 7;
    uint16_t* dst = xsh + u * kQkXPitch + 8 * part;
    reinterpret_cast<uint2*>(dst)[0] = make_uint2(v.x, v.y);
    reinterpret_cast<uint2*>(dst)[1] = make_uint2(v.z, v.w);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < K / 32; j += kQkThreads) {
    const uint16_t* xp = xsh + (j >> 1) * kQkXPitch + 32 * (j & 1);
    float s = 0.f;
#pragma unroll
    for (int v = 0; v < 16; ++v) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(xp + 2 * v);
      s += half_lo(w) + half_hi(w);
    }
    S[j] = s;
  }
  __syncthreads();
  // persistent: the CTA takes row groups g, g + gridDim.x, ... (8 rows each)
  const int64_t ngroups = (static_cast<int64_t>(N) + kQkWarps - 1) / kQkWarps;
  for (int64_t grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
  const int64_t row = grp * kQkWarps + warp;
  const uint8_t* rb = blocks + (row < N ? row : N - 1) * nblk * kQkBytes;
  float acc = 0.f;
  // two units per step, both units' loads issued before either is used
  for (int u0 = lane; u0 < U; u0 += 64) {
    const int u1 = u0 + 32;
    const bool has1 = u1 < U;
    const uint8_t* p0 = rb + (u0 >> 2) * kQkBytes;
    const uint8_t* p1 = rb + ((has1 ? u1 : u0) >> 2) * kQkBytes;
    const uint4 h0 = __ldg(reinterpret_cast<const uint4*>(p0));
    const uint4 a0 = __ldg(reinterpret_cast<const uint4*>(p0 + 16 + 32 * (u0 & 3)));
    const uint4 b0 = __ldg(reinterpret_cast<const uint4*>(p0 + 32 + 32 * (u0 & 3)));
    const uint4 h1 = __ldg(reinterpret_cast<const uint4*>(p1));
    const uint4 a1 = __ldg(reinterpret_cast<const uint4*>(p1 + 16 + 32 * ((has1 ? u1 : u0) & 3)));
    const uint4 b1 = __ldg(reinterpret_cast<const uint4*>(p1 + 32 + 32 * ((has1 ? u1 : u0) & 3)));
    {
      const uint32_t q[8] = {a0.x, a0.y, a0.z, a0.w, b0.x, b0.y, b0.z, b0.w};
      acc += q4k_unit(h0, q, xs0 + 2 * u0 * kQkXPitch, u0 & 3, S[2 * u0], S[2 * u0 + 1]);
    }
    if (has1) {
      const uint32_t q[8] = {a1.x, a1.y, a1.z, a1.w, b1.x, b1.y, b1.z, b1.w};
      acc += q4k_unit(h1, q, xs0 + 2 * u1 * kQkXPitch, u1 & 3, S[2 * u1], S[2 * u1 + 1]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0 && row < N) y[row] = __half_as_ushort(__float2half_rn(acc));
  }
}

}  // namespace

size_t q4k_gemv_smem(int K) {
  return static_cast<size_t>(K / 32) * sizeof(float) + static_cast<size_t>(K / 64) * kQkXPitch * 2;
}

cudaError_t prepare_q4k(const DeviceInfo& d) {
  (void)d;
  return cudaFuncSetAttribute(q4k_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(q4k_gemv_smem(W4A16_MAX_K)));
}

cudaError_t launch_q4k_dequant(const uint8_t* blocks, float* w, int N, int K, cudaStream_t st) {
  const int64_t nblocks = static_cast<int64_t>(N) * (K / kQkBlock);
  const int64_t threads = nblocks * 32;
  const int tpb = 256;
  q4k_dequant_kernel<<<static_cast<unsigned>((threads + tpb - 1) / tpb), tpb, 0, st>>>(blocks, w, nblocks);
  return cudaGetLastError();
}

cudaError_t launch_q4k_gemv(const uint8_t* blocks, const uint16_t* x, uint16_t* y, int N, int K, bool pdl,
                            const DeviceInfo& d, cudaStream_t st) {
  // four CTAs per SM (registers and shared memory allow it), each copying x
  // once and looping over row groups
  const int64_t groups = (static_cast<int64_t>(N) + kQkWarps - 1) / kQkWarps;
  const int64_t grid = groups < 4LL * d.sms ? groups : 4LL * d.sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kQkThreads);
  cfg.dynamicSmemBytes = q4k_gemv_smem(K);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, q4k_gemv_kernel, blocks, x, y, N, K);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace w4a16
