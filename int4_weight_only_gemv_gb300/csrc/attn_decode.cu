// attn_decode.cu -- decode attention over an fp16 KV cache (one query token,
// grouped-query heads, head dimension 128).
//
// The operation is the decode attention of the page "LLM170" (README of the
// LLM170 engine): its HIP decode kernel reads an f16 copy of the KV cache and,
// at long context, is bound by the bandwidth of reading it.  For query head h
// and its KV head g = h / (n_heads / n_kv_heads):
//   o_h = sum_t softmax_t(q_h . k_{g,t} / sqrt(128)) v_{g,t},   t < T.
// The page's kernel gives each lane one key and computes the whole dot
// product in that lane; with 7 query heads per KV head (the model shape of
// "Costruire un runtime di inference LLM da zero", "Tre bug che insegnano")
// that is about 3.5 FP32 multiply-adds per byte of cache, too many for the
// CUDA cores at HBM speed.  Here the query heads of a KV head are the rows of
// an m16n8k16 MMA (f16 x f16 -> f32), so every K/V byte read feeds all of
// them from the tensor cores.
//
// One launch (flash-decoding split over keys):
//   attn_partial_kernel   one CTA per (KV head, key range).  Warp 4 streams
//       tiles of 64 keys through an S-stage ring: per tile four 3-D TMA loads
//       (K and V, dimensions 0..63 and 64..127; 128-byte swizzle; keys at or
//       past T read as zero, so they never reach P.V as garbage).  Two groups
//       of four warps take alternate tiles, each warp 16 keys of a tile: S = Q K^T (ldmatrix from the swizzled
//       tile), scale by 1/sqrt(128), mask t >= T, an online softmax in FP32
//       (running max and sum per query head), P rounded to fp16 and
//       O += P V (ldmatrix.trans).  At the end the eight warps' (max, sum, O)
//       are merged through shared memory and written to the workspace.
//       The CTA then counts itself in on its KV head's counter (after a
//       fence); the one that completes the count merges the head's key ranges
//       in their order (max, rescale, sum), writes o in fp16 and sets the
//       counter back to zero.  No CTA waits for another.
// Every wait is bounded; a timed-out wait sets W4A16_DEV_PIPE_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kAD = 128;                    // head dimension
constexpr int kAKeys = 64;                  // keys per tile
constexpr int kAGroups = 2;                 // consumer groups, alternate tiles
constexpr int kAWarps = 4 * kAGroups;       // consumer warps, 16 keys of their group's tile each
constexpr int kAThreads = 32 * (kAWarps + 1);
constexpr int kABox = kAKeys * 128;         // one box: 64 keys x 64 dimensions fp16
constexpr int kATileBytes = 4 * kABox;      // K (two halves of the dimensions), then V
constexpr int kAStages = 4;
constexpr int kARows = 16;                  // query heads per KV head, padded (MMA M)
constexpr int kAHeader = 1024;              // barriers, then the merge flag
// per-warp merge area: max[16], sum[16], O[16][128] floats
constexpr int kAMergeBytes = kAWarps * (2 * kARows + kARows * kAD) * 4;
constexpr int kASmem = kAHeader + kAStages * kATileBytes + kAMergeBytes + 1024;

struct AttnParams {
  const uint16_t* q;  // [n_heads][128]
  uint16_t* o;        // [n_heads][128]
  unsigned* ctr;      // [n_kv_heads]: key ranges finished (zero between calls)
  float* ws_ml;       // [n_kv_heads][splits][16][2]: running max and sum
  float* ws_o;        // [n_kv_heads][splits][16][128]: unnormalised output
  int group;          // query heads per KV head (<= 16)
  int T;              // keys
  int splits;         // key ranges per KV head
  int ntiles;         // ceil(T / 64)
  uint32_t* status;
};

// L2 prefetch of one box of a 3-D tensor map (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const void* tmap, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(tmap), "r"(x), "r"(y),
               "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Shared address of 16 bytes at (key row, dimension d0, a multiple of 8) of a
// 64-key x 64-dimension box stored with the 128-byte swizzle (16-byte chunk c
// of row r at chunk c ^ (r % 8)).
__device__ __forceinline__ uint32_t box_addr(uint32_t box, int row, int d0) {
  return box + row * 128 + ((((d0 >> 3) & 7) ^ (row & 7)) << 4);
}

constexpr int kAMaxSplits = 256;  // key ranges per KV head (at most the SM count)
static_assert(kAWarps * kAMaxSplits * 4 <= kAMergeBytes, "merge scratch exceeds the merge area");
static_assert(kAMaxSplits % 32 == 0, "ranges are spread over the lanes of a warp");

// Merge the key ranges of KV head g (run by the CTA that finished last):
//   o_h = fp16_RN(sum_sp O_sp e_sp / sum_sp l_sp e_sp),  e_sp = 2^((m_sp - M) log2 e),
// M = max_sp m_sp, for the group's query heads h = g group + r, every sum
// in range order (the result does not depend on which CTA merges).  Warp w
// merges heads r = w, w + 8 alone: lane l holds the statistics of ranges
// l, l + 32, ... and sums dimensions 4 l .. 4 l + 3 over the ranges, with
// the first kB ranges' loads issued together with the statistics (two
// rounds of L2 loads for 38 ranges).  sh: kAWarps x kAMaxSplits floats.
// The workspace is read past L1 (written by other CTAs of this launch).
__device__ __forceinline__ void merge_ranges(const AttnParams& p, int g, float* sh, int t) {
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr int kB = 20;                      // ranges per round of loads
  constexpr int kPer = kAMaxSplits / 32;      // statistics per lane
  constexpr int kRangeF4 = kARows * kAD / 4;  // float4s per range
  const int lane = t & 31, warp = t >> 5;
  float* er = sh + warp * kAMaxSplits;
  const float* ml = p.ws_ml + static_cast<int64_t>(g) * p.splits * kARows * 2;
  const float* wo = p.ws_o + static_cast<int64_t>(g) * p.splits * kARows * kAD;
  const int splits = p.splits;
  for (int r = warp; r < p.group; r += kAWarps) {
    const float4* src = reinterpret_cast<const float4*>(wo + r * kAD) + lane;
    float4 v[kB];
#pragma unroll
    for (int i = 0; i < kB; ++i)
      v[i] = i < splits ? __ldcg(src + static_cast<int64_t>(i) * kRangeF4) : make_float4(0.f, 0.f, 0.f, 0.f);
    float mv[kPer], lv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int sp = lane + 32 * j;
      mv[j] = sp < splits ? __ldcg(ml + (sp * kARows + r) * 2) : -INFINITY;
      lv[j] = sp < splits ? __ldcg(ml + (sp * kARows + r) * 2 + 1) : 0.f;
    }
    float mloc = mv[0];
#pragma unroll
    for (int j = 1; j < kPer; ++j) mloc = fmaxf(mloc, mv[j]);
    for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
    const float Mu = mloc == -INFINITY ? 0.f : mloc;
    float lloc = 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int sp = lane + 32 * j;
      if (sp < splits) {
        const float e = exp2f((mv[j] - Mu) * kLog2e);
        er[sp] = e;
        lloc += lv[j] * e;
      }
    }
    for (int off = 16; off > 0; off >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, off);
    __syncwarp();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0;;) {
#pragma unroll
      for (int i = 0; i < kB; ++i) {
        if (s0 + i < splits) {
          const float e = er[s0 + i];
          acc.x += v[i].x * e;
          acc.y += v[i].y * e;
          acc.z += v[i].z * e;
          acc.w += v[i].w * e;
        }
      }
      s0 += kB;
      if (s0 >= splits) break;
#pragma unroll
      for (int i = 0; i < kB; ++i)
        v[i] = s0 + i < splits ? __ldcg(src + static_cast<int64_t>(s0 + i) * kRangeF4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const uint32_t lo = pack_half2(acc.x / lloc, acc.y / lloc), hi = pack_half2(acc.z / lloc, acc.w / lloc);
    uint2* dst = reinterpret_cast<uint2*>(p.o + (static_cast<int64_t>(g) * p.group + r) * kAD) + lane;
    if (W4A16_IN(p.status, r < p.group && g < static_cast<int>(gridDim.x) / p.splits)) *dst = make_uint2(lo, hi);
    __syncwarp();  // er is rewritten for the warp's next head
  }
}

__global__ void __launch_bounds__(kAThreads, 1)
    attn_partial_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int g = blockIdx.x / p.splits;   // KV head
  const int sp = blockIdx.x % p.splits;  // key range
  const int tb = static_cast<int>((static_cast<int64_t>(p.ntiles) * sp) / p.splits);
  const int te = static_cast<int>((static_cast<int64_t>(p.ntiles) * (sp + 1)) / p.splits);
  const int nt = te - tb;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const uint32_t base = smem_addr(smem);
  const uint32_t full0 = base;
  const uint32_t empty0 = base + 8 * kAStages;
  const uint32_t stage0 = (base + kAHeader + 1023) & ~1023u;
  const uint32_t merge0 = stage0 + kAStages * kATileBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kAWarps / kAGroups);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  // This CTA's key range is requested into L2 before the dependency wait:
  // a CTA that starts while the previous kernel is still finishing (its
  // merge runs on a few CTAs) gets its first tiles from L2.  A prefetch only
  // fills L2, the point of coherence, so a cache row the previous kernel
  // writes is read after the wait with its new value.  Measured (graphs of
  // 28 calls, cold L2): T = 8192 9.42 -> 9.05 us, T = 32768 16.25 -> 16.10,
  // T = 1024 unchanged.
  if (warp == kAWarps && lane == 0) {
    for (int i = 0; i < nt; ++i) {
      const int t0 = (tb + i) * kAKeys;
      tma_prefetch_3d(&kmap, 0, t0, g);
      tma_prefetch_3d(&kmap, 64, t0, g);
      tma_prefetch_3d(&vmap, 0, t0, g);
      tma_prefetch_3d(&vmap, 64, t0, g);
    }
  }
  pdl_wait();  // q and the cache may be the previous kernel's output

  if (warp == kAWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      for (int i = 0; i < nt; ++i) {
        const int s = i % kAStages;
        if (i >= kAStages && !mbar_wait_bounded(empty0 + 8 * s, ((i / kAStages) & 1) ^ 1, kWaitLimitNs)) {
          atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
          break;
        }
        const uint32_t st = stage0 + s * kATileBytes;
        const uint32_t bar = full0 + 8 * s;
        const int t0 = (tb + i) * kAKeys;
        mbar_arrive_expect_tx(bar, kATileBytes);
        tma_load_3d(st, &kmap, 0, t0, g, bar, pol);
        tma_load_3d(st + kABox, &kmap, 64, t0, g, bar, pol);
        tma_load_3d(st + 2 * kABox, &vmap, 0, t0, g, bar, pol);
        tma_load_3d(st + 3 * kABox, &vmap, 64, t0, g, bar, pol);
        issued = i + 1;
      }
      // the copies in flight land before the CTA can exit
      for (int i = issued - kAStages > 0 ? issued - kAStages : 0; i < issued; ++i)
        mbar_wait_bounded(full0 + 8 * (i % kAStages), (i / kAStages) & 1, kWaitLimitNs);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int g8 = lane >> 2;  // fragment row group: query heads g8 and g8 + 8
  const int t4 = lane & 3;
  // Q as the A operand (16 query heads x 128), rows past the group zero
  uint32_t qa[8][4];
  {
    const uint16_t* q0 = p.q + static_cast<int64_t>(g) * p.group * kAD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d = 16 * kk + 2 * t4;
      const bool r0 = g8 < p.group, r1 = g8 + 8 < p.group;
      qa[kk][0] = r0 ? *reinterpret_cast<const uint32_t*>(q0 + g8 * kAD + d) : 0u;
      qa[kk][1] = r1 ? *reinterpret_cast<const uint32_t*>(q0 + (g8 + 8) * kAD + d) : 0u;
      qa[kk][2] = r0 ? *reinterpret_cast<const uint32_t*>(q0 + g8 * kAD + d + 8) : 0u;
      qa[kk][3] = r1 ? *reinterpret_cast<const uint32_t*>(q0 + (g8 + 8) * kAD + d + 8) : 0u;
    }
  }
  constexpr float kLog2e = 1.4426950408889634f;
  const float kScale = 0.08838834764831845f;  // 1 / sqrt(128)
  float m_run[2] = {-INFINITY, -INFINITY};    // rows g8, g8 + 8 (scaled scores)
  float l_run[2] = {0.f, 0.f};                // this thread's share of the sums
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nd][c] = 0.f;
  bool ok = true;
  const int grp = warp / 4;         // tiles i = grp (mod kAGroups)
  const int kr = 16 * (warp % 4);   // this warp's first key row in a tile

  for (int i = grp; i < nt; i += kAGroups) {
    const int s = i % kAStages;
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(full0 + 8 * s, (i / kAStages) & 1, kWaitLimitNs));
    if (!ok) {
      if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
      break;
    }
    const uint32_t kst = stage0 + s * kATileBytes;
    const uint32_t vst = kst + 2 * kABox;
    // ---- S = Q K^T for the warp's 16 keys (two n-tiles of 8 keys)
    float sc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[j][c] = 0.f;
    {
      // ldmatrix x4: matrix mi = lane / 8 is keys kr + 8 (mi / 2) .. + 7,
      // dimensions 16 kk + 8 (mi % 2) .. + 7: b0, b1 of n-tile 0, then n-tile 1
      const int mi = lane >> 3;
      const int row = kr + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int d0 = 16 * kk + 8 * (mi & 1);
        uint32_t b00, b01, b10, b11;
        ldsm_x4(box_addr(kst + (d0 >> 6) * kABox, row, d0), b00, b01, b10, b11);
        mma16816(sc[0], qa[kk], b00, b01);
        mma16816(sc[1], qa[kk], b10, b11);
      }
    }
    // ---- online softmax (scores scaled by 1/sqrt(128); keys t >= T masked)
    const int tk = (tb + i) * kAKeys + kr;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int t = tk + 8 * j + 2 * t4 + (c & 1);
        const float v = t < p.T ? sc[j][c] * kScale : -INFINITY;
        sc[j][c] = v;
        mx[c >> 1] = fmaxf(mx[c >> 1], v);
      }
    float corr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float m_new = fmaxf(m_run[r], mx[r]);
      // with no key seen yet (m_new = -inf) every weight is 0: use 0 as the base
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      corr[r] = exp2f((m_run[r] - m_use) * kLog2e);
      m_run[r] = m_new;
      mx[r] = m_use;
    }
    uint32_t pa[4];
    {
      float pf[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) pf[j][c] = exp2f((sc[j][c] - mx[c >> 1]) * kLog2e);
#pragma unroll
      for (int r = 0; r < 2; ++r)
        l_run[r] = l_run[r] * corr[r] + (pf[0][2 * r] + pf[0][2 * r + 1]) + (pf[1][2 * r] + pf[1][2 * r + 1]);
      // A operand of P V: rows g8 / g8 + 8, keys 2 t4 (+1) and 8 + 2 t4 (+1)
      pa[0] = pack_half2(pf[0][0], pf[0][1]);
      pa[1] = pack_half2(pf[0][2], pf[0][3]);
      pa[2] = pack_half2(pf[1][0], pf[1][1]);
      pa[3] = pack_half2(pf[1][2], pf[1][3]);
    }
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
      o[nd][0] *= corr[0];
      o[nd][1] *= corr[0];
      o[nd][2] *= corr[1];
      o[nd][3] *= corr[1];
    }
    // ---- O += P V: ldmatrix.trans x4, matrix mi = lane / 8 is keys
    // kr + 8 (mi % 2) .. + 7, dimensions 8 (nd + mi / 2) .. + 7
    {
      const int mi = lane >> 3;
      const int row = kr + 8 * (mi & 1) + (lane & 7);
#pragma unroll
      for (int nd = 0; nd < 16; nd += 2) {
        const int d0 = 8 * (nd + (mi >> 1));
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(box_addr(vst + (d0 >> 6) * kABox, row, d0), b0, b1, b2, b3);
        mma16816(o[nd], pa, b0, b1);
        mma16816(o[nd + 1], pa, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }

  // ---- merge the four warps: each writes its max, sum and O to shared memory
  float* mg = reinterpret_cast<float*>(smem + (merge0 - base));
  float* wm = mg + warp * (2 * kARows + kARows * kAD);
  float* wl = wm + kARows;
  float* wo = wl + kARows;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
  }
  if (t4 == 0) {
    wm[g8] = m_run[0];
    wm[g8 + 8] = m_run[1];
    wl[g8] = l_run[0];
    wl[g8 + 8] = l_run[1];
  }
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) {
    const int d = 8 * nd + 2 * t4;
    wo[g8 * kAD + d] = o[nd][0];
    wo[g8 * kAD + d + 1] = o[nd][1];
    wo[(g8 + 8) * kAD + d] = o[nd][2];
    wo[(g8 + 8) * kAD + d + 1] = o[nd][3];
  }
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kAWarps) : "memory");
  // thread d < 128 of the consumers merges dimension d of every query head
  // and writes the key range's statistics and output to the workspace
  const int64_t slot = static_cast<int64_t>(g) * p.splits + sp;
  if (threadIdx.x < kAD) {
    const int d = threadIdx.x;
    for (int r = 0; r < p.group; ++r) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) M = fmaxf(M, mg[w * (2 * kARows + kARows * kAD) + r]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float L = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) {
        const float* b = mg + w * (2 * kARows + kARows * kAD);
        const float e = exp2f((b[r] - Mu) * kLog2e);
        L += b[kARows + r] * e;
        acc += b[2 * kARows + r * kAD + d] * e;
      }
      if (!W4A16_IN(p.status, slot < static_cast<int>(gridDim.x) && r < kARows)) break;
      p.ws_o[(slot * kARows + r) * kAD + d] = acc;
      if (d == 0) {
        p.ws_ml[(slot * kARows + r) * 2] = M;
        p.ws_ml[(slot * kARows + r) * 2 + 1] = L;
      }
    }
  }
  // Count the range in: after the CTA barrier one thread adds to the counter
  // with release and acquire semantics at GPU scope (cumulative over the
  // CTA's stores ordered before it by the barrier); the CTA that completes
  // the count (exactly one per KV head) has then acquired every range's
  // stores, and its barrier orders its threads' loads after that.
  // The flag sits in the header, past the pipeline barriers.
  volatile unsigned* s_last = reinterpret_cast<volatile unsigned*>(smem + 16 * kAStages);
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kAWarps) : "memory");
  if (threadIdx.x == 0) {
    unsigned done;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(done) : "l"(p.ctr + g) : "memory");
    const bool last = done == static_cast<unsigned>(p.splits - 1);
    *s_last = last ? 1u : 0u;
    // every range of this call has counted: ready for the next call
    if (last) atomicExch(p.ctr + g, 0u);
  }
  asm volatile("bar.sync 1, %0;" ::"r"(32 * kAWarps) : "memory");
  if (*s_last == 0) return;
  merge_ranges(p, g, mg, threadIdx.x);
}

// K or V cache as a 3-D tensor: [n_kv_heads][T][128] fp16 with head stride
// t_stride rows; box 64 dimensions x 64 keys x 1 head, 128-byte swizzle.
// Keys at or past T are outside the tensor: the copy fills them with zeros.
bool cache_map(CUtensorMap* m, const uint16_t* cache, int n_kv_heads, int T, int t_stride) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kAD), static_cast<cuuint64_t>(T),
                              static_cast<cuuint64_t>(n_kv_heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kAD) * 2,
                                 static_cast<cuuint64_t>(t_stride) * kAD * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kAKeys), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<uint16_t*>(cache), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int attn_splits(int n_kv_heads, int T, const DeviceInfo& d) {
  const int ntiles = (T + kAKeys - 1) / kAKeys;
  int per_head = d.sms / n_kv_heads;
  if (per_head < 1) per_head = 1;
  if (per_head > kAMaxSplits) per_head = kAMaxSplits;
  return ntiles < per_head ? ntiles : per_head;
}

// [counters: one per possible KV head, at a fixed place for every shape][ws_ml][ws_o]
constexpr size_t kACtrBytes = W4A16_ATTN_MAX_KV_HEADS * sizeof(unsigned);
static_assert(kACtrBytes % 16 == 0, "the statistics must stay 16-byte aligned");

size_t attn_workspace_bytes(int n_kv_heads, int splits) {
  return kACtrBytes + static_cast<size_t>(n_kv_heads) * splits * kARows * (2 + kAD) * sizeof(float);
}

cudaError_t launch_attn_decode(const AttnArgs& a, const DeviceInfo& d, cudaStream_t st) {
  const int splits = attn_splits(a.n_kv_heads, a.T, d);
  CUtensorMap kmap, vmap;
  if (!cache_map(&kmap, a.k, a.n_kv_heads, a.T, a.t_stride) ||
      !cache_map(&vmap, a.v, a.n_kv_heads, a.T, a.t_stride))
    return cudaErrorInvalidValue;
  AttnParams p;
  p.q = a.q;
  p.o = a.o;
  p.ctr = reinterpret_cast<unsigned*>(a.workspace);
  if (a.n_kv_heads > W4A16_ATTN_MAX_KV_HEADS) return cudaErrorInvalidValue;
  p.ws_ml = a.workspace + kACtrBytes / sizeof(float);
  p.ws_o = p.ws_ml + static_cast<size_t>(a.n_kv_heads) * splits * kARows * 2;
  p.group = a.n_heads / a.n_kv_heads;
  p.T = a.T;
  p.splits = splits;
  p.ntiles = (a.T + kAKeys - 1) / kAKeys;
  p.status = a.status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_kv_heads * splits);
  cfg.blockDim = dim3(kAThreads);
  cfg.dynamicSmemBytes = kASmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, attn_partial_kernel, kmap, vmap, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t prepare_attn_decode(const DeviceInfo& d) {
  (void)d;
  return cudaFuncSetAttribute(attn_partial_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kASmem);
}

}  // namespace w4a16
