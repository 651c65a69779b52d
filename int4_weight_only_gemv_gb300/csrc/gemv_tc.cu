// gemv_tc.cu -- small-batch GEMV for M = 8..16 on the 5th-generation tensor
// cores (tcgen05.mma, accumulators and the unpacked weights in tensor memory).
//
// Same operation as the other GEMV kernels ("Costruire un runtime di
// inference LLM da zero", "Tre bug che insegnano": INT4 group-128 weights x
// FP16 activations, FP32 accumulation).  From M = 8 on every weight feeds
// eight or more products, a dense contraction.  Per 128-row tile and
// 128-k group the kernel computes D[n][m] = sum_k q[n][k] x[m][k] with one
// M = 128, N = 16, K = 16 MMA per 16 k: the exact INT4 values q (fp16) are the
// A operand, read from tensor memory, and the activations (rows past M filled
// with zeros) the B operand, read from shared memory.  Each group's D is then
// scaled by the group scale in FP32 and added to per-row accumulators, so the
// result equals sum_g s[n][g] sum_{k in g} q x, as the format defines it.
//
// Roles (one CTA per SM, 320 threads):
//   warp 0      producer.  Streams the CTA's boxes through an S-stage ring:
//               per stage one 2-D TMA load of a 128-row x 128-byte box of
//               the packed weight (two groups; 128-byte swizzle; rows past
//               N and words past K read as zero) and four of the
//               activations (16 rows x 64 k each, the same swizzle; rows
//               past M and k past K zero), all on the stage's mbarrier.
//               The weights of the first S stages are requested before the
//               wait for the previous kernel, the activations after it.
//   warp 1      allocates 512 tensor-memory columns; lane 0 issues the MMAs
//               of a group once the transform warps have written its A
//               operand, commits them to the group's barrier, and releases
//               a stage once the MMAs of both its groups have completed.
//   warps 2..9  transform.  Warp w serves tensor-memory lanes 32 (w % 4) ..
//               (the rows of the tile), half (w - 2) / 4 of each group's k:
//               two 16-byte shared loads (swizzle undone), 32 fp16 pairs of
//               exact q in natural k order (PRMT + LOP3 + HFMA2 per pair),
//               one tcgen05.st of 32 columns.  kTcNB - 1 groups later they
//               read the group's D (8 columns: activation rows 8 h .. 8 h + 7),
//               scale and accumulate it.  kTcNB A and D buffers rotate.
// Split-K: when the tiles are fewer than the SMs, a cluster of KS CTAs owns
// one tile, rank r taking the r-th slice of its boxes; the ranks push their
// partial sums to the owner of each entry through distributed shared memory,
// and after one cluster barrier each owner sums them in rank order
// (deterministic, no atomics, no global workspace).
// Every wait is bounded; a role whose wait ran out stops its work, still
// takes part in the cluster barrier, and the CTA frees its tensor memory
// only after its copies and MMAs in flight have completed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kTcRows = 128;                // rows per tile = MMA M
constexpr int kTcN = 16;                    // MMA N = activation rows (padded)
constexpr int kTcTransformWarps = 16;
constexpr int kTcIssuers = 2;                // MMA-issuing warps
constexpr int kTcThreads = 32 * (1 + kTcIssuers + kTcTransformWarps);
constexpr int kTcWBytes = kTcRows * 128;    // weight box: 128 rows x 128 bytes (two groups)
constexpr int kTcXBox = kTcN * 128;         // activation box: 16 rows x 64 k
constexpr int kTcStageBytes = kTcWBytes + 4 * kTcXBox;
constexpr int kTcMaxStages = 8;
constexpr int kTcHeader = 1024;             // barriers and the tensor-memory address
// Tensor memory: kTcNB A buffers of 64 columns (128 k x 128 rows of fp16
// pairs) and kTcNB D buffers of 16 columns (fp32), so the transform warps
// run up to kTcNB - 1 groups ahead of the scaling of a group's D.
#ifndef W4A16_TC_ACC
#define W4A16_TC_ACC 2
#endif
constexpr int kTcAcc = W4A16_TC_ACC;  // independent accumulators per group (1, 2 or 4)
constexpr int kTcNB = kTcAcc == 4 ? 4 : 5;
constexpr int kTcTmemCols = 512;
constexpr int kTcColD = 64 * kTcNB;
constexpr int kTcDCols = 16 * kTcAcc;  // D columns per group
static_assert(kTcColD + kTcDCols * kTcNB <= kTcTmemCols, "tensor-memory buffers overflow the allocation");
// Dynamic shared memory is at least this much, so one CTA fits per SM: a
// second one would wait for tensor memory inside tcgen05.alloc.
constexpr int kTcMinSmem = 120 * 1024;

struct TcParams {
  GemvArgs a;
  int KS;           // CTAs per cluster (K slices); KS > 1: one tile per cluster
  int S;            // ring stages
  int part_bytes;   // owner-slot buffer (KS > 1)
  uint32_t idesc;   // MMA instruction descriptor
};

// ------------------------------------------------------------ tcgen05 / TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive (once) on a barrier of this CTA when every MMA this thread issued
// so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// The 8 MMAs of one 128-k group, k step ks into accumulator ks % kTcAcc:
// D_j (tensor memory, 16 columns at d + 16 j) = sum over ks = j mod kTcAcc
// of A_ks (tensor memory, columns a + 8 ks) x B_ks (shared memory,
// descriptor b[ks]); the first MMA into each D_j overwrites it.  Independent
// accumulators let the MMAs of a group overlap instead of each waiting for
// the previous one's D.  One asm block: the issuing thread spends its time
// on the MMAs, not on per-instruction setup.
#define W4A16_TC_MMA(A, B, P) "tcgen05.mma.cta_group::1.kind::f16 [" D_FOR(A) "], [a" #A "], %" #B ", %10, " P ";\n\t"
__device__ __forceinline__ void tc_mma_group(uint32_t d, uint32_t a, const uint64_t (&b)[8], uint32_t idesc) {
#if W4A16_TC_ACC == 4
#define D_FOR(A) "d" #A
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 a0, a1, a2, a3, a4, a5, a6, a7, d0, d1, d2, d3, d4, d5, d6, d7;\n\t"
      "setp.eq.u32 pt, %10, %10;\n\tsetp.ne.u32 pf, %10, %10;\n\t"
      "mov.u32 a0, %1;\n\tadd.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.u32 a4, %1, 32;\n\tadd.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
      "mov.u32 d0, %0;\n\tadd.u32 d1, %0, 16;\n\tadd.u32 d2, %0, 32;\n\tadd.u32 d3, %0, 48;\n\t"
      "mov.u32 d4, d0;\n\tmov.u32 d5, d1;\n\tmov.u32 d6, d2;\n\tmov.u32 d7, d3;\n\t"
      W4A16_TC_MMA(0, 2, "pf") W4A16_TC_MMA(1, 3, "pf") W4A16_TC_MMA(2, 4, "pf") W4A16_TC_MMA(3, 5, "pf")
      W4A16_TC_MMA(4, 6, "pt") W4A16_TC_MMA(5, 7, "pt") W4A16_TC_MMA(6, 8, "pt") W4A16_TC_MMA(7, 9, "pt")
      "}" ::"r"(d), "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]),
      "l"(b[7]), "r"(idesc)
      : "memory");
#undef D_FOR
#elif W4A16_TC_ACC == 2
#define D_FOR(A) "d" #A
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 a0, a1, a2, a3, a4, a5, a6, a7, d0, d1, d2, d3, d4, d5, d6, d7;\n\t"
      "setp.eq.u32 pt, %10, %10;\n\tsetp.ne.u32 pf, %10, %10;\n\t"
      "mov.u32 a0, %1;\n\tadd.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.u32 a4, %1, 32;\n\tadd.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
      "mov.u32 d0, %0;\n\tadd.u32 d1, %0, 16;\n\tmov.u32 d2, d0;\n\tmov.u32 d3, d1;\n\t"
      "mov.u32 d4, d0;\n\tmov.u32 d5, d1;\n\tmov.u32 d6, d0;\n\tmov.u32 d7, d1;\n\t"
      W4A16_TC_MMA(0, 2, "pf") W4A16_TC_MMA(1, 3, "pf") W4A16_TC_MMA(2, 4, "pt") W4A16_TC_MMA(3, 5, "pt")
      W4A16_TC_MMA(4, 6, "pt") W4A16_TC_MMA(5, 7, "pt") W4A16_TC_MMA(6, 8, "pt") W4A16_TC_MMA(7, 9, "pt")
      "}" ::"r"(d), "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]),
      "l"(b[7]), "r"(idesc)
      : "memory");
#undef D_FOR
#else
#define D_FOR(A) "%0"
  asm volatile(
      "{\n\t.reg .pred pf, pt;\n\t.reg .b32 a0, a1, a2, a3, a4, a5, a6, a7;\n\t"
      "setp.eq.u32 pt, %10, %10;\n\tsetp.ne.u32 pf, %10, %10;\n\t"
      "mov.u32 a0, %1;\n\tadd.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
      "add.u32 a4, %1, 32;\n\tadd.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
      W4A16_TC_MMA(0, 2, "pf") W4A16_TC_MMA(1, 3, "pt") W4A16_TC_MMA(2, 4, "pt") W4A16_TC_MMA(3, 5, "pt")
      W4A16_TC_MMA(4, 6, "pt") W4A16_TC_MMA(5, 7, "pt") W4A16_TC_MMA(6, 8, "pt") W4A16_TC_MMA(7, 9, "pt")
      "}" ::"r"(d), "r"(a), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]),
      "l"(b[7]), "r"(idesc)
      : "memory");
#undef D_FOR
#endif
}
#undef W4A16_TC_MMA

// 16 columns of this warp's 32 lanes, one 32-bit register per column.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
      "%13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 4 columns of this warp's 32 lanes (no wait: see tmem_wait_ld).
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand stored in 128-byte
// swizzled rows, 8-row atoms 1024 bytes apart: start address >> 4 (bits
// 0-13), leading-dimension offset 16 bytes (unused for this layout, bits
// 16-29), stride between 8-row atoms 1024 bytes (bits 32-45), descriptor
// version 1 (bits 46-48), base offset 0, layout 128-byte swizzle (bits
// 61-63 = 2).  A start inside a 128-byte row (k offsets) is the address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Exact q of one packed word as fp16 pairs in natural k order:
// {q0, q1}, {q2, q3}, {q4, q5}, {q6, q7}.  Byte i goes to both 16-bit lanes
// (PRMT); the low lane keeps its low nibble, the high lane its high nibble
// (at bits 4..7 of the lane), each turned into 1032 + q and 1152 + 16 q by
// the LOP3 of ptx.cuh, and one HFMA2 by {1, 1/16} minus {1032, 72} leaves q.
__device__ __forceinline__ void unpack_natural(uint32_t w, uint32_t* out) {
  const __half2 mul = __halves2half2(__ushort_as_half(0x3C00), __ushort_as_half(0x2C00));   // 1, 1/16
  const __half2 sub = __halves2half2(__ushort_as_half(0xE408), __ushort_as_half(0xD480));   // -1032, -72
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t t = __byte_perm(w, 0u, 0x4040u + 0x0101u * i);
    const uint32_t b = lop3_and_xor(t, 0x00F0000Fu, 0x64806408u);
    const __half2 q = __hfma2(*reinterpret_cast<const __half2*>(&b), mul, sub);
    out[i] = *reinterpret_cast<const uint32_t*>(&q);
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    gemv_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                   const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const GemvArgs& a = p.a;
  const int KS = p.KS, S = p.S;
  const int rank = KS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster = blockIdx.x / KS;
  const int nclusters = gridDim.x / KS;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const int N = a.N;
  const int G = a.K / 128;
  const int B = (G + 1) / 2;  // boxes (two groups) per row
  const int T = (N + kTcRows - 1) / kTcRows;
  const int bb = (B * rank) / KS, be = (B * (rank + 1)) / KS;
  const int nb = be - bb;                                   // boxes per tile of this rank
  const int ntl = (T - cluster + nclusters - 1) / nclusters;  // tiles of this cluster
  const int total = ntl * nb;                               // stages this CTA consumes

  // shared layout: [full S][empty S][afull NB][dfull NB][mma_done][tmem addr] |
  // owner slots | stages (1024-aligned)
  const uint32_t base = smem_addr(smem);
  const uint32_t full0 = base;
  const uint32_t empty0 = base + 8 * kTcMaxStages;
  const uint32_t afull0 = base + 16 * kTcMaxStages;
  const uint32_t dfull0 = afull0 + 8 * kTcNB;
  const uint32_t mma_done = dfull0 + 8 * kTcNB;
  const uint32_t tmem_slot = mma_done + 8;
  const uint32_t part0 = base + kTcHeader;
  const uint32_t stage0 = (part0 + p.part_bytes + 1023) & ~1023u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kTcIssuers);
    }
    for (int b = 0; b < kTcNB; ++b) {
      mbar_init(afull0 + 8 * b, kTcTransformWarps);
      mbar_init(dfull0 + 8 * b, 1);
    }
    mbar_init(mma_done, kTcIssuers);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + (tmem_slot - base));
  pdl_launch_dependents();

  // the stage of consumed box gi, its tile and box index
  auto coords = [&](int gi, int& tile, int& box) {
    tile = cluster + (gi / nb) * nclusters;
    box = bb + gi % nb;
  };
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int pre = total < S ? total : S;
      auto load_x = [&](int gi) {
        int tile, box;
        coords(gi, tile, box);
        const uint32_t st = stage0 + (gi % S) * kTcStageBytes;
        for (int j = 0; j < 4; ++j)
          tma_load_2d(st + kTcWBytes + j * kTcXBox, &xmap, box * 256 + 64 * j, 0, full0 + 8 * (gi % S), pol);
      };
      // weights of the first stages before the dependency wait: they are
      // constant; the activations may be the previous kernel's output
      for (int gi = 0; gi < pre; ++gi) {
        int tile, box;
        coords(gi, tile, box);
        mbar_arrive_expect_tx(full0 + 8 * gi, kTcStageBytes);
        tma_load_2d(stage0 + gi * kTcStageBytes, &wmap, box * 32, tile * kTcRows, full0 + 8 * gi, pol);
      }
      pdl_wait();
      for (int gi = 0; gi < pre; ++gi) load_x(gi);
      int issued = pre;
      for (int gi = pre; gi < total; ++gi) {
        const int s = gi % S;
        if (!mbar_wait_bounded(empty0 + 8 * s, ((gi / S) & 1) ^ 1, kWaitLimitNs)) {
          atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
          ok = false;
          break;
        }
        int tile, box;
        coords(gi, tile, box);
        mbar_arrive_expect_tx(full0 + 8 * s, kTcStageBytes);
        tma_load_2d(stage0 + s * kTcStageBytes, &wmap, box * 32, tile * kTcRows, full0 + 8 * s, pol);
        load_x(gi);
        issued = gi + 1;
      }
      // let the copies in flight land before the CTA can exit
      for (int gi = issued - S > 0 ? issued - S : 0; gi < issued; ++gi)
        mbar_wait_bounded(full0 + 8 * (gi % S), (gi / S) & 1, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp <= kTcIssuers) {
    // ------------------------------------------------------------ MMA issuers
    // issuer ir takes the groups gc = ir mod kTcIssuers (gc counts every
    // group of every tile); each releases a stage once its MMAs of the
    // stage have completed, so the stage's barrier counts kTcIssuers
    if (lane == 0) {
      const int ir = warp - 1;
      int gc = 0;
      for (int gi = 0; gi < total && ok; ++gi) {
        const int s = gi % S;
        if (!mbar_wait_bounded(full0 + 8 * s, (gi / S) & 1, kWaitLimitNs)) {
          atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
          ok = false;
          break;
        }
        int tile, box;
        coords(gi, tile, box);
        // descriptor of the stage's first activation box; the others and the
        // k offsets inside a 128-byte row are added to its address field
        // (>> 4; no carry: shared addresses are below 256 KB)
        const uint64_t dx = sw128_desc(stage0 + s * kTcStageBytes + kTcWBytes);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          if (2 * box + jj >= G) break;
          const int buf = gc % kTcNB;
          if (gc % kTcIssuers == ir) {
            if (!mbar_wait_bounded(afull0 + 8 * buf, (gc / kTcNB) & 1, kWaitLimitNs)) {
              atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
              ok = false;
              break;
            }
            tc_fence_after();
            uint64_t b[8];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)  // k = 16 ks: x box 2 jj + ks / 4, 32-byte offset ks % 4
              b[ks] = dx + static_cast<uint64_t>(((2 * jj + (ks >> 2)) * kTcXBox + 32 * (ks & 3)) >> 4);
            tc_mma_group(tmem + kTcColD + kTcDCols * buf, tmem + 64 * buf, b, p.idesc);
            tc_commit(dfull0 + 8 * buf);
          }
          ++gc;
        }
        tc_commit(empty0 + 8 * s);  // this issuer's reads of the stage are done
      }
      // every MMA issued has completed before tensor memory is freed
      tc_commit(mma_done);
      mbar_wait_bounded(mma_done, 0, kWaitLimitNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ transform
    const int q = warp & 3;                            // tensor-memory lane quarter
    const int h = (warp - 1 - kTcIssuers) >> 2;        // quarter of each group's k / of D's columns
    const int r = 32 * q + lane;                       // row of the tile
    const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
    const bool want_d = 4 * h < a.M;                   // D columns past M are zero
    float acc[4];
    int gc = 0;       // groups transformed (all tiles)
    int ge = 0;       // groups scaled (all tiles)
    const int g0 = 2 * bb;                             // first group of the slice
    const int ng = (2 * be < G ? 2 * be : G) - g0;     // groups per tile of the slice
    const uint16_t* srow = a.scales;
    int ge_tile = 0;     // groups of the current tile scaled so far
    float s_next = 0.f;  // scale of the next group to scale (loaded one group ahead)
    bool stored_once = false;
    // ok stays uniform across the warp (the tensor-memory accesses are
    // warp-collective): a wait that ran out in any lane stops the whole warp
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
      if (!ok) return;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, kWaitLimitNs));
      if (!ok && lane == 0) atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
    };
    // scale the oldest pending group's D (buffer ge % NB) into acc
    auto epilogue = [&]() {
      const int buf = ge % kTcNB;
      const float s = s_next;
      if (ge_tile + 1 < ng) s_next = __half2float(__ushort_as_half(ld_nc_u16(srow + g0 + ge_tile + 1)));
      ++ge_tile;
      warp_wait(dfull0 + 8 * buf, (ge / kTcNB) & 1);
      ++ge;
      tc_fence_after();
      if (ok && want_d) {
        uint32_t d[kTcAcc][4];
#pragma unroll
        for (int j = 0; j < kTcAcc; ++j) tmem_ld4(tmem + lane_addr + kTcColD + kTcDCols * buf + 16 * j + 4 * h, d[j]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float v = __uint_as_float(d[0][i]);
#pragma unroll
          for (int j = 1; j < kTcAcc; ++j) v += __uint_as_float(d[j][i]);
          acc[i] = fmaf(s, v, acc[i]);
        }
      }
    };
    for (int t = 0; t < ntl; ++t) {
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = 0.f;
      const int tile = cluster + t * nclusters;
      const int64_t row = static_cast<int64_t>(tile) * kTcRows + r;
      srow = a.scales + (row < N ? row : N - 1) * G;
      ge_tile = 0;
      s_next = __half2float(__ushort_as_half(ld_nc_u16(srow + g0)));
      for (int bi = 0; bi < nb; ++bi) {
        const int gi = t * nb + bi;
        const int s = gi % S;
        const int box = bb + bi;
        warp_wait(full0 + 8 * s, (gi / S) & 1);
        const uint32_t wrow = stage0 + s * kTcStageBytes + r * 128;
        for (int jj = 0; jj < 2; ++jj) {
          const int grp = 2 * box + jj;
          if (grp >= G) break;
          // buffer gc % NB was last used by group gc - NB: scale it first
          if (gc - ge == kTcNB) epilogue();
          const int buf = gc % kTcNB;
          if (ok) {
            // chunk 4 jj + h of the row (k = 32 h .. 32 h + 31 of the
            // group), swizzled by row % 8
            const uint4 w = lds_u4(wrow + (((4 * jj + h) ^ (r & 7)) << 4));
            uint32_t v[16];
            unpack_natural(w.x, v + 0);
            unpack_natural(w.y, v + 4);
            unpack_natural(w.z, v + 8);
            unpack_natural(w.w, v + 12);
            tmem_st16(tmem + lane_addr + 64 * buf + 16 * h, v);
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(afull0 + 8 * buf);
          ++gc;
        }
      }
      // the tile's remaining groups
      while (ge < gc) epilogue();
      // D layout: lane = row r, column 4 h + i = activation row m
      if (KS == 1) {
        if (!stored_once) {
          pdl_wait();  // y may still be read by the previous kernel
          stored_once = true;
        }
        if (row < N) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * h + i < a.M) store_out(a, 4 * h + i, row, acc[i]);
        }
      } else {
        // entry e = r * 16 + m belongs to rank e mod KS; rank q's partial
        // goes to slot (e / KS) KS + q of the owner's buffer
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int e = r * kTcN + 4 * h + i;
          const uint32_t local = part0 + 4 * static_cast<uint32_t>((e / KS) * KS + rank);
          st_cluster_f32(map_to_rank(local, static_cast<uint32_t>(e % KS)), acc[i]);
        }
      }
    }
  }

  if (KS > 1) {
    cluster_sync();  // every rank's partials have arrived at their owners
    pdl_wait();
    const int tile = cluster;  // one tile per cluster
    for (int i = threadIdx.x; i * KS + rank < kTcRows * kTcN; i += kTcThreads) {
      const int e = i * KS + rank;
      const int m = e % kTcN;
      const int64_t n = static_cast<int64_t>(tile) * kTcRows + e / kTcN;
      if (m >= a.M || n >= N) continue;
      const uint32_t addr = part0 + 4 * static_cast<uint32_t>(i * KS);
      float v = 0.f;
      for (int qq = 0; qq < KS; ++qq) v += lds_f32(addr + 4 * qq);
      store_out(a, m, n, v);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ---------------------------------------------------------------- host side

bool encode_map(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t inner, uint64_t rows,
                uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How many clusters of `ks` CTAs of the kernel fit on the GPU at once
// (a cluster must fit inside one GPC).  Cached per device.
int tc_active_clusters(int ks, int smem) {
  static std::mutex mu;
  static std::map<std::pair<int, int>, int> cache;  // (device * 16 + ks, smem) -> clusters
  int dev = 0;
  cudaGetDevice(&dev);
  const std::pair<int, int> key(dev * 16 + ks, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks * 64);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemv_tc_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

struct TcPlan {
  int KS = 0, clusters = 0, S = 0, part_bytes = 0, smem = 0;
};

// Choose the K split: the least work (boxes) for the busiest CTA, then the
// smaller split.  KS = 1: tiles spread over one CTA per SM.  KS > 1 only
// when every tile gets its own cluster (the reduction runs once, at the end).
TcPlan make_tc_plan(const GemvArgs& a, const DeviceInfo& d) {
  TcPlan best{};
  int64_t best_cost = INT64_MAX;
  const int T = (a.N + kTcRows - 1) / kTcRows;
  const int G = a.K / 128;
  const int B = (G + 1) / 2;
  for (int ks = 1; ks <= 8 && ks <= B; ++ks) {
    const int part = ks > 1 ? ((kTcRows * kTcN + ks - 1) / ks) * ks * 4 : 0;
    const int fixed = kTcHeader + part + 1023;  // stages start at the next 1024-byte boundary
    int S = (d.max_smem_optin - fixed) / kTcStageBytes;
    if (S > kTcMaxStages) S = kTcMaxStages;
    if (S < 2) continue;
    int smem = fixed + S * kTcStageBytes;
    if (smem < kTcMinSmem) smem = kTcMinSmem;
    int clusters;
    if (ks == 1) {
      clusters = T < d.sms ? T : d.sms;
    } else {
      if (tc_active_clusters(ks, smem) < T) continue;
      clusters = T;
    }
    const int64_t cost = static_cast<int64_t>((T + clusters - 1) / clusters) * ((B + ks - 1) / ks);
    if (cost < best_cost) {
      best_cost = cost;
      best.KS = ks;
      best.clusters = clusters;
      best.S = S;
      best.part_bytes = part;
      best.smem = smem;
    }
  }
  return best;
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

bool gemv_tc_supported(const GemvArgs& a) {
  return a.M >= 1 && a.M <= kTcN && a.K % 128 == 0 && a.ldx % 8 == 0 &&
         (reinterpret_cast<uintptr_t>(a.x) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.qweight) & 15u) == 0;
}

cudaError_t launch_gemv_tc(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (!gemv_tc_supported(a)) return cudaErrorInvalidValue;
  const TcPlan pl = make_tc_plan(a, d);
  if (pl.KS == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap wmap, xmap;
  // weights: uint32 [N][K/8], box 32 words x 128 rows
  if (!encode_map(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.qweight, static_cast<uint64_t>(a.K / 8),
                  static_cast<uint64_t>(a.N), static_cast<uint64_t>(a.K / 8) * 4, 32, kTcRows))
    return cudaErrorInvalidValue;
  // activations: fp16 [M][K] with row stride ldx, box 64 k x 16 rows
  if (!encode_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.x, static_cast<uint64_t>(a.K),
                  static_cast<uint64_t>(a.M), static_cast<uint64_t>(a.ldx) * 2, 64, kTcN))
    return cudaErrorInvalidValue;
  TcParams p;
  p.a = a;
  p.KS = pl.KS;
  p.S = pl.S;
  p.part_bytes = pl.part_bytes;
  // kind::f16 instruction descriptor: D f32 (bits 4-5 = 1), A and B f16
  // (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bits
  // 17-22, M >> 4 at bits 24-28
  p.idesc = (1u << 4) | (static_cast<uint32_t>(kTcN >> 3) << 17) | (static_cast<uint32_t>(kTcRows >> 4) << 24);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.clusters * pl.KS);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pl.KS > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = pl.KS;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (a.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_tc_kernel, wmap, xmap, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t prepare_gemv_tc(const DeviceInfo& d) {
  if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
  return cudaFuncSetAttribute(gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem_optin);
}

}  // namespace w4a16
