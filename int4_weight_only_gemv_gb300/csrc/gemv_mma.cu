// gemv_mma.cu -- small-batch GEMV (M = 2..16) on the tensor cores.
//
// Same operation as the other GEMV kernels ("Costruire un runtime di
// inference LLM da zero", "Tre bug che insegnano": INT4 group-128 weights x
// FP16 activations, FP32 accumulation).  With M activation rows each weight
// feeds M products, so the contraction runs on mma.sync m16n8k16
// (f16 x f16 -> f32): W is the A operand (16 weight rows), the activations
// the B operand (8 activation rows per n-tile; M <= 8 is one n-tile, M <= 16
// two sharing every unpacked A fragment).  Below M = 8 the n-tile is padded
// with zero columns: the tensor core has cycles to spare, the weight stream
// is the bound.
//
// Layout of the work.  K is cut into 256-k ranges (two groups; 128 bytes of
// a row; with an odd number of groups the last range is one group).  A
// cluster of KS CTAs owns a contiguous run of 16-row blocks; CTA rank r of
// the cluster owns ranges [r R, min(nr, (r + 1) R)), one per consumer warp,
// so the warp's activations (its B fragments for every k-step and n-tile)
// are loaded once into registers and reused for every block.
//   warp 0      producer (one lane).  Per block: ONE 3-D TMA load of the
//               rank's full ranges through a view of the packed weight as
//               [row][range][32 words] (a box of 16 rows x R ranges x 128
//               bytes, 128-byte swizzled; ranges past the row and rows past
//               N are filled with zeros, not read), a 2-D load of the last
//               half range (odd group count, last rank), and one bulk copy
//               of the block's scale rows.  A copy per block and not per
//               range: a thread's copy instructions, not the bytes, bound
//               the stream at 2 KB per copy.  S stages in flight.
//   warp 1      reducer.  Sums the consumer warps' partials of a block in
//               warp order; stores y (KS = 1) or pushes the CTA's partial to
//               the block's owner rank in the cluster (KS > 1).
//   warps 2..   consumers.  Warp w, lane (g, t) reads the 16 bytes at word
//               4 t of each group of its range in its rows pi(g) and
//               pi(g) + 8.  Rows pi(2q), pi(2q + 1) of a quarter-warp are d
//               apart with d Rb = 4 (mod 8): their 128-byte lines then differ
//               in bit 2 of the swizzle and the 8 lanes of every 16-byte load
//               hit 8 distinct chunks (no bank conflicts; R a multiple of 8
//               leaves a 2-way conflict).  Word j of those 16 bytes gives
//               two mma k-steps: halves {q0,q4},{q2,q6} (exact q) are the A
//               registers of one and {q1,q5},{q3,q7} of the other (the order
//               of k inside a contraction is free; the B fragments follow
//               it).  The second k-step's weights are left as the unpack's
//               1152 + 16 q, exact in fp16, against x / 16: each product is
//               q x + 72 x, and the chain starts from minus 72 x summed over
//               the group (FP32, computed once per warp), which saves two
//               instructions a word.  The groups' and n-tiles' mma chains are
//               interleaved; each group's partial is scaled by its scale.
// Split-K (KS > 1): owner rank of the cluster's i-th block is i mod KS; each
// rank's partial lands in its own slot of the owner's shared memory, and
// after one cluster barrier at the end the owners add the KS slots in rank
// order.  Deterministic (fixed orders, no atomics, no global workspace);
// every mbarrier wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kMmaMaxRanges = 14;  // consumer warps: 16 warps of at most 128 registers fill the register file
constexpr int kMmaMaxThreads = 32 * (2 + kMmaMaxRanges);
constexpr int kMmaMaxStages = 8;
constexpr int kMmaMaxCluster = 16;  // above the portable 8 only when K needs it
constexpr int kRangeBytes = 2048;   // one TMA box: 16 rows x 32 packed words
constexpr int kMmaBarrierBytes = 256;
constexpr int kPartialBytes = 512;  // one warp's (or CTA's) partial of a block and n-tile: 32 lanes x float4
constexpr int kRedBufs = 3;         // consumer partial buffers: consumers run up to 3 blocks ahead of the reducer
constexpr uint32_t kTailBytes = 1024;  // the half range of a block: 16 rows x 64 bytes

struct MmaParams {
  GemvArgs a;
  int KS;           // CTAs per cluster = K slices
  int R;            // ranges per rank (the last rank may have fewer) = consumer warps
  int Rb;           // ranges of the 3-D box: min(R, ranges of two groups)
  int S;            // ring stages
  int stage_bytes;  // Rb x 2048 (weights) [+ 1024: the half range] + scale rows of 16 weight rows, 1024-aligned
  int red_bytes;    // kRedBufs x R x NT x 512: consumer partials
  int part_bytes;   // owner slots (KS > 1): blocks owned x NT x KS x 512
};

// Not volatile: a pure function of its operands, so the compiler may
// interleave independent accumulator chains.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  const uint4 u = lds_u4(addr);
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

__device__ __forceinline__ void add4(float4& s, const float4 v) {
  s.x += v.x;
  s.y += v.y;
  s.z += v.z;
  s.w += v.w;
}

template <int NT>
__global__ void __launch_bounds__(kMmaMaxThreads, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_tail,
                    const __grid_constant__ MmaParams p) {
  constexpr int kCorrBytes = 64 * NT;  // a consumer warp's odd-lane corrections (two n-tiles): [group][nt][8] floats
  extern __shared__ __align__(1024) uint8_t smem[];
  const GemvArgs& a = p.a;
  const int KS = p.KS, S = p.S, R = p.R, Rb = p.Rb;
  const int rank = KS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster = blockIdx.x / KS;
  const int nclusters = gridDim.x / KS;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const int N = a.N;
  const int G = a.K / 128;
  const int nr = (G + 1) / 2;               // 256-k ranges
  const int nfull = G / 2;                  // ranges of two groups (the last one is half when G is odd)
  const int rb = rank * R;                  // this rank's ranges [rb, rb + nw)
  const int nw = (nr - rb < R ? nr - rb : R);
  const int nwf = nfull - rb < 0 ? 0 : (nfull - rb < nw ? nfull - rb : nw);  // full ones among them
  const bool has_tail = nwf < nw;           // the half range is this rank's last
  const int T16 = (N + 15) / 16;
  const int blk0 = static_cast<int>((static_cast<int64_t>(T16) * cluster) / nclusters);
  const int nblk = static_cast<int>((static_cast<int64_t>(T16) * (cluster + 1)) / nclusters) - blk0;

  // shared layout: barriers | consumer partials | corrections | owner slots | stages (1024-aligned)
  // stage: [16 rows][Rb ranges][128 bytes] swizzled | [16 rows][64 bytes] half range (odd G) | scale rows
  const uint32_t bar0 = smem_addr(smem);
  const uint32_t full0 = bar0;
  const uint32_t empty0 = bar0 + 8 * S;
  const uint32_t rfull0 = bar0 + 16 * S;
  const uint32_t rempty0 = rfull0 + 8 * kRedBufs;
  const uint32_t red0 = bar0 + kMmaBarrierBytes;
  const uint32_t corr0 = red0 + p.red_bytes;
  const uint32_t part0 = corr0 + static_cast<uint32_t>(R * kCorrBytes);
  const uint32_t stage0 = (part0 + p.part_bytes + 1023) & ~1023u;
  const uint32_t tail_off = static_cast<uint32_t>(Rb) * kRangeBytes;
  const uint32_t sc_off = tail_off + ((G & 1) ? kTailBytes : 0u);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, nw);
    }
    for (int b = 0; b < kRedBufs; ++b) {
      mbar_init(rfull0 + 8 * b, nw);
      mbar_init(rempty0 + 8 * b, 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  // Every CTA of the cluster must have started before shared memory of
  // another is written: the reducer waits for this before its first push.
  if (KS > 1) cluster_arrive_relaxed();
  pdl_launch_dependents();

  // A wait whose outcome every lane of the warp shares (the cluster barriers
  // at the end are executed by whole warps).
  auto warp_wait = [](uint32_t bar, uint32_t parity) {
    const bool r = mbar_wait_bounded(bar, parity, kWaitLimitNs);
    return __all_sync(0xffffffffu, r);
  };

  // lane's place in the mma fragments: row group g8 holds weight rows
  // pi, pi + 8 of the block; the two rows of a quarter-warp are d apart,
  // d Rb = 4 (mod 8)
  const int g8 = lane >> 2;
  const int t4 = lane & 3;
  const int pi = (Rb & 1) ? (((g8 & 1) << 2) | (g8 >> 1))                                // d = 4: 0 4 1 5 2 6 3 7
                          : ((Rb & 3) == 2 ? ((g8 & 4) | ((g8 & 1) << 1) | ((g8 >> 1) & 1))  // d = 2: 0 2 1 3 4 6 5 7
                                           : g8);                                        // d = 1

  // Where y[m][n] goes for every m: n's segment, pointer to its element of
  // activation row 0, row stride, bias (0 without); null past N.
  struct RowOut {
    uint16_t* y;
    int64_t ldy;
    float bias;
  };
  auto row_out = [&](int64_t n) {
    RowOut r{nullptr, 0, 0.f};
    if (n >= N) return r;
    int sg = 0;
    int64_t n0 = 0;
    if (a.nseg > 1 && n >= a.seg[0].n_end) {
      n0 = a.seg[0].n_end;
      sg = 1;
      if (a.nseg > 2 && n >= a.seg[1].n_end) {
        n0 = a.seg[1].n_end;
        sg = 2;
      }
    }
    r.y = a.seg[sg].y + (n - n0);
    r.ldy = a.seg[sg].ldy;
    if (a.seg[sg].bias != nullptr) r.bias = __half2float(__ushort_as_half(__ldg(a.seg[sg].bias + (n - n0))));
    return r;
  };
  // y of one block from the sums of lane's four fragment entries per
  // n-tile: rows pi, pi + 8 of the block, activation rows 8 nt + 2 t4, + 1;
  // y = fp16_RN(sum + bias)
  auto store_block = [&](int blk, const float4 (&v)[NT]) {
    const RowOut ra = row_out(16 * static_cast<int64_t>(blk) + pi);
    const RowOut rc = row_out(16 * static_cast<int64_t>(blk) + pi + 8);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int m0 = nt * 8 + 2 * t4;
      if (m0 < a.M) {
        if (ra.y) ra.y[m0 * ra.ldy] = __half_as_ushort(__float2half_rn(v[nt].x + ra.bias));
        if (rc.y) rc.y[m0 * rc.ldy] = __half_as_ushort(__float2half_rn(v[nt].z + rc.bias));
      }
      if (m0 + 1 < a.M) {
        if (ra.y) ra.y[(m0 + 1) * ra.ldy] = __half_as_ushort(__float2half_rn(v[nt].y + ra.bias));
        if (rc.y) rc.y[(m0 + 1) * rc.ldy] = __half_as_ushort(__float2half_rn(v[nt].w + rc.bias));
      }
    }
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const uint64_t pol_sc = policy_evict_normal();  // scale rows: every rank of the cluster reads them
      const uint32_t tx = (nwf > 0 ? static_cast<uint32_t>(Rb) * kRangeBytes : 0u) + (has_tail ? kTailBytes : 0u);
      bool ok = true;
      int i = 0;
      int s = 0;        // stage of block i
      uint32_t ph = 0;  // parity of the stage's round (i / S)
      uint32_t st = stage0;
      for (; i < nblk; ++i) {
        if (i >= S && !mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const int blk = blk0 + i;
        const uint32_t bar = full0 + 8 * s;
        // scale rows of the block: 16 rows x G fp16 (a whole multiple of 16
        // bytes except in a last block of fewer rows, whose last few bytes
        // are copied here before the barrier's arrival publishes them)
        const int rows = N - 16 * blk < 16 ? N - 16 * blk : 16;
        const uint32_t sc_bytes = static_cast<uint32_t>(rows) * G * 2;
        const uint32_t sc_bulk = sc_bytes & ~15u;
        const uint16_t* sc_src = a.scales + static_cast<int64_t>(blk) * 16 * G;
        for (uint32_t b = sc_bulk; b < sc_bytes; b += 2)
          sts_u16(st + sc_off + b, ld_nc_u16(sc_src + b / 2));
        mbar_arrive_expect_tx(bar, tx + sc_bulk);
        // checked build: the boxes start inside the matrix
        if (nwf > 0 && W4A16_IN(a.status, rb < nfull && 16 * blk < N))
          tma_load_3d(st, &tmap, 0, rb, 16 * blk, bar, pol);
        if (has_tail && W4A16_IN(a.status, 16 * (G - 1) < a.K / 8 && 16 * blk < N))
          tma_load_2d(st + tail_off, &tmap_tail, 16 * (G - 1), 16 * blk, bar, pol);
        if (sc_bulk > 0) bulk_g2s(st + sc_off, sc_src, sc_bulk, bar, pol_sc);
        st += p.stage_bytes;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
          st = stage0;
        }
      }
      if (!ok) {
        atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
        // the copies in flight land before the CTA may exit
        for (int j = i - S > 0 ? i - S : 0; j < i; ++j)
          mbar_wait_bounded(full0 + 8 * (j % S), (j / S) & 1, kWaitLimitNs);
      }
    }
    __syncwarp();
  } else if (warp >= 2) {
    // -------------------------------------------------------------- consumers
    const int w = warp - 2;
    const int rg = rb + w;  // this warp's range
    // TWO: a range of two groups; else the half range (one group) at the end
    // of a row with an odd group count.  Two copies of the loop, so that the
    // hot one tests nothing about it.
    auto consume = [&](auto two_tag) {
      constexpr bool TWO = decltype(two_tag)::value;
      constexpr int NG = TWO ? 2 : 1;
      pdl_wait();  // x may be the previous kernel's output
      // B fragments of the range: [nt][group jj][super-step j] =
      // {x0,x4} {x2,x6} {x1,x5} {x3,x7} of activation row 8 nt + g8 at
      // k = 128 (2 rg + jj) + 32 t4 + 8 j (zero past M); the odd-k halves
      // {x1,x5} {x3,x7} divided by 16 (unpack_mma leaves their weights as
      // 1152 + 16 q): exact in fp16 down to |x| = 2^-10, below it rounded to
      // a subnormal.
      const __half2 sixteenth = __half2half2(__ushort_as_half(0x2C00));
      uint4 bx[NT][NG][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int jj = 0; jj < NG; ++jj)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int m = nt * 8 + g8;
            const int k0 = 128 * (2 * rg + jj) + 32 * t4 + 8 * j;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m < a.M && W4A16_IN(a.status, k0 + 8 <= a.K)) v = ld_u4(a.x + m * a.ldx + k0);
            bx[nt][jj][j].x = __byte_perm(v.x, v.z, 0x5410);
            bx[nt][jj][j].y = __byte_perm(v.y, v.w, 0x5410);
            uint32_t o = __byte_perm(v.x, v.z, 0x7632);
            __half2 h = __hmul2(*reinterpret_cast<__half2*>(&o), sixteenth);
            bx[nt][jj][j].z = *reinterpret_cast<uint32_t*>(&h);
            o = __byte_perm(v.y, v.w, 0x7632);
            h = __hmul2(*reinterpret_cast<__half2*>(&o), sixteenth);
            bx[nt][jj][j].w = *reinterpret_cast<uint32_t*>(&h);
          }
      // What the biased odd lanes add per group: 1152 (x / 16) summed over
      // the group's odd k, for each activation row (FP32, exact products):
      // this lane's odd k, then the 4 lanes of row group g8.  Each block's
      // mma chains start from minus it, for the two activation rows of this
      // lane's D entries (8 nt + 2 t4, + 1): kept in registers with one
      // n-tile, in shared memory with two (registers are short there).
      float corr[NG][NT][2];
#pragma unroll
      for (int jj = 0; jj < NG; ++jj)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float c = 0.f;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            c += 1152.f * (half_lo(bx[nt][jj][j].z) + half_hi(bx[nt][jj][j].z));
            c += 1152.f * (half_lo(bx[nt][jj][j].w) + half_hi(bx[nt][jj][j].w));
          }
          c += __shfl_xor_sync(0xffffffffu, c, 1);
          c += __shfl_xor_sync(0xffffffffu, c, 2);
          if (NT == 1) {
            corr[jj][nt][0] = __shfl_sync(0xffffffffu, c, 8 * t4);
            corr[jj][nt][1] = __shfl_sync(0xffffffffu, c, 8 * t4 + 4);
          } else if (t4 == 0) {
            sts_f32(corr0 + static_cast<uint32_t>(w * kCorrBytes + ((jj * NT + nt) * 8 + g8) * 4), c);
          }
        }
      __syncwarp();
      const uint32_t corr_lane = corr0 + static_cast<uint32_t>(w * kCorrBytes + 8 * t4);
      // this lane's 16 bytes of rows pi and pi + 8 in a stage, per group
      const uint32_t line = static_cast<uint32_t>(pi * Rb + w);
      const uint32_t row_a = TWO ? line * 128 : tail_off + pi * 64;
      const uint32_t row_b = TWO ? row_a + 8 * Rb * 128 : row_a + 8 * 64;
      uint32_t chunk[NG];
#pragma unroll
      for (int jj = 0; jj < NG; ++jj)
        chunk[jj] = TWO ? ((static_cast<uint32_t>(4 * jj + t4) ^ (line & 7u)) << 4) : static_cast<uint32_t>(t4) << 4;
      const uint32_t sc_a = sc_off + 2 * (pi * G + 2 * rg);  // scale of row pi, group 2 rg
      const uint32_t sc_b = sc_a + 16 * G;                   // row pi + 8
      int s = 0;         // stage of block i
      uint32_t ph = 0;   // parity of its round
      uint32_t st = stage0;
      int b = 0;         // partial buffer of block i
      uint32_t rph = 0;  // parity of its round
      bool full_seen = false;  // block i's stage seen full at the end of block i - 1
      for (int i = 0; i < nblk; ++i) {
        if (!full_seen && !warp_wait(full0 + 8 * s, ph)) {
          if (lane == 0) atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
          break;
        }
        uint4 va[NG], vb[NG];
        float s_a[NG], s_b[NG];
#pragma unroll
        for (int jj = 0; jj < NG; ++jj) {
          va[jj] = lds_u4(st + row_a + chunk[jj]);
          vb[jj] = lds_u4(st + row_b + chunk[jj]);
          s_a[jj] = __half2float(__ushort_as_half(lds_u16(st + sc_a + 2 * jj)));
          s_b[jj] = __half2float(__ushort_as_half(lds_u16(st + sc_b + 2 * jj)));
        }
        // Accumulator chains: per group and n-tile, and with one n-tile the
        // two k-steps of a word apart too (four chains either way).  The
        // odd-k chain starts from minus the group's correction.
        constexpr int kH = NT == 1 ? 2 : 1;
        float d[kH][NG][NT][4];
#pragma unroll
        for (int jj = 0; jj < NG; ++jj)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            float c0, c1;
            if (NT == 1) {
              c0 = corr[jj][nt][0];
              c1 = corr[jj][nt][1];
            } else {
              const uint2 c = lds_u2(corr_lane + static_cast<uint32_t>((jj * NT + nt) * 32));
              c0 = __uint_as_float(c.x);
              c1 = __uint_as_float(c.y);
            }
            d[kH - 1][jj][nt][0] = -c0;
            d[kH - 1][jj][nt][1] = -c1;
            d[kH - 1][jj][nt][2] = -c0;
            d[kH - 1][jj][nt][3] = -c1;
            if (kH == 2) {
#pragma unroll
              for (int q = 0; q < 4; ++q) d[0][jj][nt][q] = 0.f;
            }
          }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          Unpacked qa[NG], qb[NG];
#pragma unroll
          for (int jj = 0; jj < NG; ++jj) {
            const uint32_t wa = j == 0 ? va[jj].x : (j == 1 ? va[jj].y : (j == 2 ? va[jj].z : va[jj].w));
            const uint32_t wb = j == 0 ? vb[jj].x : (j == 1 ? vb[jj].y : (j == 2 ? vb[jj].z : vb[jj].w));
            qa[jj] = unpack_mma(wa);
            qb[jj] = unpack_mma(wb);
          }
#pragma unroll
          for (int jj = 0; jj < NG; ++jj)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_16816(d[0][jj][nt], qa[jj].h0, qb[jj].h0, qa[jj].h2, qb[jj].h2, bx[nt][jj][j].x, bx[nt][jj][j].y);
#pragma unroll
          for (int jj = 0; jj < NG; ++jj)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_16816(d[kH - 1][jj][nt], qa[jj].h1, qb[jj].h1, qa[jj].h3, qb[jj].h3, bx[nt][jj][j].z,
                        bx[nt][jj][j].w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        st += p.stage_bytes;
        if (++s == S) {
          s = 0;
          ph ^= 1u;
          st = stage0;
        }
        // the block's partial: per D entry, the groups' sums times their scales
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v = 0.f;
#pragma unroll
            for (int jj = 0; jj < NG; ++jj) {
              const float g = kH == 2 ? d[0][jj][nt][q] + d[kH - 1][jj][nt][q] : d[0][jj][nt][q];
              v = fmaf(q < 2 ? s_a[jj] : s_b[jj], g, v);
            }
            acc[nt][q] = v;
          }
        if (i >= kRedBufs && !warp_wait(rempty0 + 8 * b, rph ^ 1u)) {
          if (lane == 0) atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
          break;
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t off = static_cast<uint32_t>(((b * R + w) * NT + nt) * kPartialBytes + 16 * lane);
          if (W4A16_IN(a.status, off + 16 <= static_cast<uint32_t>(p.red_bytes)))
            sts_u4(red0 + off, __float_as_uint(acc[nt][0]), __float_as_uint(acc[nt][1]),
                   __float_as_uint(acc[nt][2]), __float_as_uint(acc[nt][3]));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(rfull0 + 8 * b);
        if (++b == kRedBufs) {
          b = 0;
          rph ^= 1u;
        }
        full_seen = __all_sync(0xffffffffu, i + 1 < nblk && mbar_try_wait(full0 + 8 * s, ph));
      }
    };
    if (w < nwf)
      consume(std::true_type{});
    else if (w < nw)
      consume(std::false_type{});
  } else {
    // ---------------------------------------------------------------- reducer
    pdl_wait();  // y may still be read by the previous kernel
    if (KS > 1) cluster_wait();
    for (int i = 0; i < nblk; ++i) {
      const int b = i % kRedBufs;
      if (!warp_wait(rfull0 + 8 * b, (i / kRedBufs) & 1)) {
        if (lane == 0) atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
        break;
      }
      // all partials loaded, then summed in a fixed order:
      // (p0 + p2 + p4 + ...) + (p1 + p3 + ...)
      float4 v[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float4 part[kMmaMaxRanges];
#pragma unroll
        for (int w = 0; w < kMmaMaxRanges; ++w)
          if (w < nw) part[w] = lds_f4(red0 + static_cast<uint32_t>(((b * R + w) * NT + nt) * kPartialBytes + 16 * lane));
        float4 ve = part[0];
        float4 vo = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 1; w < kMmaMaxRanges; ++w)
          if (w < nw) add4((w & 1) ? vo : ve, part[w]);
        v[nt] = ve;
        add4(v[nt], vo);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty0 + 8 * b);
      if (KS == 1) {
        store_block(blk0 + i, v);
      } else {
        const uint32_t owner = static_cast<uint32_t>(i % KS);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t off =
              static_cast<uint32_t>((((i / KS) * NT + nt) * KS + rank) * kPartialBytes + 16 * lane);
          if (W4A16_IN(a.status, off + 16 <= static_cast<uint32_t>(p.part_bytes)))
            st_cluster_v4(map_to_rank(part0 + off, owner), v[nt]);
        }
      }
    }
  }

  if (KS > 1) {
    if (warp != 1) cluster_wait();
    cluster_sync();  // every rank's partials are in their owners' slots
    if (warp == 1) {
      for (int i = rank; i < nblk; i += KS) {
        float4 v[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          v[nt] = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int q = 0; q < KS; ++q)
            add4(v[nt], lds_f4(part0 + static_cast<uint32_t>((((i / KS) * NT + nt) * KS + q) * kPartialBytes +
                                                             16 * lane)));
        }
        store_block(blk0 + i, v);
      }
    }
  }
}

// ---------------------------------------------------------------- host side

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

namespace {

// Tensor maps of the packed weight (uint32 [N][K/8]).  view3: the two-group
// ranges of each row as [N][K/256][32 words], box 32 words x rb ranges x 16
// rows, 128-byte swizzle (ranges past the row's last two-group range read as
// zeros).  tail: [N][K/8] with a box of 16 words x 16 rows, no swizzle (the
// one-group range at the end of a row when K/128 is odd).
bool weight_tensor_maps(CUtensorMap* view3, CUtensorMap* tail, const uint32_t* qweight, int N, int K, int rb) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const int G = K / 128;
  *view3 = CUtensorMap{};
  *tail = CUtensorMap{};
  if (G / 2 > 0) {
    const cuuint64_t dims[3] = {32, static_cast<cuuint64_t>(G / 2), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(rb), 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(view3, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint32_t*>(qweight), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  if (G & 1) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    const cuuint32_t box[2] = {16, 16};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(tail, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(qweight), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// How many clusters of `ks` CTAs of this kernel (threads, smem bytes each)
// the GPU holds at once.  A cluster must fit inside one GPC, so large
// clusters can leave SMs idle.  Cached per device: the query is not free.
template <int NT>
int max_active_clusters(int ks, int threads, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, ks, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ks * 64);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemv_mma_kernel<NT>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

struct MmaPlan {
  int KS = 0, clusters = 0, R = 0, Rb = 0, S = 0, stage_bytes = 0, red_bytes = 0, part_bytes = 0, smem = 0;
};

// Choose the K split (cluster size).  Each split gives the ranks
// R = ceil(ranges / KS) ranges (at most kMmaMaxRanges warps; the last rank
// the rest, at least one), and as many
// clusters as the GPU holds at once share the 16-row blocks.  The critical
// path is the bytes the busiest CTA streams: blocks per cluster x (its
// ranges' weights + the blocks' scale rows); the smallest wins, ties going
// to the smaller split.  Every split needs a ring of at least 2 stages.
template <int NT>
MmaPlan make_mma_plan(const GemvArgs& a, const DeviceInfo& d, bool two_per_sm = false) {
  MmaPlan best{};
  int64_t best_cost = -1;
  const int G = a.K / 128;
  const int nr = (G + 1) / 2;
  const int T16 = (a.N + 15) / 16;
  const int cap = two_per_sm ? d.max_smem_optin / 2 - 1024 : d.max_smem_optin;
  const int rmax = two_per_sm ? kMmaMaxRanges / 2 : kMmaMaxRanges;
  const int sc_row_block = 16 * G * 2;  // scale bytes of a 16-row block
  for (int ks = 1; ks <= kMmaMaxCluster && ks <= nr; ++ks) {
    const int R = (nr + ks - 1) / ks;
    if (R > rmax || (ks - 1) * R >= nr) continue;
    const int Rb = R < G / 2 ? R : G / 2;
    const int stage = (Rb * kRangeBytes + ((G & 1) ? static_cast<int>(kTailBytes) : 0) + sc_row_block + 1023) & ~1023;
    const int red = kRedBufs * R * NT * kPartialBytes;
    const int threads = 32 * (2 + R);
    const int active = max_active_clusters<NT>(ks, threads, cap);
    if (active <= 0) continue;
    const int clusters = T16 < active ? T16 : active;
    const int nb = (T16 + clusters - 1) / clusters;  // blocks of the largest cluster
    const int part = ks > 1 ? ((nb + ks - 1) / ks) * NT * ks * kPartialBytes : 0;
    const int corr = R * 64 * NT;  // the consumer warps' odd-lane corrections
    const int avail = cap - kMmaBarrierBytes - red - corr - part - 1023;
    int S = avail / stage;
    if (S > kMmaMaxStages) S = kMmaMaxStages;
    if (S > nb) S = nb > 2 ? nb : 2;
    if (S < 2 || 16 * S + 16 * kRedBufs > kMmaBarrierBytes || avail < 2 * stage) continue;
    const int64_t cost = static_cast<int64_t>(nb) * (R * kRangeBytes + sc_row_block);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best.KS = ks;
      best.clusters = clusters;
      best.R = R;
      best.Rb = Rb;
      best.S = S;
      best.stage_bytes = stage;
      best.red_bytes = red;
      best.part_bytes = part;
      best.smem = kMmaBarrierBytes + red + corr + part + 1023 + S * stage;
    }
  }
  return best;
}

template <int NT>
cudaError_t launch_mma_nt(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  MmaPlan pl = make_mma_plan<NT>(a, d);
  // One n-tile (96 registers a thread): when K needs a cluster of ranks of
  // more than 7 ranges anyway (down, K = 18944: 6 ranks of 13), two CTAs of
  // half the warps and half the shared memory per SM, so that consecutive
  // launches overlap one's start with the other's end.  Measured (cold L2,
  // graphs of back-to-back calls): down M = 2, 4, 8 12.2, 12.4, 13.3 ->
  // 11.8, 11.9, 12.3 us; [gate;up] (one rank) and q (ranks of 5 ranges) were
  // slower that way and keep one CTA per SM.
  if (NT == 1 && pl.KS > 1 && pl.R > kMmaMaxRanges / 2) {
    const MmaPlan p2 = make_mma_plan<NT>(a, d, true);
    if (p2.KS != 0) pl = p2;
  }
  if (pl.KS == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap tmap, tmap_tail;
  if (!weight_tensor_maps(&tmap, &tmap_tail, a.qweight, a.N, a.K, pl.Rb)) return cudaErrorInvalidValue;
  MmaParams p;
  p.a = a;
  p.KS = pl.KS;
  p.R = pl.R;
  p.Rb = pl.Rb;
  p.S = pl.S;
  p.stage_bytes = pl.stage_bytes;
  p.red_bytes = pl.red_bytes;
  p.part_bytes = pl.part_bytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.clusters * pl.KS);
  cfg.blockDim = dim3(32 * (2 + pl.R));
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = pl.KS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_mma_kernel<NT>, tmap, tmap_tail, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool gemv_mma_supported(int K) {
  // ranges of a row split over at most kMmaMaxCluster ranks of kMmaMaxRanges
  return K > 0 && K % 128 == 0 && (K / 128 + 1) / 2 <= kMmaMaxCluster * kMmaMaxRanges;
}

cudaError_t launch_gemv_mma(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (a.M <= 8) return launch_mma_nt<1>(a, d, st);
  return launch_mma_nt<2>(a, d, st);
}

cudaError_t prepare_gemv_mma(const DeviceInfo& d) {
  if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
  const int limit = d.max_smem_optin;
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_mma_kernel<1>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemv_mma_kernel<2>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

}  // namespace w4a16
