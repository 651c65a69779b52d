// gemv_mma.cu -- small-batch GEMV for M = 8..16 on the tensor cores.
//
// Same operation as the other GEMV kernels ("Costruire un runtime di
// inference LLM da zero", "Tre bug che insegnano": INT4 group-128 weights x
// FP16 activations, FP32 accumulation).  From M = 8 on, each weight feeds
// eight or more products, so the contraction is dense enough for mma.sync
// m16n8k16 (f16 x f16 -> f32).  W is the A operand (16 rows per tile), the
// activations the B operand (8 activation rows per n-tile), so M = 16 is two
// n-tiles sharing every unpacked A fragment.
//
// Fragment mapping.  Lane (g = lane / 4, t = lane % 4) of a warp loads, for
// each group of 128 k, the 16 bytes (4 packed words, 32 k) at word offset 4t
// of rows g and g + 8 of its tile.  Word j of those 16 bytes is super-step j:
// its exact-q halves {q0,q4},{q2,q6} are the A registers of one mma and
// {q1,q5},{q3,q7} those of a second (the order of k inside a contraction is
// free; B is laid out to match).  The activations are staged once per CTA in
// shared memory in exactly that order, so lane (g, t) fetches its B
// fragments of a super-step with one conflict-free 16-byte load.
//
// Split-K.  A cluster of KS CTAs (KS in 1..8) shares a set of 16-row tiles;
// CTA rank r covers the r-th slice of the K groups.  Each warp owns one tile
// at a time and streams its rows' packed words with 16-byte loads, PD groups
// ahead.  Per group the mma partial is scaled by the group scales and added to
// FP32 accumulators.  After each round of tiles (one per warp) the KS partial
// tiles are summed through distributed shared memory in rank order
// (deterministic, no atomics, no global workspace) and written as fp16.
#include <cuda_fp16.h>

#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kMmaMaxWarps = 16;
constexpr int kPD = 4;  // groups in flight per warp

struct MmaPlan {
  int KS;        // CTAs per cluster = K slices
  int clusters;  // number of clusters
  int warps;     // warps per CTA
  int max_tiles; // tiles per cluster (upper bound)
  int max_groups;  // groups per K slice (upper bound)
  int smem;      // bytes
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct MmaParams {
  GemvArgs a;
  int KS, max_tiles, max_groups;
};

template <int NT>
__global__ void __launch_bounds__(kMmaMaxWarps * 32) gemv_mma_kernel(const MmaParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const GemvArgs& a = p.a;
  const int KS = p.KS;
  const int rank = KS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster = blockIdx.x / KS;
  const int nclusters = gridDim.x / KS;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g8 = lane >> 2;  // fragment row group
  const int t4 = lane & 3;   // thread in group

  const int64_t N = a.N;
  const int K = a.K;
  const int NG = K / 128;
  const int64_t T16 = (N + 15) / 16;
  const int64_t tile_begin = (T16 * cluster) / nclusters;
  const int64_t tile_end = (T16 * (cluster + 1)) / nclusters;
  const int ntiles = static_cast<int>(tile_end - tile_begin);
  const int gb = (NG * rank) / KS;
  const int ge = (NG * (rank + 1)) / KS;
  const int ng = ge - gb;

  // shared memory: B fragments [ng][NT][4 super-steps][32 lanes] x 16 B, then
  // one partial tile per warp [warps][16 rows][8 NT] f32
  uint4* xf = reinterpret_cast<uint4*>(smem);
  float* part = reinterpret_cast<float*>(smem + static_cast<size_t>(p.max_groups) * NT * 4 * 32 * 16);

  pdl_launch_dependents();
  pdl_wait();  // x may be the previous kernel's output

  // ---- stage the activations of this K slice in fragment order
  {
    const int entries = ng * NT * 4 * 32;
    for (int e = threadIdx.x; e < entries; e += blockDim.x) {
      const int ln = e & 31;
      const int j = (e >> 5) & 3;
      const int nt = (e >> 7) % NT;
      const int gl = (e >> 7) / NT;
      const int m = nt * 8 + (ln >> 2);
      const int k0 = (gb + gl) * 128 + 32 * (ln & 3) + 8 * j;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (m < a.M) v = *reinterpret_cast<const uint4*>(a.x + m * a.ldx + k0);
      uint4 f;
      f.x = __byte_perm(v.x, v.z, 0x5410);  // {x0, x4}
      f.y = __byte_perm(v.y, v.w, 0x5410);  // {x2, x6}
      f.z = __byte_perm(v.x, v.z, 0x7632);  // {x1, x5}
      f.w = __byte_perm(v.y, v.w, 0x7632);  // {x3, x7}
      xf[e] = f;
    }
  }
  __syncthreads();

  const int wpr = K / 8;
  const int rounds = (ntiles + nwarps - 1) / nwarps;
  for (int round = 0; round < rounds; ++round) {
  const int lt = round * nwarps + warp;
  if (lt < ntiles) {
    const int64_t tile = tile_begin + lt;
    const int64_t ra = tile * 16 + g8;
    const int64_t rb = ra + 8;
    const int64_t ra_c = ra < N ? ra : N - 1;  // in-bounds reads for ragged tiles
    const int64_t rb_c = rb < N ? rb : N - 1;
    const uint32_t* wa = a.qweight + ra_c * wpr + 4 * t4;
    const uint32_t* wb = a.qweight + rb_c * wpr + 4 * t4;
    const uint16_t* sa = a.scales + ra_c * NG;
    const uint16_t* sb = a.scales + rb_c * NG;

    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;

    uint4 ring_a[kPD], ring_b[kPD];
    uint16_t ring_sa[kPD], ring_sb[kPD];
#pragma unroll
    for (int i = 0; i < kPD; ++i) {
      if (i < ng) {
        ring_a[i] = ld_stream_u4(wa + (gb + i) * 16);
        ring_b[i] = ld_stream_u4(wb + (gb + i) * 16);
        ring_sa[i] = ld_nc_u16(sa + gb + i);
        ring_sb[i] = ld_nc_u16(sb + gb + i);
      }
    }
    for (int gl0 = 0; gl0 < ng; gl0 += kPD) {
#pragma unroll
      for (int i = 0; i < kPD; ++i) {
        const int gl = gl0 + i;
        if (gl < ng) {
          const uint4 va = ring_a[i];
          const uint4 vb = ring_b[i];
          const float s_a = __half2float(__ushort_as_half(ring_sa[i]));
          const float s_b = __half2float(__ushort_as_half(ring_sb[i]));
          if (gl + kPD < ng) {
            ring_a[i] = ld_stream_u4(wa + (gb + gl + kPD) * 16);
            ring_b[i] = ld_stream_u4(wb + (gb + gl + kPD) * 16);
            ring_sa[i] = ld_nc_u16(sa + gb + gl + kPD);
            ring_sb[i] = ld_nc_u16(sb + gb + gl + kPD);
          }
          float d[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) d[nt][q] = 0.f;
          const uint32_t wa4[4] = {va.x, va.y, va.z, va.w};
          const uint32_t wb4[4] = {vb.x, vb.y, vb.z, vb.w};
          const uint4* xg = xf + static_cast<size_t>(gl) * NT * 4 * 32;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const Unpacked qa = unpack_exact(wa4[j]);
            const Unpacked qb = unpack_exact(wb4[j]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 bf = xg[(nt * 4 + j) * 32 + lane];
              mma_16816(d[nt], qa.h0, qb.h0, qa.h2, qb.h2, bf.x, bf.y);
              mma_16816(d[nt], qa.h1, qb.h1, qa.h3, qb.h3, bf.z, bf.w);
            }
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[nt][0] = fmaf(s_a, d[nt][0], acc[nt][0]);
            acc[nt][1] = fmaf(s_a, d[nt][1], acc[nt][1]);
            acc[nt][2] = fmaf(s_b, d[nt][2], acc[nt][2]);
            acc[nt][3] = fmaf(s_b, d[nt][3], acc[nt][3]);
          }
        }
      }
    }

    // D layout: d[0], d[1] = row g8, columns (m) 2 t4, 2 t4 + 1; d[2], d[3] = row g8 + 8
    if (KS == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int m0 = nt * 8 + 2 * t4;
        if (ra < N) {
          if (m0 < a.M) *out_ptr(a, m0, ra) = __half_as_ushort(__float2half_rn(acc[nt][0]));
          if (m0 + 1 < a.M) *out_ptr(a, m0 + 1, ra) = __half_as_ushort(__float2half_rn(acc[nt][1]));
        }
        if (rb < N) {
          if (m0 < a.M) *out_ptr(a, m0, rb) = __half_as_ushort(__float2half_rn(acc[nt][2]));
          if (m0 + 1 < a.M) *out_ptr(a, m0 + 1, rb) = __half_as_ushort(__float2half_rn(acc[nt][3]));
        }
      }
    } else {
      float* pt = part + static_cast<size_t>(warp) * 16 * (8 * NT);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int m0 = nt * 8 + 2 * t4;
        pt[g8 * (8 * NT) + m0] = acc[nt][0];
        pt[g8 * (8 * NT) + m0 + 1] = acc[nt][1];
        pt[(g8 + 8) * (8 * NT) + m0] = acc[nt][2];
        pt[(g8 + 8) * (8 * NT) + m0 + 1] = acc[nt][3];
      }
    }
  }  // lt < ntiles
  if (KS > 1) {
    cluster_sync();  // every rank's partial tiles of this round are complete and visible
    const int per_tile = 16 * 8 * NT;
    const int in_round = (ntiles - round * nwarps) < nwarps ? (ntiles - round * nwarps) : nwarps;
    const int total = in_round * per_tile;
    // rank r finalises entries r, r + KS, ... ; sums the ranks in order 0..KS-1
    for (int e = rank + KS * static_cast<int>(threadIdx.x); e < total; e += KS * static_cast<int>(blockDim.x)) {
      const int w = e / per_tile;
      const int rem = e % per_tile;
      const int row = rem / (8 * NT);
      const int m = rem % (8 * NT);
      const int64_t n = (tile_begin + round * nwarps + w) * 16 + row;
      if (m >= a.M || n >= N) continue;
      const uint32_t addr = smem_addr(part + e);
      float v = 0.f;
      for (int q = 0; q < KS; ++q) v += ld_cluster_f32(map_to_rank(addr, q));
      *out_ptr(a, m, n) = __half_as_ushort(__float2half_rn(v));
    }
    cluster_sync();  // partials may be overwritten (next round) or freed (exit) only now
  }
  }  // rounds
}

// How many clusters of `ks` CTAs (16 warps, `smem` bytes each) the GPU can
// hold at once: clusters must fit inside one GPC, so large clusters can leave
// SMs idle.  Cached, the query is not free.
template <int NT>
int max_active_clusters(int ks, int smem) {
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
  cfg.blockDim = dim3(kMmaMaxWarps * 32);
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

// Choose the K split (cluster size) that keeps the most warps streaming: the
// SMs the co-resident clusters cover, times the warps (tiles) per CTA, capped
// at 12 warps (enough bytes in flight per SM).
template <int NT>
MmaPlan make_mma_plan(const GemvArgs& a, const DeviceInfo& d) {
  MmaPlan best{};
  int64_t best_score = -1;
  const int64_t T16 = (static_cast<int64_t>(a.N) + 15) / 16;
  const int NG = a.K / 128;
  const int smem_cap = d.max_smem_optin - 1024;
  for (int ks = 1; ks <= 8 && ks <= NG; ks *= 2) {
    const int max_groups = (NG + ks - 1) / ks;
    const int smem = max_groups * NT * 4 * 32 * 16 + (ks > 1 ? kMmaMaxWarps * 16 * 8 * NT * 4 : 0);
    if (smem > smem_cap) continue;
    const int active = max_active_clusters<NT>(ks, smem);
    if (active <= 0) continue;
    const int64_t clusters = T16 < active ? T16 : active;
    const int64_t max_tiles = (T16 + clusters - 1) / clusters;
    const int warps = static_cast<int>(max_tiles < kMmaMaxWarps ? max_tiles : kMmaMaxWarps);
    const int64_t score = clusters * ks * (warps < 12 ? warps : 12);
    if (score > best_score) {
      best_score = score;
      best.KS = ks;
      best.clusters = static_cast<int>(clusters);
      best.max_tiles = static_cast<int>(max_tiles);
      best.max_groups = max_groups;
      best.smem = smem;
      best.warps = warps;
    }
  }
  return best;
}

template <int NT>
cudaError_t launch_mma_nt(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  const MmaPlan pl = make_mma_plan<NT>(a, d);
  if (pl.KS == 0) return cudaErrorInvalidConfiguration;
  MmaParams p;
  p.a = a;
  p.KS = pl.KS;
  p.max_tiles = pl.max_tiles;
  p.max_groups = pl.max_groups;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.clusters * pl.KS);
  cfg.blockDim = dim3(pl.warps * 32);
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_mma_kernel<NT>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_mma(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (a.M <= 8) return launch_mma_nt<1>(a, d, st);
  return launch_mma_nt<2>(a, d, st);
}

cudaError_t prepare_gemv_mma(const DeviceInfo& d) {
  const int limit = d.max_smem_optin;
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
}

}  // namespace w4a16
