// gemv_mma.cu -- small-batch GEMV for M = 8..16 on the tensor cores.
//
// Same operation as the other GEMV kernels ("Costruire un runtime di
// inference LLM da zero", "Tre bug che insegnano": INT4 group-128 weights x
// FP16 activations, FP32 accumulation).  From M = 8 on, each weight feeds
// eight or more products, so the contraction is dense enough for mma.sync
// m16n8k16 (f16 x f16 -> f32).  W is the A operand (16 rows per warp), the
// activations the B operand (8 activation rows per n-tile), so M = 16 is two
// n-tiles sharing every unpacked A fragment.
//
// Layout of the work.  A cluster of KS CTAs owns a contiguous range of
// 16-row blocks; CTA rank r of the cluster covers the r-th slice [gb, ge) of
// the K groups, so it stages only that slice of x (once, in fragment order)
// and reads every weight byte of its slice exactly once.
//   warp 0      producer.  Streams the cluster's rows, W blocks (16 W rows)
//               at a time, through an S-stage shared-memory ring with one
//               2-D TMA load per stage: a box of 16 W rows x 32 packed words
//               (two groups, 128 bytes per row), 128-byte swizzled, rows past
//               N filled with zeros by the copy.
//   warps 1..W  consumers.  Warp w takes rows 16 w .. 16 w + 15 of each box;
//               lane (g, t) reads the 16 bytes of its rows g' = pi(g) and
//               g' + 8 at word offset 4 t of each group (pi = 0 4 1 5 2 6 3 7
//               puts the 8 lanes of every quarter-warp load on 8 distinct
//               swizzled 16-byte chunks: no bank conflicts).  Word j of those
//               16 bytes is super-step j: its exact-q halves {q0,q4},{q2,q6}
//               are the A registers of one mma and {q1,q5},{q3,q7} those of a
//               second (the order of k inside a contraction is free; the
//               staged B fragments follow it).  Per group the mma partial is
//               scaled by the group scales (read through L1) and added to
//               FP32 accumulators that stay in registers over the K slice.
// Split-K reduction.  Each CTA keeps its partial sums of every row of a pass
// (a bounded number of the cluster's blocks) in shared memory; after the
// pass the cluster synchronises and rank r finalises the entries r, r + KS,
// ... by summing the KS partials through distributed shared memory in rank
// order (deterministic, no atomics, no global workspace).  With KS = 1 the
// consumers write y directly.  Every wait is bounded.
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

constexpr int kMmaMaxW = 16;            // consumer warps (16-row blocks per box)
constexpr int kMmaThreads = 32 * (kMmaMaxW + 1);
constexpr int kBoxWords = 32;           // box width: 32 packed words = 2 groups = 128 bytes
constexpr int kMmaMaxStages = 8;
constexpr int kMmaBarrierBytes = 256;   // [full S][empty S]

struct MmaParams {
  GemvArgs a;
  int KS;            // CTAs per cluster = K slices
  int W;             // consumer warps = 16-row blocks per box
  int S;             // ring stages
  int pass_blocks;   // 16-row blocks per reduction pass (KS > 1)
  int x_bytes;       // bytes of the staged B fragments (max over ranks)
  int part_bytes;    // bytes of the partial buffer (KS > 1)
  int sc_bytes;      // bytes of the per-warp scale buffers (W x 16 rows x groups of a slice)
};

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

template <int NT>
__global__ void __launch_bounds__(kMmaThreads, 1)
    gemv_mma_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ MmaParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const GemvArgs& a = p.a;
  const int KS = p.KS, W = p.W, S = p.S;
  const int rank = KS > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster = blockIdx.x / KS;
  const int nclusters = gridDim.x / KS;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;

  const int N = a.N;
  const int G = a.K / 128;
  const int T16 = (N + 15) / 16;
  const int blk_begin = static_cast<int>((static_cast<int64_t>(T16) * cluster) / nclusters);
  const int blk_end = static_cast<int>((static_cast<int64_t>(T16) * (cluster + 1)) / nclusters);
  const int gb = (G * rank) / KS;
  const int ge = (G * (rank + 1)) / KS;
  const int box_first = gb / 2;                   // boxes covering groups [gb, ge)
  const int box_last = ge > gb ? (ge - 1) / 2 : box_first - 1;
  const int nbox = box_last - box_first + 1;
  const int pass_blocks = KS > 1 ? p.pass_blocks : (blk_end - blk_begin);

  // shared layout: barriers | B fragments | partials | scales | stages (1024-aligned)
  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t xf0 = full0 + kMmaBarrierBytes;
  const uint32_t part0 = xf0 + p.x_bytes;
  const uint32_t sc0 = part0 + p.part_bytes;
  const uint32_t stage0 = (sc0 + p.sc_bytes + 1023) & ~1023u;
  const uint32_t stage_bytes = 16 * W * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, W);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int s = 0, g = 0;
    uint32_t phase = 0;
    bool ok = true;
    // After a failed wait the producer issues nothing more but still takes
    // part in every cluster barrier, so no CTA of the cluster waits forever.
    for (int pb = blk_begin; pb < blk_end; pb += pass_blocks) {
      const int pe = pb + pass_blocks < blk_end ? pb + pass_blocks : blk_end;
      for (int cb = pb; cb < pe && ok; cb += W) {
        for (int b = 0; b < nbox; ++b) {
          if (g >= S && !mbar_wait_bounded(empty0 + 8 * s, phase ^ 1u, kWaitLimitNs)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            const uint32_t bar = full0 + 8 * s;
            // checked build: the box starts inside the matrix (TMA fills the
            // part of a box past the matrix with zeros)
            const bool in = W4A16_IN(a.status, (box_first + b) * kBoxWords < a.K / 8 && cb * 16 < a.N);
            mbar_arrive_expect_tx(bar, in ? stage_bytes : 0u);
            if (in) tma_load_2d(stage0 + s * stage_bytes, &tmap, (box_first + b) * kBoxWords, cb * 16, bar, pol);
          }
          __syncwarp();
          ++g;
          if (++s == S) {
            s = 0;
            phase ^= 1u;
          }
        }
      }
      if (KS > 1) {
        cluster_sync();  // the pass's partials have been pushed to their owners
        if (pe < blk_end) cluster_sync();  // and summed: the buffers may be reused
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
      for (int v = 0; v < S; ++v) {
        const int gg = g - S + v;
        if (gg >= 0) mbar_wait_bounded(full0 + 8 * ((s + v) % S), (gg / S) & 1, kWaitLimitNs);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int w = warp - 1;
  const int g8 = lane >> 2;  // fragment row group
  const int t4 = lane & 3;   // thread in group
  const int pi = ((g8 & 1) << 2) | (g8 >> 1);  // 0 4 1 5 2 6 3 7
  const int ct = threadIdx.x - 32;              // consumer thread index
  const int nct = 32 * W;

  const int ngs = ge - gb;  // groups of this rank's slice
  const uint16_t* scales = a.scales;
  // Scales of a warp's 16 rows x the slice's groups go to its own buffer:
  // [row in block][group - gb] fp16 (rows past N read row N - 1).  The
  // loads are issued in batches of 16 per lane before any of them is used.
  auto stage_scales = [&](int blk, uint32_t scw) {
    for (int i0 = lane; i0 < 16 * ngs; i0 += 16 * 32) {
      uint16_t v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int i = i0 + 32 * q;
        const int r = blk * 16 + i / ngs;
        v[q] = i < 16 * ngs ? ld_nc_u16(scales + static_cast<int64_t>(r < N ? r : N - 1) * G + gb + i % ngs)
                            : static_cast<uint16_t>(0);
      }
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (i0 + 32 * q < 16 * ngs) sts_u16(scw + 2 * (i0 + 32 * q), v[q]);
    }
  };
  const uint32_t scw = sc0 + static_cast<uint32_t>(w * 16 * ngs) * 2;
  // the first chunk's scales (weights and scales are constant: no need to
  // wait for the previous kernel)
  if (blk_begin + w < (blk_begin + pass_blocks < blk_end ? blk_begin + pass_blocks : blk_end))
    stage_scales(blk_begin + w, scw);

  pdl_wait();  // x may be the previous kernel's output
  // ---- stage this rank's slice of x as B fragments:
  // [group][nt][super-step j][lane] x 16 bytes = {x0,x4} {x2,x6} {x1,x5} {x3,x7}
  // of column m = 8 nt + lane / 4, k = 128 group + 32 (lane % 4) + 8 j
  {
    const int entries = (ge - gb) * NT * 4 * 32;
    constexpr int kBatch = 8;  // loads in flight per thread
    for (int e0 = ct; e0 < entries; e0 += kBatch * nct) {
      uint4 v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int e = e0 + i * nct;
        const int ln = e & 31;
        const int j = (e >> 5) & 3;
        const int nt = (e >> 7) % NT;
        const int gl = (e >> 7) / NT;
        const int m = nt * 8 + (ln >> 2);
        const int k0 = (gb + gl) * 128 + 32 * (ln & 3) + 8 * j;
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (e < entries && m < a.M && W4A16_IN(a.status, k0 + 8 <= a.K && 16 * e + 16 <= p.x_bytes))
          v[i] = ld_u4(a.x + m * a.ldx + k0);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int e = e0 + i * nct;
        if (e >= entries) break;
        uint4 f;
        f.x = __byte_perm(v[i].x, v[i].z, 0x5410);  // {x0, x4}
        f.y = __byte_perm(v[i].y, v[i].w, 0x5410);  // {x2, x6}
        f.z = __byte_perm(v[i].x, v[i].z, 0x7632);  // {x1, x5}
        f.w = __byte_perm(v[i].y, v[i].w, 0x7632);  // {x3, x7}
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xf0 + 16 * e), "r"(f.x), "r"(f.y),
                     "r"(f.z), "r"(f.w)
                     : "memory");
      }
    }
  }
  named_sync(1, nct);

  int s = 0;
  uint32_t phase = 0;
  // after a failed wait the warp computes nothing more but still takes part
  // in every cluster barrier
  bool ok = true;
  for (int pb = blk_begin; pb < blk_end; pb += pass_blocks) {
    const int pe = pb + pass_blocks < blk_end ? pb + pass_blocks : blk_end;
    for (int cb = pb; cb < pe; cb += W) {
      // rows of this warp in the box: 16 w + pi and 16 w + pi + 8
      const int blk = cb + w;
      const int ra = blk * 16 + pi;
      const int rb = ra + 8;
      const bool live = blk < pe;  // block inside the pass (rows < N checked at the store)
      float acc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
      // scales of this chunk (the first chunk's were staged up front)
      if (live && cb != blk_begin) {
        __syncwarp();  // the previous chunk's scales have been read
        stage_scales(blk, scw);
      }
      __syncwarp();
      for (int b = 0; b < nbox; ++b) {
        if (ok && !mbar_wait_bounded(full0 + 8 * s, phase, kWaitLimitNs)) {
          if (lane == 0) atomicOr(a.status, W4A16_DEV_PIPE_TIMEOUT);
          ok = false;
        }
        const uint32_t base = stage0 + s * stage_bytes + (16 * w + pi) * 128;
        if (live && ok) {
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int grp = 2 * (box_first + b) + jj;
            if (grp < gb || grp >= ge) continue;  // the other rank's half of a shared box
            const int c = ((4 * jj + t4) ^ pi) << 4;
            const uint4 va = lds_u4(base + c);
            const uint4 vb = lds_u4(base + 8 * 128 + c);
            const float s_a = __half2float(__ushort_as_half(lds_u16(scw + 2 * (pi * ngs + grp - gb))));
            const float s_b = __half2float(__ushort_as_half(lds_u16(scw + 2 * ((pi + 8) * ngs + grp - gb))));
            float d[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) d[nt][q] = 0.f;
            const uint32_t wa4[4] = {va.x, va.y, va.z, va.w};
            const uint32_t wb4[4] = {vb.x, vb.y, vb.z, vb.w};
            const uint32_t xg = xf0 + static_cast<uint32_t>(grp - gb) * NT * 4 * 32 * 16 + 16 * lane;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const Unpacked qa = unpack_exact(wa4[j]);
              const Unpacked qb = unpack_exact(wb4[j]);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const uint4 bf = lds_u4(xg + (nt * 4 + j) * 32 * 16);
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
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(empty0 + 8 * s);
        if (++s == S) {
          s = 0;
          phase ^= 1u;
        }
      }
      // D layout: d[0], d[1] = row g', columns 2 t, 2 t + 1; d[2], d[3] = row g' + 8
      if (live) {
        if (KS == 1) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int m0 = nt * 8 + 2 * t4;
            if (ra < N) {
              if (m0 < a.M) store_out(a, m0, ra, acc[nt][0]);
              if (m0 + 1 < a.M) store_out(a, m0 + 1, ra, acc[nt][1]);
            }
            if (rb < N) {
              if (m0 < a.M) store_out(a, m0, rb, acc[nt][2]);
              if (m0 + 1 < a.M) store_out(a, m0 + 1, rb, acc[nt][3]);
            }
          }
        } else {
          // Entry e = (row - 16 pb) 8 NT + m of the pass belongs to rank
          // e mod KS; its partial from rank q goes to slot (e / KS) KS + q of
          // the owner's buffer (remote stores, no waiting on them).
          auto push = [&](int row, int m, float v) {
            const int e = (row - 16 * pb) * 8 * NT + m;
            const uint32_t local = part0 + 4 * static_cast<uint32_t>((e / KS) * KS + rank);
            if (W4A16_IN(a.status, 4 * ((e / KS) * KS + rank) + 4 <= p.part_bytes))
              st_cluster_f32(map_to_rank(local, static_cast<uint32_t>(e % KS)), v);
          };
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int m0 = nt * 8 + 2 * t4;
            push(ra, m0, acc[nt][0]);
            push(ra, m0 + 1, acc[nt][1]);
            push(rb, m0, acc[nt][2]);
            push(rb, m0 + 1, acc[nt][3]);
          }
        }
      }
    }
    if (KS > 1) {
      cluster_sync();  // every rank's partials of the pass have arrived at their owners
      const int per_row = 8 * NT;
      const int total = (pe - pb) * 16 * per_row;
      // this rank owns entries e = rank, rank + KS, ...: sum the KS slots of
      // each in rank order (local shared memory only)
      for (int i = ct; i * KS + rank < total; i += nct) {
        const int e = i * KS + rank;
        const int row = e / per_row;
        const int m = e % per_row;
        const int n = 16 * pb + row;
        if (m >= a.M || n >= N) continue;
        const uint32_t addr = part0 + 4 * static_cast<uint32_t>(i * KS);
        float v = 0.f;
        for (int q = 0; q < KS; ++q) v += lds_f32(addr + 4 * q);
        store_out(a, m, n, v);
      }
      if (pe < blk_end) cluster_sync();  // the buffers may be rewritten by the next pass
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

// Tensor map of the packed weight as uint32 [N][K/8], box 32 words x rows,
// 128-byte swizzle.
bool weight_tensor_map(CUtensorMap* m, const uint32_t* qweight, int N, int K, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K / 8), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 8) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kBoxWords), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(qweight), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// How many clusters of `ks` CTAs of this kernel the GPU holds at once
// (clusters must fit inside one GPC, so large clusters can leave SMs idle).
// Cached per device: the query is not free.
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
  cfg.blockDim = dim3(kMmaThreads);
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
  int KS = 0, clusters = 0, W = 0, S = 0, pass_blocks = 0, x_bytes = 0, part_bytes = 0, sc_bytes = 0, smem = 0;
};

// Choose the K split (cluster size): every rank's x slice must fit next to a
// ring of at least 3 stages; among those, keep the most SMs streaming with
// enough warps (clusters x ranks x min(8, blocks per cluster)), then the
// smaller split.
template <int NT>
MmaPlan make_mma_plan(const GemvArgs& a, const DeviceInfo& d) {
  MmaPlan best{};
  int64_t best_score = -1;
  const int T16 = (a.N + 15) / 16;
  const int G = a.K / 128;
  const int smem_cap = d.max_smem_optin;
  // any cluster size up to the portable 8: a GPC holds a whole number of
  // clusters, so sizes that are not powers of two can cover more SMs
  for (int ks = 1; ks <= 8 && ks <= G; ++ks) {
    const int x_bytes = ((G + ks - 1) / ks) * NT * 4 * 32 * 16;
    const int active = max_active_clusters<NT>(ks, smem_cap);
    if (active <= 0) continue;
    const int clusters = T16 < active ? T16 : active;
    const int blocks = (T16 + clusters - 1) / clusters;  // per cluster (upper bound)
    const int W = blocks < kMmaMaxW ? blocks : kMmaMaxW;
    const int stage = 16 * W * 128;
    // partials of one pass: pass_blocks x 16 rows x 8 NT floats (KS > 1)
    int pass_blocks = ks > 1 ? blocks : 0;
    int avail = smem_cap - kMmaBarrierBytes - 1024 - x_bytes;
    if (ks > 1) {
      const int per_block = 16 * 8 * NT * 4;
      const int max_pb = (avail - 3 * stage - ks * 4) / per_block;
      if (max_pb < W) continue;
      if (pass_blocks > max_pb) pass_blocks = max_pb / W * W;
    }
    // owner slots: ceil(entries / ks) x ks floats
    const int part_bytes = ((pass_blocks * 16 * 8 * NT + ks - 1) / ks) * ks * 4;
    const int sc_bytes = (W * 16 * ((G + ks - 1) / ks) * 2 + 15) & ~15;
    avail -= part_bytes + sc_bytes;
    int S = avail / stage;
    if (S > kMmaMaxStages) S = kMmaMaxStages;
    if (S < 3) continue;
    // SMs streaming, each with up to 8 busy warps (enough to keep its share
    // of the bandwidth); ties go to the smaller split
    const int64_t score = static_cast<int64_t>(clusters) * ks * (W < 8 ? W : 8);
    if (score > best_score) {
      best_score = score;
      best.KS = ks;
      best.clusters = clusters;
      best.W = W;
      best.S = S;
      best.pass_blocks = pass_blocks;
      best.x_bytes = x_bytes;
      best.part_bytes = part_bytes;
      best.sc_bytes = sc_bytes;
      best.smem = kMmaBarrierBytes + x_bytes + part_bytes + sc_bytes + 1023 + S * stage;
    }
  }
  return best;
}

template <int NT>
cudaError_t launch_mma_nt(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  const MmaPlan pl = make_mma_plan<NT>(a, d);
  if (pl.KS == 0) return cudaErrorInvalidConfiguration;
  CUtensorMap tmap;
  if (!weight_tensor_map(&tmap, a.qweight, a.N, a.K, 16 * pl.W)) return cudaErrorInvalidValue;
  MmaParams p;
  p.a = a;
  p.KS = pl.KS;
  p.W = pl.W;
  p.S = pl.S;
  p.pass_blocks = pl.pass_blocks;
  p.x_bytes = pl.x_bytes;
  p.part_bytes = pl.part_bytes;
  p.sc_bytes = pl.sc_bytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.clusters * pl.KS);
  cfg.blockDim = dim3(32 * (pl.W + 1));
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_mma_kernel<NT>, tmap, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_mma(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (a.M <= 8) return launch_mma_nt<1>(a, d, st);
  return launch_mma_nt<2>(a, d, st);
}

cudaError_t prepare_gemv_mma(const DeviceInfo& d) {
  if (tensor_map_encoder() == nullptr) return cudaErrorNotSupported;
  const int limit = d.max_smem_optin;
  cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_mma_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
}

}  // namespace w4a16
