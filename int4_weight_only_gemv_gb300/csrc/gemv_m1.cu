// gemv_m1.cu -- the M = 1 decode GEMV: a persistent, TMA-fed, warp-specialised
// CUDA-core kernel.
//
// The operation is the INT4 x FP16 GEMV of "Costruire un runtime di inference
// LLM da zero" (datastack.it), section "Tre bug che insegnano", third bug
// (gate/up/down GEMVs unpack INT4 in-kernel against FP16 activations), with
// the group-128 symmetric format of the same section's last paragraph.
//
// Design (one CTA per SM, one pass over the weight stream):
//   warp 0      producer.  Streams tiles of RB consecutive rows into an
//               S-stage shared-memory ring with 1-D bulk copies (the tile's
//               rows are contiguous in memory: one copy, plus one for the
//               tile's scale window), completing on a per-stage mbarrier, and
//               refills a stage as soon as the consumers hold its tile in
//               registers.
//   warp 1      reducer.  Sums the consumers' per-unit partials of each tile
//               in a fixed order and writes y.
//   warps 1..   consumers.  Consumer thread c owns unit u = c mod U (64
//               consecutive k, half a group) of rows c / U + r RL (r < kRR)
//               of every tile, so its 64 activations stay in registers for
//               the whole kernel and no activation traffic touches shared
//               memory.  Per packed word
//               it does one shift, four LOP3s (nibble -> biased fp16, see
//               ptx.cuh) and eight f16 x f16 -> f32 FMAs; the biases 1032 and
//               72 are removed once per unit with the precomputed sum
//               C = 1032 sum x_even + 72 sum x_odd.
// Rows are split over the CTAs in balanced contiguous ranges (at most one row
// of imbalance).  Every wait is bounded; a timeout sets W4A16_DEV_PIPE_TIMEOUT.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

constexpr int kM1MaxThreads = 672;  // 21 warps -> the compiler may use up to 96 registers
constexpr int kM1MaxStages = 16;
constexpr int kM1SmemBudget = 200 * 1024;
constexpr int kRR = 2;  // rows per consumer thread per tile (independent chains)

struct M1Plan {
  int U;            // units (64 k) per row
  int RL;           // rows across lanes
  int RB;           // rows per tile = RL * kRR
  int T;            // consumer threads = U * RL
  int CW;           // consumer warps
  int pitch;        // shared-memory row pitch, bytes
  int sc_cap;       // bytes of the per-stage scale window
  int stage_bytes;  // RB * pitch + sc_cap
  int red_stride;   // floats per row in the partial buffer (U + 1: odd stride)
  int S;            // pipeline stages
  int smem;         // dynamic shared memory, bytes
};

__host__ __device__ inline int m1_rows_across_lanes(int U) {
  // consumer threads = U * RL: about 450-600 threads for every K
  return U > 64 ? 2 : (U > 16 ? 8 : (U > 4 ? 16 : 32));
}

M1Plan make_m1_plan(int K, int smem_limit) {
  M1Plan p{};
  p.U = K / 64;
  p.RL = m1_rows_across_lanes(p.U);
  p.RB = p.RL * kRR;
  p.T = p.U * p.RL;
  p.CW = (p.T + 31) / 32;
  p.pitch = K / 2;  // rows stored densely: a tile is one contiguous bulk copy
  p.sc_cap = ((p.RB * (K / 64) + 32) + 15) & ~15;
  p.stage_bytes = p.RB * p.pitch + p.sc_cap;
  p.red_stride = p.U + 1;
  const int per_stage = p.stage_bytes + p.RB * p.red_stride * 4;
  const int budget = (smem_limit < kM1SmemBudget ? smem_limit : kM1SmemBudget) - 512;
  p.S = budget / per_stage;
  if (p.S > kM1MaxStages) p.S = kM1MaxStages;
  p.smem = 512 + p.S * per_stage;
  return p;
}

struct M1Params {
  GemvArgs a;             // pointers, sizes and output segments
  const uint8_t* scales;  // a.scales as bytes
  int U, RL, RB, T, pitch, stage_bytes, red_stride, S;
};

__global__ void __launch_bounds__(kM1MaxThreads, 1) gemv_m1_kernel(const M1Params p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = p.S;
  const int RL = p.RL;
  const int RB = p.RB;
  // layout: barriers [full S][empty S][redfull S][redempty S] | partials
  // S*RB*red_stride f32 | stages.  All hot accesses use 32-bit shared
  // addresses (explicit ld/st.shared).
  //   full[s]      producer -> consumers: the tile's bytes landed (tx count)
  //   empty[s]     consumers -> producer: the tile is in registers, refill
  //   redfull[s]   consumers -> reducer: the tile's partial sums are written
  //   redempty[s]  reducer -> consumers: partial slot s may be rewritten
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + S;
  uint64_t* redfull = empty + S;
  uint64_t* redempty = redfull + S;
  const uint32_t smem0 = smem_addr(smem);
  const uint32_t red0 = smem0 + 512;
  const uint32_t stage0 = (red0 + S * RB * p.red_stride * 4 + 127) & ~127u;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int CW = (p.T + 31) >> 5;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), CW);
      mbar_init(smem_addr(&redfull[s]), CW);
      mbar_init(smem_addr(&redempty[s]), 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  const int64_t N = p.a.N;
  const int K = p.a.K;
  const int64_t G = gridDim.x;
  const int64_t row_begin = (N * blockIdx.x) / G;
  const int rows = static_cast<int>((N * (blockIdx.x + 1)) / G - row_begin);  // rows of this CTA
  const int ntiles = (rows + RB - 1) / RB;
  const int row_bytes = K / 2;      // packed bytes per row
  const int sc_row_bytes = K / 64;  // scale bytes per row
  // scale bytes are addressed relative to the first row of this CTA; only the
  // alignment of the absolute offset matters, and that is its low 4 bits
  const int64_t sc_cta = row_begin * sc_row_bytes;
  const int sc_cta_lo = static_cast<int>(sc_cta & 15);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    const int64_t sc_total = N * sc_row_bytes;
    const uint32_t* qrows = p.a.qweight + row_begin * (K / 8);
    // issue tile t into stage s
    auto issue = [&](int t, int s) {
      const int lr0 = t * RB;
      const int nr = rows - lr0 < RB ? rows - lr0 : RB;
      const int64_t sb0 = sc_cta + static_cast<int64_t>(lr0) * sc_row_bytes;
      const int64_t sb1 = sb0 + static_cast<int64_t>(nr) * sc_row_bytes;
      const int64_t a = sb0 & ~int64_t(15);
      int64_t e = (sb1 + 15) & ~int64_t(15);
      if (e > sc_total) e = sc_total & ~int64_t(15);  // never read past the buffer
      const int64_t ecopy = e > a ? e : a;
      const uint32_t base = stage0 + s * p.stage_bytes;
      const uint32_t scw = base + RB * p.pitch;
      const uint32_t bar = smem_addr(&full[s]);
      if (lane == 0) {
        // the last few scale bytes of the matrix, if the aligned copy stops short
        for (int64_t b = ecopy; b < sb1; b += 2)
          sts_u16(scw + static_cast<uint32_t>(b - a), ld_nc_u16(p.scales + b));
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nr * row_bytes + (ecopy - a)));
      }
      __syncwarp();
      // consecutive rows are contiguous in memory: one copy for the whole tile
      if (lane == 0)
        bulk_g2s(base, qrows + static_cast<int64_t>(lr0) * (K / 8),
                 static_cast<uint32_t>(nr * row_bytes), bar, pol);
      if (lane == 1 && ecopy > a)
        bulk_g2s(scw, p.scales + a, static_cast<uint32_t>(ecopy - a), bar, pol);
    };

    // the weights and scales are constant: stream them without waiting for
    // the previous kernel on the stream
    const int prolog = ntiles < S ? ntiles : S;
    for (int t = 0; t < prolog; ++t) issue(t, t);
    // then refill each stage as soon as the consumers hold its tile in registers
    int s = 0;
    uint32_t phase = 0;
    int t = S;
    bool ok = true;
    for (; t < ntiles; ++t) {
      if (!mbar_wait_bounded(smem_addr(&empty[s]), phase, kWaitLimitNs)) {
        ok = false;
        break;
      }
      issue(t, s);
      if (++s == S) {
        s = 0;
        phase ^= 1u;
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(p.a.status, W4A16_DEV_PIPE_TIMEOUT);
      // let the copies already in flight land before the CTA exits
      for (int v = t - S; v < t; ++v)
        if (v >= 0) mbar_wait_bounded(smem_addr(&full[v % S]), (v / S) & 1, kWaitLimitNs);
    }
    return;
  }

  if (warp == 1) {
    // ------------------------------------------------------------ reducer
    pdl_wait();  // y may still be read by the previous kernel on the stream
    const int lpr = RB >= 32 ? 1 : 32 / RB;  // reducer lanes per row
    const int rows_per_pass = 32 / lpr;
    const int part = lane % lpr;
    int s = 0;
    uint32_t phase = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!mbar_wait_bounded(smem_addr(&redfull[s]), phase, kWaitLimitNs)) {
        if (lane == 0) atomicOr(p.a.status, W4A16_DEV_PIPE_TIMEOUT);
        return;
      }
      const int lr0 = t * RB;
      const int nr = rows - lr0 < RB ? rows - lr0 : RB;
      const uint32_t rs = red0 + s * RB * p.red_stride * 4;
      for (int row = lane / lpr; row < RB; row += rows_per_pass) {
        const uint32_t rp = rs + row * p.red_stride * 4;
        // four independent running sums so the shared loads overlap; the
        // order of additions is fixed, so every run gives the same bits
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int u = part;
        for (; u + 3 * lpr < p.U; u += 4 * lpr) {
          s0 += lds_f32(rp + 4 * u);
          s1 += lds_f32(rp + 4 * (u + lpr));
          s2 += lds_f32(rp + 4 * (u + 2 * lpr));
          s3 += lds_f32(rp + 4 * (u + 3 * lpr));
        }
        for (; u < p.U; u += lpr) s0 += lds_f32(rp + 4 * u);
        float sum = (s0 + s1) + (s2 + s3);
        for (int o = lpr >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (part == 0 && row < nr)
          *out_ptr(p.a, 0, row_begin + lr0 + row) = __half_as_ushort(__float2half_rn(sum));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&redempty[s]));
      if (++s == S) {
        s = 0;
        phase ^= 1u;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // consecutive threads take consecutive 64-k units of one row, so a warp
  // reads 32 x 32 contiguous bytes; threads whose unit index has bit 2 set
  // read their two 16-byte chunks in the opposite order, which makes every
  // quarter-warp phase of the 16-byte shared loads hit 8 distinct bank groups
  const int c = tid - 64;
  const bool active = c < p.T;
  const int u = c % p.U;
  const int rl = active ? c / p.U : 0;
  const int rot = ((u >> 2) & 1) * 16;

  // activations of this thread's 64 k, paired to match the unpacked lanes
  // (x may be the previous kernel's output: wait for it first)
  pdl_wait();
  XPairs X[8];
  float C = 0.f;
  {
    const uint16_t* xp = p.a.x + u * 64;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // X[j] pairs with the j-th word as this thread loads them: with the
      // chunk order rotated, words 4..7 come first
      const int jj = rot ? (j ^ 4) : j;
      const uint4 v = *reinterpret_cast<const uint4*>(xp + 8 * jj);
      X[j] = pair_activations(v);
      const float even = (half_lo(X[j].p0) + half_hi(X[j].p0)) + (half_lo(X[j].p2) + half_hi(X[j].p2));
      const float odd = (half_lo(X[j].p1) + half_hi(X[j].p1)) + (half_lo(X[j].p3) + half_hi(X[j].p3));
      C = fmaf(1032.f, even, fmaf(72.f, odd, C));
    }
  }

  // per-thread offsets inside a stage (32-bit, fixed for the whole kernel):
  // this thread handles rows rl + r RL, r < kRR, of every tile
  const int w_off = rl * p.pitch + u * 32;
  const int w_row_step = RL * p.pitch;
  const int sc_off = RB * p.pitch + rl * sc_row_bytes + (u >> 1) * 2;
  const int sc_row_step = RL * sc_row_bytes;
  const int red_off = 4 * (rl * p.red_stride + u);
  const int red_row_step = 4 * RL * p.red_stride;
  const int sc_tile_step = RB * sc_row_bytes;
  int sc_lo = sc_cta_lo;  // low 4 bits of the absolute scale offset of the tile

  int s = 0;
  uint32_t phase = 0;
  for (int t = 0; t < ntiles; ++t) {
    if (!mbar_wait_bounded(smem_addr(&full[s]), phase, kWaitLimitNs)) {
      if (lane == 0) atomicOr(p.a.status, W4A16_DEV_PIPE_TIMEOUT);
      return;
    }
    const int nr = rows - t * RB;  // rows of this tile (may exceed RB)
    const uint32_t base = stage0 + s * p.stage_bytes;
    const uint32_t rs = red0 + s * RB * p.red_stride * 4;
    // the tile's bytes go to registers; the stage is then free for a refill
    uint32_t w[kRR][8];
    float sc[kRR];
    const bool work = active && rl < nr;
    if (work) {
#pragma unroll
      for (int r = 0; r < kRR; ++r) {
        if (r == 0 || rl + r * RL < nr) {
          const uint4 lo = lds_u4(base + w_off + r * w_row_step + rot);
          const uint4 hi = lds_u4(base + w_off + r * w_row_step + (16 - rot));
          w[r][0] = lo.x; w[r][1] = lo.y; w[r][2] = lo.z; w[r][3] = lo.w;
          w[r][4] = hi.x; w[r][5] = hi.y; w[r][6] = hi.z; w[r][7] = hi.w;
          sc[r] = __half2float(__ushort_as_half(lds_u16(base + sc_off + r * sc_row_step + sc_lo)));
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) w[r][j] = 0u;
          sc[r] = 0.f;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty[s]));
    float res[kRR];
    if (work) {
      float e0[kRR], e1[kRR], o0[kRR], o1[kRR];
#pragma unroll
      for (int r = 0; r < kRR; ++r) e0[r] = e1[r] = o0[r] = o1[r] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int r = 0; r < kRR; ++r) {
          const Unpacked h = unpack_biased(w[r][j]);
          fma_f32_f16x2(e0[r], e1[r], h.h0, X[j].p0);
          fma_f32_f16x2(o0[r], o1[r], h.h1, X[j].p1);
          fma_f32_f16x2(e0[r], e1[r], h.h2, X[j].p2);
          fma_f32_f16x2(o0[r], o1[r], h.h3, X[j].p3);
        }
      }
#pragma unroll
      for (int r = 0; r < kRR; ++r) res[r] = (fmaf(0.0625f, o0[r] + o1[r], e0[r] + e1[r]) - C) * sc[r];
    }
    // partial slot s still holds tile t - S until the reducer has read it
    if (t >= S && !mbar_wait_bounded(smem_addr(&redempty[s]), phase ^ 1u, kWaitLimitNs)) {
      if (lane == 0) atomicOr(p.a.status, W4A16_DEV_PIPE_TIMEOUT);
      return;
    }
    if (work) {
#pragma unroll
      for (int r = 0; r < kRR; ++r)
        if (r == 0 || rl + r * RL < nr) sts_f32(rs + red_off + r * red_row_step, res[r]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&redfull[s]));
    sc_lo = (sc_lo + sc_tile_step) & 15;
    if (++s == S) {
      s = 0;
      phase ^= 1u;
    }
  }
}

}  // namespace

bool gemv_m1_supported(int K) {
  if (K <= 0 || K % 128 != 0) return false;
  const int U = K / 64;
  const int T = U * m1_rows_across_lanes(U);
  return T + 64 <= kM1MaxThreads;
}

cudaError_t launch_gemv_m1(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  const M1Plan plan = make_m1_plan(a.K, d.max_smem_optin);
  if (plan.S < 2) return cudaErrorInvalidConfiguration;
  M1Params p;
  p.a = a;
  p.scales = reinterpret_cast<const uint8_t*>(a.scales);
  p.U = plan.U;
  p.RL = plan.RL;
  p.RB = plan.RB;
  p.T = plan.T;
  p.pitch = plan.pitch;
  p.stage_bytes = plan.stage_bytes;
  p.red_stride = plan.red_stride;
  p.S = plan.S;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.N < d.sms ? a.N : d.sms);
  cfg.blockDim = dim3(64 + plan.CW * 32);
  cfg.dynamicSmemBytes = plan.smem + 128;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_m1_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t prepare_gemv_m1(const DeviceInfo& d) {
  const int limit = d.max_smem_optin < kM1SmemBudget + 1024 ? d.max_smem_optin : kM1SmemBudget + 1024;
  return cudaFuncSetAttribute(gemv_m1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
}

}  // namespace w4a16
