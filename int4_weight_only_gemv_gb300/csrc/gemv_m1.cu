// gemv_m1.cu -- the M = 1 decode GEMV: a persistent, TMA-fed, warp-specialised
// CUDA-core kernel that runs a list of GEMVs in one launch.
//
// The operation is the INT4 x FP16 GEMV of "Costruire un runtime di inference
// LLM da zero" (datastack.it), section "Tre bug che insegnano", third bug
// (gate/up/down GEMVs unpack INT4 in-kernel against FP16 activations), with
// the group-128 symmetric format of the same section's last paragraph.  The
// second bug of that section is the cost of launching every kernel of a
// decode step on its own; here a list of GEMVs (a decode step's projections)
// runs as one persistent launch whose weight stream does not stop between
// GEMVs.  A single GEMV is a list of one.
//
// Design (one CTA per SM; every CTA takes a balanced contiguous range of the
// rows of every task, at most one row of imbalance):
//   warp 0      producer.  Streams tiles of RB consecutive rows into an
//               S-stage shared-memory ring: one 1-D bulk copy for the tile's
//               rows (contiguous in memory) and one for its scale window,
//               completing on the stage's mbarrier.  It runs ahead across
//               task boundaries and never waits for a dependency: weights
//               and scales are constant.
//   warp 1      reducer.  Sums the consumers' per-unit partials of each tile
//               in a fixed order and writes y; after a task's last tile it
//               publishes the CTA's completion of the task (fence + atomic
//               on the task's counter).  Before a task that reads another
//               task's output it waits until every CTA has published that
//               task, then releases the consumers through an mbarrier.
//   warps 2..   consumers.  Consumer thread c owns unit u = c mod U (64
//               consecutive k, half a group) of rows c / U + r RL (r < 4) of
//               every tile, so its 64 activations stay in registers for the
//               whole task.  Per packed word: one shift, four LOP3s (nibble
//               -> biased fp16, see ptx.cuh) and eight f16 x f16 -> f32 FMAs;
//               the biases 1032 and 72 are removed once per unit and row with
//               the precomputed C = 1032 sum x_even + 72 sum x_odd.
// W4A8 variant (kFmt = kFmtW4A8, the INT8-activation GEMV that the same section's third
// bug compares with): each consumer thread quantises its own 64-activation
// unit when it loads it (scale max|x| / 127 and codes round(x 127 / max|x|)
// in FP32, ties to even), so no pass over x runs first and x stays
// fp16 in memory.  Per packed word: one shift, two LOP3s (nibbles + 8 as
// bytes, even and odd k) and two dp4a against the unit's codes; the bias 8 is
// removed once per unit and row with 8 sum(codes), and the integer sum is
// scaled by group scale x activation scale in FP32.
// Q4_K variant (kFmt = kFmtQ4K, a single GEMV): the tile is RB whole rows of
// GGUF Q4_K super-blocks (144 bytes per 256 weights, scales inside the
// blocks, so there is no scale window).  Unit u is chunk u mod 4 of block
// u / 4; per row the thread reads the block's 16-byte header and the chunk's
// 32 code bytes, forms D_j = sum (1024 + q) x for its two sub-blocks with
// mask-and-OR unpacking (the high nibbles in place, as 1024 + 16 q), and
// returns d sc_j (D_j - 1024 S_j) - dmin m_j S_j summed over them, S_j =
// sum x over the sub-block computed once per task.
// Every wait is bounded; on a timeout the kernel sets W4A16_DEV_PIPE_TIMEOUT
// and the CTA returns once its copies in flight have landed.
#include <cuda_fp16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "w4a16.h"

namespace w4a16 {
namespace {

// 16 warps: the producer (lane 0 of warp 0; for W4A16, lanes 1..31 of the
// same warp stage the activations of the next task into shared memory), the
// reducer and 14 consumer warps.  Registers are handed out to warps in groups
// of four, so 16 warps leave up to 128 registers per thread.
constexpr int kM1MaxThreads = 512;
constexpr int kM1MaxConsumers = kM1MaxThreads - 64;
constexpr int kM1MaxStages = 8;
constexpr int kM1SmemBudget = 227 * 1024;

// Weight formats of the kernel: the INT4 group-128 layout with FP16 or
// in-kernel INT8 activations, and GGUF Q4_K blocks (144 bytes per 256
// weights, scales inside the blocks).
constexpr int kFmtW4A16 = 0;
constexpr int kFmtW4A8 = 1;
constexpr int kFmtQ4K = 2;

// First consumer warp and consumer threads.
__host__ __device__ constexpr int first_consumer_warp(int) { return 2; }
__host__ __device__ constexpr int max_consumers(int fmt) { return kM1MaxThreads - 32 * first_consumer_warp(fmt); }

// A consumer thread's unit of K and its rows per tile, by format.  W4A16:
// one whole 128-k group (its 128 activations in 64 registers, the group scale
// applied once per row), two rows per tile.  W4A8: 64 k, one activation
// block; Q4_K: 64 k, one chunk of a block; four rows per tile.
__host__ __device__ constexpr int unit_k(int fmt) { return fmt == kFmtW4A16 ? 128 : 64; }
__host__ __device__ constexpr int rows_per_thread(int fmt) { return fmt == kFmtW4A16 ? 2 : 4; }

// Rows of one CTA a K-split task may have (its first part's sums wait in
// shared memory for the second part).
constexpr int kM1PartRows = 256;

// Per-task tiling, a pure function of the task's K, its format and whether
// it is half of a K-split GEMV (U <= max_consumers(fmt)).
struct TaskPlan {
  int U;             // units (unit_k(fmt) k) per row
  int RL;            // rows across consumer threads
  int RB;            // rows per tile = RL * rows_per_thread(fmt)
  int T;             // consumer threads = U * RL
  int row_bytes;     // K / 2: packed bytes of a row's K range, also the row pitch in a stage
  int sc_row_bytes;  // K / 64: scale bytes of a row's K range
  int pitch;         // bytes between rows in memory (row_bytes times the parts of the split)
  int sc_pitch;      // scale bytes between rows in memory
  int red_stride;    // floats per row in a partial slot (U + 1)
};

// a / b for a >= 0, b >= 1, computed at task starts.  On the device, below
// a = 2^21, through the approximate float reciprocal: (a + 0.5) / b lies at
// least 0.5 / b from an integer, and the reciprocal's and the product's
// rounding (relative 2^-22 together) move it by less than (a + 0.5) / b x
// 2^-22, under that margin while a < 2^21.  It keeps a long integer-division
// sequence off the producer's and consumers' path between two tasks.
// Integer division elsewhere.
__host__ __device__ inline int small_div(int a, int b) {
#ifdef __CUDA_ARCH__
  if (a >= (1 << 21)) return a / b;
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(static_cast<float>(b)));
  return static_cast<int>((static_cast<float>(a) + 0.5f) * r);
#else
  return a / b;
#endif
}

__host__ __device__ inline TaskPlan task_plan(int K, int fmt, int parts = 1) {
  TaskPlan p;
  const int cons = max_consumers(fmt);
  p.U = K / unit_k(fmt);
  p.RL = p.U >= cons ? 1 : small_div(cons, p.U);
  p.RB = p.RL * rows_per_thread(fmt);
  p.T = p.U * p.RL;
  // Q4_K: 144 bytes per 256 weights (a multiple of 16), no separate scales
  p.row_bytes = fmt == kFmtQ4K ? (K >> 8) * 144 : K >> 1;
  p.sc_row_bytes = fmt == kFmtQ4K ? 0 : K >> 6;
  p.pitch = p.row_bytes * parts;
  p.sc_pitch = p.sc_row_bytes * parts;
  p.red_stride = p.U + 1;
  return p;
}

__host__ __device__ inline int task_parts(const M1Task& tk) { return tk.split ? 2 : 1; }

// Bytes of a stage's scale window: RB rows at the task's scale pitch plus up
// to 15 bytes of alignment slack on each side, rounded to 16.
__host__ __device__ inline int sc_window_cap(const TaskPlan& tp) {
  return (tp.RB * tp.sc_pitch + 32 + 15) & ~15;
}

// Bytes of one W4A16 activation slot for a task of U units: per unit its 128
// activations paired as the consumers use them (256 bytes), then one FP32
// bias sum per unit.
__host__ __device__ inline int xslot_bytes(int U) { return (U * 260 + 15) & ~15; }

// Units the stager converts in one pass (one per lane 1..31).
constexpr int kStagers = 31;

// W4A16: whether the stager may stage task i (its activations come through
// the shared-memory slot), given its activation vector x, whether it is the
// first task with rows on the CTA and whether the launch runs a task list
// (the layer sequence's kernel instantiation) or one GEMV.  The stager's
// 16-byte copies need x 16-byte aligned (the ABI asks for it; an unaligned
// x is loaded by the consumers instead).  In a single-GEMV launch the first
// task is staged only when one pass of the stager converts it (nothing runs
// before it to hide a longer staging: a standalone down, 148 units, is
// 0.7 us faster on the consumers' own loads).  In a list every other task
// is: measured, the step took 0.676 ms with the list's first task held to
// the same rule and 0.670 ms without it (its first task is [gate; up],
// staged either way; the simpler test is what differs).  The test runs on
// the device too, so the list kernel keeps the consumers' own-load path:
// with staging known at compile time the compiler's schedule of the list
// kernel ran the step 3 % slower.
__host__ __device__ inline bool may_stage(const uint16_t* x, int U, bool first, bool list) {
  return (reinterpret_cast<uintptr_t>(x) & 15) == 0 && (list || !first || U <= kStagers);
}

// Sizes shared by every task of a launch.
struct RingPlan {
  int stage_bytes;  // max over tasks of RB * row_bytes + scale window, 128-aligned
  int red_bytes;    // max over tasks of RB * red_stride * 4, 16-aligned
  int xslot;        // bytes of one activation slot (W4A16 tasks the stager may stage), 16-aligned; or 0
  int CW;           // consumer warps = max over tasks of ceil(T / 32)
  int S;            // stages
  int smem;         // dynamic shared memory, bytes
};

// dependency-signal barriers: the reducer signals up to kXReady - 1
// dependent tasks ahead of the consumers.  Measured on the 28-layer step
// (same box): 4 0.667 ms, 8 0.663, 12 0.660, 16 0.663.
constexpr int kXReady = 12;
constexpr int kXSlots = 1;          // activation slots (W4A16)
// The stager's pause between pieces of work.  The 28-layer step (same box):
// 0.6311 ms at 64 ns, 0.6298-0.6300 at 0, 8, 16 and 32 ns; with no sleep
// instruction at all the producer lane starves.
constexpr unsigned kStagerYieldNs = 32;
// [full S][empty S][redfull S][redempty S][xready kXReady][xfull kXSlots][xempty kXSlots]
constexpr int kBarrierBytes = 512;
static_assert(32 * kM1MaxStages + 8 * kXReady + 16 * kXSlots <= kBarrierBytes, "barriers overflow their area");
constexpr int kPartBytes = 4 * kM1PartRows;
// The first task's stages are filled at each CTA's share of this HBM rate
// (bytes per microsecond) rather than all at once.  Copies in flight share
// the bandwidth, so S tiles issued together land together, late; paced, the
// first tile lands early and the consumers start on it.  Measured on
// standalone GEMVs (graphs of back-to-back calls, cold L2; same box):
// down 3584 x 18944 12.5 -> 11.6 us, [gate; up] 37888 x 3584 15.9 -> 15.6 us
// (0.8x and 1.25x this rate: 11.7 / 15.7 and 11.5 / 15.7 us).
constexpr float kPaceBytesPerUs = 6800.f * 1000.f;

// Bytes of the kept gate outputs (one fp16 per row of a CTA) of a list with
// SwiGLU, after the stages.
constexpr int kGateBytes = 2 * kM1PartRows;

// Shared layout: barriers | K-split partial sums | xslots | S partial slots |
// S stages (128-aligned) | kept gate outputs (lists with SwiGLU).
RingPlan make_ring_plan(const M1Task* tasks, int n, int smem_limit, int fmt, bool list) {
  RingPlan r{};
  int gate = 0;
  for (int i = 0; i < n; ++i) {
    if (tasks[i].swiglu != 0) gate = kGateBytes;
    const TaskPlan tp = task_plan(tasks[i].K, fmt, task_parts(tasks[i]));
    const int st = tp.RB * tp.row_bytes + sc_window_cap(tp);
    const int rb = tp.RB * tp.red_stride * 4;
    const int cw = (tp.T + 31) / 32;
    // any task but the list's first may be some CTA's first with rows
    const int xs = fmt == kFmtW4A16 && may_stage(tasks[i].x, tp.U, i == 0, list) ? xslot_bytes(tp.U) : 0;
    if (st > r.stage_bytes) r.stage_bytes = st;
    if (rb > r.red_bytes) r.red_bytes = rb;
    if (cw > r.CW) r.CW = cw;
    if (xs > r.xslot) r.xslot = xs;
  }
  r.stage_bytes = (r.stage_bytes + 127) & ~127;
  r.red_bytes = (r.red_bytes + 15) & ~15;
  const int per_stage = r.stage_bytes + r.red_bytes;
  const int fixed = kBarrierBytes + kPartBytes + kXSlots * r.xslot + 128 + gate;  // 128: stage alignment slack
  const int budget = (smem_limit < kM1SmemBudget ? smem_limit : kM1SmemBudget) - fixed;
  r.S = budget / per_stage;
  if (r.S > kM1MaxStages) r.S = kM1MaxStages;
  r.smem = fixed + r.S * per_stage;
  return r;
}

// K-split of a W4A16 GEMV: two tasks over the two halves of each row's K
// when that fills the consumer threads markedly better (K = 18944: 148
// units use 2 x 148 = 296 of 416 threads, 74 use 5 x 74 = 370) and a CTA's
// rows fit the partial-sum buffer.  A pure function of K, N and the grid, so
// a GEMV is split the same way alone and inside a task list.
int split_parts(int K, int N, int grid) {
  const int cons = max_consumers(kFmtW4A16);
  if (K % 256 != 0 || (N + grid - 1) / grid > kM1PartRows) return 1;
  auto used = [&](int U) { return U >= cons ? cons : (cons / U) * U; };
  const int U = K / 128;
  return 10 * used(U / 2) > 11 * used(U) ? 2 : 1;
}

template <int MAXT>
struct M1Params {
  int ntasks;
  int S, stage_bytes, red_bytes, xslot, CW;
  float pace;        // ns per byte of the first task's initial stage fill (this CTA's share)
  int* done;         // per-task completion counters (null: no task has a dependency)
  uint32_t* status;  // device status word
  M1Task task[MAXT];
};

// This CTA's rows of a task: [row_begin, row_begin + return value).  The
// launcher split the N rows as rq per CTA plus one for the first rr CTAs.
__device__ __forceinline__ int cta_rows(const M1Task& tk, int64_t* row_begin) {
  const int b = blockIdx.x;
  *row_begin = static_cast<int64_t>(b) * tk.rq + (b < tk.rr ? b : tk.rr);
  return tk.rq + (b < tk.rr ? 1 : 0);
}

__device__ __forceinline__ bool cta_has_rows(const M1Task& tk) {
  return tk.rq > 0 || static_cast<int>(blockIdx.x) < tk.rr;
}

// Bounded wait until *counter >= target (acquire).  False if the bound ran out.
// Polls every 64 ns (the 28-layer step: 0.659 ms at 256 ns, 0.658 at 128,
// 0.657 at 64; 0.788 ms at 2 us).
__device__ __forceinline__ bool wait_count(const int* counter, int target, uint64_t limit_ns) {
  if (ld_acquire_gpu(counter) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(counter) >= target) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// SwiGLU of one element: fp16_RN(silu(g) u), silu(g) = g / (1 + e^-g),
// computed in FP32 from the fp16 inputs with the fast exponential and
// division (relative error ~1e-6, far below the fp16 result's 2^-11).
__device__ __forceinline__ uint16_t swiglu1(uint16_t g, uint16_t u) {
  const float g0 = __half2float(__ushort_as_half(g));
  const float h0 = __fdividef(g0, 1.f + __expf(-g0)) * __half2float(__ushort_as_half(u));
  return __half_as_ushort(__float2half_rn(h0));
}

// Bias sums of a W4A16 unit, C = 1032 sum x(k even) + 72 sum x(k odd) (the
// dot product of its activations with a word of zero nibbles), in one
// canonical order: each 4-word chunk (32 activations, words in natural
// order) into its own even and odd sums, then the chunks in natural order.
// Both ways of staging a unit's activations (the stager, or each consumer
// thread for itself) use it, so a row's sum does not depend on the way.
__device__ __forceinline__ void chunk_bias(const XPairs* q, float& e, float& o) {
  float e0 = 0.f, e1 = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    fma_f32_f16x2(e0, e1, 0x64086408u, q[i].p0);
    fma_f32_f16x2(o0, o1, 0x64806480u, q[i].p1);
    fma_f32_f16x2(e0, e1, 0x64086408u, q[i].p2);
    fma_f32_f16x2(o0, o1, 0x64806480u, q[i].p3);
  }
  e = e0 + e1;
  o = o0 + o1;
}
__device__ __forceinline__ float unit_bias(const float (&e)[4], const float (&o)[4]) {
  return fmaf(0.0625f, (o[0] + o[1]) + (o[2] + o[3]), (e[0] + e[1]) + (e[2] + e[3]));
}

// The stager's conversion of one W4A16 unit in shared memory, in place: word
// w of the unit (activations 8 w .. 8 w + 7) sits at 16-byte slot
// w ^ (u mod 16) of its 256 bytes both raw (the copies land there) and as
// the pairs dot_unit128 uses.  The swizzle puts the same word of eight
// consecutive units in eight distinct bank groups, for the stager's reads
// here and for the consumers' rotated reads.  Returns the unit's bias sum.
__device__ __forceinline__ float convert_unit128(uint32_t dst, int u) {
  uint4 v[16];
#pragma unroll
  for (int w = 0; w < 16; ++w) v[w] = lds_u4(dst + ((w ^ (u & 15)) << 4));
  float e[4], o[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    XPairs q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int w = 4 * c + i;
      q[i] = pair_activations(v[w]);
      sts_u4(dst + ((w ^ (u & 15)) << 4), q[i].p0, q[i].p1, q[i].p2, q[i].p3);
    }
    chunk_bias(q, e[c], o[c]);
  }
  return unit_bias(e, o);
}

// x[(c - f) mod 4] for c = 0..3 (a runtime rotation of four registers).
__device__ __forceinline__ void unrotate4(const float (&x)[4], int f, float (&out)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int j = (c - f) & 3;
    out[c] = j == 0 ? x[0] : (j == 1 ? x[1] : (j == 2 ? x[2] : x[3]));
  }
}

// The 16 packed words of one row's 128-k unit at a stage address: four
// 16-byte shared loads, chunk (j + f) mod 4 into words 4j .. 4j + 3.
__device__ __forceinline__ void load_unit128(uint32_t addr, int f, uint32_t (&w)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 v = lds_u4(addr + 16 * ((j + f) & 3));
    w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
  }
}

// Dot product of one row's 128-k unit (16 packed words) with this thread's
// 128 activations: sum_k (1032 + q or 1152 + 16 q) x, the second kind scaled
// back by 1/16, i.e. sum_k q x + C.
__device__ __forceinline__ float dot_unit128(const uint32_t (&w)[16], const XPairs (&X)[16]) {
  float e0 = 0.f, e1 = 0.f, o0 = 0.f, o1 = 0.f;
  float e2 = 0.f, e3 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const Unpacked a = unpack_biased(w[j]);
    const Unpacked b = unpack_biased(w[j + 1]);
    fma_f32_f16x2(e0, e1, a.h0, X[j].p0);
    fma_f32_f16x2(e2, e3, b.h0, X[j + 1].p0);
    fma_f32_f16x2(o0, o1, a.h1, X[j].p1);
    fma_f32_f16x2(o2, o3, b.h1, X[j + 1].p1);
    fma_f32_f16x2(e0, e1, a.h2, X[j].p2);
    fma_f32_f16x2(e2, e3, b.h2, X[j + 1].p2);
    fma_f32_f16x2(o0, o1, a.h3, X[j].p3);
    fma_f32_f16x2(o2, o3, b.h3, X[j + 1].p3);
  }
  return fmaf(0.0625f, (o0 + o1) + (o2 + o3), (e0 + e1) + (e2 + e3));
}

// W4A8: integer dot products of two rows (8 packed words each) with this
// thread's 64 activation codes, xe[j] / xo[j] the codes of the even / odd k of
// word j as 4 bytes.  Nibble n becomes n ^ 8 = q + 8 (0..15) in a byte, so the
// sums are sum_k (q + 8) xq; the caller subtracts 8 sum(xq).
__device__ __forceinline__ void dot_pair_a8(const uint32_t (&wa)[8], const uint32_t (&wb)[8],
                                            const uint32_t (&xe)[8], const uint32_t (&xo)[8], int& ra,
                                            int& rb) {
  int a = 0, b = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a = __dp4a(static_cast<int>(lop3_and_xor(wa[j], 0x0F0F0F0Fu, 0x08080808u)), static_cast<int>(xe[j]), a);
    b = __dp4a(static_cast<int>(lop3_and_xor(wb[j], 0x0F0F0F0Fu, 0x08080808u)), static_cast<int>(xe[j]), b);
    a = __dp4a(static_cast<int>(lop3_and_xor(wa[j] >> 4, 0x0F0F0F0Fu, 0x08080808u)), static_cast<int>(xo[j]), a);
    b = __dp4a(static_cast<int>(lop3_and_xor(wb[j] >> 4, 0x0F0F0F0Fu, 0x08080808u)), static_cast<int>(xo[j]), b);
  }
  ra = a;
  rb = b;
}

// Q4_K: dot products of one 64-weight unit (chunk c of a block: code word t
// holds weights 4t .. 4t + 3 in its low nibbles and 32 + 4t .. + 3 in its
// high nibbles) with this thread's activations, paired as X[t] = {x(4t),
// x(4t+2)}, {x(4t+1), x(4t+3)}, {x(32+4t), x(32+4t+2)}, {x(32+4t+1),
// x(32+4t+3)}.  A low nibble becomes fp16 1024 + q and a high nibble, left
// in place, 1024 + 16 q (bits 4-7 are still mantissa), one LOP3 each,
// written as the explicit lop3 (the mask and the constant share no bit, so
// the OR is the XOR).  Written as a C++ mask-and-OR, the [gate; up] GEMV
// counted 9.2 LOP3 per packed word in ncu and took 19.6 us; as lop3, 17.8 us.
// Returns D0 = sum (1024 + q) x over sub-block 2c and D1 = sum (1024 + 16 q) x
// over sub-block 2c + 1.
__device__ __forceinline__ void q4k_dot(const uint32_t (&q)[8], const XPairs (&X)[8], float& D0, float& D1) {
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const uint32_t v = q[t], v8 = v >> 8;
    fma_f32_f16x2(a0, a1, lop3_and_xor(v, 0x000F000Fu, 0x64006400u), X[t].p0);
    fma_f32_f16x2(a0, a1, lop3_and_xor(v8, 0x000F000Fu, 0x64006400u), X[t].p1);
    fma_f32_f16x2(b0, b1, lop3_and_xor(v, 0x00F000F0u, 0x64006400u), X[t].p2);
    fma_f32_f16x2(b0, b1, lop3_and_xor(v8, 0x00F000F0u, 0x64006400u), X[t].p3);
  }
  D0 = a0 + a1;
  D1 = b0 + b1;
}

// Q4_K: the 6-bit scales and minima of sub-blocks 2c and 2c + 1 from the
// header words h.y, h.z, h.w (packed bytes 0-11) as bytes {sc0, sc1, m0, m1}
// of one word.  Both cases start from bytes {2c', 2c'+1, 2c'+4, 2c'+5},
// c' = c mod 2 (selector selp): for c < 2 these are the values' 6 bits;
// for c >= 2 their top two bits are the values' bits 4-5, and the low four
// come from the nibbles of bytes 8 + 2c', 9 + 2c' (selector selq: scale in
// the low nibble, minimum in the high).
__device__ __forceinline__ uint32_t q4k_scales_pair(const uint4 h, uint32_t selp, uint32_t selq, bool hi) {
  const uint32_t p = __byte_perm(h.y, h.z, selp);
  const uint32_t q = __byte_perm(h.w, h.w, selq);
  const uint32_t low = (q & 0x00000F0Fu) | ((q >> 4) & 0x0F0F0000u);
  return hi ? (low | ((p >> 2) & 0x30303030u)) : (p & 0x3F3F3F3Fu);
}

// Q4_K: one row's partial of the unit from its block header h:
// d sc0 (D0 - 1024 S0) + d sc1 (D1 - 1024 S1) / 16 - dmin (m0 S0 + m1 S1).
__device__ __forceinline__ float q4k_combine(const uint4 h, uint32_t selp, uint32_t selq, bool hi, float D0,
                                             float D1, float S0, float S1) {
  const uint32_t sm = q4k_scales_pair(h, selp, selq, hi);
  const float sc0 = static_cast<float>(sm & 0xFFu), sc1 = static_cast<float>((sm >> 8) & 0xFFu);
  const float m0 = static_cast<float>((sm >> 16) & 0xFFu), m1 = static_cast<float>(sm >> 24);
  const float d = half_lo(h.x), dmin = half_hi(h.x);
  float r = (d * sc0) * fmaf(-1024.f, S0, D0);
  r = fmaf((d * 0.0625f) * sc1, fmaf(-1024.f, S1, D1), r);
  return fmaf(-dmin, fmaf(m0, S0, m1 * S1), r);
}

// The low bytes of four ints as one word (byte i from argument i).
__device__ __forceinline__ uint32_t pack_bytes(int a, int b, int c, int d) {
  const uint32_t lo = __byte_perm(static_cast<uint32_t>(a), static_cast<uint32_t>(b), 0x0040u);
  const uint32_t hi = __byte_perm(static_cast<uint32_t>(c), static_cast<uint32_t>(d), 0x0040u);
  return __byte_perm(lo, hi, 0x5410u);
}

// The 8 packed words of one row at a stage address: two 16-byte shared loads,
// the second chunk first when rot = 16.
__device__ __forceinline__ void load_row(uint32_t addr, int rot, uint32_t (&w)[8]) {
  const uint4 lo = lds_u4(addr + rot);
  const uint4 hi = lds_u4(addr + (16 - rot));
  w[0] = lo.x; w[1] = lo.y; w[2] = lo.z; w[3] = lo.w;
  w[4] = hi.x; w[5] = hi.y; w[6] = hi.z; w[7] = hi.w;
}

// kAct: some task of the list takes part in a SwiGLU (swiglu set).  The
// instantiation without it carries no trace of that path, so the plain task
// lists compile exactly as they would without the feature.  kFmt: the
// weight format (kFmtW4A16, kFmtW4A8, kFmtQ4K).
template <int MAXT, bool kAct, int kFmt>
__global__ void __launch_bounds__(kM1MaxThreads, 1)
    gemv_m1_kernel(const __grid_constant__ M1Params<MAXT> p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int S = p.S;
  constexpr int CW0 = first_consumer_warp(kFmt);
  // shared layout: barriers | K-split row sums | activation slots (W4A16) |
  // S partial slots of red_bytes | S stages of stage_bytes (128-aligned).
  // All hot accesses use 32-bit shared addresses.
  //   full[s]      producer -> consumers: the tile's bytes landed (tx count)
  //   empty[s]     consumers -> producer: the stage may be refilled
  //   redfull[s]   consumers -> reducer: the tile's partial sums are written
  //   redempty[s]  reducer -> consumers: partial slot s may be rewritten
  //   xready[kXReady] reducer -> stager (W4A16) or consumers: a dependent task's
  //                input is complete (a ring of kXReady barriers, so the
  //                reducer may signal up to kXReady - 1 dependent tasks ahead)
  //   xfull[2]     stager -> consumers: activation slot written (W4A16)
  //   xempty[2]    consumers -> stager: activation slot read (W4A16)
  const uint32_t full0 = smem_addr(smem);
  const uint32_t empty0 = full0 + 8 * S;
  const uint32_t redfull0 = full0 + 16 * S;
  const uint32_t redempty0 = full0 + 24 * S;
  const uint32_t xready0 = full0 + 32 * S;
  const uint32_t xfull0 = xready0 + 8 * kXReady;
  const uint32_t xempty0 = xfull0 + 8 * kXSlots;
  const uint32_t part0 = full0 + kBarrierBytes;
  const uint32_t xslot0 = part0 + kPartBytes;
  const uint32_t red0 = xslot0 + kXSlots * p.xslot;
  const uint32_t stage0 = (red0 + S * p.red_bytes + 127) & ~127u;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, p.CW);
      mbar_init(redfull0 + 8 * s, p.CW);
      mbar_init(redempty0 + 8 * s, 1);
    }
    for (int b = 0; b < kXReady; ++b) mbar_init(xready0 + 8 * b, 1);
    for (int b = 0; b < kXSlots; ++b) {
      mbar_init(xfull0 + 8 * b, 1);
      mbar_init(xempty0 + 8 * b, p.CW);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  // W4A16: whether task i's activations come through the stager's slot
  // (may_stage) or each consumer thread loads its own
  int first_task = 0;
  while (first_task < p.ntasks && !cta_has_rows(p.task[first_task])) ++first_task;
  auto staged = [&](const M1Task& tk, int i) {
    return kFmt == kFmtW4A16 && may_stage(tk.x, tk.K / unit_k(kFmt), i == first_task, MAXT > 2);
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int s = 0, g = 0;  // stage, tiles issued so far (all tasks)
    uint32_t phase = 0;
    uint32_t base = stage0;
    bool ok = true;
    uint64_t t_fill = 0;  // when the first tile was issued
    uint32_t filled = 0;  // bytes issued into the first task's first S tiles
    for (int i = 0; i < p.ntasks && ok; ++i) {
      const M1Task& tk = p.task[i];
      const TaskPlan tp = task_plan(tk.K, kFmt, task_parts(tk));
      int64_t row_begin;
      const int rows = cta_rows(tk, &row_begin);
      const int ntiles = (rows + tp.RB - 1) / tp.RB;
      const uint8_t* wsrc = reinterpret_cast<const uint8_t*>(tk.qweight) + row_begin * tp.pitch;
      // the task's scales: rows sc_pitch apart from its first one; the buffer
      // they sit in ends N rows after its start (a second half starts
      // sc_row_bytes into it)
      const uint8_t* scb = reinterpret_cast<const uint8_t*>(tk.scales);
      const uintptr_t sc_end = reinterpret_cast<uintptr_t>(scb) - (tk.split == 2 ? tp.sc_row_bytes : 0) +
                               static_cast<uintptr_t>(tk.N) * tp.sc_pitch;
      for (int t = 0; t < ntiles; ++t) {
        // stage s still holds tile g - S until every consumer warp is done with it
        if (g >= S && !mbar_wait_bounded(empty0 + 8 * s, phase ^ 1u, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const int lr0 = t * tp.RB;
        const int nr = rows - lr0 < tp.RB ? rows - lr0 : tp.RB;
        // scale window: from the tile's first scale byte to past its last,
        // widened to 16-byte boundaries but never past the buffer
        const uintptr_t f = reinterpret_cast<uintptr_t>(scb) + static_cast<uintptr_t>(row_begin + lr0) * tp.sc_pitch;
        const uintptr_t l = f + static_cast<uintptr_t>(nr - 1) * tp.sc_pitch + tp.sc_row_bytes;
        const uintptr_t a = f & ~uintptr_t(15);
        uintptr_t e = (l + 15) & ~uintptr_t(15);
        if (e > sc_end) e = sc_end & ~uintptr_t(15);
        const uintptr_t ecopy = e > a ? e : a;
        const uint32_t scw = base + tp.RB * tp.row_bytes;
        const uint32_t bar = full0 + 8 * s;
        // checked build: the tile's rows and its scale window inside the
        // task and the stage (else nothing is copied and the tile is garbage)
        const bool in = W4A16_IN(p.status, row_begin + lr0 + nr <= tk.N && nr <= tp.RB &&
                                               tp.RB * tp.row_bytes + (l - a) <= static_cast<uintptr_t>(p.stage_bytes) &&
                                               a + (tk.split == 2 ? tp.sc_row_bytes : 0) >= reinterpret_cast<uintptr_t>(scb));
        // the last few scale bytes of the matrix, where the aligned copy stops short
        for (uintptr_t b = ecopy; in && b < l; b += 2)
          sts_u16(scw + static_cast<uint32_t>(b - a), ld_nc_u16(reinterpret_cast<const void*>(b)));
        if (i == first_task && g < S) {
          // paced initial fill: tile g leaves once the bytes before it have had
          // their time at this CTA's share of the bandwidth (a wait of at most
          // S stages' worth, a few microseconds)
          if (g == 0) {
            t_fill = global_timer_ns();
          } else {
            const uint64_t due = t_fill + static_cast<uint64_t>(p.pace * static_cast<float>(filled));
            while (global_timer_ns() < due) __nanosleep(32);
          }
          filled += static_cast<uint32_t>(nr * tp.row_bytes + (ecopy - a));
        }
        mbar_arrive_expect_tx(bar, in ? static_cast<uint32_t>(nr * tp.row_bytes + (ecopy - a)) : 0u);
        if (!in) {
        } else if (tk.split) {
          // a half of each row: one copy per row
          for (int r = 0; r < nr; ++r)
            bulk_g2s(base + r * tp.row_bytes, wsrc + static_cast<int64_t>(lr0 + r) * tp.pitch,
                     static_cast<uint32_t>(tp.row_bytes), bar, pol);
        } else {
          // consecutive rows are contiguous in memory: one copy for the whole tile
          bulk_g2s(base, wsrc + static_cast<int64_t>(lr0) * tp.row_bytes, static_cast<uint32_t>(nr * tp.row_bytes),
                   bar, pol);
        }
        if (in && ecopy > a) bulk_g2s(scw, reinterpret_cast<const void*>(a), static_cast<uint32_t>(ecopy - a), bar, pol);
        ++g;
        base += p.stage_bytes;
        if (++s == S) {
          s = 0;
          phase ^= 1u;
          base = stage0;
        }
      }
    }
    if (!ok) {
      atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
      // let the copies in flight land before the CTA exits: the last S tiles
      // issued sit in stages s, s + 1, ... (mod S)
      for (int v = 0; v < S; ++v) {
        const int gg = g - S + v;  // index of the tile in stage (s + v) mod S
        if (gg >= 0) mbar_wait_bounded(full0 + 8 * ((s + v) % S), (gg / S) & 1, kWaitLimitNs);
      }
    }
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ stager
    // Lanes 1..31 of the producer's warp (W4A16; idle for the other
    // formats): the activations of each task it stages (may_stage), one task
    // ahead of the consumers (the slot is refilled once they have read it).
    // After the task's dependency signal, the raw activations come in with
    // 16-byte asynchronous copies from every lane at once (through L2: the
    // reducer's acquire made the other CTAs' writes visible), then each unit
    // is paired in place and its bias sum stored.
    if (kFmt != kFmtW4A16) return;
    constexpr unsigned kStagerMask = 0xFFFFFFFEu;  // lanes 1..31
    const int sl0 = lane - 1;
    pdl_wait();  // x may be the previous kernel's output
    int n = 0, nw = 0;  // slot uses, dependency signals waited on
    const uint16_t* xprev = nullptr;
    int kprev = 0;
    for (int i = 0; i < p.ntasks; ++i) {
      const M1Task& tk = p.task[i];
      if (!cta_has_rows(tk)) continue;
      const TaskPlan tp = task_plan(tk.K, kFmt, task_parts(tk));
      if (tk.dep >= 0 && p.done != nullptr) {
        // every dependent task's signal, in order, staged here or not
        if (!mbar_wait_bounded(xready0 + 8 * (nw % kXReady), (nw / kXReady) & 1, kWaitLimitNs)) {
          if (lane == 1) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
          return;
        }
        ++nw;
      }
      if (!staged(tk, i)) continue;
      const int sl = n % kXSlots;
      if (n >= kXSlots && !mbar_wait_bounded(xempty0 + 8 * sl, ((n / kXSlots) - 1) & 1, kWaitLimitNs)) {
        if (lane == 1) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
        return;
      }
      const uint32_t xs = xslot0 + sl * p.xslot;
      // the slot already holds these activations (the previous task staged
      // here read the same vector over the same K): keep it
      const bool same = n > 0 && tk.x == xprev && tk.K == kprev;
      xprev = tk.x;
      kprev = tk.K;
      if (!same) {
        const int chunks = tp.U * 16;  // 16-byte chunks of the task's activations
        for (int q = sl0; q < chunks; q += kStagers)
          // chunk q = word q mod 16 of unit q / 16, to its swizzled slot
          if (W4A16_IN(p.status, 16 * q + 16 <= p.xslot && 8 * q + 8 <= tk.K))
            cp_async_16(xs + 16 * ((q & ~15) | ((q ^ (q >> 4)) & 15)), tk.x + 8 * q);
        cp_async_wait_all();
        __syncwarp(kStagerMask);
        // the producer shares this warp: after the launch's first task, a
        // short sleep after each unit lets its lane issue the next weight
        // copies
        const bool yield = i != first_task;
        for (int u = sl0; u < tp.U; u += kStagers) {
          sts_f32(xs + tp.U * 256 + 4 * u, convert_unit128(xs + u * 256, u));
          if (yield) __nanosleep(kStagerYieldNs);
        }
        __syncwarp(kStagerMask);
      }
      if (lane == 1) mbar_arrive(xfull0 + 8 * sl);
      ++n;
    }
    return;
  }

  if (warp == 1) {
    // ------------------------------------------------------------ reducer
    pdl_wait();  // y may still be read by the previous kernel on the stream
    int s = 0;
    uint32_t phase = 0;
    uint32_t rs = red0;
    // A task that reads task dep's output starts once every CTA has
    // published dep.  The reducer checks (acquire) and tells the stager
    // (W4A16) or the consumers (release), the n-th such task with rows here
    // on xready[n % kXReady], in task order.  At the start of task i it
    // signals, ahead of time, every next such task whose producer is older
    // than i (so this CTA has published it), up to kXReady - 1 signals beyond
    // what has been used; the polls of one batch run in parallel lanes.  In
    // an interleaved layer sequence a dependent task is signalled a few tasks
    // early, off the consumers' path.
    int nsig = 0;    // signals sent
    int nused = 0;   // dependent tasks with rows here before task i (consumed)
    int jnext = 0;   // next task that may need a signal
    auto needs_signal = [&](int j) {
      return p.done != nullptr && p.task[j].dep >= 0 && cta_has_rows(p.task[j]);
    };
    for (int i = 0; i < p.ntasks; ++i) {
      const M1Task& tk = p.task[i];
      const TaskPlan tp = task_plan(tk.K, kFmt, task_parts(tk));
      int64_t row_begin;
      const int rows = cta_rows(tk, &row_begin);
      const int ntiles = (rows + tp.RB - 1) / tp.RB;
      {
        int nc = 0, my_dep = -1;
        while (nc < kXReady) {
          while (jnext < p.ntasks && !needs_signal(jnext)) ++jnext;
          if (jnext >= p.ntasks || p.task[jnext].dep >= i || nsig + nc >= nused + kXReady) break;
          if (lane == nc) my_dep = p.task[jnext].dep;
          ++nc;
          ++jnext;
        }
        if (nc > 0) {
          const int ok = my_dep < 0 ||
                         wait_count(p.done + my_dep, static_cast<int>(gridDim.x), kWaitLimitNs);
          if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
            return;
          }
          if (lane == 0)
            for (int c = 0; c < nc; ++c) mbar_arrive(xready0 + 8 * ((nsig + c) % kXReady));
          nsig += nc;
        }
      }
      if (needs_signal(i)) ++nused;
      // the task's output segments, in registers for the whole task
      const int64_t e0 = tk.nseg < 2 ? INT64_MAX : tk.seg[0].n_end;
      const int64_t e1 = tk.nseg < 3 ? INT64_MAX : tk.seg[1].n_end;
      uint16_t* const y0 = tk.seg[0].y;
      uint16_t* const y1 = tk.seg[1].y;
      uint16_t* const y2 = tk.seg[2].y;
      const uint16_t* const b0 = tk.seg[0].bias;
      const uint16_t* const b1 = tk.seg[1].bias;
      const uint16_t* const b2 = tk.seg[2].bias;
      const bool has_bias = b0 != nullptr || b1 != nullptr || b2 != nullptr;
      // lanes per row: a power of two (for the butterfly) with lpr * RB <= 32
      int lpr = 1;
      while (2 * lpr * tp.RB <= 32) lpr *= 2;
      const int rows_per_pass = 32 / lpr;
      const int part = lane & (lpr - 1);
      for (int t = 0; t < ntiles; ++t) {
        if (!mbar_wait_bounded(redfull0 + 8 * s, phase, kWaitLimitNs)) {
          if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
          return;
        }
        const int lr0 = t * tp.RB;
        const int nr = rows - lr0 < tp.RB ? rows - lr0 : tp.RB;
        // every lane runs every pass: the shuffles take the whole warp
        for (int row0 = 0; row0 < tp.RB; row0 += rows_per_pass) {
          const int row = row0 + lane / lpr;
          const uint32_t rp = rs + row * tp.red_stride * 4;
          // four running sums so the shared loads overlap; the order of the
          // additions is fixed, so every run gives the same bits
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
          if (row < tp.RB) {
            int u = part;
            for (; u + 3 * lpr < tp.U; u += 4 * lpr) {
              s0 += lds_f32(rp + 4 * u);
              s1 += lds_f32(rp + 4 * (u + lpr));
              s2 += lds_f32(rp + 4 * (u + 2 * lpr));
              s3 += lds_f32(rp + 4 * (u + 3 * lpr));
            }
            for (; u < tp.U; u += lpr) s0 += lds_f32(rp + 4 * u);
          }
          float sum = (s0 + s1) + (s2 + s3);
          for (int o = lpr >> 1; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
          if (part == 0 && row < nr &&
              W4A16_IN(p.status, row_begin + lr0 + row < tk.N && (tk.split == 0 || lr0 + row < kM1PartRows))) {
            const uint32_t pa = part0 + 4 * static_cast<uint32_t>(lr0 + row);
            if (tk.split == 1) {
              // the first half of a K-split row: kept for the second half
              sts_f32(pa, sum);
            } else {
              // y[n] = fp16_RN(first half + sum + bias), routed to n's segment
              if (tk.split == 2) sum = lds_f32(pa) + sum;
              const int64_t n = row_begin + lr0 + row;
              const int seg = n < e0 ? 0 : (n < e1 ? 1 : 2);
              const int64_t j = seg == 0 ? n : (seg == 1 ? n - e0 : n - e1);
              if (has_bias) {
                const uint16_t* b = seg == 0 ? b0 : (seg == 1 ? b1 : b2);
                if (b != nullptr) sum += __half2float(__ushort_as_half(__ldg(b + j)));
              }
              uint16_t* y = seg == 0 ? y0 : (seg == 1 ? y1 : y2);
              const uint16_t yb = __half_as_ushort(__float2half_rn(sum));
              y[j] = yb;
              if (kAct && tk.swiglu != 0) {
                // SwiGLU: the gate task keeps its rounded outputs after the
                // stages, one per row of this CTA; the up task's epilogue
                // reads the same row's (this warp wrote it in an earlier
                // task: the __syncwarp of each tile orders the two)
                const uint32_t ga = stage0 + static_cast<uint32_t>(S * p.stage_bytes + 2 * (lr0 + row));
                if (W4A16_IN(p.status, lr0 + row < kM1PartRows)) {
                  if (tk.swiglu == 1)
                    sts_u16(ga, yb);
                  else
                    tk.epi_h[j] = swiglu1(lds_u16(ga), yb);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(redempty0 + 8 * s);
        rs += p.red_bytes;
        if (++s == S) {
          s = 0;
          phase ^= 1u;
          rs = red0;
        }
      }
      if (p.done != nullptr && tk.publish) {
        // this CTA's rows of task i are written: publish them to the grid
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.done + i, 1);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int c = tid - 32 * CW0;
  const int cw = warp - CW0;
  pdl_wait();  // x may be the previous kernel's output
  int s = 0, g = 0;  // stage, tiles consumed so far (all tasks)
  uint32_t phase = 0;
  int nwait = 0;  // dependent tasks with rows here so far (the next one's signal index)
  int nx = 0;     // activation slots used (W4A16)
  uint32_t base = stage0, rs = red0;
  for (int i = 0; i < p.ntasks; ++i) {
    const M1Task& tk = p.task[i];
    const TaskPlan tp = task_plan(tk.K, kFmt, task_parts(tk));
    int64_t row_begin;
    const int rows = cta_rows(tk, &row_begin);
    const int ntiles = small_div(rows + tp.RB - 1, tp.RB);
    if (ntiles == 0) continue;

    // Consecutive threads take consecutive units of one row, so a warp reads
    // 32 units' contiguous bytes of a stage.  The 16-byte chunks of a unit
    // are read in a rotated order so that every quarter-warp phase of the
    // 16-byte shared loads touches 8 distinct bank groups (except where the
    // quarter-warp spans two rows): W4A16 (four chunks of a 64-byte unit)
    // starts at chunk f = (u / 2) mod 4; the 64-k formats (two chunks of a
    // 32-byte unit) swap them when bit 2 of the unit is set.  The order is a
    // function of the unit alone, so a row's sum is the same whichever
    // thread and CTA compute it.  Threads past T (in a partly used warp)
    // compute on unit 0 of row 0 and store nothing; wholly unused warps only
    // keep the barrier counts.
    constexpr int kR = rows_per_thread(kFmt);
    const bool wact = cw * 32 < tp.T;
    // checked build: a thread whose rows, unit and partial slot do not fit
    // the stage and the slots computes on unit 0 of row 0 and stores nothing
    const bool active =
        c < tp.T && W4A16_IN(p.status, (c / tp.U + (kR - 1) * tp.RL + 1) * tp.row_bytes <= tp.RB * tp.row_bytes &&
                                           4 * ((c / tp.U + (kR - 1) * tp.RL) * tp.red_stride + c % tp.U + 1) <= p.red_bytes &&
                                           (kFmt != kFmtW4A16 || !staged(tk, i) || tp.U * 260 <= p.xslot));
    const int cq = small_div(c, tp.U);
    const int u = active ? c - cq * tp.U : 0;
    const int rl = active ? cq : 0;
    const int rot = ((u >> 2) & 1) * 16;
    const int f = (u >> 1) & 3;

    // this thread's activations (W4A16: 128, else 64), paired to match the
    // unpacked lanes
    XPairs X[kFmt == kFmtW4A16 ? 16 : 8];
    float C = 0.f;
    // the index of this task's dependency signal (every dependent task with
    // rows here has one, in order)
    const int sig = tk.dep >= 0 && p.done != nullptr ? nwait++ : -1;
    if constexpr (kFmt == kFmtW4A16) if (!staged(tk, i)) {
      // this thread's own 128 activations, loaded from global memory:
      // X[4 j + i] pairs with word 4 ((j + f) mod 4) + i of the unit, the
      // order in which the tiles' words are read.  Plain loads through L1:
      // x of a dependent task is read after the reducer's acquire.
      if (sig >= 0 && !mbar_wait_bounded(xready0 + 8 * (sig % kXReady), (sig / kXReady) & 1, kWaitLimitNs)) {
        if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
        return;
      }
      if (wact) {
        const uint16_t* xp = tk.x + u * 128;
        float es[4], os[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int ch = (j + f) & 3;
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            X[4 * j + i4] = pair_activations(ld_u4(xp + 32 * ch + 8 * i4));
          }
          chunk_bias(&X[4 * j], es[j], os[j]);
        }
        float e[4], o[4];
        unrotate4(es, f, e);
        unrotate4(os, f, o);
        C = unit_bias(e, o);
      }
    } else {
      // from the stager's slot: X[4 j + i] pairs with word 4 ((j + f) mod 4) + i
      // of the unit, the order in which the tiles' words are read
      const int sl = nx % kXSlots;
      if (!mbar_wait_bounded(xfull0 + 8 * sl, (nx / kXSlots) & 1, kWaitLimitNs)) {
        if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
        return;
      }
      const uint32_t xs = xslot0 + sl * p.xslot;
      if (wact) {
        const uint32_t xu = xs + u * 256;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int w0 = 4 * ((j + f) & 3);
#pragma unroll
          for (int i4 = 0; i4 < 4; ++i4) {
            const uint4 v = lds_u4(xu + (((w0 + i4) ^ (u & 15)) << 4));
            X[4 * j + i4] = XPairs{v.x, v.y, v.z, v.w};
          }
        }
        C = lds_f32(xs + tp.U * 256 + 4 * u);
      }
      // the slot's values are in registers once these reads are issued
      // (release order): the stager may refill it
      __syncwarp();
      if (lane == 0) mbar_arrive(xempty0 + 8 * sl);
      ++nx;
    }
    if (kFmt != kFmtW4A16 && sig >= 0 &&
        !mbar_wait_bounded(xready0 + 8 * (sig % kXReady), (sig / kXReady) & 1, kWaitLimitNs)) {
      if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
      return;
    }
    // W4A8: the unit's int8 codes (even / odd k of each word as 4 bytes), 8
    // times their sum, and the unit's activation scale
    uint32_t xe[8], xo[8];
    int C8 = 0;
    float s_act = 0.f;
    if constexpr (kFmt == kFmtW4A8) if (wact) {
      const uint16_t* xp = tk.x + u * 64;
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = rot ? (j ^ 4) : j;
        v[j] = ld_u4(xp + 8 * jj);
      }
      // max |x| with packed fp16 operations (exact), as a tree
      __half2 m2[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const __half2 a = __habs2(*reinterpret_cast<const __half2*>(&v[j].x));
        const __half2 b = __habs2(*reinterpret_cast<const __half2*>(&v[j].y));
        const __half2 c = __habs2(*reinterpret_cast<const __half2*>(&v[j].z));
        const __half2 d = __habs2(*reinterpret_cast<const __half2*>(&v[j].w));
        m2[j] = __hmax2(__hmax2(a, b), __hmax2(c, d));
      }
      const __half2 mm = __hmax2(__hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3])),
                                 __hmax2(__hmax2(m2[4], m2[5]), __hmax2(m2[6], m2[7])));
      const float amax = fmaxf(__low2float(mm), __high2float(mm));
      s_act = amax > 0.f ? amax / 127.f : 0.f;
      const float inv = amax > 0.f ? 127.f / amax : 0.f;
      // codes: one FP32 product and one round-to-nearest-even conversion each
      // (|x inv| <= 127 (1 + 2^-23): no clamp), packed 4 to a word; their sum
      // through dp4a with ones
      int csum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
        int ce[4], co[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          ce[i] = __float2int_rn(half_lo(w4[i]) * inv);
          co[i] = __float2int_rn(half_hi(w4[i]) * inv);
        }
        xe[j] = pack_bytes(ce[0], ce[1], ce[2], ce[3]);
        xo[j] = pack_bytes(co[0], co[1], co[2], co[3]);
        csum = __dp4a(static_cast<int>(xe[j]), 0x01010101, csum);
        csum = __dp4a(static_cast<int>(xo[j]), 0x01010101, csum);
      }
      C8 = 8 * csum;
    }
    // Q4_K: the pairs above and the two 32-activation sums
    float S0 = 0.f, S1 = 0.f;
    if constexpr (kFmt == kFmtQ4K) if (wact) {
      const uint4* xp = reinterpret_cast<const uint4*>(tk.x + u * 64);
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = ld_u4(xp + j);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint4 lo = v[t >> 1], hi = v[4 + (t >> 1)];
        const uint32_t la = (t & 1) ? lo.z : lo.x, lb = (t & 1) ? lo.w : lo.y;
        const uint32_t ha = (t & 1) ? hi.z : hi.x, hb = (t & 1) ? hi.w : hi.y;
        X[t].p0 = __byte_perm(la, lb, 0x5410u);
        X[t].p1 = __byte_perm(la, lb, 0x7632u);
        X[t].p2 = __byte_perm(ha, hb, 0x5410u);
        X[t].p3 = __byte_perm(ha, hb, 0x7632u);
        S0 += (half_lo(la) + half_hi(la)) + (half_lo(lb) + half_hi(lb));
        S1 += (half_lo(ha) + half_hi(ha)) + (half_lo(hb) + half_hi(hb));
      }
    }
    // per-thread offsets inside a stage and a partial slot: rows rl + r RL
    const int w_off = rl * tp.row_bytes + u * (unit_k(kFmt) / 2);
    const int w_row_step = tp.RL * tp.row_bytes;
    const int sc_off = tp.RB * tp.row_bytes + rl * tp.sc_pitch + (kFmt == kFmtW4A16 ? u : (u >> 1)) * 2;
    const int sc_row_step = tp.RL * tp.sc_pitch;
    const int red_off = 4 * (rl * tp.red_stride + u);
    const int red_row_step = 4 * tp.RL * tp.red_stride;
    const int sc_tile_step = tp.RB * tp.sc_pitch;
    // offset of the tile's first scale byte in its 16-byte-aligned window
    int sc_lo = static_cast<int>((reinterpret_cast<uintptr_t>(tk.scales) + row_begin * tp.sc_pitch) & 15);

    // 64-k formats: the next task with rows here has its activations go to
    // L1 ahead of time, one 128-byte line per thread (K / 64 lines), right
    // away when it reads nothing written in this launch, else once its
    // signal has arrived (W4A16: the stager loads them).
    int inext = i + 1;
    while (inext < p.ntasks && !cta_has_rows(p.task[inext])) ++inext;
    const uint16_t* xnext = nullptr;
    bool pending = false;
    if (kFmt != kFmtW4A16 && inext < p.ntasks && c < (p.task[inext].K >> 6)) {
      xnext = p.task[inext].x + c * 64;
      if (p.task[inext].dep < 0 || p.done == nullptr) {
        prefetch_l1(xnext);
      } else {
        pending = true;
      }
    }

    // whether tile t's stage was already seen full, at the end of tile t - 1
    bool full_seen = false;
    for (int t = 0; t < ntiles; ++t) {
      if (!full_seen && !mbar_wait_bounded(full0 + 8 * s, phase, kWaitLimitNs)) {
        if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
        return;
      }
      const int nr = rows - t * tp.RB;  // rows of this tile (may exceed RB)
      if (pending && mbar_try_wait(xready0 + 8 * (nwait % kXReady), (nwait / kXReady) & 1)) {
        prefetch_l1(xnext);
        pending = false;
      }
      float res[kR];
      if (!wact) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
      } else if constexpr (kFmt == kFmtQ4K) {
        // rows rl + r RL: the unit's block header and 32 code bytes
        const uint32_t ua = base + rl * tp.row_bytes + (u >> 2) * 144;
        const int cc = u & 3;
        const uint32_t selp = (cc & 1) ? 0x7632u : 0x5410u, selq = (cc & 1) ? 0x3232u : 0x1010u;
        const bool hi = cc >= 2;
        uint4 h[2], qa, qb;
        uint32_t q[8];
        float D0, D1;
#pragma unroll
        for (int r = 0; r < kR; ++r) {
          const uint32_t ra = ua + r * w_row_step;
          h[r & 1] = lds_u4(ra);
          qa = lds_u4(ra + 16 + 32 * cc);
          qb = lds_u4(ra + 32 + 32 * cc);
          if (r == kR - 1) {
            // the last reads of the stage are issued: release it
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * s);
          }
          q[0] = qa.x; q[1] = qa.y; q[2] = qa.z; q[3] = qa.w;
          q[4] = qb.x; q[5] = qb.y; q[6] = qb.z; q[7] = qb.w;
          q4k_dot(q, X, D0, D1);
          res[r] = q4k_combine(h[r & 1], selp, selq, hi, D0, D1, S0, S1);
        }
      } else if constexpr (kFmt == kFmtW4A16) {
        // rows rl and rl + RL: one scale and 16 words each.  The second row
        // is skipped by a warp none of whose threads has it in this tile (a
        // tile's last rows).
        const uint32_t sa = base + sc_off + sc_lo;
        const uint32_t wa = base + w_off;
        const float sc0 = __half2float(__ushort_as_half(lds_u16(sa)));
        const float sc1 = __half2float(__ushort_as_half(lds_u16(sa + sc_row_step)));
        uint32_t w[16];
        load_unit128(wa, f, w);
        res[0] = (dot_unit128(w, X) - C) * sc0;
        const bool any1 = __any_sync(0xffffffffu, active && rl + tp.RL < nr);
        if (any1) load_unit128(wa + w_row_step, f, w);
        // the last reads of the stage are issued: release it (release order)
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        res[1] = any1 ? (dot_unit128(w, X) - C) * sc1 : 0.f;
      } else {
        const uint32_t sa = base + sc_off + sc_lo;
        float sc[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) sc[r] = __half2float(__ushort_as_half(lds_u16(sa + r * sc_row_step)));
        const uint32_t wa = base + w_off;
        uint32_t w0[8], w1[8];
        load_row(wa, rot, w0);
        load_row(wa + w_row_step, rot, w1);
        int i0, i1;
        dot_pair_a8(w0, w1, xe, xo, i0, i1);
        res[0] = static_cast<float>(i0 - C8) * (sc[0] * s_act);
        res[1] = static_cast<float>(i1 - C8) * (sc[1] * s_act);
        load_row(wa + 2 * w_row_step, rot, w0);
        load_row(wa + 3 * w_row_step, rot, w1);
        // the last reads of the stage are issued: release it (release order)
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * s);
        dot_pair_a8(w0, w1, xe, xo, i0, i1);
        res[2] = static_cast<float>(i0 - C8) * (sc[2] * s_act);
        res[3] = static_cast<float>(i1 - C8) * (sc[3] * s_act);
      }
      // partial slot s still holds tile g - S until the reducer has read it
      if (g >= S && !mbar_wait_bounded(redempty0 + 8 * s, phase ^ 1u, kWaitLimitNs)) {
        if (lane == 0) atomicOr(p.status, W4A16_DEV_PIPE_TIMEOUT);
        return;
      }
      if (active) {
#pragma unroll
        for (int r = 0; r < kR; ++r)
          if (rl + r * tp.RL < nr) sts_f32(rs + red_off + r * red_row_step, res[r]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(redfull0 + 8 * s);
      sc_lo = (sc_lo + sc_tile_step) & 15;
      ++g;
      base += p.stage_bytes;
      rs += p.red_bytes;
      if (++s == S) {
        s = 0;
        phase ^= 1u;
        base = stage0;
        rs = red0;
      }
      // A non-blocking look at the next tile's stage (acquire): when it has
      // landed, the next tile starts without the blocking wait.  Measured on
      // the 28-layer step (same box): 0.6640 -> 0.6580 ms.
      full_seen = t + 1 < ntiles && mbar_try_wait(full0 + 8 * s, phase);
    }
  }
}

template <int MAXT>
cudaError_t launch_tasks(const M1Params<MAXT>& p, const RingPlan& rp, int grid, bool pdl, bool act, int fmt,
                         cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(32 * (first_consumer_warp(fmt) + rp.CW));
  cfg.dynamicSmemBytes = rp.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (p.done != nullptr) {
    // CTAs wait on each other's completion counters: the launch must make
    // every CTA resident at once, or fail (e.g. when fewer SMs are free)
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t e;
  if constexpr (MAXT == 1) {
    // Q4_K runs as a single task without an activation epilogue
    if (fmt != kFmtQ4K || act) return cudaErrorInvalidValue;
    e = cudaLaunchKernelEx(&cfg, gemv_m1_kernel<MAXT, false, kFmtQ4K>, p);
  } else {
    if (fmt == kFmtQ4K) return cudaErrorInvalidValue;
    if (fmt == kFmtW4A8)
      e = act ? cudaLaunchKernelEx(&cfg, gemv_m1_kernel<MAXT, true, kFmtW4A8>, p)
              : cudaLaunchKernelEx(&cfg, gemv_m1_kernel<MAXT, false, kFmtW4A8>, p);
    else
      e = act ? cudaLaunchKernelEx(&cfg, gemv_m1_kernel<MAXT, true, kFmtW4A16>, p)
              : cudaLaunchKernelEx(&cfg, gemv_m1_kernel<MAXT, false, kFmtW4A16>, p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Shared checks and plan of a task list; fills the launch fields of p.
template <int MAXT>
bool plan_tasks(M1Params<MAXT>& p, const M1Task* tasks, int ntasks, int fmt, const DeviceInfo& d, int grid,
                RingPlan* rp) {
  *rp = make_ring_plan(tasks, ntasks, d.max_smem_optin, fmt, MAXT > 2);
  if (rp->S < 2) return false;
  p.S = rp->S;
  p.stage_bytes = rp->stage_bytes;
  p.red_bytes = rp->red_bytes;
  p.xslot = rp->xslot;
  p.CW = rp->CW;
  p.pace = static_cast<float>(grid) * 1000.f / kPaceBytesPerUs;
  return true;
}

// ---------------------------------------------------------------- short rows
// A standalone M = 1 GEMV with K <= 4096 (at most 32 units of 128 k per row)
// and few bytes is bound by the task kernel's fixed costs (its ring, its
// roles, its one CTA per SM).  This kernel computes the same bits with a
// short latency: one warp per row, lane u < U owns unit u.  Each lane does
// what a consumer thread of gemv_m1_kernel does for the unit -- the 16 words
// in the rotated order f = (u / 2) mod 4, the 128 activations paired and
// their bias sum C in the same order, (dot - C) x scale -- and lanes 0..3
// form the task kernel's reducer for such a row (one lane per row when
// K <= 4096): four running sums over the units u = q (mod 4), the units
// past the last whole four added to the first, combined as
// (s0 + s1) + (s2 + s3), then the bias and one rounding.  So a call gives
// the same bits here as inside a layer sequence.
constexpr int kShortWarps = 8;

__global__ void __launch_bounds__(32 * kShortWarps) gemv_m1_short_kernel(const GemvArgs a) {
  __shared__ float part[kShortWarps][32];
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int U = a.K / 128;
  const int G = a.K / 128;
  const int u = lane;
  const bool act = u < U;
  const int f = (u >> 1) & 3;
  const int64_t N = a.N;
  const int64_t step = static_cast<int64_t>(gridDim.x) * kShortWarps;
  int64_t n = static_cast<int64_t>(blockIdx.x) * kShortWarps + warp;

  // this lane's 16 words of row `row` (chunk (j + f) mod 4 into words
  // 4 j .. 4 j + 3, as load_unit128 reads a stage) and its scale
  auto load_row = [&](int64_t row, uint32_t (&w)[16], float& sc) {
    // checked build: the unit's 16 words and its scale inside the row
    if (act && row < N && W4A16_IN(a.status, 16 * u + 16 <= a.K / 8 && u < G)) {
      const uint4* src = reinterpret_cast<const uint4*>(a.qweight + row * (a.K / 8) + 16 * u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = ld_stream_u4(src + ((j + f) & 3));
        w[4 * j] = v.x;
        w[4 * j + 1] = v.y;
        w[4 * j + 2] = v.z;
        w[4 * j + 3] = v.w;
      }
      sc = __half2float(__ushort_as_half(ld_nc_u16(a.scales + row * G + u)));
    }
  };
  uint32_t w[16] = {};
  float sc = 0.f;
  load_row(n, w, sc);  // weights and scales are constant: before the dependency wait
  pdl_wait();          // x may be the previous kernel's output; y may still be read by it

  // the lane's 128 activations, paired as the task kernel's consumers pair
  // them (X[4 j + i] with word 4 ((j + f) mod 4) + i), and their bias sum
  XPairs X[16];
  float C = 0.f;
  if (act && W4A16_IN(a.status, 128 * u + 128 <= a.K)) {
    const uint16_t* xp = a.x + u * 128;
    float es[4], os[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int ch = (j + f) & 3;
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) X[4 * j + i4] = pair_activations(ld_u4(xp + 32 * ch + 8 * i4));
      chunk_bias(&X[4 * j], es[j], os[j]);
    }
    float e[4], o[4];
    unrotate4(es, f, e);
    unrotate4(os, f, o);
    C = unit_bias(e, o);
  }
  const int u4 = U & ~3;  // units in whole fours
  for (; n < N; n += step) {
    const float res = act ? (dot_unit128(w, X) - C) * sc : 0.f;
    load_row(n + step, w, sc);  // the next row's words, in flight during the sum
    part[warp][lane] = res;
    __syncwarp();
    float s = 0.f;
    if (lane < 4) {
      for (int v = lane; v < u4; v += 4) s += part[warp][v];
      if (lane == 0)
        for (int v = u4; v < U; ++v) s += part[warp][v];
    }
    const float s1 = __shfl_sync(0xffffffffu, s, 1);
    const float s2 = __shfl_sync(0xffffffffu, s, 2);
    const float s3 = __shfl_sync(0xffffffffu, s, 3);
    if (lane == 0 && W4A16_IN(a.status, n < N)) store_out(a, 0, n, (s + s1) + (s2 + s3));
    __syncwarp();
  }
}

}  // namespace

bool gemv_m1_supported(int K) {
  return K > 0 && K % 128 == 0 && K / 64 <= kM1MaxConsumers;
}

bool gemv_m1_short_supported(int K) { return K > 0 && K % 128 == 0 && K / 128 <= 32; }

cudaError_t launch_gemv_m1_short(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (a.M != 1 || a.a8 || !gemv_m1_short_supported(a.K)) return cudaErrorInvalidValue;
  const int64_t rows_per_cta = kShortWarps;
  int64_t grid = (static_cast<int64_t>(a.N) + rows_per_cta - 1) / rows_per_cta;
  if (grid > 2 * d.sms) grid = 2 * d.sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(32 * kShortWarps);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemv_m1_short_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int gemv_m1_split_tasks(const M1Task& t, bool a8, const DeviceInfo& d, M1Task* out) {
  out[0] = t;
  out[0].split = 0;
  if (a8 || split_parts(t.K, t.N, d.sms) == 1) return 1;
  const int h = t.K / 2;
  out[0].K = h;
  out[0].split = 1;
  out[0].publish = 0;
  out[1] = t;
  out[1].K = h;
  out[1].split = 2;
  out[1].qweight = t.qweight + h / 8;
  out[1].scales = t.scales + h / 128;
  out[1].x = t.x + h;
  out[0].swiglu = 0;  // the first half writes nothing
  return 2;
}

cudaError_t launch_gemv_m1(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st) {
  if (!gemv_m1_supported(a.K) || a.M != 1) return cudaErrorInvalidValue;
  M1Task t{};
  t.qweight = a.qweight;
  t.scales = a.scales;
  t.x = a.x;
  t.N = a.N;
  t.K = a.K;
  t.swiglu = 0;
  t.nseg = static_cast<uint8_t>(a.nseg);
  t.dep = -1;
  t.publish = 0;
  for (int s = 0; s < kMaxSegs; ++s) t.seg[s] = M1Seg{a.seg[s].y, a.seg[s].bias, a.seg[s].n_end};
  M1Params<2> p{};
  p.ntasks = gemv_m1_split_tasks(t, a.a8, d, p.task);
  p.done = nullptr;
  p.status = a.status;
  // no dependency counting: CTAs beyond N would have no rows
  const int grid = a.N < d.sms ? a.N : d.sms;
  for (int i = 0; i < p.ntasks; ++i) {
    p.task[i].rq = a.N / grid;
    p.task[i].rr = a.N % grid;
  }
  const int fmt = a.a8 ? kFmtW4A8 : kFmtW4A16;
  RingPlan rp;
  if (!plan_tasks(p, p.task, p.ntasks, fmt, d, grid, &rp)) return cudaErrorInvalidConfiguration;
  return launch_tasks(p, rp, grid, a.pdl, false, fmt, st);
}

bool gemv_m1_q4k_supported(int K) {
  return K > 0 && K % 256 == 0 && K / 64 <= kM1MaxConsumers;
}

cudaError_t launch_gemv_m1_q4k(const uint8_t* blocks, const uint16_t* x, uint16_t* y, int N, int K, bool pdl,
                               uint32_t* status, const DeviceInfo& d, cudaStream_t st) {
  if (!gemv_m1_q4k_supported(K) || N <= 0) return cudaErrorInvalidValue;
  M1Params<1> p{};
  p.ntasks = 1;
  p.done = nullptr;
  p.status = status;
  M1Task& tk = p.task[0];
  tk.qweight = reinterpret_cast<const uint32_t*>(blocks);
  tk.scales = nullptr;
  tk.x = x;
  tk.N = N;
  tk.K = K;
  tk.swiglu = 0;
  tk.nseg = 1;
  tk.dep = -1;
  tk.publish = 0;
  tk.split = 0;
  tk.seg[0] = M1Seg{y, nullptr, N};
  for (int s = 1; s < kMaxSegs; ++s) tk.seg[s] = M1Seg{nullptr, nullptr, N};
  const int grid = N < d.sms ? N : d.sms;
  tk.rq = N / grid;
  tk.rr = N % grid;
  RingPlan rp;
  if (!plan_tasks(p, p.task, 1, kFmtQ4K, d, grid, &rp)) return cudaErrorInvalidConfiguration;
  return launch_tasks(p, rp, grid, pdl, false, kFmtQ4K, st);
}

cudaError_t launch_gemv_m1_tasks(const M1Task* tasks, int ntasks, int* done, uint32_t* status,
                                 bool pdl, bool a8, const DeviceInfo& d, cudaStream_t st) {
  if (tasks == nullptr || ntasks <= 0 || ntasks > kM1MaxTasks) return cudaErrorInvalidValue;
  static thread_local M1Params<kM1MaxTasks> p;  // ~28 KB: kept off the stack
  for (int i = 0; i < ntasks; ++i) {
    const M1Task& t = tasks[i];
    if (!gemv_m1_supported(t.K * task_parts(t)) || t.N <= 0) return cudaErrorInvalidValue;
    if (t.dep >= i || (t.dep >= 0 && done == nullptr)) return cudaErrorInvalidValue;
    // a K split is two consecutive halves of one GEMV, small enough per CTA
    if (t.split > 2 || (t.split != 0 && (a8 || (t.N + d.sms - 1) / d.sms > kM1PartRows))) return cudaErrorInvalidValue;
    // a SwiGLU pair keeps one gate output per row of a CTA
    if (t.swiglu > 2 || (t.swiglu != 0 && (t.nseg != 1 || (t.N + d.sms - 1) / d.sms > kM1PartRows)) ||
        (t.swiglu == 2 && t.epi_h == nullptr))
      return cudaErrorInvalidValue;
    if (t.split == 1 && (i + 1 >= ntasks || tasks[i + 1].split != 2 || tasks[i + 1].N != t.N ||
                         tasks[i + 1].K != t.K))
      return cudaErrorInvalidValue;
    if (t.split == 2 && (i == 0 || tasks[i - 1].split != 1)) return cudaErrorInvalidValue;
    p.task[i] = t;
    p.task[i].rq = t.N / d.sms;
    p.task[i].rr = t.N % d.sms;
    p.task[i].publish = 0;
  }
  bool act = false;
  for (int i = 0; i < ntasks; ++i) {
    if (tasks[i].dep >= 0) p.task[tasks[i].dep].publish = 1;
    act = act || tasks[i].swiglu != 0;
  }
  p.ntasks = ntasks;
  p.done = done;
  p.status = status;
  const int fmt = a8 ? kFmtW4A8 : kFmtW4A16;
  RingPlan rp;
  if (!plan_tasks(p, p.task, ntasks, fmt, d, d.sms, &rp)) return cudaErrorInvalidConfiguration;
  // one CTA per SM: every CTA must be resident for the dependency counts
  return launch_tasks(p, rp, d.sms, pdl, act, fmt, st);
}

bool gemv_m1_swiglu_fits(int ffn, const DeviceInfo& d) { return (ffn + d.sms - 1) / d.sms <= kM1PartRows; }

bool gemv_m1_tasks_fit(const M1Task* tasks, int n, bool a8, const DeviceInfo& d) {
  if (tasks == nullptr || n <= 0) return false;
  for (int i = 0; i < n; ++i)
    if (!gemv_m1_supported(tasks[i].K * task_parts(tasks[i]))) return false;
  // a table's plan takes the largest stage of its tasks: the plan over all of
  // them bounds every subset's
  return make_ring_plan(tasks, n, d.max_smem_optin, a8 ? kFmtW4A8 : kFmtW4A16, true).S >= 2;
}

cudaError_t prepare_gemv_m1(const DeviceInfo& d) {
  const int limit = d.max_smem_optin < kM1SmemBudget ? d.max_smem_optin : kM1SmemBudget;
  const void* fns[] = {
      reinterpret_cast<const void*>(gemv_m1_kernel<1, false, kFmtQ4K>),
      reinterpret_cast<const void*>(gemv_m1_kernel<2, false, kFmtW4A16>),
      reinterpret_cast<const void*>(gemv_m1_kernel<2, true, kFmtW4A16>),
      reinterpret_cast<const void*>(gemv_m1_kernel<2, false, kFmtW4A8>),
      reinterpret_cast<const void*>(gemv_m1_kernel<2, true, kFmtW4A8>),
      reinterpret_cast<const void*>(gemv_m1_kernel<kM1MaxTasks, false, kFmtW4A16>),
      reinterpret_cast<const void*>(gemv_m1_kernel<kM1MaxTasks, true, kFmtW4A16>),
      reinterpret_cast<const void*>(gemv_m1_kernel<kM1MaxTasks, false, kFmtW4A8>),
      reinterpret_cast<const void*>(gemv_m1_kernel<kM1MaxTasks, true, kFmtW4A8>)};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace w4a16
