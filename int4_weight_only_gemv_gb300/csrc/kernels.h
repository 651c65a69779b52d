// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "w4a16.h"

namespace w4a16 {

// Where output row n of activation row m goes.  A GEMV over a weight made of
// up to three stacked matrices (e.g. [W_q; W_k; W_v]) can write each part to
// its own buffer: rows [n_begin(s), n_end(s)) go to seg[s].y with row stride
// seg[s].ldy (elements), n_begin(0) = 0, n_begin(s) = seg[s-1].n_end.  With
// a bias, y = fp16_RN(sum + bias[n - n_begin(s)]) (the fp16 bias added to the
// FP32 sum before the one rounding).
struct OutSeg {
  uint16_t* y;
  int64_t ldy;
  int64_t n_end;
  const uint16_t* bias;  // fp16 bits, one per row of the segment, or null
};
constexpr int kMaxSegs = 3;

// One GEMV: y[m][n] = sum_k x[m*ldx + k] * q[n][k] * s[n][k/128].
struct GemvArgs {
  const uint32_t* qweight;  // [N][K/8]
  const uint16_t* scales;   // [N][K/128] fp16 bits
  const uint16_t* x;        // [M][ldx] fp16 bits (first K used per row)
  int M, N, K;
  int64_t ldx;              // row stride of x in elements (K for a dense x)
  int nseg;                 // 1..kMaxSegs
  OutSeg seg[kMaxSegs];
  uint32_t* status;         // device status word (W4A16_DEV_* bits)
  // Programmatic dependent launch: the kernel may start while the previous
  // kernel on the stream is still running; it reads only the (constant)
  // weights and scales before waiting for that kernel to finish.
  bool pdl;
  // W4A8: int8 activations quantised per 64-element unit inside the M = 1
  // kernel (gemv_m1.cu); only that kernel supports it.
  bool a8;
  // M = 1 layer sequences only: the task's SwiGLU role (M1Task::swiglu) and,
  // for the up projection (2), where h goes.
  int swiglu;
  uint16_t* epi_h;
};

#ifdef __CUDACC__
// Epilogue: y[m][n] = fp16_RN(v + bias), routed to n's segment.
__device__ __forceinline__ void store_out(const GemvArgs& a, int m, int64_t n, float v) {
  int s = 0;
  int64_t n0 = 0;
  if (a.nseg > 1 && n >= a.seg[0].n_end) {
    n0 = a.seg[0].n_end;
    s = 1;
    if (a.nseg > 2 && n >= a.seg[1].n_end) {
      n0 = a.seg[1].n_end;
      s = 2;
    }
  }
  const OutSeg& sg = a.seg[s];
  if (sg.bias != nullptr) v += __half2float(__ushort_as_half(__ldg(sg.bias + (n - n0))));
  sg.y[m * sg.ldy + (n - n0)] = __half_as_ushort(__float2half_rn(v));
}
#endif

// One GEMV (M = 1) of a task list that a single launch of the M = 1 kernel
// runs in order.  Task i may read the output of an earlier task `dep` of the
// same list as its activations: its consumer warps then start once every CTA
// of the launch has written that output.  Weights and scales of every task
// must stay constant for the whole launch (they are streamed ahead of any
// dependency wait).
// An output segment of an M = 1 task (one activation row: no row stride).
struct M1Seg {
  uint16_t* y;
  const uint16_t* bias;  // fp16 bits or null (as OutSeg::bias)
  int64_t n_end;
};

struct M1Task {
  const uint32_t* qweight;  // [N][K/8]
  const uint16_t* scales;   // [N][K/128] fp16 bits
  const uint16_t* x;        // [K] fp16 bits
  uint16_t* epi_h;          // SwiGLU up task (swiglu = 2): where h goes; else null
  int N, K;
  int dep;                  // index of the task whose output x is, or -1
  int rq, rr;               // rows per CTA (set by the launcher): rq, one more for CTAs < rr
  uint8_t nseg;             // 1..kMaxSegs
  uint8_t publish;          // a later task reads this one's output (set by the launcher)
  // K-split of one GEMV into two consecutive tasks over the halves of each
  // row's K (rows of pitch 2 K): 1 = the first half (its row sums wait in
  // shared memory, nothing is written), 2 = the second half (adds them, then
  // the bias and the rounding; qweight, scales and x point at the half).
  // 0 = a whole GEMV.
  uint8_t split;
  // SwiGLU across two tasks over the same rows (one output segment each):
  // 1 = the gate, whose rounded outputs the CTA also keeps in shared memory;
  // 2 = the up projection, whose epilogue writes h[n] = fp16_RN(silu(g) y[n])
  // to epi_h[n] after y[n] is rounded, g the value the last gate task kept
  // for the same row; 0 = neither (set by the sequence builder).
  uint8_t swiglu;
  M1Seg seg[kMaxSegs];
};
static_assert(sizeof(M1Task) == 128, "a task record is 128 bytes (the table is kernel parameters)");
constexpr int kM1MaxTasks = 224;  // the task table travels in the kernel parameters

#ifdef __CUDACC__
// Epilogue of an M = 1 task: y[n] = fp16_RN(v + bias), routed to n's segment
// (selects, not an indexed segment: keeps the task table in parameter space).
__device__ __forceinline__ void store_out(const M1Task& a, int64_t n, float v) {
  const int64_t e0 = a.seg[0].n_end, e1 = a.seg[1].n_end;
  const bool s0 = a.nseg < 2 || n < e0;
  const bool s1 = !s0 && (a.nseg < 3 || n < e1);
  const int64_t j = s0 ? n : (s1 ? n - e0 : n - e1);
  uint16_t* y = s0 ? a.seg[0].y : (s1 ? a.seg[1].y : a.seg[2].y);
  const uint16_t* b = s0 ? a.seg[0].bias : (s1 ? a.seg[1].bias : a.seg[2].bias);
  if (b != nullptr) v += __half2float(__ushort_as_half(__ldg(b + j)));
  y[j] = __half_as_ushort(__float2half_rn(v));
}
#endif

// Device facts the launchers size their grids with.
struct DeviceInfo {
  int sms;
  int max_smem_optin;  // bytes of dynamic shared memory a block may opt into
};

// Kernel families.  Each returns cudaSuccess or the launch error.
// M = 1, K within the pipelined kernel's limit (see gemv_m1_supported).
bool gemv_m1_supported(int K);
cudaError_t launch_gemv_m1(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// M = 1 with K <= 4096: a warp-per-row kernel with the task kernel's exact
// per-unit arithmetic and row-sum order (the same bits as gemv_m1_kernel), for
// standalone GEMVs whose launch the task kernel's fixed costs would dominate.
bool gemv_m1_short_supported(int K);
cudaError_t launch_gemv_m1_short(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// The same kernel on GGUF Q4_K blocks (K a multiple of 256, blocks 16-byte
// aligned, one CTA per SM).
bool gemv_m1_q4k_supported(int K);
cudaError_t launch_gemv_m1_q4k(const uint8_t* blocks, const uint16_t* x, uint16_t* y, int N, int K, bool pdl,
                               uint32_t* status, const DeviceInfo& d, cudaStream_t st);
// A task list (1 <= ntasks <= kM1MaxTasks, every K supported, M = 1) in one
// launch of one CTA per SM.  done: ntasks ints, zero before the launch
// (per-task completion counters); required when a task has a dependency,
// may be null otherwise.  pdl: as GemvArgs::pdl.  A K-split GEMV is two
// consecutive tasks (M1Task::split), made by gemv_m1_split_tasks.
cudaError_t launch_gemv_m1_tasks(const M1Task* tasks, int ntasks, int* done, uint32_t* status,
                                 bool pdl, bool a8, const DeviceInfo& d, cudaStream_t st);
// Host-only: whether task lists over these tasks (any subset of them, in
// tables of up to kM1MaxTasks) pass launch_gemv_m1_tasks's own checks of K
// and the shared-memory plan on this device.
bool gemv_m1_tasks_fit(const M1Task* tasks, int n, bool a8, const DeviceInfo& d);
// Whether a SwiGLU over ffn-row gate and up tasks fits the task lists (the
// CTA keeps one gate output per row of its share).
bool gemv_m1_swiglu_fits(int ffn, const DeviceInfo& d);
// Host-only: the tasks of one M = 1 GEMV (its K, N, pointers in t, split 0):
// one task, or (W4A16 only, when split_parts says so) its two K halves.
// Writes 1 or 2 tasks to out and returns the count; dep and publish are
// copied to both.
int gemv_m1_split_tasks(const M1Task& t, bool a8, const DeviceInfo& d, M1Task* out);
// M = 1 (any K; used when K is beyond the M = 1 kernel's range): CUDA-core
// kernel with 8 warps per row block.
cudaError_t launch_gemv_rows(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// M = 2..16: mma.sync tensor-core kernel with cluster split-K, for every K
// that gemv_mma_supported accepts.
bool gemv_mma_supported(int K);
cudaError_t launch_gemv_mma(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// Decode attention (attn_decode.cu): head dimension 128, at most 16 query
// heads per KV head; arguments checked by the caller.
struct AttnArgs {
  const uint16_t* q;   // [n_heads][128]
  const uint16_t* k;   // [n_kv_heads][t_stride][128]
  const uint16_t* v;
  uint16_t* o;         // [n_heads][128]
  float* workspace;    // attn_workspace_bytes(n_kv_heads, attn_splits(...))
  int n_heads, n_kv_heads, T, t_stride;
  bool pdl;
  uint32_t* status;
};
int attn_splits(int n_kv_heads, int T, const DeviceInfo& d);
size_t attn_workspace_bytes(int n_kv_heads, int splits);
cudaError_t launch_attn_decode(const AttnArgs& a, const DeviceInfo& d, cudaStream_t st);
// GGUF Q4_K (q4k.cu): K a multiple of 256, blocks 16-byte aligned.
cudaError_t launch_q4k_dequant(const uint8_t* blocks, float* w, int N, int K, cudaStream_t st);
cudaError_t launch_q4k_gemv(const uint8_t* blocks, const uint16_t* x, uint16_t* y, int N, int K, bool pdl,
                            const DeviceInfo& d, cudaStream_t st);
size_t q4k_gemv_smem(int K);
cudaError_t prepare_q4k(const DeviceInfo& d);
// cuTensorMapEncodeTiled from the driver (null if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// h[m][j] = fp16_RN(silu(g[m*ld + j]) u[m*ld + j]) for j < n, rows of h with
// stride n (the SwiGLU step of an unfused layer sequence).
cudaError_t launch_swiglu(const uint16_t* g, const uint16_t* u, int64_t ld, uint16_t* h, int M, int n,
                          bool pdl, cudaStream_t st);
cudaError_t launch_dequant(const uint32_t* qweight, const uint16_t* scales, uint16_t* w_out,
                           int N, int K, cudaStream_t st);
cudaError_t launch_quantize(const float* w, uint32_t* qweight, uint16_t* scales, int N, int K,
                            uint32_t* status, cudaStream_t st);

// One thread waits (bounded by limit_ns) on an mbarrier nothing arrives on.
cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, uint32_t* status, cudaStream_t st);

// Set per-device function attributes (dynamic shared memory opt-in); each
// must run once per device before the first launch and outside stream capture.
cudaError_t prepare_gemv_m1(const DeviceInfo& d);
cudaError_t prepare_gemv_mma(const DeviceInfo& d);
cudaError_t prepare_attn_decode(const DeviceInfo& d);

// Wall-clock bound on any in-kernel wait (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

#ifdef __CUDACC__
// Index checks of the checked build (compiled with W4A16_CHECKED): when cond
// is false, W4A16_DEV_INDEX is set in the device status word and the caller
// skips the access.  In the normal build every check is the constant true and
// compiles to nothing.
#ifdef W4A16_CHECKED
__device__ __forceinline__ bool w4a16_check(uint32_t* status, bool cond) {
  if (!cond) atomicOr(status, W4A16_DEV_INDEX);
  return cond;
}
#define W4A16_IN(status, cond) ::w4a16::w4a16_check((status), (cond))
#else
#define W4A16_IN(status, cond) true
#endif
#endif

}  // namespace w4a16
