// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

// Where output row n of activation row m goes.  A GEMV over a weight made of
// up to three stacked matrices (e.g. [W_q; W_k; W_v]) can write each part to
// its own buffer: rows [n_begin(s), n_end(s)) go to seg[s].y with row stride
// seg[s].ldy (elements), n_begin(0) = 0, n_begin(s) = seg[s-1].n_end.
struct OutSeg {
  uint16_t* y;
  int64_t ldy;
  int64_t n_end;
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
};

#ifdef __CUDACC__
__device__ __forceinline__ uint16_t* out_ptr(const GemvArgs& a, int m, int64_t n) {
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
  return a.seg[s].y + m * a.seg[s].ldy + (n - n0);
}
#endif

// One GEMV (M = 1) of a task list that a single launch of the M = 1 kernel
// runs in order.  Task i may read the output of an earlier task `dep` of the
// same list as its activations: its consumer warps then start once every CTA
// of the launch has written that output.  Weights and scales of every task
// must stay constant for the whole launch (they are streamed ahead of any
// dependency wait).
struct M1Task {
  const uint32_t* qweight;  // [N][K/8]
  const uint16_t* scales;   // [N][K/128] fp16 bits
  const uint16_t* x;        // [K] fp16 bits
  int N, K;
  int nseg;                 // 1..kMaxSegs
  int dep;                  // index of the task whose output x is, or -1
  int rq, rr;               // rows per CTA (set by the launcher): rq, one more for CTAs < rr
  int publish;              // a later task reads this one's output (set by the launcher)
  OutSeg seg[kMaxSegs];     // ldy unused (one activation row)
};
constexpr int kM1MaxTasks = 224;  // the task table travels in the kernel parameters

#ifdef __CUDACC__
__device__ __forceinline__ uint16_t* out_ptr(const M1Task& a, int64_t n) {
  // selects, not an indexed segment: keeps the task table in parameter space
  const int64_t e0 = a.seg[0].n_end, e1 = a.seg[1].n_end;
  if (a.nseg < 2 || n < e0) return a.seg[0].y + n;
  if (a.nseg < 3 || n < e1) return a.seg[1].y + (n - e0);
  return a.seg[2].y + (n - e1);
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
// A task list (1 <= ntasks <= kM1MaxTasks, every K supported, M = 1) in one
// launch of one CTA per SM.  done: ntasks ints, zero before the launch
// (per-task completion counters); required when a task has a dependency,
// may be null otherwise.  pdl: as GemvArgs::pdl.
cudaError_t launch_gemv_m1_tasks(const M1Task* tasks, int ntasks, int* done, uint32_t* status,
                                 bool pdl, const DeviceInfo& d, cudaStream_t st);
// M = 1..7 (any K): warp-per-row-block CUDA-core kernel.
cudaError_t launch_gemv_rows(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// M = 8..16: mma.sync tensor-core kernel with cluster split-K.
cudaError_t launch_gemv_mma(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);

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

// Wall-clock bound on any in-kernel wait (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

}  // namespace w4a16
