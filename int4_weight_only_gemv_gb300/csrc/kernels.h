// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w4a16 {

// One GEMV: y[m][n] = sum_k x[m*ldx + k] * q[n][k] * s[n][k/128].
struct GemvArgs {
  const uint32_t* qweight;  // [N][K/8]
  const uint16_t* scales;   // [N][K/128] fp16 bits
  const uint16_t* x;        // [M][ldx] fp16 bits (first K used per row)
  uint16_t* y;              // [M][N] fp16 bits
  int M, N, K;
  int64_t ldx;              // row stride of x in elements (K for a dense x)
  uint32_t* status;         // device status word (W4A16_DEV_* bits)
};

// Device facts the launchers size their grids with.
struct DeviceInfo {
  int sms;
  int max_smem_optin;  // bytes of dynamic shared memory a block may opt into
};

// Kernel families.  Each returns cudaSuccess or the launch error.
// M = 1, K within the pipelined kernel's limit (see gemv_m1_supported).
bool gemv_m1_supported(int K);
cudaError_t launch_gemv_m1(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// M = 1..7 (any K): warp-per-row-block CUDA-core kernel.
cudaError_t launch_gemv_rows(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);
// M = 8..16: mma.sync tensor-core kernel with cluster split-K.
cudaError_t launch_gemv_mma(const GemvArgs& a, const DeviceInfo& d, cudaStream_t st);

cudaError_t launch_dequant(const uint32_t* qweight, const uint16_t* scales, uint16_t* w_out,
                           int N, int K, cudaStream_t st);
cudaError_t launch_quantize(const float* w, uint32_t* qweight, uint16_t* scales, int N, int K,
                            uint32_t* status, cudaStream_t st);

// Set per-device function attributes (dynamic shared memory opt-in); each
// must run once per device before the first launch and outside stream capture.
cudaError_t prepare_gemv_m1(const DeviceInfo& d);
cudaError_t prepare_gemv_mma(const DeviceInfo& d);

// Wall-clock bound on any in-kernel wait (nanoseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

}  // namespace w4a16
