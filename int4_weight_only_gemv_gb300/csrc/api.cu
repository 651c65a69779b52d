// api.cu -- the C ABI of include/w4a16.h: argument checks, kernel dispatch,
// the per-device status word and the graph-captured layer sequence.
//
// Every argument is checked on the host before anything is enqueued.  The
// only device memory the library allocates is a layer_seq's completion
// counters (one int per GEMV, M = 1), next to its CUDA graph, stream and event.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <thread>
#include <chrono>
#include <vector>

#include "kernels.h"
#include "w4a16.h"

namespace w4a16 {
namespace {

// Per-device word into which kernels OR the W4A16_DEV_* bits.
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  DeviceInfo info{};
  uint32_t* status = nullptr;  // device address of g_device_status on this device
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Query and cache the facts and attributes of the current device.  Runs
// cudaFuncSetAttribute, so the first call per device must not be made during
// stream capture; every entry point calls it before launching anything.
w4a16_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int sms = 0, smem = 0;
    void* addr = nullptr;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
    d.info.sms = sms;
    d.info.max_smem_optin = smem;
    d.status = static_cast<uint32_t*>(addr);
    if (prepare_gemv_m1(d.info) != cudaSuccess || prepare_gemv_mma(d.info) != cudaSuccess ||
        prepare_attn_decode(d.info) != cudaSuccess || prepare_q4k(d.info) != cudaSuccess) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
    d.ready = true;
  }
  *out = &d;
  return W4A16_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
  if (abytes == 0 || bbytes == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

// Shape / group checks shared by every weight-taking entry point.
w4a16_status check_weight_shape(int N, int K, int group) {
  if (group != W4A16_GROUP) return W4A16_ERR_GROUP;
  if (N < 0 || N > W4A16_MAX_N) return W4A16_ERR_SHAPE;
  if (K <= 0 || K % W4A16_GROUP != 0 || K > W4A16_MAX_K) return W4A16_ERR_SHAPE;
  return W4A16_OK;
}

// Full validation of one GEMV; x has row stride ldx (== K for the public call).
w4a16_status check_gemv(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                        const uint16_t* y, int M, int N, int K, int group, int64_t ldx) {
  w4a16_status s = check_weight_shape(N, K, group);
  if (s != W4A16_OK) return s;
  if (M < 0 || M > W4A16_MAX_M) return W4A16_ERR_M_RANGE;
  if (M == 0 || N == 0) return W4A16_OK;  // empty product
  if (!qweight || !scales || !x || !y) return W4A16_ERR_NULL;
  if (!aligned16(qweight) || !aligned16(scales) || !aligned16(x) || !aligned16(y))
    return W4A16_ERR_ALIGN;
  if (ldx < K || ldx % 8 != 0) return W4A16_ERR_SHAPE;
  const size_t wbytes = static_cast<size_t>(N) * (K / 2);
  const size_t sbytes = static_cast<size_t>(N) * (K / W4A16_GROUP) * 2;
  const size_t xbytes = (static_cast<size_t>(M - 1) * ldx + K) * 2;
  const size_t ybytes = static_cast<size_t>(M) * N * 2;
  if (overlaps(y, ybytes, x, xbytes) || overlaps(y, ybytes, qweight, wbytes) ||
      overlaps(y, ybytes, scales, sbytes))
    return W4A16_ERR_ALIAS;
  return W4A16_OK;
}

// Standalone M = 1 GEMVs with short rows and at most this many bytes of
// packed weights run on the warp-per-row kernel (the same bits as the task
// kernel); larger ones stream through the task kernel's ring.  Measured in
// graphs of back-to-back calls (cold L2): 512 x 1024 4.55 -> 3.41 us; at
// 512 x 3584 (0.9 MB) the two are even (4.63 / 4.72 us) and from 3584 x 3584
// on the ring is faster (5.0 / 6.2 us).
constexpr int64_t kShortMaxWeightBytes = 512 << 10;

// Enqueue one checked GEMV (M, N > 0) whose output rows go to the segments
// of `a` (pointers, sizes, strides and segments already filled in).
w4a16_status enqueue(const DeviceState& d, GemvArgs a, cudaStream_t st) {
  a.status = d.status;
  cudaError_t e;
  if (a.M == 1 && gemv_m1_short_supported(a.K) &&
      static_cast<int64_t>(a.N) * (a.K / 2) <= kShortMaxWeightBytes)
    e = launch_gemv_m1_short(a, d.info, st);
  else if (a.M == 1 && gemv_m1_supported(a.K))
    e = launch_gemv_m1(a, d.info, st);
  else if (a.M == 1)
    e = launch_gemv_rows(a, d.info, st);
  else if (gemv_mma_supported(a.K))
    e = launch_gemv_mma(a, d.info, st);
  else
    e = cudaErrorInvalidValue;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

GemvArgs plain_args(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                    uint16_t* y, int M, int N, int K, int64_t ldx, int64_t ldy) {
  GemvArgs a{};
  a.qweight = qweight;
  a.scales = scales;
  a.x = x;
  a.M = M;
  a.N = N;
  a.K = K;
  a.ldx = ldx;
  a.nseg = 1;
  a.seg[0] = OutSeg{y, ldy, N, nullptr};
  a.pdl = false;
  return a;
}

}  // namespace
}  // namespace w4a16

using namespace w4a16;

extern "C" {

const char* w4a16_status_str(w4a16_status s) {
  switch (s) {
    case W4A16_OK: return "ok";
    case W4A16_ERR_NULL: return "null pointer";
    case W4A16_ERR_SHAPE: return "bad shape (N, K or stride out of range, or K not a multiple of 128)";
    case W4A16_ERR_ALIGN: return "pointer not 16-byte aligned";
    case W4A16_ERR_GROUP: return "group size is not 128";
    case W4A16_ERR_M_RANGE: return "M outside 0..16";
    case W4A16_ERR_ALIAS: return "output overlaps an input";
    case W4A16_ERR_CUDA: return "CUDA runtime error";
    case W4A16_ERR_TIMEOUT: return "wait timed out";
    case W4A16_ERR_STATE: return "invalid object handle";
    case W4A16_ERR_DEVICE: return "a kernel reported an error in the device status word";
    case W4A16_ERR_LIMIT:
      return "beyond the fixed limits of w4a16_layer_seq_run_static (GEMV count or K)";
  }
  return "unknown status";
}

int w4a16_abi_version(void) { return W4A16_ABI_VERSION; }

w4a16_status w4a16_gemv(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                        uint16_t* y, int M, int N, int K, int group, void* stream) {
  w4a16_status s = check_gemv(qweight, scales, x, y, M, N, K, group, K);
  if (s != W4A16_OK) return s;
  if (M == 0 || N == 0) return W4A16_OK;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  // a programmatic dependent of the previous kernel on the stream: the
  // kernels read only the constant weights and scales before waiting for it
  GemvArgs ga = plain_args(qweight, scales, x, y, M, N, K, K, N);
  ga.pdl = true;
  return enqueue(*d, ga, static_cast<cudaStream_t>(stream));
}

namespace {
constexpr int kAttnMaxT = 1 << 24;

w4a16_status check_attn_shape(int n_heads, int n_kv_heads, int head_dim, int T) {
  if (head_dim != 128 || n_heads <= 0 || n_kv_heads <= 0 || n_kv_heads > W4A16_ATTN_MAX_KV_HEADS ||
      n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > 16 || T < 1 || T > kAttnMaxT)
    return W4A16_ERR_SHAPE;
  return W4A16_OK;
}
}  // namespace

w4a16_status w4a16_attn_decode_workspace(int n_heads, int n_kv_heads, int head_dim, int T,
                                         size_t* bytes) {
  if (!bytes) return W4A16_ERR_NULL;
  *bytes = 0;
  w4a16_status s = check_attn_shape(n_heads, n_kv_heads, head_dim, T);
  if (s != W4A16_OK) return s;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  *bytes = attn_workspace_bytes(n_kv_heads, attn_splits(n_kv_heads, T, d->info));
  return W4A16_OK;
}

w4a16_status w4a16_attn_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                               uint16_t* o, int n_heads, int n_kv_heads, int head_dim, int T,
                               int t_stride, float* workspace, size_t workspace_bytes, void* stream) {
  w4a16_status s = check_attn_shape(n_heads, n_kv_heads, head_dim, T);
  if (s != W4A16_OK) return s;
  if (t_stride < T || t_stride > kAttnMaxT) return W4A16_ERR_SHAPE;
  if (!q || !k_cache || !v_cache || !o || !workspace) return W4A16_ERR_NULL;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(workspace))
    return W4A16_ERR_ALIGN;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  const size_t need = attn_workspace_bytes(n_kv_heads, attn_splits(n_kv_heads, T, d->info));
  if (workspace_bytes < need) return W4A16_ERR_SHAPE;
  const size_t qo = static_cast<size_t>(n_heads) * head_dim * 2;
  const size_t cache = static_cast<size_t>(n_kv_heads) * t_stride * head_dim * 2;
  if (overlaps(o, qo, q, qo) || overlaps(o, qo, k_cache, cache) || overlaps(o, qo, v_cache, cache) ||
      overlaps(o, qo, workspace, need) || overlaps(workspace, need, q, qo) ||
      overlaps(workspace, need, k_cache, cache) || overlaps(workspace, need, v_cache, cache))
    return W4A16_ERR_ALIAS;
  AttnArgs a;
  a.q = q;
  a.k = k_cache;
  a.v = v_cache;
  a.o = o;
  a.workspace = workspace;
  a.n_heads = n_heads;
  a.n_kv_heads = n_kv_heads;
  a.T = T;
  a.t_stride = t_stride;
  a.pdl = true;  // the partial kernel reads q and the caches only after its wait
  a.status = d->status;
  if (launch_attn_decode(a, d->info, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_gemv_a8(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                           uint16_t* y, int M, int N, int K, int group, void* stream) {
  w4a16_status s = check_gemv(qweight, scales, x, y, M, N, K, group, K);
  if (s != W4A16_OK) return s;
  if (M > 1) return W4A16_ERR_M_RANGE;
  if (!gemv_m1_supported(K)) return W4A16_ERR_SHAPE;
  if (M == 0 || N == 0) return W4A16_OK;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  GemvArgs a = plain_args(qweight, scales, x, y, M, N, K, K, N);
  a.a8 = true;
  a.pdl = true;  // as w4a16_gemv
  a.status = d->status;
  if (launch_gemv_m1(a, d->info, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

namespace {
w4a16_status check_q4k(const void* blocks, int N, int K) {
  if (K <= 0 || K % 256 != 0 || K > W4A16_MAX_K || N < 0 || N > W4A16_MAX_N) return W4A16_ERR_SHAPE;
  if (N > 0 && !blocks) return W4A16_ERR_NULL;
  if (N > 0 && !aligned16(blocks)) return W4A16_ERR_ALIGN;
  return W4A16_OK;
}
}  // namespace

w4a16_status w4a16_q4k_gemv(const uint8_t* blocks, const uint16_t* x, uint16_t* y, int N, int K,
                            void* stream) {
  w4a16_status s = check_q4k(blocks, N, K);
  if (s != W4A16_OK) return s;
  if (N == 0) return W4A16_OK;
  if (!x || !y) return W4A16_ERR_NULL;
  if (!aligned16(x) || !aligned16(y)) return W4A16_ERR_ALIGN;
  const size_t bbytes = static_cast<size_t>(N) * (K / 256) * 144;
  if (overlaps(y, static_cast<size_t>(N) * 2, blocks, bbytes) ||
      overlaps(y, static_cast<size_t>(N) * 2, x, static_cast<size_t>(K) * 2))
    return W4A16_ERR_ALIAS;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  // the persistent TMA-fed kernel where K fits its consumer threads, else the
  // warp-per-row kernel
  const cudaError_t e =
      gemv_m1_q4k_supported(K)
          ? launch_gemv_m1_q4k(blocks, x, y, N, K, true, d->status, d->info, static_cast<cudaStream_t>(stream))
          : launch_q4k_gemv(blocks, x, y, N, K, true, d->info, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_q4k_dequant(const uint8_t* blocks, float* w_out, int N, int K, void* stream) {
  w4a16_status s = check_q4k(blocks, N, K);
  if (s != W4A16_OK) return s;
  if (N == 0) return W4A16_OK;
  if (!w_out) return W4A16_ERR_NULL;
  if (!aligned16(w_out)) return W4A16_ERR_ALIGN;
  if (overlaps(w_out, static_cast<size_t>(N) * K * 4, blocks, static_cast<size_t>(N) * (K / 256) * 144))
    return W4A16_ERR_ALIAS;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  if (launch_q4k_dequant(blocks, w_out, N, K, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_dequant(const uint32_t* qweight, const uint16_t* scales, uint16_t* w_out,
                           int N, int K, int group, void* stream) {
  w4a16_status s = check_weight_shape(N, K, group);
  if (s != W4A16_OK) return s;
  if (N == 0) return W4A16_OK;
  if (!qweight || !scales || !w_out) return W4A16_ERR_NULL;
  if (!aligned16(qweight) || !aligned16(scales) || !aligned16(w_out)) return W4A16_ERR_ALIGN;
  const size_t obytes = static_cast<size_t>(N) * K * 2;
  if (overlaps(w_out, obytes, qweight, static_cast<size_t>(N) * (K / 2)) ||
      overlaps(w_out, obytes, scales, static_cast<size_t>(N) * (K / W4A16_GROUP) * 2))
    return W4A16_ERR_ALIAS;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  if (launch_dequant(qweight, scales, w_out, N, K, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_quantize(const float* w, uint32_t* qweight, uint16_t* scales, int N, int K,
                            int group, void* stream) {
  w4a16_status s = check_weight_shape(N, K, group);
  if (s != W4A16_OK) return s;
  if (N == 0) return W4A16_OK;
  if (!w || !qweight || !scales) return W4A16_ERR_NULL;
  if (!aligned16(w) || !aligned16(qweight) || !aligned16(scales)) return W4A16_ERR_ALIGN;
  const size_t wbytes = static_cast<size_t>(N) * K * 4;
  const size_t qbytes = static_cast<size_t>(N) * (K / 2);
  const size_t sbytes = static_cast<size_t>(N) * (K / W4A16_GROUP) * 2;
  if (overlaps(qweight, qbytes, w, wbytes) || overlaps(scales, sbytes, w, wbytes) ||
      overlaps(qweight, qbytes, scales, sbytes))
    return W4A16_ERR_ALIAS;
  DeviceState* d = nullptr;
  if ((s = device_state(&d)) != W4A16_OK) return s;
  if (launch_quantize(w, qweight, scales, N, K, d->status, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_selftest_wait_timeout(int limit_us, void* stream) {
  if (limit_us < 0 || limit_us > 10000000) return W4A16_ERR_SHAPE;
  DeviceState* d = nullptr;
  w4a16_status s = device_state(&d);
  if (s != W4A16_OK) return s;
  if (launch_wait_timeout_selftest(static_cast<uint64_t>(limit_us) * 1000u, d->status,
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_device_status(uint32_t* flags, int clear) {
  if (!flags) return W4A16_ERR_NULL;
  DeviceState* d = nullptr;
  w4a16_status s = device_state(&d);
  if (s != W4A16_OK) return s;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  uint32_t v = 0;
  if (cudaMemcpy(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  if (clear && v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
  }
  *flags = v;
  return v ? W4A16_ERR_DEVICE : W4A16_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- layer_seq

struct w4a16_layer_seq {
  int device = 0;
  int n_layers = 0, M = 0, hidden = 0, kv_dim = 0, ffn = 0;
  int launches = 0;
  w4a16_seq_io io{};
  cudaStream_t capture_stream = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaEvent_t done = nullptr;
  int* task_done = nullptr;  // per-GEMV completion counters of the task lists (M = 1)
  uint16_t* hbuf = nullptr;  // SwiGLU activations h (sequences with SwiGLU)
};

namespace {

void seq_free(w4a16_layer_seq* s) {
  if (!s) return;
  if (s->exec) cudaGraphExecDestroy(s->exec);
  if (s->graph) cudaGraphDestroy(s->graph);
  if (s->done) cudaEventDestroy(s->done);
  if (s->capture_stream) cudaStreamDestroy(s->capture_stream);
  if (s->task_done) cudaFree(s->task_done);
  if (s->hbuf) cudaFree(s->hbuf);
  delete s;
}

struct ProjSpec {
  int idx;        // W4A16_Q..W4A16_DOWN
  int N, K;
};

// Argument checks of a layer sequence: every GEMV of every layer is checked
// exactly as w4a16_gemv would check it.
w4a16_status check_seq_args(const w4a16_layer_weights* layers, int n_layers, int M, int hidden,
                            int kv_dim, int ffn, int group, const w4a16_seq_io* io) {
  if (!layers || !io) return W4A16_ERR_NULL;
  if (group != W4A16_GROUP) return W4A16_ERR_GROUP;
  if (n_layers <= 0) return W4A16_ERR_SHAPE;
  if (M <= 0 || M > W4A16_MAX_M) return W4A16_ERR_M_RANGE;
  if (hidden <= 0 || kv_dim <= 0 || ffn <= 0) return W4A16_ERR_SHAPE;
  if (!io->x || !io->y_q || !io->y_k || !io->y_v || !io->y_o || !io->y_gu || !io->y_down)
    return W4A16_ERR_NULL;

  const ProjSpec specs[W4A16_NPROJ] = {
      {W4A16_Q, hidden, hidden},   {W4A16_K, kv_dim, hidden}, {W4A16_V, kv_dim, hidden},
      {W4A16_O, hidden, hidden},   {W4A16_GATE, ffn, hidden}, {W4A16_UP, ffn, hidden},
      {W4A16_DOWN, hidden, ffn}};
  const int64_t Mh = static_cast<int64_t>(M) * hidden, Mkv = static_cast<int64_t>(M) * kv_dim,
                Mgu = static_cast<int64_t>(M) * 2 * ffn;
  for (int l = 0; l < n_layers; ++l) {
    const w4a16_layer_weights& w = layers[l];
    const uint16_t* xl = io->x + l * Mh;
    const uint16_t* yq = io->y_q + l * Mh;
    const uint16_t* ygu = io->y_gu + l * Mgu;
    const uint16_t* yout[W4A16_NPROJ] = {yq, io->y_k + l * Mkv, io->y_v + l * Mkv,
                                         io->y_o + l * Mh, ygu, ygu + ffn, io->y_down + l * Mh};
    const uint16_t* xin[W4A16_NPROJ] = {xl, xl, xl, yq, xl, xl, ygu};
    const int64_t ldx[W4A16_NPROJ] = {hidden, hidden, hidden, hidden, hidden, hidden, 2 * ffn};
    for (int pj = 0; pj < W4A16_NPROJ; ++pj) {
      const ProjSpec& ps = specs[pj];
      // the up projection writes the second half of each y_gu row: check it
      // as a GEMV with output row stride 2 ffn by treating rows as M = 1 views
      for (int m = 0; m < (pj == W4A16_GATE || pj == W4A16_UP ? M : 1); ++m) {
        const int mm = (pj == W4A16_GATE || pj == W4A16_UP) ? 1 : M;
        const uint16_t* yy = (pj == W4A16_GATE || pj == W4A16_UP) ? yout[pj] + m * 2 * ffn : yout[pj];
        const uint16_t* xx = xin[pj] + ((pj == W4A16_GATE || pj == W4A16_UP) ? m * ldx[pj] : 0);
        w4a16_status s = check_gemv(w.qweight[pj], w.scales[pj], xx, yy, mm, ps.N, ps.K, group,
                                    ldx[pj]);
        if (s != W4A16_OK) return s;
      }
    }
  }
  return W4A16_OK;
}

// The GEMVs of a checked layer sequence, in order.  Per layer: [q; k; v] as
// one GEMV when the three weights are stacked in one allocation (outputs
// still go to y_q, y_k, y_v), o, [gate; up] as one GEMV when stacked, down.
// dep[i] is the GEMV whose output GEMV i reads (o reads y_q, down the gate
// half of y_gu), or -1; layer_first[l] is the index of layer l's first GEMV
// (layer_first[n_layers] = number of GEMVs).
// Checks of the optional biases: 16-byte aligned, and no output of the
// sequence overlapping any bias.
w4a16_status check_seq_biases(const w4a16_layer_bias* biases, int n_layers, int M, int hidden,
                              int kv_dim, int ffn, const w4a16_seq_io* io) {
  if (biases == nullptr) return W4A16_OK;
  const int width[W4A16_NPROJ] = {hidden, kv_dim, kv_dim, hidden, ffn, ffn, hidden};
  const size_t L = static_cast<size_t>(n_layers) * M * 2;  // bytes per element x rows x layers
  const struct {
    const void* p;
    size_t bytes;
  } outs[6] = {{io->y_q, L * hidden},  {io->y_k, L * kv_dim},  {io->y_v, L * kv_dim},
               {io->y_o, L * hidden},  {io->y_gu, L * 2 * ffn}, {io->y_down, L * hidden}};
  for (int l = 0; l < n_layers; ++l)
    for (int pj = 0; pj < W4A16_NPROJ; ++pj) {
      const uint16_t* b = biases[l].bias[pj];
      if (b == nullptr) continue;
      if (!aligned16(b)) return W4A16_ERR_ALIGN;
      for (const auto& o : outs)
        if (overlaps(o.p, o.bytes, b, static_cast<size_t>(width[pj]) * 2)) return W4A16_ERR_ALIAS;
    }
  return W4A16_OK;
}

// Epilogue options of a layer sequence (w4a16_layer_seq_create2).
struct SeqOptions {
  const w4a16_layer_bias* biases = nullptr;  // n_layers entries or null
  unsigned flags = 0;                        // W4A16_SEQ_*
  uint16_t* hbuf = nullptr;  // SwiGLU activations h [n_layers][M][ffn], or null
};

// The SwiGLU step before a down GEMV outside the M = 1 task lists (there
// up's epilogue writes h): h[m][j] = fp16_RN(silu(g[m][j]) u[m][j]) for
// j < n (rows of g, u have stride ld, rows of h stride n).
struct ActOp {
  const uint16_t* g = nullptr;
  const uint16_t* u = nullptr;
  int64_t ld = 0;
  uint16_t* h = nullptr;  // null: no step
  int M = 0, n = 0;
};

// The GEMVs of a checked layer sequence, in order.  Per layer: [q; k; v] as
// one GEMV when the three weights are stacked in one allocation (outputs
// still go to y_q, y_k, y_v), o, [gate; up] as one GEMV when stacked, down.
// With SwiGLU fused into the M = 1 task lists (fuse_swiglu): up then gate as
// two GEMVs, up carrying the epilogue that writes h, and down reading h.
// dep[i] is the GEMV whose output GEMV i reads (o reads y_q; down the gate
// half of y_gu, or h: written by up's epilogue, or by a separate step after
// both halves, when dep2[i] is the other of gate and up if they are separate
// GEMVs), or -1; act[i] the separate SwiGLU step before GEMV i (unfused path);
// layer_first[l] is the index of layer l's first GEMV (layer_first[n_layers]
// = number of GEMVs).  Biases go to the output segments.
void build_seq_gemvs(const w4a16_layer_weights* layers, const SeqOptions& opt, int n_layers, int M,
                     int hidden, int kv_dim, int ffn, const w4a16_seq_io* io, bool fuse_swiglu,
                     std::vector<GemvArgs>* gemvs, std::vector<int>* dep, std::vector<int>* dep2,
                     std::vector<ActOp>* act,
                     std::vector<int>* layer_first) {
  gemvs->clear();
  dep->clear();
  dep2->clear();
  act->clear();
  layer_first->clear();
  const int64_t Mh = static_cast<int64_t>(M) * hidden, Mkv = static_cast<int64_t>(M) * kv_dim,
                Mgu = static_cast<int64_t>(M) * 2 * ffn;
  const size_t hw = static_cast<size_t>(hidden) / 8, hg = static_cast<size_t>(hidden) / W4A16_GROUP;
  const bool swiglu = (opt.flags & W4A16_SEQ_SWIGLU) != 0;
  auto stacked = [&](const w4a16_layer_weights& w, int first, int second, int rows_first) {
    return w.qweight[second] == w.qweight[first] + static_cast<size_t>(rows_first) * hw &&
           w.scales[second] == w.scales[first] + static_cast<size_t>(rows_first) * hg;
  };
  auto add = [&](const GemvArgs& a, int d) {
    gemvs->push_back(a);
    dep->push_back(d);
    dep2->push_back(-1);
    act->push_back(ActOp{});
    return static_cast<int>(gemvs->size()) - 1;
  };
  for (int l = 0; l < n_layers; ++l) {
    layer_first->push_back(static_cast<int>(gemvs->size()));
    const w4a16_layer_weights& w = layers[l];
    const uint16_t* const* bias = opt.biases != nullptr ? opt.biases[l].bias : nullptr;
    auto b = [&](int pj) { return bias != nullptr ? bias[pj] : nullptr; };
    const uint16_t* xl = io->x + l * Mh;
    uint16_t* yq = io->y_q + l * Mh;
    uint16_t* yk = io->y_k + l * Mkv;
    uint16_t* yv = io->y_v + l * Mkv;
    uint16_t* ygu = io->y_gu + l * Mgu;
    int iq;
    if (stacked(w, W4A16_Q, W4A16_K, hidden) && stacked(w, W4A16_K, W4A16_V, kv_dim)) {
      GemvArgs a = plain_args(w.qweight[W4A16_Q], w.scales[W4A16_Q], xl, yq, M,
                              hidden + 2 * kv_dim, hidden, hidden, hidden);
      a.nseg = 3;
      a.seg[0] = OutSeg{yq, hidden, hidden, b(W4A16_Q)};
      a.seg[1] = OutSeg{yk, kv_dim, static_cast<int64_t>(hidden) + kv_dim, b(W4A16_K)};
      a.seg[2] = OutSeg{yv, kv_dim, static_cast<int64_t>(hidden) + 2 * kv_dim, b(W4A16_V)};
      iq = add(a, -1);
    } else {
      GemvArgs a = plain_args(w.qweight[W4A16_Q], w.scales[W4A16_Q], xl, yq, M, hidden, hidden, hidden,
                              hidden);
      a.seg[0].bias = b(W4A16_Q);
      iq = add(a, -1);
      a = plain_args(w.qweight[W4A16_K], w.scales[W4A16_K], xl, yk, M, kv_dim, hidden, hidden, kv_dim);
      a.seg[0].bias = b(W4A16_K);
      add(a, -1);
      a = plain_args(w.qweight[W4A16_V], w.scales[W4A16_V], xl, yv, M, kv_dim, hidden, hidden, kv_dim);
      a.seg[0].bias = b(W4A16_V);
      add(a, -1);
    }
    {
      GemvArgs a = plain_args(w.qweight[W4A16_O], w.scales[W4A16_O], yq, io->y_o + l * Mh, M, hidden,
                              hidden, hidden, hidden);
      a.seg[0].bias = b(W4A16_O);
      add(a, iq);
    }
    // y_gu rows are [gate | up]: row stride 2 ffn
    int ilast;       // the GEMV down waits for
    int ialso = -1;  // and, with SwiGLU over separate gate and up, the other one
    const int64_t ldgu = 2 * static_cast<int64_t>(ffn);
    uint16_t* const hl = swiglu ? opt.hbuf + static_cast<int64_t>(l) * M * ffn : nullptr;
    if (swiglu && fuse_swiglu) {
      // The task lists: gate and up as two GEMVs over the same rows of the
      // same CTAs; up's epilogue forms h from its own rounded output and the
      // gate output this CTA wrote earlier, and down reads h.  up is added
      // first: a table emits a layer's GEMVs that read x in reverse order,
      // so gate runs before up.
      GemvArgs u = plain_args(w.qweight[W4A16_UP], w.scales[W4A16_UP], xl, ygu + ffn, M, ffn, hidden, hidden,
                              ldgu);
      u.seg[0].bias = b(W4A16_UP);
      u.swiglu = 2;
      u.epi_h = hl;
      ilast = add(u, -1);
      GemvArgs g = plain_args(w.qweight[W4A16_GATE], w.scales[W4A16_GATE], xl, ygu, M, ffn, hidden, hidden,
                              ldgu);
      g.seg[0].bias = b(W4A16_GATE);
      g.swiglu = 1;
      add(g, -1);
    } else if (stacked(w, W4A16_GATE, W4A16_UP, ffn)) {
      GemvArgs a = plain_args(w.qweight[W4A16_GATE], w.scales[W4A16_GATE], xl, ygu, M, 2 * ffn, hidden,
                              hidden, ldgu);
      a.nseg = 2;
      a.seg[0] = OutSeg{ygu, ldgu, ffn, b(W4A16_GATE)};
      a.seg[1] = OutSeg{ygu + ffn, ldgu, 2 * static_cast<int64_t>(ffn), b(W4A16_UP)};
      ilast = add(a, -1);
    } else {
      GemvArgs a = plain_args(w.qweight[W4A16_GATE], w.scales[W4A16_GATE], xl, ygu, M, ffn, hidden, hidden,
                              ldgu);
      a.seg[0].bias = b(W4A16_GATE);
      ilast = add(a, -1);
      a = plain_args(w.qweight[W4A16_UP], w.scales[W4A16_UP], xl, ygu + ffn, M, ffn, hidden, hidden, ldgu);
      a.seg[0].bias = b(W4A16_UP);
      const int iu = add(a, -1);
      if (swiglu) {
        // down reads both halves: it waits for whichever of the two a task
        // table runs later (each CTA publishes its tasks in table order)
        ialso = ilast;
        ilast = iu;
      }
    }
    {
      GemvArgs a = plain_args(w.qweight[W4A16_DOWN], w.scales[W4A16_DOWN], ygu, io->y_down + l * Mh, M,
                              hidden, ffn, ldgu, hidden);
      a.seg[0].bias = b(W4A16_DOWN);
      ActOp op;
      if (swiglu) {
        // down reads h (written by up's epilogue, or by a separate step)
        if (!fuse_swiglu) op = ActOp{ygu, ygu + ffn, ldgu, hl, M, ffn};
        a.x = hl;
        a.ldx = ffn;
      }
      const int id = add(a, ilast);
      (*dep2)[id] = ialso;
      (*act)[id] = op;
    }
  }
  layer_first->push_back(static_cast<int>(gemvs->size()));
}

// The GEMVs of layers [l0, l1) as one task table, in launch order.  Layers
// are independent of each other, so the table interleaves them: stage A of
// a layer (the GEMVs that read the layer's x) runs one layer ahead of its
// stage B (o and down, which read stage A's outputs), so that a dependent
// GEMV finds its producer finished a whole cycle earlier by the whole grid.
// W4A16 alternates the two stages, largest first:
//   gate_up(l+1) down(l) qkv(l+1) o(l)
// (the M = 1 kernel stages each task's activations into shared memory while
// the task before it runs; down's, K = 18944, take the longest to stage and
// follow [gate; up], the longest task; with separate q, k, v or gate, up
// weights the longer stage continues after the shorter one runs out).  W4A8,
// whose consumer threads load their own activations, runs
//   gate_up(l+1) qkv(l+1) o(l) down(l)
// which puts the shortest set-up after down, its most CUDA-core-bound task.
// Dependencies become task indices within the table (the done counters are
// per table slot); a producer before l0 is met by the launch order.  A GEMV
// whose K the M = 1 kernel splits becomes two consecutive tasks; a GEMV that
// reads its output depends on the second.
void seq_tasks(const DeviceState& d, const std::vector<GemvArgs>& gemvs, const std::vector<int>& dep,
               const std::vector<int>& dep2, const std::vector<int>& layer_first, int l0, int l1, bool a8, std::vector<M1Task>* tasks) {
  tasks->clear();
  static thread_local std::vector<int> slot;  // table slot of each emitted GEMV (capacity kept)
  slot.assign(gemvs.size(), -1);
  auto emit_one = [&](int i) {
    {
      const GemvArgs& a = gemvs[i];
      M1Task tk{};
      tk.qweight = a.qweight;
      tk.scales = a.scales;
      tk.x = a.x;
      tk.swiglu = static_cast<uint8_t>(a.swiglu);
      tk.N = a.N;
      tk.K = a.K;
      tk.nseg = static_cast<uint8_t>(a.nseg);
      // with two producers, the one later in the table (its publication on
      // every CTA implies the other's)
      tk.dep = dep[i] < 0 ? -1 : slot[dep[i]];
      if (dep2[i] >= 0 && slot[dep2[i]] > tk.dep) tk.dep = slot[dep2[i]];
      for (int g = 0; g < kMaxSegs; ++g) tk.seg[g] = M1Seg{a.seg[g].y, a.seg[g].bias, a.seg[g].n_end};
      tk.epi_h = a.epi_h;  // h of the SwiGLU epilogue (up tasks)
      M1Task parts[2];
      const int np = gemv_m1_split_tasks(tk, a8, d.info, parts);
      for (int q = 0; q < np; ++q) tasks->push_back(parts[q]);
      slot[i] = static_cast<int>(tasks->size()) - 1;
    }
  };
  // a layer's stage A (reads x) and stage B (reads stage A), each in reverse
  // GEMV order: [gate; up] before [q; k; v], down before o
  static thread_local std::vector<int> stage_a, stage_b;
  auto stage = [&](int l, bool b, std::vector<int>* out) {
    out->clear();
    for (int i = layer_first[l + 1] - 1; i >= layer_first[l]; --i)
      if ((dep[i] >= 0) == b) out->push_back(i);
  };
  stage(l0, false, &stage_a);
  for (int i : stage_a) emit_one(i);
  for (int l = l0; l < l1; ++l) {
    if (l + 1 < l1)
      stage(l + 1, false, &stage_a);
    else
      stage_a.clear();
    stage(l, true, &stage_b);
    if (a8) {
      for (int i : stage_a) emit_one(i);
      for (auto it = stage_b.rbegin(); it != stage_b.rend(); ++it) emit_one(*it);  // o, down
      continue;
    }
    const size_t n = stage_a.size() > stage_b.size() ? stage_a.size() : stage_b.size();
    for (size_t k = 0; k < n; ++k) {
      if (k < stage_a.size()) emit_one(stage_a[k]);
      if (k < stage_b.size()) emit_one(stage_b[k]);
    }
  }
}

// Whether a checked sequence runs as task lists of the M = 1 kernel.
bool seq_uses_tasks(int M, const std::vector<GemvArgs>& gemvs) {
  if (M != 1) return false;
  for (const GemvArgs& a : gemvs)
    if (!gemv_m1_supported(a.K)) return false;
  return true;
}

// The task lists of a checked M = 1 sequence: task_first[l] is the index of
// layer l's first task (task_first[n_layers] = tasks, one completion counter
// each), every layer within one task table, every task within the M = 1
// kernel's limits on this device.  Host-only: nothing is enqueued.
// scratch: the caller's buffer (its capacity is reused).
w4a16_status check_seq_tasks(const DeviceState& d, const std::vector<GemvArgs>& gemvs,
                             const std::vector<int>& dep, const std::vector<int>& dep2,
                             const std::vector<int>& layer_first, bool a8, std::vector<M1Task>* scratch,
                             std::vector<int>* task_first) {
  const int n_layers = static_cast<int>(layer_first.size()) - 1;
  for (const GemvArgs& a : gemvs)
    if (a.N <= 0) return W4A16_ERR_SHAPE;
  task_first->assign(1, 0);
  for (int l = 0; l < n_layers; ++l) {
    int n = 0;
    for (int i = layer_first[l]; i < layer_first[l + 1]; ++i) {
      M1Task t{};
      t.K = gemvs[i].K;
      t.N = gemvs[i].N;
      M1Task parts[2];
      n += gemv_m1_split_tasks(t, a8, d.info, parts);
    }
    if (n > kM1MaxTasks) return W4A16_ERR_SHAPE;  // one layer beyond a task table
    task_first->push_back(task_first->back() + n);
  }
  seq_tasks(d, gemvs, dep, dep2, layer_first, 0, n_layers, a8, scratch);
  return gemv_m1_tasks_fit(scratch->data(), static_cast<int>(scratch->size()), a8, d.info) ? W4A16_OK
                                                                                          : W4A16_ERR_SHAPE;
}

// Enqueue a sequence's task lists: as many whole layers per launch as fit in
// one task table, each launch after the first a programmatic dependent of the
// previous one.  done: one zeroed counter per task (task_first from
// check_seq_tasks, which must have passed: a launch that fails here leaves
// the launches before it enqueued); tasks: the caller's table buffer (its
// capacity is reused).  Returns the launch count through *launches.
w4a16_status enqueue_seq_tasks(const DeviceState& d, const std::vector<GemvArgs>& gemvs,
                               const std::vector<int>& dep, const std::vector<int>& dep2,
                               const std::vector<int>& layer_first, const std::vector<int>& task_first,
                               int* done, bool a8, cudaStream_t st, std::vector<M1Task>* tasks, int* launches) {
  const int n_layers = static_cast<int>(layer_first.size()) - 1;
  int l0 = 0;
  *launches = 0;
  while (l0 < n_layers) {
    int l1 = l0 + 1;
    while (l1 < n_layers && task_first[l1 + 1] - task_first[l0] <= kM1MaxTasks) ++l1;
    const int t0 = task_first[l0], t1 = task_first[l1];
    if (t1 - t0 > kM1MaxTasks) return W4A16_ERR_SHAPE;  // one layer beyond a task table
    seq_tasks(d, gemvs, dep, dep2, layer_first, l0, l1, a8, tasks);
    const cudaError_t e =
        launch_gemv_m1_tasks(tasks->data(), t1 - t0, done + t0, d.status, *launches > 0, a8, d.info, st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
    ++*launches;
    l0 = l1;
  }
  return W4A16_OK;
}

}  // namespace

extern "C" {

w4a16_status w4a16_layer_seq_create(const w4a16_layer_weights* layers, int n_layers, int M,
                                    int hidden, int kv_dim, int ffn, int group,
                                    const w4a16_seq_io* io, w4a16_layer_seq** out) {
  return w4a16_layer_seq_create2(layers, nullptr, 0u, n_layers, M, hidden, kv_dim, ffn, group, io, out);
}

w4a16_status w4a16_layer_seq_create2(const w4a16_layer_weights* layers, const w4a16_layer_bias* biases,
                                     unsigned flags, int n_layers, int M, int hidden, int kv_dim, int ffn,
                                     int group, const w4a16_seq_io* io, w4a16_layer_seq** out) {
  if (!out) return W4A16_ERR_NULL;
  *out = nullptr;
  if ((flags & ~static_cast<unsigned>(W4A16_SEQ_SWIGLU | W4A16_SEQ_ACT_INT8)) != 0) return W4A16_ERR_SHAPE;
  w4a16_status st = check_seq_args(layers, n_layers, M, hidden, kv_dim, ffn, group, io);
  if (st != W4A16_OK) return st;
  if ((st = check_seq_biases(biases, n_layers, M, hidden, kv_dim, ffn, io)) != W4A16_OK) return st;
  // W4A8 runs only in the M = 1 task-list kernel
  if ((flags & W4A16_SEQ_ACT_INT8) != 0) {
    if (M != 1) return W4A16_ERR_M_RANGE;
    if (!gemv_m1_supported(hidden) || !gemv_m1_supported(ffn)) return W4A16_ERR_SHAPE;
  }

  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != W4A16_OK) return st;

  // M = 1 with every K in the M = 1 kernel's range: task lists, SwiGLU in
  // up's epilogue; otherwise one launch per GEMV and, with SwiGLU, a separate
  // activation step.  Either way h goes to a buffer this object owns.
  const bool swiglu = (flags & W4A16_SEQ_SWIGLU) != 0;
  const bool tasks = M == 1 && gemv_m1_supported(hidden) && gemv_m1_supported(ffn) &&
                     (!swiglu || gemv_m1_swiglu_fits(ffn, d->info));
  const bool a8 = (flags & W4A16_SEQ_ACT_INT8) != 0;
  if (a8 && !tasks) return W4A16_ERR_SHAPE;  // W4A8 runs only in the task lists
  SeqOptions opt;
  opt.biases = biases;
  opt.flags = flags;

  w4a16_layer_seq* s = new (std::nothrow) w4a16_layer_seq();
  if (!s) return W4A16_ERR_CUDA;
  cudaGetDevice(&s->device);
  s->n_layers = n_layers;
  s->M = M;
  s->hidden = hidden;
  s->kv_dim = kv_dim;
  s->ffn = ffn;
  s->io = *io;
  if (cudaStreamCreateWithFlags(&s->capture_stream, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&s->done, cudaEventDisableTiming) != cudaSuccess ||
      (swiglu &&
       cudaMalloc(&s->hbuf, sizeof(uint16_t) * static_cast<size_t>(n_layers) * M * ffn) != cudaSuccess)) {
    cudaGetLastError();
    seq_free(s);
    return W4A16_ERR_CUDA;
  }
  opt.hbuf = s->hbuf;
  std::vector<GemvArgs> gemvs;
  std::vector<int> dep, dep2, layer_first;
  std::vector<ActOp> act;
  build_seq_gemvs(layers, opt, n_layers, M, hidden, kv_dim, ffn, io, tasks, &gemvs, &dep, &dep2, &act,
                  &layer_first);
  // M = 1: the task lists, checked on the host before anything is captured
  std::vector<M1Task> table;
  std::vector<int> task_first;
  if (tasks && (st = check_seq_tasks(*d, gemvs, dep, dep2, layer_first, a8, &table, &task_first)) != W4A16_OK) {
    seq_free(s);
    return st;
  }
  const size_t ntasks = tasks ? static_cast<size_t>(task_first.back()) : 0;
  if (tasks && cudaMalloc(&s->task_done, sizeof(int) * ntasks) != cudaSuccess) {
    cudaGetLastError();
    seq_free(s);
    return W4A16_ERR_CUDA;
  }
  if (cudaStreamBeginCapture(s->capture_stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaGetLastError();
    seq_free(s);
    return W4A16_ERR_CUDA;
  }
  // M = 1: the whole sequence runs as task lists of the persistent M = 1
  // kernel; its per-GEMV completion counters are zeroed by a memset node
  // before every replay.  M > 1: one launch per GEMV, each after the first a
  // programmatic dependent of its predecessor (it streams its constant
  // weights while the previous GEMV finishes and waits for it before reading
  // activations or writing outputs).
  w4a16_status cap = W4A16_OK;
  int launches = 0;
  if (tasks) {
    if (cudaMemsetAsync(s->task_done, 0, sizeof(int) * ntasks, s->capture_stream) != cudaSuccess)
      cap = W4A16_ERR_CUDA;
    else
      cap = enqueue_seq_tasks(*d, gemvs, dep, dep2, layer_first, task_first, s->task_done, a8,
                              s->capture_stream, &table, &launches);
  } else {
    for (size_t i = 0; i < gemvs.size() && cap == W4A16_OK; ++i) {
      if (act[i].h != nullptr) {
        const ActOp& op = act[i];
        if (launch_swiglu(op.g, op.u, op.ld, op.h, op.M, op.n, launches > 0, s->capture_stream) !=
            cudaSuccess) {
          cudaGetLastError();
          cap = W4A16_ERR_CUDA;
          break;
        }
        ++launches;
      }
      GemvArgs a = gemvs[i];
      a.pdl = launches > 0;
      cap = enqueue(*d, a, s->capture_stream);
      ++launches;
    }
  }
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(s->capture_stream, &graph);
  if (cap != W4A16_OK || ec != cudaSuccess) {
    cudaGetLastError();
    if (graph) cudaGraphDestroy(graph);
    seq_free(s);
    return cap != W4A16_OK ? cap : W4A16_ERR_CUDA;
  }
  s->graph = graph;
  if (cudaGraphInstantiate(&s->exec, graph, 0) != cudaSuccess) {
    cudaGetLastError();
    seq_free(s);
    return W4A16_ERR_CUDA;
  }
  s->launches = launches;
  *out = s;
  return W4A16_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- allocation-free run
//
// For callers that cannot allocate device memory (a serving process whose
// device memory all belongs to its own pool, or code that must not call
// cudaFree, which waits for the whole device): the counters of the task
// lists live in a fixed array of this library's device image instead of a
// cudaMalloc'd buffer, and no CUDA graph is built.

namespace w4a16 {
namespace {

// In host code this name is only a stand-in for the device symbol, not an
// address a kernel may be given: the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) int g_static_task_done[W4A16_STATIC_MAX_GEMVS];

int* g_static_task_done_addr[kMaxDevices];  // device address per device, under g_mu

// Device address of g_static_task_done on the current device (looked up once
// per device, with that device current).
w4a16_status static_task_done(int** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_static_task_done_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_task_done);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
    g_static_task_done_addr[dev] = static_cast<int*>(p);
  }
  *out = g_static_task_done_addr[dev];
  return W4A16_OK;
}

}  // namespace
}  // namespace w4a16

extern "C" w4a16_status w4a16_layer_seq_run_static(const w4a16_layer_weights* layers, int n_layers,
                                                   int hidden, int kv_dim, int ffn, int group,
                                                   const w4a16_seq_io* io, void* stream) {
  w4a16_status st = check_seq_args(layers, n_layers, 1, hidden, kv_dim, ffn, group, io);
  if (st != W4A16_OK) return st;
  if (n_layers > W4A16_STATIC_MAX_GEMVS / 4) return W4A16_ERR_LIMIT;  // >= 4 GEMVs per layer

  // host tables: thread-local, their capacity kept from call to call
  static thread_local std::vector<GemvArgs> gemvs;
  static thread_local std::vector<int> dep, dep2, layer_first;
  static thread_local std::vector<ActOp> act;
  static thread_local std::vector<M1Task> tasks;
  static thread_local std::vector<int> task_first;
  build_seq_gemvs(layers, SeqOptions{}, n_layers, 1, hidden, kv_dim, ffn, io, true, &gemvs, &dep, &dep2,
                  &act, &layer_first);
  if (!seq_uses_tasks(1, gemvs)) return W4A16_ERR_LIMIT;

  DeviceState* d = nullptr;
  if ((st = device_state(&d)) != W4A16_OK) return st;
  int* done = nullptr;
  if ((st = static_task_done(&done)) != W4A16_OK) return st;

  // every task table is checked on the host before anything is enqueued
  if ((st = check_seq_tasks(*d, gemvs, dep, dep2, layer_first, false, &tasks, &task_first)) != W4A16_OK)
    return st;
  const int n = task_first.back();  // one counter per task
  if (n > W4A16_STATIC_MAX_GEMVS) return W4A16_ERR_LIMIT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the counters keep the previous call's values: zero the ones this call uses
  if (cudaMemsetAsync(done, 0, sizeof(int) * n, s) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  int launches = 0;
  return enqueue_seq_tasks(*d, gemvs, dep, dep2, layer_first, task_first, done, false, s, &tasks, &launches);
}

extern "C" {

int w4a16_layer_seq_num_launches(const w4a16_layer_seq* seq) { return seq ? seq->launches : 0; }

w4a16_status w4a16_layer_seq_run(w4a16_layer_seq* seq, void* stream) {
  if (!seq || !seq->exec) return W4A16_ERR_STATE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaGraphLaunch(seq->exec, st) != cudaSuccess || cudaEventRecord(seq->done, st) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

w4a16_status w4a16_layer_seq_run_host(w4a16_layer_seq* seq, const w4a16_seq_io* host, void* stream) {
  if (!seq || !seq->exec) return W4A16_ERR_STATE;
  if (!host) return W4A16_ERR_NULL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t L = static_cast<size_t>(seq->n_layers) * seq->M * 2;  // bytes per element x rows x layers
  const size_t bh = L * seq->hidden, bkv = L * seq->kv_dim, bgu = L * 2 * seq->ffn;
  bool ok = true;
  if (host->x)
    ok = ok && cudaMemcpyAsync(const_cast<uint16_t*>(seq->io.x), host->x, bh, cudaMemcpyHostToDevice, st) == cudaSuccess;
  ok = ok && cudaGraphLaunch(seq->exec, st) == cudaSuccess;
  struct {
    uint16_t* h;
    const uint16_t* d;
    size_t bytes;
  } outs[6] = {{host->y_q, seq->io.y_q, bh},   {host->y_k, seq->io.y_k, bkv},
               {host->y_v, seq->io.y_v, bkv},  {host->y_o, seq->io.y_o, bh},
               {host->y_gu, seq->io.y_gu, bgu}, {host->y_down, seq->io.y_down, bh}};
  for (auto& o : outs)
    if (o.h) ok = ok && cudaMemcpyAsync(o.h, o.d, o.bytes, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  ok = ok && cudaEventRecord(seq->done, st) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}

}  // extern "C"

namespace {

// After a replay has completed: W4A16_ERR_DEVICE if the device status word of
// the sequence's device holds W4A16_DEV_PIPE_TIMEOUT (a pipeline or
// dependency wait inside a GEMV ran out, so outputs may be wrong), else OK.
// The word is read on the sequence's own stream and left as it is.
w4a16_status seq_device_check(w4a16_layer_seq* seq) {
  uint32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (seq->device >= 0 && seq->device < kMaxDevices) status = g_dev[seq->device].status;
  }
  if (status == nullptr) return W4A16_ERR_STATE;
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, status, sizeof(v), cudaMemcpyDeviceToHost, seq->capture_stream) != cudaSuccess ||
      cudaStreamSynchronize(seq->capture_stream) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return (v & W4A16_DEV_PIPE_TIMEOUT) ? W4A16_ERR_DEVICE : W4A16_OK;
}

}  // namespace

extern "C" {

w4a16_status w4a16_layer_seq_sync(w4a16_layer_seq* seq, int timeout_ms) {
  if (!seq || !seq->done) return W4A16_ERR_STATE;
  if (timeout_ms < 0) {
    if (cudaEventSynchronize(seq->done) != cudaSuccess) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
    return seq_device_check(seq);
  }
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t e = cudaEventQuery(seq->done);
    if (e == cudaSuccess) return seq_device_check(seq);
    if (e != cudaErrorNotReady) {
      cudaGetLastError();
      return W4A16_ERR_CUDA;
    }
    const auto ms = std::chrono::duration_cast<std::chrono::milliseconds>(
                        std::chrono::steady_clock::now() - t0).count();
    if (ms >= timeout_ms) return W4A16_ERR_TIMEOUT;
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

void w4a16_layer_seq_destroy(w4a16_layer_seq* seq) {
  if (!seq) return;
  if (seq->done) cudaEventSynchronize(seq->done);
  seq_free(seq);
}

}  // extern "C"
