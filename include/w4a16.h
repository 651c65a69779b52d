/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) INT4 weight-only GEMV library.
 *
 * The operation.  y[m][n] = sum_k x[m][k] * w_hat[n][k] with
 * w_hat[n][k] = q[n][k] * s[n][k / 128]: INT4 weights, symmetric and
 * group-wise with group 128 along K and one FP16 scale per group, times FP16
 * activations, unpacked inside the kernel and accumulated in FP32.  This is
 * the weight format of the page "Costruire un runtime di inference LLM da
 * zero" (datastack.it), section "Tre bug che insegnano": last paragraph (INT4
 * symmetric group-wise, group 128, on the seven per-layer projections) and
 * third bug (the gate/up/down GEMVs unpack INT4 in-kernel and multiply FP16
 * activations).  The page gives no layout; this library's layout is:
 *
 *   qweight  uint32[N][K/8]   nibble i (bits 4i..4i+3) of word j of row n is
 *                             q[n][8j + i], 4-bit two's complement in [-8, 7]
 *   scales   fp16[N][K/128]   row-major, s[n][g] for k in [128g, 128g + 128)
 *   x        fp16[M][K]       row-major activations
 *   y        fp16[M][N]       row-major output, fp16 round-to-nearest of the
 *                             FP32 accumulator
 *
 * fp16 values travel as uint16_t bit patterns.  W is stored like an
 * nn.Linear weight (out x in).
 *
 * Conventions for every entry point
 *   - All data pointers are DEVICE pointers unless the name says host.  The
 *     caller owns every buffer; no entry point frees or keeps a caller buffer
 *     beyond the call, except layer_seq (which records the pointers it is
 *     given in a CUDA graph: they must stay valid until it is destroyed).
 *   - Every data pointer must be 16-byte aligned (W4A16_ERR_ALIGN otherwise).
 *   - group must be 128 (W4A16_ERR_GROUP); K must be a positive multiple of
 *     128 and at most W4A16_MAX_K (W4A16_ERR_SHAPE); 0 <= N <= W4A16_MAX_N.
 *   - Arguments are checked on the host before anything is enqueued; a bad
 *     argument returns its status and enqueues nothing.
 *   - Work is enqueued on `stream` (a cudaStream_t; 0 = legacy default
 *     stream) and the call returns without waiting.  W4A16_ERR_CUDA means a
 *     launch or runtime call failed (cudaGetLastError is cleared).
 *   - No entry point traps or asserts on the device.  Kernels whose internal
 *     waits are bounded record a run-time failure in a per-device status word
 *     instead; read it with w4a16_device_status.
 *   - The current CUDA device is the one the pointers belong to.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_ABI_VERSION 1
#define W4A16_GROUP 128
#define W4A16_MAX_M 16
#define W4A16_MAX_K 32768
#define W4A16_MAX_N (1 << 24)
/* Decode attention: most KV heads per call (the workspace's counter block
 * holds one counter per possible KV head). */
#define W4A16_ATTN_MAX_KV_HEADS 256

typedef enum {
  W4A16_OK = 0,
  W4A16_ERR_NULL = 1,       /* a required pointer is NULL */
  W4A16_ERR_SHAPE = 2,      /* N, K out of range, or K not a multiple of 128 */
  W4A16_ERR_ALIGN = 3,      /* a data pointer is not 16-byte aligned */
  W4A16_ERR_GROUP = 4,      /* group != 128 */
  W4A16_ERR_M_RANGE = 5,    /* M outside 0..16 */
  W4A16_ERR_ALIAS = 6,      /* an output buffer overlaps an input buffer */
  W4A16_ERR_CUDA = 7,       /* a CUDA runtime call or kernel launch failed */
  W4A16_ERR_TIMEOUT = 8,    /* a bounded host wait ran out */
  W4A16_ERR_STATE = 9,      /* NULL or unusable object handle */
  W4A16_ERR_DEVICE = 10,    /* a kernel recorded a failure (see w4a16_device_status) */
  W4A16_ERR_LIMIT = 11      /* beyond the fixed limits of w4a16_layer_seq_run_static */
} w4a16_status;

/* Bits of the per-device status word written by kernels. */
#define W4A16_DEV_NONFINITE 0x1u     /* w4a16_quantize met a non-finite weight   */
#define W4A16_DEV_SCALE_OVERFLOW 0x2u /* w4a16_quantize: max|w|/7 overflows fp16 */
#define W4A16_DEV_PIPE_TIMEOUT 0x4u  /* a GEMV pipeline wait ran past its bound  */
/* Only in the index-checked build of the library (compiled with
 * W4A16_CHECKED, for tests): a kernel's index or address check failed and the
 * access was skipped instead of made (the results are then undefined). */
#define W4A16_DEV_INDEX 0x8u

/* Human-readable name of a status code (static string, never NULL). */
const char* w4a16_status_str(w4a16_status s);

/* Returns W4A16_ABI_VERSION of the loaded library. */
int w4a16_abi_version(void);

/*
 * w4a16_gemv -- y = x . w_hat^T for 1 <= M <= 16 activation rows (the decode
 * GEMV of the third bug of "Tre bug che insegnano"; M > 1 is small-batch
 * decode).  M == 0 or N == 0 is an empty product: OK, nothing is launched.
 *   qweight, scales  the packed weight of N output rows and K inputs
 *   x                fp16 [M][K]
 *   y                fp16 [M][N]; must not overlap x, qweight or scales
 * Dispatch: M = 1 with K <= 28672 runs the persistent TMA-fed CUDA-core
 * kernel; other M in 1..7 the CUDA-core small-batch kernel (nibble unpack in
 * registers, FP32 accumulation); M in 8..16 the tensor-core kernel (mma.sync
 * over each group of 128, FP32 accumulators).  The result is deterministic:
 * the same inputs give the same bits on every call.  Never allocates, never
 * synchronises.  The kernel is launched as a programmatic dependent of the
 * previous kernel on the stream: if that kernel lets dependents start early
 * (griddepcontrol.launch_dependents), this one may read qweight and scales
 * before it completes, but reads x and writes y only after it has completed
 * (kernels that do not opt in are simply waited for).  The first call of any
 * entry point on a device does a one-time set-up (device queries, kernel
 * attributes); make it outside CUDA stream capture.  After that, w4a16_gemv
 * may be captured.
 */
w4a16_status w4a16_gemv(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                        uint16_t* y, int M, int N, int K, int group, void* stream);

/*
 * w4a16_gemv_a8 -- the W4A8 variant of w4a16_gemv: INT4 weights against
 * INT8 activations with int8 dot products (dp4a), the variant that the third
 * bug of "Tre bug che insegnano" reports measuring against the FP16 path.
 * x stays fp16 in memory; the kernel quantises each block of 64 consecutive
 * activations of a row as it loads it:
 *   s_b = max|x_b| / 127,  xq = round_to_nearest_even(x * (127 / max|x_b|))
 * (FP32 divisions and product, |xq| <= 127; an all-zero block gives s_b = 0,
 * xq = 0), and
 *   y[n] = fp16_RN( sum_b s_w[n][b / 2] s_b sum_{k in b} q[n][k] xq[k] )
 * with exact integer block sums and FP32 scaling and accumulation.  The
 * result differs from w4a16_gemv by the activation rounding (about 1 % of
 * |y| on Gaussian activations).  Arguments and checks as w4a16_gemv, plus:
 * M must be 0 or 1 (W4A16_ERR_M_RANGE) and K within the M = 1 kernel's range
 * (at most 28672; W4A16_ERR_SHAPE).  Deterministic; never allocates.
 */
w4a16_status w4a16_gemv_a8(const uint32_t* qweight, const uint16_t* scales, const uint16_t* x,
                           uint16_t* y, int M, int N, int K, int group, void* stream);

/*
 * w4a16_dequant -- debugging aid: w_out fp16[N][K] = fp16_RN(q * s) (exact
 * product, one rounding).  w_out must not overlap qweight or scales.
 */
w4a16_status w4a16_dequant(const uint32_t* qweight, const uint16_t* scales, uint16_t* w_out,
                           int N, int K, int group, void* stream);

/*
 * w4a16_quantize -- the load-time encoder: fp32 W[N][K] -> (qweight, scales).
 * Per row n and group g:  s = fp16_RN(fp32(max|w| / 7));
 *                         q = clamp(round_half_away(w / s), -8, 7)  (s = 0: q = 0)
 * The rounding decision is the one of the exact quotient w / s.  A
 * non-finite weight sets W4A16_DEV_NONFINITE and a group whose scale would
 * overflow fp16 sets W4A16_DEV_SCALE_OVERFLOW in the device status word (that
 * group is written as zeros); call w4a16_device_status after the stream
 * completes to learn of it.  Outputs must not overlap w.
 */
w4a16_status w4a16_quantize(const float* w, uint32_t* qweight, uint16_t* scales, int N, int K,
                            int group, void* stream);

/*
 * w4a16_device_status -- read (and if clear != 0, reset) the status word of
 * the current device.  Synchronises the device first (it is a debugging and
 * test call, not for the hot path).  *flags gets the W4A16_DEV_* bits seen
 * since the last reset.  Returns W4A16_ERR_DEVICE if any bit is set, OK
 * otherwise, W4A16_ERR_CUDA if the device could not be read.
 */
w4a16_status w4a16_device_status(uint32_t* flags, int clear);

/*
 * w4a16_selftest_wait_timeout -- exercise the failure path of the bounded
 * in-kernel waits without any fault: one GPU thread waits on a barrier that
 * nothing arrives on, gives up after limit_us microseconds (0..10,000,000),
 * sets W4A16_DEV_PIPE_TIMEOUT in the device status word and returns.  The
 * context stays usable.  Returns after enqueue.
 */
w4a16_status w4a16_selftest_wait_timeout(int limit_us, void* stream);

/* ------------------------------------------------------------------------
 * layer_seq -- the seven projections of a Qwen-7B-shaped decoder layer,
 * repeated for n_layers, captured once as one CUDA graph and replayed.  The
 * second bug of "Tre bug che insegnano" is that eager decode pays a launch
 * overhead per kernel (about 119 -> 17 ms/token once captured); this is the
 * GEMV part of such a captured decode step.
 *
 * Per layer l (M activation rows):
 *   y_q    = gemv(W_q,  x_l)        N = hidden, K = hidden
 *   y_k    = gemv(W_k,  x_l)        N = kv_dim, K = hidden
 *   y_v    = gemv(W_v,  x_l)        N = kv_dim, K = hidden
 *   y_o    = gemv(W_o,  y_q)        N = hidden, K = hidden
 *   y_gu   = gemv([W_gate; W_up], x_l)   N = 2 ffn, K = hidden (one GEMV
 *            when the up weight directly follows the gate weight in memory,
 *            two otherwise)
 *   y_down = gemv(W_down, gate half of y_gu)   N = hidden, K = ffn
 * Layers are independent (each takes its own x_l), so magnitudes stay in the
 * fp16 range for any depth.
 * ---------------------------------------------------------------------- */
typedef struct w4a16_layer_seq w4a16_layer_seq;

enum { W4A16_Q = 0, W4A16_K = 1, W4A16_V = 2, W4A16_O = 3, W4A16_GATE = 4, W4A16_UP = 5,
       W4A16_DOWN = 6, W4A16_NPROJ = 7 };

typedef struct {
  const uint32_t* qweight[W4A16_NPROJ]; /* indexed by W4A16_Q .. W4A16_DOWN */
  const uint16_t* scales[W4A16_NPROJ];
} w4a16_layer_weights;

/* Activation / output buffers of all layers, each [n_layers][M][width]. */
typedef struct {
  const uint16_t* x; /* width hidden */
  uint16_t* y_q;     /* width hidden */
  uint16_t* y_k;     /* width kv_dim */
  uint16_t* y_v;     /* width kv_dim */
  uint16_t* y_o;     /* width hidden */
  uint16_t* y_gu;    /* width 2 * ffn: gate then up */
  uint16_t* y_down;  /* width hidden */
} w4a16_seq_io;

/*
 * Validate every weight and io pointer (as w4a16_gemv would), capture the
 * sequence into a CUDA graph on a private stream and instantiate it.
 * layers[l] holds the weights of layer l.  [q; k; v] run as one GEMV when
 * the three weights are stacked in one allocation, [gate; up] likewise.
 *   M = 1:  the GEMVs run as task lists of the persistent M = 1 kernel, whole
 *           layers per launch and up to 224 GEMVs per launch (28 Qwen-7B-
 *           shaped layers with stacked weights: one launch), after a memset
 *           node that zeroes one completion counter per GEMV.  A GEMV that
 *           reads another's output (o, down) starts once every CTA has
 *           written that output.  Such a launch is cooperative (one CTA per
 *           SM, all resident at once): where that cannot be had (fewer free
 *           SMs, e.g. under MPS limits), the launch fails and so does the
 *           replay, instead of CTAs waiting on ones that never start.
 *   M > 1:  one launch per GEMV, each a programmatic dependent of the
 *           previous one.
 * The library allocates the graph, a stream, an event and, for M = 1, one
 * int of device memory per task (the counters: one per GEMV, two for a GEMV
 * whose K the M = 1 kernel splits in halves); nothing else.  The pointers
 * are recorded in the graph and must outlive the object.  Blocks until
 * instantiation is done (a set-up call, not a hot-path call).  *out is NULL
 * on failure.
 */
w4a16_status w4a16_layer_seq_create(const w4a16_layer_weights* layers, int n_layers, int M,
                                    int hidden, int kv_dim, int ffn, int group,
                                    const w4a16_seq_io* io, w4a16_layer_seq** out);

/* ------------------------------------------------------------------------
 * Fused layer epilogues (w4a16_layer_seq_create2): the steps either side of
 * the GEMVs in a Qwen2 decoder layer, as the page on hipfire describes its
 * Qwen2 decoder ("Overview of hipfire-arch-qwen2", "Key Technical
 * Specifications": a SwiGLU feed-forward and attention_bias on the Q, K and
 * V projections).
 * ---------------------------------------------------------------------- */

/* Flag: down reads h = silu(gate) * up instead of the gate half of y_gu:
 * h[m][j] = fp16_RN(silu(g) u), g = y_gu[m][j], u = y_gu[m][ffn + j] (fp16),
 * silu(g) = g / (1 + e^-g), evaluated in FP32.  y_gu is still written. */
#define W4A16_SEQ_SWIGLU 0x1u
/* Flag: every GEMV of the sequence is the W4A8 variant (see w4a16_gemv_a8);
 * M = 1 with every K within the M = 1 kernel's range only (W4A16_ERR_M_RANGE
 * for M > 1, W4A16_ERR_SHAPE otherwise). */
#define W4A16_SEQ_ACT_INT8 0x2u

/* Optional per-layer output biases, fp16 bits, one per output row of a
 * projection (NULL: none), indexed by W4A16_Q .. W4A16_DOWN.  A bias is
 * added to the FP32 sum before the fp16 rounding: y = fp16_RN(sum + b[n]).
 * 16-byte aligned; must not overlap any output of the sequence. */
typedef struct {
  const uint16_t* bias[W4A16_NPROJ];
} w4a16_layer_bias;

/*
 * w4a16_layer_seq_create with epilogues: biases (n_layers entries, or NULL
 * for none) and flags (W4A16_SEQ_SWIGLU, W4A16_SEQ_ACT_INT8 or both; other
 * bits return W4A16_ERR_SHAPE).  With SwiGLU, h goes to a device buffer of
 * n_layers x M x ffn fp16 values that the object allocates and frees, and
 * down reads it.  At M = 1 (every K within the M = 1 kernel's range) gate
 * and up run as two GEMVs of the layer's one task list and up's epilogue
 * writes h as each row of y_up is rounded; otherwise a separate kernel
 * writes h after the [gate; up] GEMV.  Everything else as
 * w4a16_layer_seq_create (which is this call with no biases and no flags).
 */
w4a16_status w4a16_layer_seq_create2(const w4a16_layer_weights* layers, const w4a16_layer_bias* biases,
                                     unsigned flags, int n_layers, int M, int hidden, int kv_dim, int ffn,
                                     int group, const w4a16_seq_io* io, w4a16_layer_seq** out);

/* Number of kernel launches one replay performs. */
int w4a16_layer_seq_num_launches(const w4a16_layer_seq* seq);

/* Enqueue one replay of the graph on `stream`; returns after enqueue. */
w4a16_status w4a16_layer_seq_run(w4a16_layer_seq* seq, void* stream);

/*
 * End-to-end replay with HOST buffers: on `stream`, copy host->x (if
 * host->x is not NULL) into the device x buffer, replay the graph, copy each
 * non-NULL host output pointer of `host` back from the matching device output.
 * Each host buffer has the size of its device counterpart.  Host buffers
 * should be page-locked for the copies to be asynchronous.  Returns after
 * enqueue; wait with w4a16_layer_seq_sync before reading the host outputs.
 */
w4a16_status w4a16_layer_seq_run_host(w4a16_layer_seq* seq, const w4a16_seq_io* host,
                                      void* stream);

/*
 * Wait for the most recent run / run_host of `seq`: timeout_ms < 0 waits
 * without bound, timeout_ms >= 0 polls and returns W4A16_ERR_TIMEOUT if the
 * replay has not finished in that time (the replay keeps running; call again
 * to keep waiting).  Once it has finished, the device status word of the
 * sequence's device is read (on the sequence's own stream): if it holds
 * W4A16_DEV_PIPE_TIMEOUT -- a pipeline or dependency wait inside a GEMV ran
 * past its bound, so outputs may be wrong -- the call returns
 * W4A16_ERR_DEVICE.  The word is shared by every call on the device and is
 * left set (later syncs return W4A16_ERR_DEVICE too) until
 * w4a16_device_status reads and clears it.
 */
w4a16_status w4a16_layer_seq_sync(w4a16_layer_seq* seq, int timeout_ms);

/* Free the graph, stream, event and counters.  NULL is a no-op.  Waits for
 * pending replays. */
void w4a16_layer_seq_destroy(w4a16_layer_seq* seq);

/* GEMVs one call of w4a16_layer_seq_run_static may run (its fixed scratch). */
#define W4A16_STATIC_MAX_GEMVS 512

/*
 * w4a16_layer_seq_run_static -- run the layer sequence once, M = 1, without
 * allocating anything.  The page has no counterpart of this entry point: it
 * exists for callers that cannot allocate device memory, such as a serving
 * process that hands all free device memory to its own pool (a KV cache)
 * up front, so that any cudaMalloc outside the pool fails or breaks its
 * budget, or code that must not call cudaFree (it waits for the whole device).
 * w4a16_layer_seq_create allocates its completion counters and a CUDA graph;
 * this call uses neither.
 *
 * Arguments and checks are those of w4a16_layer_seq_create with M = 1; the
 * work is the same task-list launches (one per up to 224 GEMVs), enqueued on
 * `stream` directly, so the outputs are the same bits.  Limits: at most
 * W4A16_STATIC_MAX_GEMVS tasks per call -- one per GEMV (4 per layer with
 * stacked [q; k; v] and [gate; up], up to 7 otherwise), two for a GEMV whose
 * K the M = 1 kernel splits in halves (a K = 18944 down projection) -- and
 * every K at most 28672 (the M = 1 kernel's range); beyond either the call
 * returns W4A16_ERR_LIMIT and
 * enqueues nothing.  Every task table is also checked against the kernel's
 * limits on this device before anything is enqueued; W4A16_ERR_CUDA after
 * that means a launch itself failed, and the memset and any launches before
 * it may have been enqueued (the outputs are then undefined).
 *
 * Scratch: the per-task completion counters are one fixed device array of
 * W4A16_STATIC_MAX_GEMVS ints (2 KB) inside the library, held on every device
 * that loads the library until the process exits.  Each call zeroes the
 * counters it uses with a memset on `stream` before its launches.  All calls
 * on a device share that array: calls whose work overlaps on the GPU (on
 * different streams, or from different host threads) race on it and give
 * wrong results; order them (one stream, or events).
 *
 * The first call on a device does a one-time set-up (device queries, kernel
 * attributes, the device address of the counter array); make that first call
 * before any CUDA stream capture.  Host-side tables are thread-local and keep
 * their capacity, so later calls allocate no host memory either.  Returns
 * after enqueue.
 */
w4a16_status w4a16_layer_seq_run_static(const w4a16_layer_weights* layers, int n_layers,
                                        int hidden, int kv_dim, int ffn, int group,
                                        const w4a16_seq_io* io, void* stream);

/*
 * Decode attention over an fp16 KV cache -- the bandwidth-bound kernel next
 * to the GEMV in a decode step (the page "LLM170", README of the LLM170
 * engine: its HIP decode attention reads an f16 copy of the KV cache and is
 * bound by that read at long context).  For one query token and query head h
 * reading KV head g = h / (n_heads / n_kv_heads) (grouped-query attention):
 *   o_h = sum_{t < T} softmax_t(q_h . k_{g,t} / sqrt(head_dim)) v_{g,t}
 * with FP32 scores, FP32 softmax statistics, the softmax weights rounded to
 * fp16 for the product with V (FP32 accumulation) and o rounded to fp16.
 *   q          fp16 [n_heads][head_dim]
 *   k_cache,   fp16 [n_kv_heads][t_stride][head_dim]; keys 0 .. T-1 of each
 *   v_cache    head are read, rows T .. t_stride-1 are never touched
 *   o          fp16 [n_heads][head_dim]; must not overlap q, the caches or
 *              the workspace
 *   workspace  device scratch of at least the size that
 *              w4a16_attn_decode_workspace returns for the same shape, owned
 *              by the caller; must not overlap q or the caches.  It must be
 *              zero-filled before its first use: its first
 *              4 * W4A16_ATTN_MAX_KV_HEADS bytes count the finished key
 *              ranges of each KV head, and every call leaves them zero
 *              again, so it can be reused for any shape it is large enough
 *              for.  After a call that set W4A16_DEV_PIPE_TIMEOUT, zero it
 *              again.  Two calls that overlap on the GPU must not share it.
 * Limits: head_dim == 128, n_heads a multiple of n_kv_heads with at most 16
 * query heads per KV head, n_kv_heads <= W4A16_ATTN_MAX_KV_HEADS, 1 <= T <= t_stride <= 2^24 (W4A16_ERR_SHAPE
 * otherwise, also for a workspace smaller than required); every pointer
 * 16-byte aligned (W4A16_ERR_ALIGN).  One kernel launch on `stream`, a
 * programmatic dependent of the kernel before it (it reads q and the caches
 * only after the previous kernel has completed): the key ranges of each KV
 * head are merged, in a fixed order, by the CTA that finishes last.  Never
 * allocates, never synchronises, deterministic.
 */
w4a16_status w4a16_attn_decode_workspace(int n_heads, int n_kv_heads, int head_dim, int T,
                                         size_t* bytes);
w4a16_status w4a16_attn_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                               uint16_t* o, int n_heads, int n_kv_heads, int head_dim, int T,
                               int t_stride, float* workspace, size_t workspace_bytes, void* stream);

/*
 * GGUF Q4_K super-blocks (the format the page "VTE" dequantises byte for
 * byte in llama.cpp's layout; the hipEngine page serves GGUF Q4_K_M files).
 * A row of K weights (K a positive multiple of 256, at most W4A16_MAX_K) is
 * K / 256 blocks of 144 bytes, rows back to back (`blocks` N * K / 256 * 144
 * bytes, 16-byte aligned):
 *   bytes 0-1 d, 2-3 dmin (fp16); bytes 4-15 eight 6-bit scales sc_j and
 *   minima m_j (j < 4: sc_j = b[j] & 63, m_j = b[j + 4] & 63; j >= 4:
 *   sc_j = (b[j + 4] & 15) | (b[j - 4] >> 6) << 4, m_j = (b[j + 4] >> 4) |
 *   (b[j] >> 6) << 4, b = bytes 4-15); bytes 16-143 unsigned 4-bit codes,
 *   chunk c of 32 bytes holding sub-block 2c in the low nibbles and 2c + 1
 *   in the high nibbles (weight 64 c + i, i < 32: low nibble of byte i).
 * The weight is w = d sc_j q - dmin m_j.  The blocks are read as stored (no
 * repack).
 *
 * w4a16_q4k_gemv   y[n] = fp16_RN(sum_k x[k] w[n][k]) for one activation
 *                  row x (fp16 [K]), y fp16 [N] (must not overlap x or the
 *                  blocks); FP32 accumulation; a programmatic dependent of
 *                  the previous kernel on the stream as w4a16_gemv.
 * w4a16_q4k_dequant  w_out float [N][K] = (d sc_j) q - dmin m_j in FP32 with
 *                  three roundings (the reference dequantisation; must not
 *                  overlap the blocks).
 * N == 0: OK, nothing launched.  Errors: W4A16_ERR_SHAPE, _NULL, _ALIGN,
 * _ALIAS, _CUDA as for w4a16_gemv.  Never allocate, never synchronise.
 */
w4a16_status w4a16_q4k_gemv(const uint8_t* blocks, const uint16_t* x, uint16_t* y, int N, int K,
                            void* stream);
w4a16_status w4a16_q4k_dequant(const uint8_t* blocks, float* w_out, int N, int K, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* W4A16_H */
