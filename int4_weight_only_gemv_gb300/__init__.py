"""Python binding of the W4A16 GEMV library (include/w4a16.h).

Argument marshalling only: every function passes device pointers, sizes and
the current CUDA stream of torch to the C ABI of libw4a16.so, and raises
W4A16Error on a non-OK status.  No step of the computation runs in Python or
in torch; if the compiled library is missing, importing the functions raises
instead of falling back to anything.

Tensors: qweight int32 [N][K/8] (the uint32 bit patterns), scales float16
[N][K/128], x float16 [M][K], y float16 [M][N], all CUDA, contiguous and
16-byte aligned.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "W4A16Error", "lib", "w4a16_gemv", "w4a16_dequant", "w4a16_quantize", "w4a16_device_status",
    "w4a16_selftest_wait_timeout", "w4a16_layer_seq_run_static", "STATIC_MAX_GEMVS",
    "LayerSeq", "GROUP", "MAX_M", "MAX_K", "DEV_NONFINITE", "DEV_SCALE_OVERFLOW",
    "DEV_PIPE_TIMEOUT", "DEV_INDEX", "STATUS", "EXPORTED_SYMBOLS", "w4a16_attn_decode", "attn_decode_workspace",
    "attn_decode_new_workspace", "w4a16_gemv_a8", "SEQ_ACT_INT8", "w4a16_q4k_gemv", "w4a16_q4k_dequant",
]

HERE = os.path.dirname(os.path.abspath(__file__))
# W4A16_LIBRARY=checked selects the index-checked build (build(checked=True)),
# whose kernels record W4A16_DEV_INDEX instead of an out-of-range access.
LIB_PATH = (os.path.join(HERE, "_lib", "checked", "libw4a16_checked.so")
            if os.environ.get("W4A16_LIBRARY") == "checked" else os.path.join(HERE, "_lib", "libw4a16.so"))

GROUP = 128
MAX_M = 16
MAX_K = 32768
DEV_NONFINITE = 0x1
DEV_SCALE_OVERFLOW = 0x2
DEV_PIPE_TIMEOUT = 0x4
DEV_INDEX = 0x8
SEQ_SWIGLU = 0x1
SEQ_ACT_INT8 = 0x2
NPROJ = 7
STATIC_MAX_GEMVS = 512

STATUS = {
    0: "W4A16_OK", 1: "W4A16_ERR_NULL", 2: "W4A16_ERR_SHAPE", 3: "W4A16_ERR_ALIGN",
    4: "W4A16_ERR_GROUP", 5: "W4A16_ERR_M_RANGE", 6: "W4A16_ERR_ALIAS", 7: "W4A16_ERR_CUDA",
    8: "W4A16_ERR_TIMEOUT", 9: "W4A16_ERR_STATE", 10: "W4A16_ERR_DEVICE", 11: "W4A16_ERR_LIMIT",
}

# Every function include/w4a16.h declares.
EXPORTED_SYMBOLS = (
    "w4a16_status_str", "w4a16_abi_version", "w4a16_gemv", "w4a16_dequant", "w4a16_quantize",
    "w4a16_device_status", "w4a16_selftest_wait_timeout", "w4a16_layer_seq_create", "w4a16_layer_seq_num_launches",
    "w4a16_layer_seq_run", "w4a16_layer_seq_run_host", "w4a16_layer_seq_sync",
    "w4a16_layer_seq_destroy", "w4a16_layer_seq_run_static", "w4a16_layer_seq_create2",
    "w4a16_attn_decode_workspace", "w4a16_attn_decode", "w4a16_gemv_a8", "w4a16_q4k_gemv",
    "w4a16_q4k_dequant",
)


class W4A16Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.name}")


class _LayerWeights(ctypes.Structure):
    _fields_ = [("qweight", ctypes.c_void_p * NPROJ), ("scales", ctypes.c_void_p * NPROJ)]


class _LayerBias(ctypes.Structure):
    _fields_ = [("bias", ctypes.c_void_p * NPROJ)]


class _SeqIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("x", "y_q", "y_k", "y_v", "y_o", "y_gu", "y_down")]


_LIB = None


def lib() -> ctypes.CDLL:
    """The loaded libw4a16.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m int4_weight_only_gemv_gb300.build` "
                "(or __graft_entry__.build()); there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        p, i = ctypes.c_void_p, ctypes.c_int
        L.w4a16_status_str.argtypes = [i]
        L.w4a16_status_str.restype = ctypes.c_char_p
        L.w4a16_abi_version.argtypes = []
        L.w4a16_abi_version.restype = i
        L.w4a16_gemv.argtypes = [p, p, p, p, i, i, i, i, p]
        L.w4a16_gemv_a8.argtypes = [p, p, p, p, i, i, i, i, p]
        L.w4a16_q4k_gemv.argtypes = [p, p, p, i, i, p]
        L.w4a16_q4k_dequant.argtypes = [p, p, i, i, p]
        L.w4a16_dequant.argtypes = [p, p, p, i, i, i, p]
        L.w4a16_quantize.argtypes = [p, p, p, i, i, i, p]
        L.w4a16_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), i]
        L.w4a16_selftest_wait_timeout.argtypes = [i, p]
        L.w4a16_layer_seq_create.argtypes = [ctypes.POINTER(_LayerWeights), i, i, i, i, i, i,
                                             ctypes.POINTER(_SeqIO), ctypes.POINTER(p)]
        L.w4a16_layer_seq_create2.argtypes = [ctypes.POINTER(_LayerWeights), ctypes.POINTER(_LayerBias),
                                              ctypes.c_uint, i, i, i, i, i, i, ctypes.POINTER(_SeqIO),
                                              ctypes.POINTER(p)]
        L.w4a16_layer_seq_num_launches.argtypes = [p]
        L.w4a16_layer_seq_num_launches.restype = i
        L.w4a16_layer_seq_run.argtypes = [p, p]
        L.w4a16_layer_seq_run_host.argtypes = [p, ctypes.POINTER(_SeqIO), p]
        L.w4a16_layer_seq_sync.argtypes = [p, i]
        L.w4a16_layer_seq_destroy.argtypes = [p]
        L.w4a16_layer_seq_destroy.restype = None
        L.w4a16_layer_seq_run_static.argtypes = [ctypes.POINTER(_LayerWeights), i, i, i, i, i,
                                                 ctypes.POINTER(_SeqIO), p]
        L.w4a16_attn_decode_workspace.argtypes = [i, i, i, i, ctypes.POINTER(ctypes.c_size_t)]
        L.w4a16_attn_decode.argtypes = [p, p, p, p, i, i, i, i, i, p, ctypes.c_size_t, p]
        for f in ("w4a16_gemv", "w4a16_gemv_a8", "w4a16_q4k_gemv", "w4a16_q4k_dequant", "w4a16_dequant", "w4a16_quantize", "w4a16_device_status",
                  "w4a16_selftest_wait_timeout",
                  "w4a16_layer_seq_create", "w4a16_layer_seq_run", "w4a16_layer_seq_run_host",
                  "w4a16_layer_seq_sync", "w4a16_layer_seq_run_static", "w4a16_layer_seq_create2",
                  "w4a16_attn_decode_workspace", "w4a16_attn_decode"):
            getattr(L, f).restype = i
        _LIB = L
    return _LIB


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise W4A16Error(rc, what)


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def w4a16_gemv(qweight, scales, x, y=None, stream=None):
    """y[M][N] = x[M][K] . w_hat^T.  Allocates y (float16) if not given."""
    import torch
    M, K = x.shape
    N = qweight.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(lib().w4a16_gemv(_ptr(qweight), _ptr(scales), _ptr(x), _ptr(y), M, N, K, GROUP,
                            _stream(stream)), "w4a16_gemv")
    return y


def w4a16_gemv_a8(qweight, scales, x, y=None, stream=None):
    """W4A8 GEMV (M = 1): activations quantised to int8 per 64-element block
    inside the kernel; y float16 [1][N] (allocated if not given)."""
    import torch
    M, K = x.shape
    N = qweight.shape[0]
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check(lib().w4a16_gemv_a8(_ptr(qweight), _ptr(scales), _ptr(x), _ptr(y), M, N, K, GROUP,
                               _stream(stream)), "w4a16_gemv_a8")
    return y


def w4a16_q4k_gemv(blocks, x, N, K, y=None, stream=None):
    """GGUF Q4_K GEMV (M = 1): blocks uint8 CUDA tensor of N * K / 256 * 144
    bytes, x float16 [K] or [1][K]; returns y float16 [N]."""
    import torch
    if y is None:
        y = torch.empty((N,), dtype=torch.float16, device=x.device)
    _check(lib().w4a16_q4k_gemv(_ptr(blocks), _ptr(x), _ptr(y), N, K, _stream(stream)), "w4a16_q4k_gemv")
    return y


def w4a16_q4k_dequant(blocks, N, K, w_out=None, stream=None):
    """GGUF Q4_K blocks -> float32 [N][K] (the FP32 reference dequantisation)."""
    import torch
    if w_out is None:
        w_out = torch.empty((N, K), dtype=torch.float32, device=blocks.device)
    _check(lib().w4a16_q4k_dequant(_ptr(blocks), _ptr(w_out), N, K, _stream(stream)), "w4a16_q4k_dequant")
    return w_out


def w4a16_gemv_raw(qw_ptr, sc_ptr, x_ptr, y_ptr, M, N, K, group=GROUP, stream=None) -> int:
    """Unchecked status passthrough (tests of the argument checks use it)."""
    return lib().w4a16_gemv(qw_ptr, sc_ptr, x_ptr, y_ptr, M, N, K, group, stream)


def attn_decode_workspace(n_heads, n_kv_heads, T, head_dim=128) -> int:
    """Bytes of device scratch w4a16_attn_decode needs for this shape."""
    n = ctypes.c_size_t(0)
    _check(lib().w4a16_attn_decode_workspace(n_heads, n_kv_heads, head_dim, T, ctypes.byref(n)),
           "w4a16_attn_decode_workspace")
    return n.value


def attn_decode_new_workspace(n_heads, n_kv_heads, T, device, head_dim=128):
    """A zero-filled workspace for w4a16_attn_decode of this shape (or any
    shape needing no more bytes); calls leave it zero-filled where it must
    be, so it can be reused."""
    import torch
    return torch.zeros(attn_decode_workspace(n_heads, n_kv_heads, T, head_dim) // 4, dtype=torch.float32,
                       device=device)


def w4a16_attn_decode(q, k_cache, v_cache, T=None, o=None, workspace=None, stream=None):
    """Decode attention of one token: q float16 [H][128], caches float16
    [Hkv][t_stride][128] (keys t < T, default all), o float16 [H][128]
    (allocated if not given); workspace a CUDA tensor of at least
    attn_decode_workspace(...) bytes, zero-filled before its first use
    (attn_decode_new_workspace; allocated if not given)."""
    import torch
    H, D = q.shape
    Hkv, t_stride, _ = k_cache.shape
    T = t_stride if T is None else T
    if o is None:
        o = torch.empty((H, D), dtype=torch.float16, device=q.device)
    if workspace is None:
        workspace = attn_decode_new_workspace(H, Hkv, T, q.device, D)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().w4a16_attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), H, Hkv, D, T, t_stride,
                                   _ptr(workspace), nbytes, _stream(stream)), "w4a16_attn_decode")
    return o


def w4a16_attn_decode_raw(q_ptr, k_ptr, v_ptr, o_ptr, H, Hkv, D, T, t_stride, ws_ptr, ws_bytes,
                          stream=None) -> int:
    """Unchecked status passthrough (tests of the argument checks use it)."""
    return lib().w4a16_attn_decode(q_ptr, k_ptr, v_ptr, o_ptr, H, Hkv, D, T, t_stride, ws_ptr, ws_bytes,
                                   stream)


def w4a16_dequant(qweight, scales, w_out=None, stream=None):
    import torch
    N = qweight.shape[0]
    K = qweight.shape[1] * 8
    if w_out is None:
        w_out = torch.empty((N, K), dtype=torch.float16, device=qweight.device)
    _check(lib().w4a16_dequant(_ptr(qweight), _ptr(scales), _ptr(w_out), N, K, GROUP,
                               _stream(stream)), "w4a16_dequant")
    return w_out


def w4a16_quantize(w, qweight=None, scales=None, stream=None):
    """fp32 W[N][K] -> (qweight int32 [N][K/8], scales float16 [N][K/128])."""
    import torch
    N, K = w.shape
    if qweight is None:
        qweight = torch.empty((N, K // 8), dtype=torch.int32, device=w.device)
    if scales is None:
        scales = torch.empty((N, K // GROUP), dtype=torch.float16, device=w.device)
    _check(lib().w4a16_quantize(_ptr(w), _ptr(qweight), _ptr(scales), N, K, GROUP,
                                _stream(stream)), "w4a16_quantize")
    return qweight, scales


def w4a16_device_status(clear: bool = True) -> int:
    """The W4A16_DEV_* bits recorded by kernels on the current device."""
    flags = ctypes.c_uint32(0)
    rc = lib().w4a16_device_status(ctypes.byref(flags), int(clear))
    if rc not in (0, 10):
        raise W4A16Error(rc, "w4a16_device_status")
    return int(flags.value)


def w4a16_selftest_wait_timeout(limit_us: int = 20000, stream=None) -> None:
    """Run the bounded-wait self-test kernel (sets DEV_PIPE_TIMEOUT)."""
    _check(lib().w4a16_selftest_wait_timeout(limit_us, _stream(stream)),
           "w4a16_selftest_wait_timeout")


def _layer_tables(layers, io):
    arr = (_LayerWeights * len(layers))()
    for li, lw in enumerate(layers):
        for pj, name in enumerate(LayerSeq.NAMES):
            qw, sc = lw[name]
            arr[li].qweight[pj] = qw.data_ptr()
            arr[li].scales[pj] = sc.data_ptr()
    return arr, _SeqIO(*[io[n].data_ptr() for n in LayerSeq.IO])


def w4a16_layer_seq_run_static(layers, io, hidden, kv_dim, ffn, stream=None) -> None:
    """Run the M = 1 layer sequence once on `stream` through the entry point
    that allocates nothing (for callers that cannot allocate device memory:
    its scratch is a fixed array inside the library, W4A16_ERR_LIMIT beyond
    STATIC_MAX_GEMVS GEMVs).  Same layers / io conventions as LayerSeq, M = 1.
    Calls that overlap on the GPU share that scratch and race."""
    arr, sio = _layer_tables(layers, io)
    _check(lib().w4a16_layer_seq_run_static(arr, len(layers), hidden, kv_dim, ffn, GROUP,
                                            ctypes.byref(sio), _stream(stream)),
           "w4a16_layer_seq_run_static")


class LayerSeq:
    """n_layers x {q, k, v, o, gate+up, down} GEMVs captured as one CUDA graph.

    layers: list of dicts name -> (qweight, scales) with names q, k, v, o,
    gate, up, down; io: dict of device tensors x, y_q, y_k, y_v, y_o, y_gu,
    y_down, each [n_layers][M][width].  Optional epilogues
    (w4a16_layer_seq_create2): biases, a list of dicts name -> fp16 tensor of
    the projection's output width (missing names: no bias); swiglu=True makes
    down read silu(gate) * up; act_int8=True runs every GEMV as the W4A8
    variant (M = 1).  The tensors must outlive the object.
    """

    NAMES = ("q", "k", "v", "o", "gate", "up", "down")
    IO = ("x", "y_q", "y_k", "y_v", "y_o", "y_gu", "y_down")

    def __init__(self, layers, io, M, hidden, kv_dim, ffn, biases=None, swiglu=False, act_int8=False):
        arr = (_LayerWeights * len(layers))()
        for li, lw in enumerate(layers):
            for pj, name in enumerate(self.NAMES):
                qw, sc = lw[name]
                arr[li].qweight[pj] = qw.data_ptr()
                arr[li].scales[pj] = sc.data_ptr()
        sio = _SeqIO(*[io[n].data_ptr() for n in self.IO])
        handle = ctypes.c_void_p(None)
        self._keep = (layers, io, biases)
        if biases is None and not swiglu and not act_int8:
            _check(lib().w4a16_layer_seq_create(arr, len(layers), M, hidden, kv_dim, ffn, GROUP,
                                                ctypes.byref(sio), ctypes.byref(handle)),
                   "w4a16_layer_seq_create")
        else:
            barr = None
            if biases is not None:
                barr = (_LayerBias * len(layers))()
                for li, lb in enumerate(biases):
                    for pj, name in enumerate(self.NAMES):
                        barr[li].bias[pj] = _ptr(lb.get(name))
            flags = (SEQ_SWIGLU if swiglu else 0) | (SEQ_ACT_INT8 if act_int8 else 0)
            _check(lib().w4a16_layer_seq_create2(arr, barr, flags, len(layers), M,
                                                 hidden, kv_dim, ffn, GROUP, ctypes.byref(sio),
                                                 ctypes.byref(handle)),
                   "w4a16_layer_seq_create2")
        self.handle = handle
        self.io = io

    @property
    def num_launches(self) -> int:
        return lib().w4a16_layer_seq_num_launches(self.handle)

    def run(self, stream=None) -> None:
        _check(lib().w4a16_layer_seq_run(self.handle, _stream(stream)), "w4a16_layer_seq_run")

    def run_host(self, host: dict, stream=None) -> None:
        """host: dict of pinned CPU tensors (any subset of IO names)."""
        hio = _SeqIO(*[_ptr(host.get(n)) for n in self.IO])
        _check(lib().w4a16_layer_seq_run_host(self.handle, ctypes.byref(hio), _stream(stream)),
               "w4a16_layer_seq_run_host")

    def sync(self, timeout_ms: int = -1) -> int:
        """0 when done; W4A16_ERR_TIMEOUT (8) if the bound ran out; raises otherwise."""
        rc = lib().w4a16_layer_seq_sync(self.handle, timeout_ms)
        if rc not in (0, 8):
            raise W4A16Error(rc, "w4a16_layer_seq_sync")
        return rc

    def close(self) -> None:
        if self.handle is not None and self.handle.value:
            lib().w4a16_layer_seq_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 -- interpreter shutdown
            pass
