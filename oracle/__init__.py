"""CPU oracle for the W4A16 GEMV: ctypes binding to the plain C implementation.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference leg may import this package.  The GPU library in
int4_weight_only_gemv_gb300/ never imports it and shares no code with it.

Every function takes and returns numpy arrays.  fp16 data travels as uint16 bit
patterns so that no conversion happens outside the C code.  The semantics of
each function are documented in w4a16_oracle.c; the tolerance check follows the
bound stated for the GEMV (maximum error and relative L2 error, below).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None

ORC_OK = 0
ORC_ERR_SHAPE = 1
ORC_ERR_NONFINITE = 2
ORC_ERR_SCALE_OVERFLOW = 3

# Tolerances of the GEMV check: per activation row m,
#   max_n |y - y_ref| <= ABS_SLOPE * ||x_m||_2 * max_n ||w_hat_n||_2 + ABS_FLOOR
# and over the whole output ||y - y_ref||_2 / ||y_ref||_2 <= REL_L2.
ABS_SLOPE = 2e-3
ABS_FLOOR = 1e-3
REL_L2 = 1e-3


def lib(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library."""
    global _LIB
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _LIB is None:
        _LIB = _bind(ctypes.CDLL(_build.build()))
    return _LIB


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, u16 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint16
    L.orc_half_to_double.argtypes = [u16]
    L.orc_half_to_double.restype = ctypes.c_double
    L.orc_double_to_half.argtypes = [ctypes.c_double]
    L.orc_double_to_half.restype = u16
    L.orc_float_to_half.argtypes = [ctypes.c_float]
    L.orc_float_to_half.restype = u16
    L.orc_double_to_half_array.argtypes = [p, i64, p]
    L.orc_double_to_half_array.restype = None
    L.orc_half_to_double_array.argtypes = [p, i64, p]
    L.orc_half_to_double_array.restype = None
    L.orc_quantize.argtypes = [p, i64, i64, i64, p, p]
    L.orc_unpack.argtypes = [p, i64, i64, p]
    L.orc_dequant.argtypes = [p, p, i64, i64, i64, p]
    L.orc_dequant_f64.argtypes = [p, p, i64, i64, i64, p]
    L.orc_gemv.argtypes = [p, p, p, i64, i64, i64, i64, p]
    L.orc_gemv_rows.argtypes = [p, p, p, i64, i64, i64, i64, p, i64, p]
    L.orc_silu.argtypes = [ctypes.c_double]
    L.orc_silu.restype = ctypes.c_double
    L.orc_swiglu.argtypes = [p, p, i64, p]
    L.orc_swiglu.restype = None
    L.orc_attn_decode.argtypes = [p, p, p, i64, i64, i64, i64, i64, p]
    L.orc_attn_decode.restype = ctypes.c_int
    L.orc_quantize_act_a8.argtypes = [p, i64, p, p]
    L.orc_quantize_act_a8.restype = ctypes.c_int
    L.orc_gemv_w4a8.argtypes = [p, p, p, i64, i64, i64, i64, p]
    L.orc_gemv_w4a8.restype = ctypes.c_int
    L.orc_q4k_dequant.argtypes = [p, i64, i64, p]
    L.orc_q4k_dequant.restype = ctypes.c_int
    L.orc_q4k_gemv.argtypes = [p, p, i64, i64, i64, p]
    L.orc_q4k_gemv.restype = ctypes.c_int
    for f in ("orc_quantize", "orc_unpack", "orc_dequant", "orc_dequant_f64", "orc_gemv",
              "orc_gemv_rows"):
        getattr(L, f).restype = ctypes.c_int
    return L


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != ORC_OK:
        raise OracleError(f"{what} failed with oracle status {rc}")


def half_to_double(h: np.ndarray, L=None) -> np.ndarray:
    L = L or lib()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float64)
    L.orc_half_to_double_array(_ptr(h), h.size, _ptr(out))
    return out


def double_to_half(v: np.ndarray, L=None) -> np.ndarray:
    L = L or lib()
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    L.orc_double_to_half_array(_ptr(v), v.size, _ptr(out))
    return out


def quantize(w: np.ndarray, group: int = 128, L=None) -> tuple[np.ndarray, np.ndarray]:
    """fp32 W[N][K] -> (qweight uint32[N][K/8], scales uint16(fp16 bits)[N][K/G])."""
    L = L or lib()
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    qw = np.zeros((N, K // 8), np.uint32)
    sc = np.zeros((N, K // group), np.uint16)
    _check(L.orc_quantize(_ptr(w), N, K, group, _ptr(qw), _ptr(sc)), "quantize")
    return qw, sc


def unpack(qweight: np.ndarray, L=None) -> np.ndarray:
    L = L or lib()
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    N, K8 = qweight.shape
    q = np.empty((N, K8 * 8), np.int8)
    _check(L.orc_unpack(_ptr(qweight), N, K8 * 8, _ptr(q)), "unpack")
    return q


def dequant(qweight: np.ndarray, scales: np.ndarray, group: int = 128, L=None) -> np.ndarray:
    """fp16 bits [N][K] = fp16_RN(q * s)."""
    L = L or lib()
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    N, K8 = qweight.shape
    out = np.empty((N, K8 * 8), np.uint16)
    _check(L.orc_dequant(_ptr(qweight), _ptr(scales), N, K8 * 8, group, _ptr(out)), "dequant")
    return out


def dequant_f64(qweight: np.ndarray, scales: np.ndarray, group: int = 128, L=None) -> np.ndarray:
    """Exact q * s as float64 [N][K]."""
    L = L or lib()
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    N, K8 = qweight.shape
    out = np.empty((N, K8 * 8), np.float64)
    _check(L.orc_dequant_f64(_ptr(qweight), _ptr(scales), N, K8 * 8, group, _ptr(out)),
           "dequant_f64")
    return out


def gemv(qweight: np.ndarray, scales: np.ndarray, x: np.ndarray, group: int = 128,
         L=None) -> np.ndarray:
    """FP64 y[M][N] = x[M][K] . w_hat[N][K]^T; x given as fp16 bit patterns (uint16)."""
    L = L or lib()
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    N, K8 = qweight.shape
    M = x.shape[0]
    assert x.shape[1] == K8 * 8
    y = np.empty((M, N), np.float64)
    _check(L.orc_gemv(_ptr(qweight), _ptr(scales), _ptr(x), M, N, K8 * 8, group, _ptr(y)), "gemv")
    return y


def gemv_rows(qweight: np.ndarray, scales: np.ndarray, x: np.ndarray, rows: np.ndarray,
              group: int = 128, L=None) -> np.ndarray:
    """FP64 y[M][len(rows)] for the selected output rows only."""
    L = L or lib()
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    if x.ndim == 1:
        x = x[None, :]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    N, K8 = qweight.shape
    M = x.shape[0]
    y = np.empty((M, rows.size), np.float64)
    _check(L.orc_gemv_rows(_ptr(qweight), _ptr(scales), _ptr(x), M, N, K8 * 8, group,
                           _ptr(rows), rows.size, _ptr(y)), "gemv_rows")
    return y


def silu(v: float, L=None) -> float:
    """silu(v) = v / (1 + e^-v) in double (the SwiGLU activation)."""
    return float((L or lib()).orc_silu(float(v)))


def swiglu(g: np.ndarray, u: np.ndarray, L=None) -> np.ndarray:
    """h = fp16_RN(silu(g) * u) elementwise from fp16 bit patterns (uint16),
    in double with one rounding."""
    g = np.ascontiguousarray(g, dtype=np.uint16)
    u = np.ascontiguousarray(u, dtype=np.uint16)
    if g.shape != u.shape:
        raise ValueError("g and u differ in shape")
    h = np.empty(g.shape, dtype=np.uint16)
    (L or lib()).orc_swiglu(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def attn_decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, T: int | None = None, L=None) -> np.ndarray:
    """Decode attention of one token (see orc_attn_decode): q uint16 (fp16 bits)
    [H][D], k and v uint16 [Hkv][t_stride][D] (keys t < T used, default all);
    returns o float64 [H][D]."""
    L = L or lib()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    H, D = q.shape
    Hkv, t_stride, Dk = k.shape
    assert Dk == D and v.shape == k.shape
    T = t_stride if T is None else T
    o = np.empty((H, D), np.float64)
    _check(L.orc_attn_decode(_ptr(q), _ptr(k), _ptr(v), H, Hkv, D, T, t_stride, _ptr(o)), "attn_decode")
    return o


def quantize_act_a8(x: np.ndarray, L=None) -> tuple[np.ndarray, np.ndarray]:
    """One fp16 activation row (uint16 bits [K]) -> (int8 codes [K], float32
    block scales [K / 64]), see orc_quantize_act_a8."""
    L = L or lib()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    xq = np.empty(x.shape, np.int8)
    s = np.empty(x.size // 64, np.float32)
    _check(L.orc_quantize_act_a8(_ptr(x), x.size, _ptr(xq), _ptr(s)), "quantize_act_a8")
    return xq, s


def gemv_w4a8(qweight: np.ndarray, scales: np.ndarray, x: np.ndarray, group: int = 128, L=None) -> np.ndarray:
    """W4A8 GEMV (activations quantised per 64-element block), float64 [M][N]."""
    L = L or lib()
    qweight = np.ascontiguousarray(qweight, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    N, K8 = qweight.shape
    M = x.shape[0]
    y = np.empty((M, N), np.float64)
    _check(L.orc_gemv_w4a8(_ptr(qweight), _ptr(scales), _ptr(x), M, N, K8 * 8, group, _ptr(y)), "gemv_w4a8")
    return y


def q4k_dequant(blocks: np.ndarray, N: int, K: int, L=None) -> np.ndarray:
    """GGUF Q4_K blocks (uint8, N * K / 256 * 144 bytes) -> float32 [N][K]
    (the FP32 reference dequantisation, see orc_q4k_dequant)."""
    L = L or lib()
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    assert blocks.size == N * (K // 256) * 144
    w = np.empty((N, K), np.float32)
    _check(L.orc_q4k_dequant(_ptr(blocks), N, K, _ptr(w)), "q4k_dequant")
    return w


def q4k_gemv(blocks: np.ndarray, x: np.ndarray, N: int, K: int, L=None) -> np.ndarray:
    """y[M][N] = x . w^T over GGUF Q4_K blocks with exact weights, FP64."""
    L = L or lib()
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M = x.shape[0]
    y = np.empty((M, N), np.float64)
    _check(L.orc_q4k_gemv(_ptr(blocks), _ptr(x), M, N, K, _ptr(y)), "q4k_gemv")
    return y


# Tolerance of the decode-attention check, per query head h reading KV head g:
#   max_d |o - o_ref| <= ATTN_SLOPE * max_{t < T, d} |v_g[t][d]| + ATTN_FLOOR.
# The GPU rounds the softmax weights to fp16 for the P.V product (relative
# error <= 2^-11 per weight, so <= 2^-11 max|v| on o) and o to fp16 (another
# 2^-11 max|v|); scores and sums are FP32.  2e-3 is about twice their sum.
ATTN_SLOPE = 2e-3
ATTN_FLOOR = 1e-5


def check_attn(o: np.ndarray, o_ref: np.ndarray, v: np.ndarray, n_heads: int, T: int,
               slope: float = ATTN_SLOPE, floor: float = ATTN_FLOOR) -> dict:
    """o, o_ref [H][D] float64; v uint16 [Hkv][t_stride][D].  Returns a report
    with 'ok'.  Query head h reads KV head h / (n_heads / Hkv); its bound is
    slope * max|v| over that KV head's keys t < T, plus floor."""
    Hkv = v.shape[0]
    group = n_heads // Hkv
    vmax = np.abs(half_to_double(v[:, :T, :])).reshape(Hkv, -1).max(axis=1)
    bound = slope * vmax[np.arange(n_heads) // group] + floor
    err = np.abs(o - o_ref).max(axis=1)
    finite = bool(np.isfinite(o).all())
    return {"ok": finite and bool((err <= bound).all()), "finite": finite,
            "max_err": err.tolist(), "bound": bound.tolist()}


def row_norms(qweight: np.ndarray, scales: np.ndarray, group: int = 128, L=None) -> np.ndarray:
    """||w_hat_n||_2 for every output row n (exact dequantised weights)."""
    w = dequant_f64(qweight, scales, group, L)
    return np.sqrt(np.sum(w * w, axis=1))


def check_gemv(y: np.ndarray, y_ref: np.ndarray, x_f64: np.ndarray, max_row_norm: float,
               rel_l2: float = REL_L2, abs_slope: float = ABS_SLOPE,
               abs_floor: float = ABS_FLOOR) -> dict:
    """The GEMV tolerance.

    y      -- the result under test, float64 [M][n] (fp16 values widened)
    y_ref  -- the oracle's FP64 result, same shape
    x_f64  -- the activations as float64 [M][K]
    max_row_norm -- max_n ||w_hat_n||_2 over the rows of the weight matrix
    Returns a report dict with 'ok' and the measured figures.
    """
    y = np.atleast_2d(np.asarray(y, np.float64))
    y_ref = np.atleast_2d(np.asarray(y_ref, np.float64))
    x_f64 = np.atleast_2d(np.asarray(x_f64, np.float64))
    assert y.shape == y_ref.shape and x_f64.shape[0] == y.shape[0]
    err = np.abs(y - y_ref)
    bound = abs_slope * np.sqrt(np.sum(x_f64 * x_f64, axis=1)) * max_row_norm + abs_floor
    max_err = err.max(axis=1) if err.size else np.zeros(y.shape[0])
    denom = np.sqrt(np.sum(y_ref * y_ref))
    rel = float(np.sqrt(np.sum(err * err)) / denom) if denom > 0 else float(np.sqrt(np.sum(err * err)))
    finite = bool(np.all(np.isfinite(y)))
    ok = finite and bool(np.all(max_err <= bound)) and rel <= rel_l2
    return {"ok": ok, "finite": finite, "rel_l2": rel, "max_err": max_err.tolist(),
            "bound": bound.tolist()}
