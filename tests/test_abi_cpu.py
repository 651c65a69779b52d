"""The C-ABI library on a host without a GPU: it loads, exports every function
include/w4a16.h declares, and rejects bad arguments with the documented
status before touching CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import int4_weight_only_gemv_gb300 as w4
from int4_weight_only_gemv_gb300 import build as wbuild

HEADER = os.path.join(wbuild.ROOT, "include", "w4a16.h")


@pytest.fixture(scope="module")
def L():
    wbuild.build()
    return w4.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_match_binding_list():
    assert declared_functions() == sorted(w4.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_library_is_built_for_sm_103a_only():
    # the architecture flags of the build: one -gencode, sm_103a
    assert wbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_abi_version_and_status_strings(L):
    assert L.w4a16_abi_version() == 1
    for code, name in w4.STATUS.items():
        s = L.w4a16_status_str(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert L.w4a16_status_str(999) == b"unknown status"


# fake, never-dereferenced device addresses: argument checks only look at values
A = 0x10000
B = 0x20000
C = 0x40000
D = 0x80000


@pytest.mark.parametrize("args,expect", [
    ((0, B, C, D, 1, 8, 128, 128), 1),          # null qweight
    ((A, 0, C, D, 1, 8, 128, 128), 1),          # null scales
    ((A, B, 0, D, 1, 8, 128, 128), 1),          # null x
    ((A, B, C, 0, 1, 8, 128, 128), 1),          # null y
    ((A, B, C, D, 1, 8, 128, 64), 4),           # group != 128
    ((A, B, C, D, 1, 8, 100, 128), 2),          # K not a multiple of 128
    ((A, B, C, D, 1, 8, 0, 128), 2),            # K = 0
    ((A, B, C, D, 1, 8, 32768 + 128, 128), 2),  # K above the maximum
    ((A, B, C, D, 1, -1, 128, 128), 2),         # negative N
    ((A, B, C, D, 17, 8, 128, 128), 5),         # M above 16
    ((A, B, C, D, -1, 8, 128, 128), 5),         # negative M
    ((A + 4, B, C, D, 1, 8, 128, 128), 3),      # misaligned qweight
    ((A, B + 2, C, D, 1, 8, 128, 128), 3),      # misaligned scales
    ((A, B, C + 8, D, 1, 8, 128, 128), 3),      # misaligned x
    ((A, B, C, D + 2, 1, 8, 128, 128), 3),      # misaligned y
    ((A, B, C, C, 1, 8, 128, 128), 6),          # y overlaps x
    ((A, B, C, A + 16, 1, 8, 128, 128), 6),     # y overlaps qweight
    ((A, B, C, B, 1, 8, 128, 128), 6),          # y overlaps scales
    ((0, 0, 0, 0, 0, 8, 128, 128), 0),          # M = 0: empty product, nothing launched
    ((0, 0, 0, 0, 4, 0, 128, 128), 0),          # N = 0: empty product
])
def test_gemv_argument_checks(L, args, expect):
    qw, sc, x, y, M, N, K, g = args
    assert L.w4a16_gemv(qw, sc, x, y, M, N, K, g, None) == expect


def test_dequant_and_quantize_argument_checks(L):
    assert L.w4a16_dequant(0, B, C, 8, 128, 128, None) == 1
    assert L.w4a16_dequant(A, B, C, 8, 128, 96, None) == 4
    assert L.w4a16_dequant(A, B, C, 8, 200, 128, None) == 2
    assert L.w4a16_dequant(A, B, C + 2, 8, 128, 128, None) == 3
    assert L.w4a16_dequant(A, B, A, 8, 128, 128, None) == 6
    assert L.w4a16_dequant(0, 0, 0, 0, 128, 128, None) == 0
    assert L.w4a16_quantize(0, B, C, 8, 128, 128, None) == 1
    assert L.w4a16_quantize(A, B, C, 8, 129, 128, None) == 2
    assert L.w4a16_quantize(A, B + 2, C, 8, 128, 128, None) == 3
    assert L.w4a16_quantize(A, A + 64, C, 8, 128, 128, None) == 6   # qweight inside w
    assert L.w4a16_quantize(0, 0, 0, 0, 128, 128, None) == 0


def test_layer_seq_argument_checks(L):
    out = ctypes.c_void_p(None)
    lw = (w4._LayerWeights * 1)()
    io = w4._SeqIO()
    assert L.w4a16_layer_seq_create(lw, 1, 1, 3584, 512, 18944, 128, ctypes.byref(io), None) == 1
    assert L.w4a16_layer_seq_create(None, 1, 1, 3584, 512, 18944, 128, ctypes.byref(io), ctypes.byref(out)) == 1
    assert L.w4a16_layer_seq_create(lw, 0, 1, 3584, 512, 18944, 128, ctypes.byref(io), ctypes.byref(out)) == 2
    assert L.w4a16_layer_seq_create(lw, 1, 0, 3584, 512, 18944, 128, ctypes.byref(io), ctypes.byref(out)) == 5
    assert L.w4a16_layer_seq_create(lw, 1, 1, 3584, 512, 18944, 64, ctypes.byref(io), ctypes.byref(out)) == 4
    # io pointers NULL
    assert L.w4a16_layer_seq_create(lw, 1, 1, 3584, 512, 18944, 128, ctypes.byref(io), ctypes.byref(out)) == 1
    assert out.value is None
    # weights NULL with valid-looking io
    io2 = w4._SeqIO(*[0x100000 * (i + 1) for i in range(7)])
    assert L.w4a16_layer_seq_create(lw, 1, 1, 256, 128, 512, 128, ctypes.byref(io2), ctypes.byref(out)) == 1
    # NULL handles
    assert L.w4a16_layer_seq_run(None, None) == 9
    assert L.w4a16_layer_seq_run_host(None, ctypes.byref(io), None) == 9
    assert L.w4a16_layer_seq_sync(None, 0) == 9
    assert L.w4a16_layer_seq_num_launches(None) == 0
    L.w4a16_layer_seq_destroy(None)  # no-op


def test_layer_seq_run_static_argument_checks(L):
    """The allocation-free entry point checks everything on the host, limits
    included, before touching the device."""
    io = w4._SeqIO(*[0x20_0000_0000 + 0x1000_0000 * i for i in range(7)])

    def layers(n, hidden, kv, ffn):
        arr = (w4._LayerWeights * n)()
        for l in range(n):
            for pj in range(7):
                arr[l].qweight[pj] = 0x10_0000_0000 + (7 * l + pj) * 0x100_0000
                arr[l].scales[pj] = 0x10_0000_0000 + (7 * l + pj) * 0x100_0000 + 0x80_0000
        return arr

    lw = layers(1, 256, 128, 512)
    assert L.w4a16_layer_seq_run_static(None, 1, 256, 128, 512, 128, ctypes.byref(io), None) == 1
    assert L.w4a16_layer_seq_run_static(lw, 1, 256, 128, 512, 128, None, None) == 1
    assert L.w4a16_layer_seq_run_static(lw, 0, 256, 128, 512, 128, ctypes.byref(io), None) == 2
    assert L.w4a16_layer_seq_run_static(lw, 1, 256, 128, 512, 64, ctypes.byref(io), None) == 4
    # more GEMVs than the fixed scratch holds (at least 4 per layer)
    n = w4.STATIC_MAX_GEMVS // 4 + 1
    assert L.w4a16_layer_seq_run_static(layers(n, 128, 128, 256), n, 128, 128, 256, 128,
                                        ctypes.byref(io), None) == 11
    # a K beyond the M = 1 kernel (down: K = ffn = 28800 > 28672)
    assert L.w4a16_layer_seq_run_static(layers(1, 128, 128, 28800), 1, 128, 128, 28800, 128,
                                        ctypes.byref(io), None) == 11
    assert L.w4a16_status_str(11) and b"limit" in L.w4a16_status_str(11)


def test_layer_seq_create2_argument_checks(L):
    """Epilogue options are checked on the host: unknown flag bits, misaligned
    biases and biases overlapping an output are rejected before any device
    work."""
    lw = (w4._LayerWeights * 1)()
    for pj in range(7):
        lw[0].qweight[pj] = 0x10_0000_0000 + pj * 0x100_0000
        lw[0].scales[pj] = 0x10_0000_0000 + pj * 0x100_0000 + 0x80_0000
    io = w4._SeqIO(*[0x20_0000_0000 + 0x1000_0000 * i for i in range(7)])
    out = ctypes.c_void_p(None)
    args = (1, 1, 256, 128, 512, 128, ctypes.byref(io), ctypes.byref(out))
    assert L.w4a16_layer_seq_create2(lw, None, 0x4, *args) == 2
    b = (w4._LayerBias * 1)()
    b[0].bias[0] = 0x30_0000_0008  # not 16-byte aligned
    assert L.w4a16_layer_seq_create2(lw, b, 0, *args) == 3
    b[0].bias[0] = 0x20_0000_0000 + 0x1000_0000 * 5 + 64  # inside y_gu
    assert L.w4a16_layer_seq_create2(lw, b, 1, *args) == 6
    assert L.w4a16_layer_seq_create2(lw, None, 0, 1, 1, 256, 128, 512, 128, ctypes.byref(io), None) == 1
    # W4A8 sequences: M = 1 only, and every K within the M = 1 kernel's range
    assert L.w4a16_layer_seq_create2(lw, None, 0x2, 1, 2, 256, 128, 512, 128, ctypes.byref(io),
                                     ctypes.byref(out)) == 5
    assert L.w4a16_layer_seq_create2(lw, None, 0x2, 1, 1, 256, 128, 32768, 128, ctypes.byref(io),
                                     ctypes.byref(out)) == 2


def test_gemv_a8_argument_checks(L):
    assert L.w4a16_gemv_a8(0, B, C, D, 1, 8, 128, 128, None) == 1          # null qweight
    assert L.w4a16_gemv_a8(A, B, C, D, 2, 8, 128, 128, None) == 5          # M > 1
    assert L.w4a16_gemv_a8(A, B, C, D, 1, 8, 32768, 128, None) == 2        # K beyond the M = 1 kernel
    assert L.w4a16_gemv_a8(A, B, C, C, 1, 8, 128, 128, None) == 6          # y overlaps x
    assert L.w4a16_gemv_a8(0, 0, 0, 0, 0, 8, 128, 128, None) == 0          # M = 0


def test_device_status_null(L):
    assert L.w4a16_device_status(None, 0) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(w4, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(w4, "_LIB", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        w4.lib()


def test_attn_decode_argument_checks(L):
    """Shape, null and alignment checks come before any CUDA call.  Q, K, V, O
    and the workspace are fake 16-byte aligned addresses far apart (never
    dereferenced: each call below fails its checks first)."""
    Q, K, V, O, W = 1 << 20, 1 << 30, 1 << 31, 1 << 32, 1 << 33
    f = L.w4a16_attn_decode
    assert f(Q, K, V, O, 28, 4, 64, 100, 100, W, 1 << 20, None) == 2     # head_dim != 128
    assert f(Q, K, V, O, 28, 5, 128, 100, 100, W, 1 << 20, None) == 2    # heads not a multiple
    assert f(Q, K, V, O, 34, 2, 128, 100, 100, W, 1 << 20, None) == 2    # 17 heads per KV head
    assert f(Q, K, V, O, 257, 257, 128, 100, 100, W, 1 << 20, None) == 2  # KV heads past the counter block
    assert f(Q, K, V, O, 28, 4, 128, 0, 100, W, 1 << 20, None) == 2      # T = 0
    assert f(Q, K, V, O, 28, 4, 128, 100, 99, W, 1 << 20, None) == 2     # t_stride < T
    assert f(0, K, V, O, 28, 4, 128, 100, 100, W, 1 << 20, None) == 1    # null q
    assert f(Q, K, V, O, 28, 4, 128, 100, 100, 0, 1 << 20, None) == 1    # null workspace
    assert f(Q, K + 2, V, O, 28, 4, 128, 100, 100, W, 1 << 20, None) == 3  # misaligned k
    assert f(Q, K, V, O + 8, 28, 4, 128, 100, 100, W, 1 << 20, None) == 3  # misaligned o
    n = ctypes.c_size_t(7)
    assert L.w4a16_attn_decode_workspace(28, 4, 128, 0, ctypes.byref(n)) == 2 and n.value == 0
    assert L.w4a16_attn_decode_workspace(28, 4, 128, 10, None) == 1


def test_q4k_argument_checks(L):
    assert L.w4a16_q4k_gemv(A, C, D, 8, 100, None) == 2        # K not a multiple of 256
    assert L.w4a16_q4k_gemv(A, C, D, 8, 32768 + 256, None) == 2
    assert L.w4a16_q4k_gemv(0, C, D, 8, 256, None) == 1        # null blocks
    assert L.w4a16_q4k_gemv(A + 8, C, D, 8, 256, None) == 3    # misaligned blocks
    assert L.w4a16_q4k_gemv(A, C, C, 8, 256, None) == 6        # y overlaps x
    assert L.w4a16_q4k_gemv(0, 0, 0, 0, 256, None) == 0        # N = 0
    assert L.w4a16_q4k_dequant(A, 0, 8, 256, None) == 1
    assert L.w4a16_q4k_dequant(A, A, 8, 256, None) == 6        # output overlaps the blocks


def test_checked_build_compiles_and_exports_every_declared_symbol():
    """The index-checked build (W4A16_CHECKED: kernels record
    W4A16_DEV_INDEX instead of an out-of-range access) compiles for sm_103a
    and exports the same entry points."""
    path = wbuild.build(checked=True)
    assert path.endswith("libw4a16_checked.so") and os.path.exists(path)
    Lc = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(Lc, name), name
