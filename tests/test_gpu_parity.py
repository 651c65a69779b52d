"""GPU parity: the CUDA library against the CPU oracle, through the C ABI.

dequant and quantise are bit-exact; the GEMV is within the stated tolerance
(per-row max error <= 2e-3 ||x|| max||w_hat_row|| + 1e-3 and relative L2
error <= 1e-3) on every workload shape, on ragged and edge shapes, at every
M in 1..16, deterministic run to run, with untouched guard bands around y.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_gemv_gb300 as w4
import oracle
import synth
from gpu_helpers import Case, to_np_u16, to_np_u32

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    oracle.lib()
    assert torch.cuda.is_available()
    w4.w4a16_device_status(clear=True)
    yield
    assert w4.w4a16_device_status(clear=True) == 0


# ------------------------------------------------------------------ quantise

@pytest.mark.parametrize("N,K", [(1, 128), (3, 384), (17, 256), (512, 1024), (3584, 3584),
                                 (512, 3584), (100, 18944)])
def test_quantize_bit_exact(N, K):
    c = Case(N, K, 1, seed=N + K)
    assert c.packed_equal()


@pytest.mark.parametrize("cfg", [synth.GATE_UP, synth.DOWN_SWEEP[0]], ids=lambda c: c.name)
def test_quantize_bit_exact_full_size(cfg):
    c = Case(cfg.N, cfg.K, 1, seed=cfg.seed)
    assert c.packed_equal()


def test_quantize_edge_values():
    """Exact half-integer quotients, zero groups, subnormal and largest scales."""
    K = 256
    w = np.zeros((6, K), np.float32)
    w[0, :8] = [7.0, 2.5, -2.5, 0.5, -0.5, 2.4999998, -6.5, 3.5]      # ties -> away from 0
    w[1, 128] = -0.25                                                   # one non-zero group
    w[2, :128] = np.float32(3e-7) * np.arange(128)                      # subnormal-range scale
    w[3, :] = np.float32(7.0 * 65504.0)                                 # largest finite scale
    w[4, :] = np.linspace(-1, 1, K, dtype=np.float32)
    w[5, 0] = np.float32(1e-30)                                         # scale rounds to 0
    c = Case(6, K, 1, seed=0, w_cpu=torch.from_numpy(w), x_cpu=torch.zeros(1, K, dtype=torch.float16))
    assert c.packed_equal()


def test_quantize_flags_bad_input():
    w = torch.zeros(4, 256)
    w[1, 7] = float("inf")
    w[2, 130] = 7.0 * 65520.0
    qw, sc = w4.w4a16_quantize(w.to(DEV))
    flags = w4.w4a16_device_status(clear=True)
    assert flags == w4.DEV_NONFINITE | w4.DEV_SCALE_OVERFLOW
    # the bad groups are written as zeros, the others as usual
    assert to_np_u16(sc)[1, 0] == 0 and to_np_u16(sc)[2, 1] == 0
    assert w4.w4a16_device_status(clear=True) == 0


# ------------------------------------------------------------------ dequant

@pytest.mark.parametrize("cfg", [synth.TINY, synth.Q_PROJ, synth.KV_PROJ, synth.GATE_UP,
                                 synth.DOWN_SWEEP[0]], ids=lambda c: c.name)
def test_dequant_bit_exact(cfg):
    c = Case(cfg.N, cfg.K, 1, seed=cfg.seed)
    assert c.packed_equal()
    got = to_np_u16(w4.w4a16_dequant(c.qw, c.sc))
    want = oracle.dequant(c.qw_ref, c.sc_ref)
    assert np.array_equal(got, want)


def test_dequant_every_nibble_and_scale():
    """All 16 nibble values in all 8 positions, random fp16 scales incl. subnormal."""
    rng = np.random.default_rng(5)
    N, K = 64, 256
    qw = rng.integers(0, 2**32, (N, K // 8), dtype=np.uint64).astype(np.uint32)
    qw[0, :] = 0x76543210
    qw[1, :] = 0xFEDCBA98
    sc = rng.integers(0, 0x7BFF, (N, K // 128)).astype(np.uint16)
    sc[2, 0] = 0x0001
    got = to_np_u16(w4.w4a16_dequant(torch.from_numpy(qw.view(np.int32)).to(DEV),
                                     torch.from_numpy(sc.view(np.int16)).view(torch.float16).to(DEV)))
    assert np.array_equal(got, oracle.dequant(qw, sc))


# ------------------------------------------------------------------ GEMV

def _run_and_check(c, rows=None):
    y = c.gemv()
    y2 = c.gemv()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16)), "not deterministic"
    rep = c.check(y, rows=rows)
    assert rep["ok"], rep
    return y


@pytest.mark.parametrize("cfg", [synth.TINY, synth.Q_PROJ, synth.KV_PROJ], ids=lambda c: c.name)
def test_gemv_small_configs_full(cfg):
    c = Case(cfg.N, cfg.K, cfg.M, seed=cfg.seed)
    assert c.packed_equal()
    _run_and_check(c)


def test_gemv_gate_up_full_size():
    """[gate; up] at full size, every one of the 37,888 outputs against the
    oracle (about 136 M multiply-adds on the host)."""
    cfg = synth.GATE_UP
    c = Case(cfg.N, cfg.K, cfg.M, seed=cfg.seed)
    assert c.packed_equal()
    _run_and_check(c)


@pytest.mark.parametrize("cfg", synth.DOWN_SWEEP, ids=lambda c: c.name)
def test_gemv_down_sweep_full_size(cfg):
    """down at full size, every output of every batch row against the oracle
    (M = 16: about 1.1 G multiply-adds on the host)."""
    c = Case(cfg.N, cfg.K, cfg.M, seed=cfg.seed)
    assert c.packed_equal()
    _run_and_check(c)


@pytest.mark.parametrize("M", list(range(1, 17)))
@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (33, 1024), (100, 3584), (37, 18944),
                                 (20, 19456), (9, 19584), (3, 28672), (4, 28800), (5, 32768)])
def test_gemv_shapes_and_batch(M, N, K):
    """Every M with ragged N and K across all three kernel families and their
    limits: at M = 1, K = 19456 takes the persistent kernel's K split and
    19584 does not; 28672 is that kernel's largest K and 28800 the rows
    kernel's smallest."""
    c = Case(N, K, M, seed=1000 * M + N)
    _run_and_check(c)


@pytest.mark.parametrize("N", [1, 2, 15, 16, 17, 151, 152, 153, 304, 1217, 4097])
def test_gemv_ragged_rows_m1_and_m16(N):
    for M in (1, 16):
        c = Case(N, 1024, M, seed=N)
        _run_and_check(c)


def test_gemv_guard_bands_and_poisoned_output():
    """y prefilled with NaN inside a larger buffer: every element is written,
    nothing outside y is."""
    for M, N, K in [(1, 1000, 3584), (4, 333, 1024), (16, 777, 2048)]:
        c = Case(N, K, M, seed=M)
        pad = 64
        buf = torch.full((M * N + 2 * pad,), float("nan"), dtype=torch.float16, device=DEV)
        buf[:pad] = 7.0
        buf[-pad:] = -7.0
        y = buf[pad:pad + M * N].view(M, N)
        assert y.data_ptr() % 16 == 0
        c.gemv(y=y)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == 7.0) and torch.all(buf[-pad:] == -7.0)
        assert not torch.isnan(y).any()
        assert c.check(y)["ok"]


def test_gemv_special_values():
    """Zero scales, zero activations, one-hot activations (a column of W_hat)."""
    N, K = 64, 1024
    c = Case(N, K, 1, seed=3)
    x0 = torch.zeros(1, K, dtype=torch.float16, device=DEV)
    assert torch.all(w4.w4a16_gemv(c.qw, c.sc, x0) == 0)
    dq = w4.w4a16_dequant(c.qw, c.sc).float()
    for k in (0, 1, 127, 128, 517, K - 1):
        e = torch.zeros(1, K, dtype=torch.float16, device=DEV)
        e[0, k] = 1.0
        y = w4.w4a16_gemv(c.qw, c.sc, e)
        assert torch.equal(y[0].float(), dq[:, k]), k
        e16 = e.repeat(16, 1)
        y16 = w4.w4a16_gemv(c.qw, c.sc, e16)
        assert torch.equal(y16[5].float(), dq[:, k]), k


def test_gemv_m_consistency():
    """A batch of M rows equals M single-row GEMVs (within tolerance; the
    kernels differ)."""
    c = Case(1000, 3584, 16, seed=9)
    y = c.gemv()
    for m in (0, 7, 15):
        ym = w4.w4a16_gemv(c.qw, c.sc, c.x_dev[m:m + 1].contiguous())
        d = (y[m].double() - ym[0].double()).abs().max().item()
        assert d <= 2e-3 * float(c.x_dev[m].double().norm()) * c.max_row_norm() + 1e-3


def test_fused_gate_up_equals_separate():
    """[gate; up] as one N = 2 ffn GEMV equals gate and up run separately
    (bitwise for M = 1: each row's sum does not depend on the row split)."""
    K, F = 3584, 4096
    wg = synth.weights(F, K, 31)
    wu = synth.weights(F, K, 32)
    x = synth.activations(1, K, 31).to(DEV)
    qg, sg = w4.w4a16_quantize(wg.to(DEV))
    qu, su = w4.w4a16_quantize(wu.to(DEV))
    qgu, sgu = w4.w4a16_quantize(torch.cat([wg, wu]).to(DEV))
    y = w4.w4a16_gemv(qgu, sgu, x)
    y_sep = torch.cat([w4.w4a16_gemv(qg, sg, x), w4.w4a16_gemv(qu, su, x)], dim=1)
    assert torch.equal(y.view(torch.int16), y_sep.view(torch.int16))


def test_gemv_on_side_stream():
    c = Case(3584, 3584, 1, seed=11)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = c.gemv()
    s.synchronize()
    assert c.check(y)["ok"]


def test_gemv_rejects_bad_args_on_gpu():
    c = Case(64, 256, 1, seed=1)
    with pytest.raises(w4.W4A16Error, match="ALIGN"):
        w4.w4a16_gemv(c.qw, c.sc, c.x_dev, torch.empty(64 * 2 + 1, dtype=torch.float16, device=DEV)[1:].view(1, 128)[:, :64])
    with pytest.raises(w4.W4A16Error, match="ALIAS"):
        w4.w4a16_gemv(c.qw, c.sc, c.x_dev, c.x_dev.view(1, 256)[:, :64])


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait on a barrier nothing arrives on gives up after its bound, sets
    DEV_PIPE_TIMEOUT, and the device keeps working."""
    assert w4.w4a16_device_status(clear=True) == 0
    w4.w4a16_selftest_wait_timeout(20000)
    assert w4.w4a16_device_status(clear=True) == w4.DEV_PIPE_TIMEOUT
    c = Case(256, 1024, 1, seed=2)
    assert c.check(c.gemv())["ok"]
    assert w4.w4a16_device_status(clear=True) == 0
