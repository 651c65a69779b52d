"""GPU parity of the GGUF Q4_K path (w4a16_q4k_dequant, w4a16_q4k_gemv)
against the oracle through the C ABI: the FP32 reference dequantisation bit
for bit, and the M = 1 GEMV within the GEMV tolerance of the oracle's FP64
sum over the exact weights.  Blocks are random bytes (every code, scale and
minimum pattern occurs) with d and dmin drawn in [1e-3, 0.05]."""
import numpy as np
import pytest
import torch

import int4_weight_only_gemv_gb300 as w4
import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    oracle.lib()
    w4.w4a16_device_status(clear=True)
    yield
    assert w4.w4a16_device_status(clear=True) == 0


def _blocks(N, K, seed):
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 256, (N * (K // 256), 144)).astype(np.uint8)
    d = rng.uniform(1e-3, 0.05, (b.shape[0], 2)).astype(np.float16)
    b[:, 0:4] = d.view(np.uint8).reshape(-1, 4)
    return b.reshape(-1)


@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (33, 3584), (300, 18944)])
def test_q4k_dequant_bit_exact(N, K):
    b = _blocks(N, K, N + K)
    w = w4.w4a16_q4k_dequant(torch.from_numpy(b).to(DEV), N, K)
    torch.cuda.synchronize()
    ref = oracle.q4k_dequant(b, N, K)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def _max_row_norm(b, N, K):
    rows = b.reshape(N, -1)
    wn = 0.0
    for r0 in range(0, N, 4096):
        r1 = min(N, r0 + 4096)
        w = oracle.q4k_dequant(np.ascontiguousarray(rows[r0:r1]).reshape(-1), r1 - r0, K)
        wn = max(wn, float(np.linalg.norm(w.astype(np.float64), axis=1).max()))
    return wn


# K up to 28672 runs on the persistent TMA-fed kernel (1000 x 256: 448-row
# tiles; 100 x 3584: fewer rows than SMs; 3584 x 3584 and the full gate+up
# and down shapes: ragged row split over the SMs), larger K on the
# warp-per-row kernel (28928, 32768).
@pytest.mark.parametrize("N,K", [(1, 256), (7, 512), (1000, 256), (100, 3584), (37, 18944), (3584, 3584),
                                 (37888, 3584), (3584, 18944), (64, 28672), (64, 28928), (129, 32768)])
def test_q4k_gemv_against_oracle(N, K):
    b = _blocks(N, K, 3 * N + K)
    x = np.random.default_rng(N * K).standard_normal(K).astype(np.float16)
    y = w4.w4a16_q4k_gemv(torch.from_numpy(b).to(DEV), torch.from_numpy(x).to(DEV), N, K)
    torch.cuda.synchronize()
    y_ref = oracle.q4k_gemv(b, x.view(np.uint16)[None, :], N, K)
    wn = _max_row_norm(b, N, K)
    rep = oracle.check_gemv(y.double().cpu().numpy()[None, :], y_ref, x.astype(np.float64)[None, :], wn)
    assert rep["ok"], rep


def test_q4k_gemv_zero_and_deterministic():
    N, K = 64, 1024
    b = torch.from_numpy(_blocks(N, K, 5)).to(DEV)
    assert torch.all(w4.w4a16_q4k_gemv(b, torch.zeros(K, dtype=torch.float16, device=DEV), N, K) == 0)
    x = torch.from_numpy(np.random.default_rng(6).standard_normal(K).astype(np.float16)).to(DEV)
    a, c = w4.w4a16_q4k_gemv(b, x, N, K), w4.w4a16_q4k_gemv(b, x, N, K)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))
