"""GPU parity of the W4A8 variant (w4a16_gemv_a8 and the W4A16_SEQ_ACT_INT8
layer sequence) against the oracle's W4A8 GEMV (orc_gemv_w4a8), through the C
ABI.  Both sides quantise the activations per 64-element block with the same
FP32 steps, so the integer codes agree and the remaining difference is the
FP32 accumulation; the GEMV tolerance applies.  The distance from the W4A16
result (the activation rounding) is bounded as well."""
import numpy as np
import pytest
import torch

import int4_weight_only_gemv_gb300 as w4
import oracle
import synth
from gpu_helpers import Case, sample_rows, to_np_u16, to_np_u32

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, KV, F = synth.HIDDEN, synth.KV_DIM, synth.FFN


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    oracle.lib()
    w4.w4a16_device_status(clear=True)
    yield
    assert w4.w4a16_device_status(clear=True) == 0


@pytest.mark.parametrize("N,K", [(1, 128), (7, 256), (33, 1024), (100, 3584), (37, 18944), (3584, 3584),
                                 (153, 19456), (512, 1024)])
def test_gemv_a8_against_oracle(N, K):
    c = Case(N, K, 1, seed=7 * N + K)
    y = w4.w4a16_gemv_a8(c.qw, c.sc, c.x_dev)
    torch.cuda.synchronize()
    y_ref = oracle.gemv_w4a8(c.qw_ref, c.sc_ref, c.x_u16)
    rep = oracle.check_gemv(y.double().cpu().numpy(), y_ref, c.x_f64, c.max_row_norm())
    assert rep["ok"], rep
    # the activation rounding moves the result by about 1 % of |y|
    y16 = oracle.gemv(c.qw_ref, c.sc_ref, c.x_u16)
    assert np.linalg.norm(y_ref - y16) <= 0.03 * np.linalg.norm(y16) + 1e-6


def test_gemv_a8_special_cases():
    c = Case(64, 1024, 1, seed=3)
    x0 = torch.zeros(1, 1024, dtype=torch.float16, device=DEV)
    assert torch.all(w4.w4a16_gemv_a8(c.qw, c.sc, x0) == 0)
    # block maxima 127 and integer activations quantise exactly: equals W4A16
    xi = torch.randint(-126, 127, (1, 1024), generator=torch.Generator().manual_seed(4)).half()
    xi[:, ::64] = 127.0
    a = w4.w4a16_gemv_a8(c.qw, c.sc, xi.to(DEV)).double().cpu().numpy()
    y_ref = oracle.gemv(c.qw_ref, c.sc_ref, xi.view(torch.int16).numpy().view(np.uint16))
    assert oracle.check_gemv(a, y_ref, xi.double().numpy(), c.max_row_norm())["ok"]
    # deterministic
    b = w4.w4a16_gemv_a8(c.qw, c.sc, c.x_dev)
    b2 = w4.w4a16_gemv_a8(c.qw, c.sc, c.x_dev)
    assert torch.equal(b.view(torch.int16), b2.view(torch.int16))


def test_gemv_a8_argument_ranges():
    c = Case(16, 256, 2, seed=1)
    y = torch.empty((2, 16), dtype=torch.float16, device=DEV)
    L = w4.lib()
    assert L.w4a16_gemv_a8(c.qw.data_ptr(), c.sc.data_ptr(), c.x_dev.data_ptr(), y.data_ptr(), 2, 16, 256, 128,
                           None) == 5  # M > 1
    big = Case(4, 32768, 1, seed=2)
    yb = torch.empty((1, 4), dtype=torch.float16, device=DEV)
    assert L.w4a16_gemv_a8(big.qw.data_ptr(), big.sc.data_ptr(), big.x_dev.data_ptr(), yb.data_ptr(), 1, 4,
                           32768, 128, None) == 2  # K beyond the M = 1 kernel


NL = 2
WIDTH = {"q": H, "k": KV, "v": KV, "o": H, "gate": F, "up": F, "down": H}


def _layers():
    layers = []
    for l in range(NL):
        lw = {}
        for names, idx in ((("q", "k", "v"), (0, 1, 2)), (("gate", "up"), (4, 5))):
            ws = [synth.weights(*synth.proj_shape(n), synth.layer_seed(l, i), DEV) for n, i in zip(names, idx)]
            qw, sc = w4.w4a16_quantize(torch.cat(ws))
            r = 0
            for n, wt in zip(names, ws):
                lw[n] = (qw[r:r + wt.shape[0]], sc[r:r + wt.shape[0]])
                r += wt.shape[0]
        for pj, n in enumerate(synth.PROJ_NAMES):
            if n not in lw:
                lw[n] = w4.w4a16_quantize(synth.weights(*synth.proj_shape(n), synth.layer_seed(l, pj), DEV))
        layers.append(lw)
    return layers


def _io():
    x = torch.cat([synth.activations(1, H, synth.layer_seed(l, 7)) for l in range(NL)])
    io = {"x": x.view(NL, 1, H).to(DEV)}
    for name, width in (("y_q", H), ("y_k", KV), ("y_v", KV), ("y_o", H), ("y_gu", 2 * F), ("y_down", H)):
        io[name] = torch.full((NL, 1, width), float("nan"), dtype=torch.float16, device=DEV)
    return io


@pytest.mark.parametrize("epilogues", [False, True])
def test_layer_seq_act_int8(epilogues):
    layers = _layers()
    io = _io()
    biases = None
    if epilogues:
        g = torch.Generator().manual_seed(9)
        biases = [{n: (torch.randn(WIDTH[n], generator=g) * 0.5).half().to(DEV) for n in ("q", "k", "v")}
                  for _ in range(NL)]
    seq = w4.LayerSeq(layers, io, 1, H, KV, F, biases=biases, swiglu=epilogues, act_int8=True)
    assert seq.num_launches == 1
    seq.run()
    assert seq.sync() == 0
    for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert not torch.isnan(io[name]).any(), name
    for l in range(NL):
        lw = layers[l]
        x = to_np_u16(io["x"][l])
        ygu = io["y_gu"][l]
        down_in = (oracle.swiglu(to_np_u16(ygu[:, :F]), to_np_u16(ygu[:, F:])) if epilogues
                   else to_np_u16(ygu[:, :F]))
        cases = {"q": (x, io["y_q"][l]), "k": (x, io["y_k"][l]), "v": (x, io["y_v"][l]),
                 "o": (to_np_u16(io["y_q"][l]), io["y_o"][l]), "gate": (x, ygu[:, :F]),
                 "up": (x, ygu[:, F:]), "down": (down_in, io["y_down"][l])}
        for i, (name, (xin, yout)) in enumerate(cases.items()):
            qw, sc = to_np_u32(lw[name][0]), to_np_u16(lw[name][1])
            rows = sample_rows(qw.shape[0], 48, 10 * l + i)
            y_ref = oracle.gemv_w4a8(qw[rows], sc[rows], xin)
            if biases is not None and name in biases[l]:
                y_ref = y_ref + to_np_u16(biases[l][name]).view(np.float16).astype(np.float64)[rows][None, :]
            y = yout.to(torch.float64).cpu().numpy()[:, rows]
            rep = oracle.check_gemv(y, y_ref, xin.view(np.float16).astype(np.float64),
                                    float(oracle.row_norms(qw[rows], sc[rows]).max()))
            assert rep["ok"], (l, name, rep)
    seq.close()
