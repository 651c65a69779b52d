"""GPU tests of the fused layer epilogues (w4a16_layer_seq_create2): output
biases and SwiGLU between [gate; up] and down, as the Qwen2 decoder of the
page on hipfire has them ("Overview of hipfire-arch-qwen2", "Key Technical
Specifications": SwiGLU feed-forward, attention_bias on Q, K, V).

Each projection of each layer is checked on sampled rows against the oracle:
y_ref = sum_k x w_hat (FP64) + bias, with the GPU's own fp16 intermediates as
inputs (o reads y_q; down reads h = fp16_RN(silu(gate) up) computed by the
oracle from the GPU's y_gu), within the GEMV tolerance.  M = 1 runs the task
list (gate and up as two tasks, h written by up's epilogue), M = 3 and M = 9
the tensor-core kernel (SwiGLU as a separate kernel).
"""
import numpy as np
import pytest
import torch

import int4_weight_only_gemv_gb300 as w4
import oracle
import synth
from gpu_helpers import sample_rows, to_np_u16, to_np_u32

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, KV, F = synth.HIDDEN, synth.KV_DIM, synth.FFN
NL = 2
WIDTH = {"q": H, "k": KV, "v": KV, "o": H, "gate": F, "up": F, "down": H}


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    oracle.lib()
    w4.w4a16_device_status(clear=True)
    yield
    assert w4.w4a16_device_status(clear=True) == 0


def _layers(stacked: bool):
    """Packed weights of NL layers; stacked: [q; k; v] and [gate; up] share one
    allocation each (one GEMV each in the sequence)."""
    layers = []
    for l in range(NL):
        lw = {}
        groups = ((("q", "k", "v"), (0, 1, 2)), (("gate", "up"), (4, 5))) if stacked else ()
        for names, idx in groups:
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


def _biases(seed: int):
    g = torch.Generator().manual_seed(seed)
    return [{n: (torch.randn(WIDTH[n], generator=g) * 0.5).to(torch.float16).to(DEV) for n in WIDTH}
            for _ in range(NL)]


def _io(M):
    x = torch.cat([synth.activations(M, H, synth.layer_seed(l, 7)) for l in range(NL)])
    io = {"x": x.view(NL, M, H).to(DEV)}
    for name, width in (("y_q", H), ("y_k", KV), ("y_v", KV), ("y_o", H), ("y_gu", 2 * F), ("y_down", H)):
        io[name] = torch.full((NL, M, width), float("nan"), dtype=torch.float16, device=DEV)
    return io


def _check(lw, name, x_u16, y_gpu, bias, seed):
    qw, sc = lw[name]
    qw_np, sc_np = to_np_u32(qw), to_np_u16(sc)
    rows = sample_rows(qw_np.shape[0], 48, seed)
    y_ref = oracle.gemv_rows(qw_np, sc_np, x_u16, rows)
    if bias is not None:
        y_ref = y_ref + to_np_u16(bias).view(np.float16).astype(np.float64)[rows][None, :]
    y = y_gpu.to(torch.float64).cpu().numpy()[:, rows]
    x_f64 = x_u16.view(np.float16).astype(np.float64)
    rep = oracle.check_gemv(y, y_ref, x_f64, float(oracle.row_norms(qw_np, sc_np).max()))
    assert rep["ok"], (name, rep)


@pytest.mark.parametrize("M,stacked", [(1, True), (1, False), (3, True), (9, False)])
def test_bias_and_swiglu_against_oracle(M, stacked):
    layers = _layers(stacked)
    biases = _biases(100 + M)
    io = _io(M)
    seq = w4.LayerSeq(layers, io, M, H, KV, F, biases=biases, swiglu=True)
    if M == 1:
        assert seq.num_launches == 1  # SwiGLU inside the task list
    seq.run()
    assert seq.sync() == 0
    for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert not torch.isnan(io[name]).any(), name
    for l in range(NL):
        lw, b = layers[l], biases[l]
        x = to_np_u16(io["x"][l])
        ygu = io["y_gu"][l]
        h = oracle.swiglu(to_np_u16(ygu[:, :F]), to_np_u16(ygu[:, F:]))
        cases = {"q": (x, io["y_q"][l]), "k": (x, io["y_k"][l]), "v": (x, io["y_v"][l]),
                 "o": (to_np_u16(io["y_q"][l]), io["y_o"][l]), "gate": (x, ygu[:, :F]),
                 "up": (x, ygu[:, F:]), "down": (h, io["y_down"][l])}
        for i, (name, (xin, yout)) in enumerate(cases.items()):
            _check(lw, name, xin, yout, b[name], seed=10 * l + i)
    seq.close()


def test_bias_subset_and_no_swiglu():
    """Biases on some projections only, no SwiGLU: down reads the gate half."""
    M = 1
    layers = _layers(True)
    full = _biases(7)
    biases = [{"q": full[l]["q"], "v": full[l]["v"], "down": full[l]["down"]} for l in range(NL)]
    io = _io(M)
    seq = w4.LayerSeq(layers, io, M, H, KV, F, biases=biases, swiglu=False)
    seq.run()
    assert seq.sync() == 0
    for l in range(NL):
        lw, b = layers[l], biases[l]
        x = to_np_u16(io["x"][l])
        _check(lw, "q", x, io["y_q"][l], b["q"], 1)
        _check(lw, "k", x, io["y_k"][l], None, 2)
        _check(lw, "v", x, io["y_v"][l], b["v"], 3)
        _check(lw, "down", to_np_u16(io["y_gu"][l][:, :F]), io["y_down"][l], b["down"], 4)
    seq.close()


@pytest.mark.parametrize("M", [1, 9])
def test_create2_without_options_equals_create(M):
    """No biases and no flags: the same graph as w4a16_layer_seq_create, bit for bit."""
    layers = _layers(True)
    io_a, io_b = _io(M), _io(M)
    a = w4.LayerSeq(layers, io_a, M, H, KV, F)
    b = w4.LayerSeq(layers, io_b, M, H, KV, F, biases=[{} for _ in range(NL)], swiglu=False)
    a.run()
    b.run()
    assert a.sync() == 0 and b.sync() == 0
    for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert torch.equal(io_a[name].view(torch.int16), io_b[name].view(torch.int16)), name
    a.close()
    b.close()


def test_swiglu_waits_for_both_halves_small_layers():
    """SwiGLU over separate gate and up GEMVs: down reads both halves of y_gu,
    so it must wait for both producers, whichever order the task table runs
    them in.  Small layers make each cycle of the table short, so a down task
    that waited for only one of them would read NaN from the poisoned half.
    Every output of every layer, on several replays, within tolerance of the
    oracle (h from the GPU's own y_gu)."""
    h, kv, ffn, n = 256, 128, 512, 6
    widths = {"q": (h, h), "k": (kv, h), "v": (kv, h), "o": (h, h), "gate": (ffn, h), "up": (ffn, h),
              "down": (h, ffn)}
    layers, keep = [], []
    for l in range(n):
        lw = {}
        for pj, name in enumerate(synth.PROJ_NAMES):
            lw[name] = w4.w4a16_quantize(synth.weights(*widths[name], 82000 + 8 * l + pj).to(DEV))
            keep.append(torch.empty(4096, dtype=torch.uint8, device=DEV))  # no two weights adjacent
        layers.append(lw)
    io = {"x": synth.activations(n, h, 82999).view(n, 1, h).to(DEV)}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn), ("y_down", h)):
        io[name] = torch.empty((n, 1, width), dtype=torch.float16, device=DEV)
    seq = w4.LayerSeq(layers, io, 1, h, kv, ffn, swiglu=True)
    assert seq.num_launches == 1
    for rep in range(4):
        for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
            io[name].fill_(float("nan"))
        seq.run()
        assert seq.sync() == 0
        for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
            assert not torch.isnan(io[name]).any(), (rep, name)
        for l in range(n):
            ygu = io["y_gu"][l]
            hh = oracle.swiglu(to_np_u16(ygu[:, :ffn]), to_np_u16(ygu[:, ffn:]))
            qw, sc = layers[l]["down"]
            qw_np, sc_np = to_np_u32(qw), to_np_u16(sc)
            y_ref = oracle.gemv(qw_np, sc_np, hh)
            rep_ = oracle.check_gemv(io["y_down"][l].double().cpu().numpy(), y_ref,
                                     hh.view(np.float16).astype(np.float64),
                                     float(oracle.row_norms(qw_np, sc_np).max()))
            assert rep_["ok"], (rep, l, rep_)
    seq.close()
