"""GPU test of w4a16_layer_seq_run_static, the entry point that allocates
nothing.

Some callers cannot allocate device memory when they run the model: a
serving process that has handed all free device memory to its own pool (a
KV cache) cannot take a cudaMalloc outside it, and code that must not stall
cannot call cudaFree (it waits for the whole device).  layer_seq allocates
its completion counters and a CUDA graph at creation; run_static instead
keeps its counters in a fixed array inside the library and enqueues the
launches directly.  Here it must give the same outputs as a LayerSeq replay
(within the GEMV tolerance, and in fact bit for bit: same kernel, same task
table) on two calls in a row, each into outputs poisoned with NaN, so a
counter left over from the first call would show up in the second.

This file is collected last on purpose and stands alone: it builds the
library and draws its own inputs.
"""
import pytest
import torch

import int4_weight_only_gemv_gb300 as w4
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, KV, F = synth.HIDDEN, synth.KV_DIM, synth.FFN
N_LAYERS = 3
OUTS = (("y_q", H), ("y_k", KV), ("y_v", KV), ("y_o", H), ("y_gu", 2 * F), ("y_down", H))


@pytest.fixture(scope="module")
def model():
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    layers = []
    for l in range(N_LAYERS):
        lw = {}
        # layers 0 and 1: [q; k; v] and [gate; up] stacked (4 GEMVs per layer);
        # layer 2: seven separate weights (o then waits on q three GEMVs back)
        if l < 2:
            ws = [synth.weights(*synth.proj_shape(n), synth.layer_seed(l, i), DEV)
                  for i, n in enumerate(("q", "k", "v"))]
            qw, sc = w4.w4a16_quantize(torch.cat(ws))
            lw["q"], lw["k"], lw["v"] = (qw[:H], sc[:H]), (qw[H:H + KV], sc[H:H + KV]), (qw[H + KV:], sc[H + KV:])
            ws = [synth.weights(*synth.proj_shape(n), synth.layer_seed(l, 4 + i), DEV)
                  for i, n in enumerate(("gate", "up"))]
            qw, sc = w4.w4a16_quantize(torch.cat(ws))
            lw["gate"], lw["up"] = (qw[:F], sc[:F]), (qw[F:], sc[F:])
        for pj, name in enumerate(synth.PROJ_NAMES):
            if name not in lw:
                lw[name] = w4.w4a16_quantize(synth.weights(*synth.proj_shape(name),
                                                           synth.layer_seed(l, pj), DEV))
        layers.append(lw)
    x = torch.cat([synth.activations(1, H, synth.layer_seed(l, 7)) for l in range(N_LAYERS)])
    return layers, x.view(N_LAYERS, 1, H).to(DEV)


def _poisoned_io(x):
    io = {"x": x}
    for name, width in OUTS:
        io[name] = torch.full((N_LAYERS, 1, width), float("nan"), dtype=torch.float16, device=DEV)
    return io


def _bound(layers, l, name, xin):
    """The GEMV tolerance of the parity tests, for one projection of layer l:
    2e-3 ||x|| max_n ||w_hat_n|| + 1e-3."""
    w_hat = w4.w4a16_dequant(*layers[l][name]).double()
    return 2e-3 * float(xin.double().norm()) * float(w_hat.norm(dim=1).max()) + 1e-3


def test_run_static_matches_layer_seq_on_two_calls(model):
    layers, x = model
    io_ref = _poisoned_io(x)
    seq = w4.LayerSeq(layers, io_ref, 1, H, KV, F)
    seq.run()
    assert seq.sync() == 0
    seq.close()

    io = _poisoned_io(x)
    for call in range(2):
        for name, _ in OUTS:
            io[name].fill_(float("nan"))
        w4.w4a16_layer_seq_run_static(layers, io, H, KV, F)
        torch.cuda.synchronize()
        for name, _ in OUTS:
            assert not torch.isnan(io[name]).any(), (call, name)
        for l in range(N_LAYERS):
            views = {"q": ("y_q", slice(None), io_ref["x"][l]), "k": ("y_k", slice(None), io_ref["x"][l]),
                     "v": ("y_v", slice(None), io_ref["x"][l]), "o": ("y_o", slice(None), io_ref["y_q"][l]),
                     "gate": ("y_gu", slice(0, F), io_ref["x"][l]),
                     "up": ("y_gu", slice(F, 2 * F), io_ref["x"][l]),
                     "down": ("y_down", slice(None), io_ref["y_gu"][l][:, :F])}
            for name, (out, cols, xin) in views.items():
                got = io[out][l][:, cols].double()
                ref = io_ref[out][l][:, cols].double()
                d = (got - ref).abs().max().item()
                assert d <= _bound(layers, l, name, xin), (call, l, name, d)
        # same kernel, same task table: the bits agree too
        for name, _ in OUTS:
            assert torch.equal(io[name].view(torch.int16), io_ref[name].view(torch.int16)), (call, name)
    assert w4.w4a16_device_status(clear=True) == 0


def test_run_static_takes_no_device_memory(model):
    """The property the entry point exists for: after a first round of calls
    (which may set up the library on this device, and lets torch cache what
    the comparisons below need), further calls -- with another layer count,
    and on another stream -- leave both the device's free memory and torch's
    allocator untouched, and give the same bits on a side stream as on the
    default stream."""
    layers, x = model
    io = _poisoned_io(x)
    side = torch.cuda.Stream()
    io2 = {k: v[:2] for k, v in io.items()}
    w4.w4a16_layer_seq_run_static(layers, io, H, KV, F)
    torch.cuda.synchronize()
    ref = {name: io[name].clone() for name, _ in OUTS}

    def one_call(kind):
        for name, _ in OUTS:
            io[name].fill_(float("nan"))
        torch.cuda.synchronize()
        if kind == "fewer_layers":
            w4.w4a16_layer_seq_run_static(layers[:2], io2, H, KV, F)
        elif kind == "side_stream":
            with torch.cuda.stream(side):
                w4.w4a16_layer_seq_run_static(layers, io, H, KV, F, stream=side)
            side.synchronize()
        else:
            w4.w4a16_layer_seq_run_static(layers, io, H, KV, F)
        torch.cuda.synchronize()
        n = 2 if kind == "fewer_layers" else N_LAYERS
        return all(torch.equal(io[name][:n].view(torch.int16), ref[name][:n].view(torch.int16))
                   for name, _ in OUTS)

    kinds = ("default", "fewer_layers", "side_stream", "default")
    for kind in kinds:  # warm-up round: first use of every path
        assert one_call(kind), kind
    free0 = torch.cuda.mem_get_info()[0]
    alloc0 = torch.cuda.memory_allocated()
    for kind in kinds:
        assert one_call(kind), kind
        assert torch.cuda.mem_get_info()[0] == free0, kind
        assert torch.cuda.memory_allocated() == alloc0, kind
    assert w4.w4a16_device_status(clear=True) == 0


def test_run_static_rejects_k_beyond_the_kernel(model):
    """An FFN width whose down projection (K = 28800) is beyond the M = 1
    kernel's K range: W4A16_ERR_LIMIT, and the outputs keep their NaN."""
    h, kv, ffn = 128, 128, 28800
    lw = {}
    for pj, name in enumerate(synth.PROJ_NAMES):
        N, K = {"q": (h, h), "k": (kv, h), "v": (kv, h), "o": (h, h), "gate": (ffn, h), "up": (ffn, h),
                "down": (h, ffn)}[name]
        lw[name] = w4.w4a16_quantize(synth.weights(N, K, 71000 + pj, DEV))
    io = {"x": synth.activations(1, h, 71999).view(1, 1, h).to(DEV)}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn), ("y_down", h)):
        io[name] = torch.full((1, 1, width), float("nan"), dtype=torch.float16, device=DEV)
    with pytest.raises(w4.W4A16Error, match="LIMIT"):
        w4.w4a16_layer_seq_run_static([lw], io, h, kv, ffn)
    torch.cuda.synchronize()
    for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert torch.isnan(io[name]).all(), name


def test_run_static_rejects_beyond_its_limits(model):
    """More GEMVs than the fixed scratch holds, or a K beyond the M = 1
    kernel: W4A16_ERR_LIMIT, and nothing is written."""
    layers, x = model
    n = w4.STATIC_MAX_GEMVS // 4 + 1
    h, kv, ffn = 128, 128, 256
    small = {}
    for pj, name in enumerate(synth.PROJ_NAMES):
        N, K = {"q": (h, h), "k": (kv, h), "v": (kv, h), "o": (h, h), "gate": (ffn, h),
                "up": (ffn, h), "down": (h, ffn)}[name]
        small[name] = w4.w4a16_quantize(synth.weights(N, K, 70000 + pj, DEV))
    io = {"x": synth.activations(n, h, 7).view(n, 1, h).to(DEV)}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn),
                        ("y_down", h)):
        io[name] = torch.full((n, 1, width), float("nan"), dtype=torch.float16, device=DEV)
    with pytest.raises(w4.W4A16Error, match="LIMIT"):
        w4.w4a16_layer_seq_run_static([small] * n, io, h, kv, ffn)
    torch.cuda.synchronize()
    assert torch.isnan(io["y_q"]).all()
    # the same tables within the limit run
    m = w4.STATIC_MAX_GEMVS // 7
    io_m = {k: v[:m] for k, v in io.items()}
    w4.w4a16_layer_seq_run_static([small] * m, io_m, h, kv, ffn)
    torch.cuda.synchronize()
    assert not torch.isnan(io_m["y_down"]).any()
    assert w4.w4a16_device_status(clear=True) == 0
