"""GPU tests of layer_seq: the seven projections of a Qwen-7B-shaped layer,
28 layers, captured as one CUDA graph.

Layers 0, 14 and 27 are drawn on the CPU and checked against the oracle on
sampled rows (each GEMV alone: o and down take the GPU's own fp16
intermediate as their input); every layer is checked bit for bit against
separate w4a16_gemv calls; run_host, the fused/unfused gate+up paths, M > 1
and the bounded sync are covered too.
"""
import numpy as np
import pytest
import torch

import int4_weight_only_gemv_gb300 as w4
import oracle
import synth
from gpu_helpers import to_np_u16, to_np_u32

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, KV, F, L = synth.HIDDEN, synth.KV_DIM, synth.FFN, synth.N_LAYERS
CHECKED_LAYERS = (0, L // 2, L - 1)


def _layer_weights(layer, fused=True, cpu=False, qkv=False):
    """One layer's packed weights.  fused: gate and up share one allocation;
    qkv: q, k and v share one allocation (both are launched as one GEMV)."""
    out, w_cpu = {}, {}
    dev_gen = "cpu" if cpu else DEV

    def draw(pj):
        N, K = synth.proj_shape(synth.PROJ_NAMES[pj])
        return synth.weights(N, K, synth.layer_seed(layer, pj), dev_gen)

    def stack(names, idx):
        ws = [draw(i) for i in idx]
        qw, sc = w4.w4a16_quantize(torch.cat(ws).to(DEV))
        r = 0
        for name, wt in zip(names, ws):
            n = wt.shape[0]
            out[name] = (qw[r:r + n], sc[r:r + n])
            w_cpu[name] = wt.cpu()
            r += n

    if qkv:
        stack(("q", "k", "v"), (0, 1, 2))
    if fused:
        stack(("gate", "up"), (4, 5))
    for pj, name in enumerate(synth.PROJ_NAMES):
        if name in out:
            continue
        w = draw(pj)
        out[name] = w4.w4a16_quantize(w.to(DEV))
        w_cpu[name] = w.cpu()
    return out, (w_cpu if cpu else None)


def _adjacent(first, second):
    """True when `second`'s packed weight and scales directly follow `first`'s."""
    (qa, sa), (qb, sb) = first, second
    return (qb.data_ptr() == qa.data_ptr() + qa.numel() * 4
            and sb.data_ptr() == sa.data_ptr() + sa.numel() * 2)


def _io(M, n_layers):
    x = torch.cat([synth.activations(M, H, synth.layer_seed(l, 7)) for l in range(n_layers)])
    io = {"x": x.view(n_layers, M, H).to(DEV)}
    for name, width in (("y_q", H), ("y_k", KV), ("y_v", KV), ("y_o", H), ("y_gu", 2 * F),
                        ("y_down", H)):
        io[name] = torch.full((n_layers, M, width), float("nan"), dtype=torch.float16, device=DEV)
    return io


@pytest.fixture(scope="module")
def seq28():
    from int4_weight_only_gemv_gb300 import build as wbuild
    wbuild.build()
    layers, cpu_w = [], {}
    for l in range(L):
        lw, wc = _layer_weights(l, fused=True, cpu=l in CHECKED_LAYERS, qkv=True)
        layers.append(lw)
        if wc is not None:
            cpu_w[l] = wc
    io = _io(1, L)
    seq = w4.LayerSeq(layers, io, 1, H, KV, F)
    seq.run()
    assert seq.sync() == 0
    torch.cuda.synchronize()
    yield seq, layers, io, cpu_w
    seq.close()


def test_layer_seq_launch_count(seq28):
    seq = seq28[0]
    # M = 1: the 4 x 28 GEMVs ([q; k; v] and [gate; up] stacked) are one task list
    assert seq.num_launches == 1


def test_layer_seq_outputs_written(seq28):
    _, _, io, _ = seq28
    for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert not torch.isnan(io[name]).any(), name


def test_layer_seq_equals_separate_calls(seq28):
    """Every projection of every layer equals a separate w4a16_gemv (bitwise:
    same kernels, same inputs)."""
    _, layers, io, _ = seq28
    for l in range(L):
        lw = layers[l]
        x = io["x"][l]
        pairs = [("q", x, io["y_q"][l]), ("k", x, io["y_k"][l]), ("v", x, io["y_v"][l]),
                 ("o", io["y_q"][l], io["y_o"][l]),
                 ("down", io["y_gu"][l][:, :F].contiguous(), io["y_down"][l])]
        for name, xin, yout in pairs:
            y = w4.w4a16_gemv(*lw[name], xin)
            assert torch.equal(y.view(torch.int16), yout.view(torch.int16)), (l, name)
        for name, half in (("gate", slice(0, F)), ("up", slice(F, 2 * F))):
            y = w4.w4a16_gemv(*lw[name], x)
            assert torch.equal(y.view(torch.int16), io["y_gu"][l][:, half].view(torch.int16)), (l, name)


@pytest.mark.parametrize("layer", CHECKED_LAYERS)
def test_layer_seq_against_oracle(seq28, layer):
    """Packed weights bit-exact, and every output of every GEMV of the layer
    within tolerance of the oracle (the full-size graph, as timed)."""
    _, layers, io, cpu_w = seq28
    lw, wc = layers[layer], cpu_w[layer]
    x_l = io["x"][layer].cpu()
    inputs = {"q": x_l, "k": x_l, "v": x_l, "gate": x_l, "up": x_l,
              "o": io["y_q"][layer].cpu(), "down": io["y_gu"][layer][:, :F].cpu()}
    outputs = {"q": io["y_q"][layer], "k": io["y_k"][layer], "v": io["y_v"][layer],
               "o": io["y_o"][layer], "gate": io["y_gu"][layer][:, :F],
               "up": io["y_gu"][layer][:, F:], "down": io["y_down"][layer]}
    for name in synth.PROJ_NAMES:
        qw_ref, sc_ref = oracle.quantize(wc[name].numpy())
        qw, sc = lw[name]
        assert np.array_equal(to_np_u32(qw), qw_ref) and np.array_equal(to_np_u16(sc), sc_ref), name
        xin = inputs[name].contiguous()
        x_u16 = xin.view(torch.int16).numpy().view(np.uint16)
        rows = np.arange(qw_ref.shape[0])
        y_ref = oracle.gemv_rows(qw_ref, sc_ref, x_u16, rows)
        y = outputs[name].to(torch.float64).cpu().numpy()[:, rows]
        norms = oracle.row_norms(qw_ref, sc_ref)
        rep = oracle.check_gemv(y, y_ref, xin.to(torch.float64).numpy(), float(norms.max()))
        assert rep["ok"], (name, rep)


def test_layer_seq_replay_is_deterministic(seq28):
    seq, _, io, _ = seq28
    before = {k: v.clone() for k, v in io.items() if k != "x"}
    seq.run()
    seq.sync()
    for k, v in before.items():
        assert torch.equal(v.view(torch.int16), io[k].view(torch.int16)), k


def test_layer_seq_run_host(seq28):
    """End-to-end replay with host buffers: x in, every output back."""
    seq, _, io, _ = seq28
    host = {"x": io["x"].cpu().pin_memory()}
    for k in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        host[k] = torch.empty(io[k].shape, dtype=torch.float16).pin_memory()
    seq.run_host(host)
    assert seq.sync() == 0
    for k in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert torch.equal(host[k].view(torch.int16), io[k].cpu().view(torch.int16)), k


def test_layer_seq_sync_timeout(seq28):
    """A zero-millisecond bound on a replay that cannot have finished returns
    W4A16_ERR_TIMEOUT; waiting without bound then completes."""
    seq = seq28[0]
    for _ in range(20):  # ~20 x 0.5 ms of queued work
        seq.run()
    assert seq.sync(0) == 8
    assert seq.sync(-1) == 0


def test_layer_seq_sync_reports_device_failure():
    """A bounded wait that ran out on the device (here the self-test's wait on
    a barrier nothing arrives on) makes the next sync return
    W4A16_ERR_DEVICE instead of OK; once the status word is cleared, a replay
    syncs OK again.  No kernel is left waiting: the self-test's wait ends at
    its 20 ms bound."""
    h, kv, ffn, n = 256, 128, 512, 2
    layers = []
    for l in range(n):
        lw = {}
        for pj, name in enumerate(synth.PROJ_NAMES):
            N, K = {"q": (h, h), "k": (kv, h), "v": (kv, h), "o": (h, h), "gate": (ffn, h), "up": (ffn, h),
                    "down": (h, ffn)}[name]
            lw[name] = w4.w4a16_quantize(synth.weights(N, K, 81000 + 8 * l + pj).to(DEV))
        layers.append(lw)
    io = {"x": synth.activations(n, h, 81999).view(n, 1, h).to(DEV)}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn), ("y_down", h)):
        io[name] = torch.empty((n, 1, width), dtype=torch.float16, device=DEV)
    seq = w4.LayerSeq(layers, io, 1, h, kv, ffn)
    assert w4.w4a16_device_status(clear=True) == 0
    seq.run()
    assert seq.sync() == 0
    w4.w4a16_selftest_wait_timeout(20000)
    seq.run()
    with pytest.raises(w4.W4A16Error, match="DEVICE"):
        seq.sync()
    with pytest.raises(w4.W4A16Error, match="DEVICE"):
        seq.sync(1000)  # the word stays set until it is read and cleared
    assert w4.w4a16_device_status(clear=True) == w4.DEV_PIPE_TIMEOUT
    seq.run()
    assert seq.sync() == 0
    seq.close()


@pytest.mark.parametrize("M,fused,qkv", [(1, False, False), (3, True, True), (3, False, False),
                                         (16, True, False), (8, False, True)])
def test_layer_seq_small(M, fused, qkv):
    """Two layers, stacked or separate weights, batched activations, vs
    separate calls."""
    n = 2
    layers = [_layer_weights(l, fused=fused, qkv=qkv)[0] for l in range(n)]
    io = _io(M, n)
    seq = w4.LayerSeq(layers, io, M, H, KV, F)
    # separately allocated weights may still land back to back in memory, in
    # which case the library launches them as one stack: count what is adjacent
    expect_launches = 0
    for lw in layers:
        q_k = _adjacent(lw["q"], lw["k"]) and _adjacent(lw["k"], lw["v"])
        g_u = _adjacent(lw["gate"], lw["up"])
        expect_launches += (1 if q_k else 3) + 1 + (1 if g_u else 2) + 1
        assert q_k or not qkv
        assert g_u or not fused
    # M = 1 runs the whole sequence as one task list
    assert seq.num_launches == (1 if M == 1 else expect_launches)
    seq.run()
    assert seq.sync() == 0
    for l in range(n):
        lw = layers[l]
        x = io["x"][l]
        for name in ("q", "k", "v"):
            y = w4.w4a16_gemv(*lw[name], x)
            ref = io["y_" + name][l]
            if qkv and M == 1:
                # one launch over [q; k; v]: per-row sums do not depend on the split
                assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), (l, name)
            else:
                d = (y.double() - ref.double()).abs().max().item()
                assert (d == 0.0) if not qkv else d < 0.05, (l, name, d)
        y = w4.w4a16_gemv(*lw["down"], io["y_gu"][l][:, :F].contiguous())
        assert torch.equal(y.view(torch.int16), io["y_down"][l].view(torch.int16))
        stacked_gu = _adjacent(lw["gate"], lw["up"])
        for name, half in (("gate", slice(0, F)), ("up", slice(F, 2 * F))):
            y = w4.w4a16_gemv(*lw[name], x)
            ref = io["y_gu"][l][:, half]
            if stacked_gu and M > 7:
                # the split of K in the tensor-core kernel depends on N: tolerance
                d = (y.double() - ref.double()).abs().max().item()
                assert d < 0.05, (l, name, d)
            else:
                assert torch.equal(y.view(torch.int16), ref.contiguous().view(torch.int16)), (l, name)
    seq.close()


def test_layer_seq_task_lists_split_between_layers():
    """M = 1 with more GEMVs than one task table holds: the sequence is split
    between layers into several launches (each a programmatic dependent of the
    previous one); every GEMV equals a separate call bit for bit, outputs
    prefilled with NaN are all written, and two replays agree."""
    h, kv, ffn, n = 256, 128, 512, 60
    layers = []
    for l in range(n):
        lw = {}
        ws = [synth.weights(N, h, 50000 + 8 * l + i) for i, N in enumerate((h, kv, kv))]
        qw, sc = w4.w4a16_quantize(torch.cat(ws).to(DEV))
        lw["q"], lw["k"], lw["v"] = (qw[:h], sc[:h]), (qw[h:h + kv], sc[h:h + kv]), (qw[h + kv:], sc[h + kv:])
        ws = [synth.weights(ffn, h, 50000 + 8 * l + 4 + i) for i in range(2)]
        qw, sc = w4.w4a16_quantize(torch.cat(ws).to(DEV))
        lw["gate"], lw["up"] = (qw[:ffn], sc[:ffn]), (qw[ffn:], sc[ffn:])
        lw["o"] = w4.w4a16_quantize(synth.weights(h, h, 50000 + 8 * l + 3).to(DEV))
        lw["down"] = w4.w4a16_quantize(synth.weights(h, ffn, 50000 + 8 * l + 6).to(DEV))
        layers.append(lw)
    x = torch.cat([synth.activations(1, h, 60000 + l) for l in range(n)]).view(n, 1, h).to(DEV)
    io = {"x": x}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn),
                        ("y_down", h)):
        io[name] = torch.full((n, 1, width), float("nan"), dtype=torch.float16, device=DEV)
    seq = w4.LayerSeq(layers, io, 1, h, kv, ffn)
    assert seq.num_launches == 2  # 4 GEMVs per layer, 224 per task table
    seq.run()
    assert seq.sync() == 0
    for name in ("y_q", "y_k", "y_v", "y_o", "y_gu", "y_down"):
        assert not torch.isnan(io[name]).any(), name
    first = {k: v.clone() for k, v in io.items() if k != "x"}
    for l in range(n):
        lw = layers[l]
        pairs = [("q", io["x"][l], io["y_q"][l]), ("k", io["x"][l], io["y_k"][l]),
                 ("v", io["x"][l], io["y_v"][l]), ("o", io["y_q"][l], io["y_o"][l]),
                 ("gate", io["x"][l], io["y_gu"][l][:, :ffn]), ("up", io["x"][l], io["y_gu"][l][:, ffn:]),
                 ("down", io["y_gu"][l][:, :ffn].contiguous(), io["y_down"][l])]
        for name, xin, yout in pairs:
            y = w4.w4a16_gemv(*lw[name], xin)
            assert torch.equal(y.view(torch.int16), yout.contiguous().view(torch.int16)), (l, name)
    seq.run()
    assert seq.sync() == 0
    for k, v in first.items():
        assert torch.equal(v.view(torch.int16), io[k].view(torch.int16)), k
    assert w4.w4a16_device_status(clear=True) == 0
    seq.close()


@pytest.mark.parametrize("h,kv,ffn", [(640, 128, 1280), (1024, 256, 2048)])
def test_short_rows_kernel_matches_sequence(h, kv, ffn):
    """A standalone M = 1 GEMV small enough for the warp-per-row kernel (at
    most 512 KB of packed weights, K <= 4096) gives the same bits as the same
    projection inside a layer sequence (the task kernel).  h = 640: five
    units of 128 k per row, so the row sum's units past the last whole four
    are exercised."""
    n = 2
    layers = []
    for l in range(n):
        lw = {}
        for pj, name in enumerate(synth.PROJ_NAMES):
            NN, KK = {"q": (h, h), "k": (kv, h), "v": (kv, h), "o": (h, h), "gate": (ffn, h), "up": (ffn, h),
                      "down": (h, ffn)}[name]
            lw[name] = w4.w4a16_quantize(synth.weights(NN, KK, 92000 + 8 * l + pj).to(DEV))
        layers.append(lw)
    io = {"x": synth.activations(n, h, 92999).view(n, 1, h).to(DEV)}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn), ("y_down", h)):
        io[name] = torch.full((n, 1, width), float("nan"), dtype=torch.float16, device=DEV)
    seq = w4.LayerSeq(layers, io, 1, h, kv, ffn)
    seq.run()
    seq.sync()
    small = 0
    for l in range(n):
        x = io["x"][l]
        for name, xin, yout in (("q", x, io["y_q"][l]), ("k", x, io["y_k"][l]), ("v", x, io["y_v"][l]),
                                ("o", io["y_q"][l], io["y_o"][l]),
                                ("down", io["y_gu"][l][:, :ffn].contiguous(), io["y_down"][l])):
            qw = layers[l][name][0]
            small += qw.numel() * 4 <= 512 * 1024 and qw.shape[1] * 8 <= 4096
            y = w4.w4a16_gemv(*layers[l][name], xin)
            assert torch.equal(y.view(torch.int16), yout.view(torch.int16)), (h, l, name)
    seq.close()
    assert small >= 4 * n  # q, k, v, o of each layer took the warp-per-row kernel
