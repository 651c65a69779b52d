"""GPU parity of the decode attention (w4a16_attn_decode) against the oracle
(orc_attn_decode, FP64), through the C ABI.

Shapes span one key, partial and full 64-key tiles, ragged tails, a cache
stride larger than T, multi-head (group 1), the Qwen-7B grouped shape (28
query heads over 4 KV heads) up to T = 8192 and the widest group (16 query
heads per KV head).  Inputs: q, k, v ~ N(0, 1) in fp16 (synthetic, seeded);
a scaled-up q gives sharp softmax weights.  The tolerance (oracle.check_attn)
covers the fp16 rounding of the softmax weights and of o.
"""
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


def _inputs(H, Hkv, T, t_stride, seed, q_scale=1.0, poison=True):
    rng = np.random.default_rng(seed)
    q = (rng.standard_normal((H, 128)) * q_scale).astype(np.float16)
    k = rng.standard_normal((Hkv, t_stride, 128)).astype(np.float16)
    v = rng.standard_normal((Hkv, t_stride, 128)).astype(np.float16)
    if poison and t_stride > T:  # rows past T must never be read
        k[:, T:] = np.nan
        v[:, T:] = np.nan
    return q, k, v


def _run(q, k, v, T):
    qd, kd, vd = (torch.from_numpy(a).to(DEV) for a in (q, k, v))
    o = w4.w4a16_attn_decode(qd, kd, vd, T)
    torch.cuda.synchronize()
    return o


def _check(q, k, v, T, o):
    H = q.shape[0]
    ref = oracle.attn_decode(q.view(np.uint16), k.view(np.uint16), v.view(np.uint16), T)
    rep = oracle.check_attn(o.double().cpu().numpy(), ref, v.view(np.uint16), H, T)
    assert rep["ok"], {k_: rep[k_] for k_ in ("finite",)} | {"worst": max(
        e / b for e, b in zip(rep["max_err"], rep["bound"]))}
    return rep


# The key ranges per KV head are min(tiles of 64 keys, SMs / n_kv_heads):
# 1 (T <= 64) up to 38 for 4 KV heads; 76 for 2 KV heads (2 x 9000) and
# every SM for one KV head (16 x 1 x 16384: 152 ranges merged by one CTA).
@pytest.mark.parametrize("H,Hkv,T,t_stride", [
    (28, 4, 1, 1), (28, 4, 63, 64), (28, 4, 64, 64), (28, 4, 65, 100), (28, 4, 129, 129),
    (28, 4, 1000, 1024), (8, 8, 300, 300), (16, 1, 777, 800), (7, 1, 5000, 5000),
    (28, 4, 8192, 8192), (2, 2, 9000, 9000), (16, 1, 16384, 16384),
])
def test_attn_against_oracle(H, Hkv, T, t_stride):
    q, k, v = _inputs(H, Hkv, T, t_stride, seed=H * 100003 + T)
    o = _run(q, k, v, T)
    assert torch.isfinite(o).all()
    _check(q, k, v, T, o)


@pytest.mark.parametrize("T", [17, 2048])
def test_attn_sharp_softmax(T):
    """q scaled by 4: scores of spread ~4, weights concentrated on few keys."""
    q, k, v = _inputs(28, 4, T, T, seed=T, q_scale=4.0)
    _check(q, k, v, T, _run(q, k, v, T))


def test_attn_single_key_is_value_row():
    """T = 1: every weight is 1, so o is the KV head's value row (rounded to
    fp16 it is the value itself, bit for bit)."""
    q, k, v = _inputs(28, 4, 1, 8, seed=5)
    o = _run(q, k, v, 1).cpu().numpy()
    for h in range(28):
        assert np.array_equal(o[h].view(np.uint16), v[h // 7, 0].view(np.uint16)), h


def test_attn_deterministic_and_prefix():
    """Two calls give the same bits; T keys of a longer cache give the same o
    as a cache holding just those T keys (the tail is never read)."""
    q, k, v = _inputs(28, 4, 3000, 4096, seed=11, poison=False)
    a = _run(q, k, v, 3000)
    b = _run(q, k, v, 3000)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = _run(q, k[:, :3000].copy(), v[:, :3000].copy(), 3000)
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_attn_rejects_bad_workspace_and_alias():
    q, k, v = _inputs(28, 4, 500, 500, seed=3)
    qd, kd, vd = (torch.from_numpy(a).to(DEV) for a in (q, k, v))
    need = w4.attn_decode_workspace(28, 4, 500)
    assert need > 0
    o = torch.empty((28, 128), dtype=torch.float16, device=DEV)
    ws = w4.attn_decode_new_workspace(28, 4, 500, DEV)
    rc = w4.w4a16_attn_decode_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), 28, 4, 128, 500,
                                  500, ws.data_ptr(), need - 16)
    assert rc == 2  # workspace too small
    rc = w4.w4a16_attn_decode_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), qd.data_ptr(), 28, 4, 128,
                                  500, 500, ws.data_ptr(), need)
    assert rc == 6  # o overlaps q
    rc = w4.w4a16_attn_decode_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), 28, 4, 128, 500,
                                  500, ws.data_ptr(), need)
    assert rc == 0
    torch.cuda.synchronize()
    _check(q, k, v, 500, o)


def test_attn_workspace_reused_and_left_zero():
    """The workspace's range counters are zero after every call: one zeroed
    workspace serves calls of different shapes in turn, each matching the
    oracle and a fresh workspace bit for bit."""
    big = w4.attn_decode_new_workspace(28, 4, 8192, DEV)
    ws_u32 = big.view(torch.int32)
    for H, Hkv, T in ((28, 4, 8192), (8, 8, 300), (16, 1, 777), (28, 4, 65), (28, 4, 8192)):
        assert w4.attn_decode_workspace(H, Hkv, T) <= big.numel() * 4
        q, k, v = _inputs(H, Hkv, T, T, seed=7 * T + H, poison=False)
        qd, kd, vd = (torch.from_numpy(a).to(DEV) for a in (q, k, v))
        a = w4.w4a16_attn_decode(qd, kd, vd, T, workspace=big)
        b = w4.w4a16_attn_decode(qd, kd, vd, T)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert int(ws_u32[:256].abs().sum()) == 0  # the whole counter block
        _check(q, k, v, T, a)


def test_attn_graph_of_calls_sharing_a_workspace():
    """28 calls captured in one CUDA graph over distinct caches with one
    workspace (the bench's layout), replayed twice: every output equals its
    call made alone."""
    H, Hkv, T = 28, 4, 1000
    ins = [_inputs(H, Hkv, T, T, seed=1000 + i, poison=False) for i in range(28)]
    dev_ins = [tuple(torch.from_numpy(a).to(DEV) for a in t) for t in ins]
    ws = w4.attn_decode_new_workspace(H, Hkv, T, DEV)
    outs = [torch.empty((H, 128), dtype=torch.float16, device=DEV) for _ in ins]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for (q, k, v), o in zip(dev_ins, outs):
            w4.w4a16_attn_decode(q, k, v, T, o=o, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for (q, k, v), o in zip(dev_ins, outs):
            w4.w4a16_attn_decode(q, k, v, T, o=o, workspace=ws)
    for _ in range(2):
        for o in outs:
            o.zero_()
        g.replay()
        torch.cuda.synchronize()
        for (q, k, v), o in zip(dev_ins, outs):
            alone = w4.w4a16_attn_decode(q, k, v, T)
            torch.cuda.synchronize()
            assert torch.equal(o.view(torch.int16), alone.view(torch.int16))
    _check(*ins[5], T, outs[5])
