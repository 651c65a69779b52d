"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each pin takes an oracle library handle (so the same pins can be run against
deliberately broken builds of the oracle, see test_oracle_mutants.py) and
raises AssertionError when the oracle disagrees with:
  - the IEEE 754 binary16 definition (exhaustive over all 65,536 patterns,
    every midpoint between neighbours, and numpy's float16 conversion);
  - the hand-decoded words and hand-computed GEMVs under tests/golden/;
  - the quantiser's closed-form properties (scale = fp16_RN(max|w| / 7),
    q in [-8, 7], |w - q s| <= s / 2, exact recovery of w = q s);
  - numpy's float64 matmul on a dense matrix built directly from chosen (q, s).
"""
from __future__ import annotations

import os

import math

import numpy as np

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------- fp16

def pin_half_to_double_exhaustive(L):
    """All 65,536 binary16 patterns decode to numpy's float16 value."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_to_double(h, L)
    want = h.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # the sign of zero is kept
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def pin_half_roundtrip(L):
    """double(h) -> half gives back h for every non-NaN pattern."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = h.view(np.float16).astype(np.float64)
    keep = ~np.isnan(v)
    back = oracle.double_to_half(v[keep], L)
    assert np.array_equal(back, h[keep])


def pin_half_midpoints_ties_to_even(L):
    """The exact midpoint between two neighbouring finite halves rounds to the
    one with the even fraction (IEEE 754 ties-to-even); a hair above/below
    rounds up/down."""
    h = np.arange(0, 0x7bff, dtype=np.uint32).astype(np.uint16)  # 0 .. 65504's predecessor
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2.0  # exact in double
    got = oracle.double_to_half(mid, L)
    even = np.where(h % 2 == 0, h, h + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    up = oracle.double_to_half(np.nextafter(mid, np.inf), L)
    down = oracle.double_to_half(np.nextafter(mid, -np.inf), L)
    assert np.array_equal(up, (h + 1).astype(np.uint16))
    assert np.array_equal(down, h)
    # negative side mirrors
    gotn = oracle.double_to_half(-mid, L)
    assert np.array_equal(gotn, (even | 0x8000).astype(np.uint16))


def pin_half_overflow_and_specials(L):
    cases = [
        (65504.0, 0x7BFF), (65519.99, 0x7BFF), (65520.0, 0x7C00), (1e9, 0x7C00),
        (-65520.0, 0xFC00), (2.0 ** -24, 0x0001), (2.0 ** -25, 0x0000),
        (1.5 * 2.0 ** -24, 0x0002), (2.0 ** -14, 0x0400), (1.0, 0x3C00), (-2.0, 0xC000),
        (0.0, 0x0000), (-0.0, 0x8000), (float("inf"), 0x7C00), (float("-inf"), 0xFC00),
        (1.0 + 2.0 ** -11, 0x3C00), (1.0 + 3 * 2.0 ** -11, 0x3C02),
    ]
    v = np.array([c[0] for c in cases], np.float64)
    got = oracle.double_to_half(v, L)
    want = [c[1] for c in cases]
    assert [int(g) for g in got] == want, (got, want)
    nan = oracle.double_to_half(np.array([np.nan]), L)
    assert (int(nan[0]) & 0x7C00) == 0x7C00 and (int(nan[0]) & 0x3FF) != 0


def pin_half_vs_numpy_random(L):
    """Random doubles and floats over the whole binary16 range agree with numpy."""
    rng = np.random.default_rng(12345)
    mag = np.exp2(rng.uniform(-30, 17, 200000))
    v = mag * rng.choice([-1.0, 1.0], mag.size)
    got = oracle.double_to_half(v, L)
    with np.errstate(over="ignore"):  # values past 65520 become inf, as they should
        want = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)
    f = v.astype(np.float32)
    got32 = np.array([L.orc_float_to_half(float(t)) for t in f[:5000]], np.uint16)
    with np.errstate(over="ignore"):
        want32 = f[:5000].astype(np.float16).view(np.uint16)
    assert np.array_equal(got32, want32)


# --------------------------------------------------------------------------- format

def read_hand_words():
    rows = []
    with open(os.path.join(GOLDEN, "hand_words.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            rows.append((int(parts[0], 16), [int(t) for t in parts[1:]]))
    return rows


def pin_hand_words(L):
    for word, q in read_hand_words():
        got = oracle.unpack(np.array([[word]], np.uint32), L)
        assert got.tolist() == [q], (hex(word), got.tolist(), q)


def pin_dequant_half_scale(L):
    """s = 0.5: w_hat = q / 2, exact in fp16."""
    for word, q in read_hand_words():
        qw = np.full((1, 16), word, np.uint32)
        sc = np.array([[0x3800]], np.uint16)  # 0.5
        got = oracle.dequant(qw, sc, 128, L)
        want = np.tile(np.array(q, np.float64) * 0.5, 16).astype(np.float16).view(np.uint16)
        assert np.array_equal(got[0], want)


def _parse_scale(tok: str, n: int) -> float:
    if tok == "2^-n":
        return 2.0 ** -n
    if tok.startswith("2^"):
        return 2.0 ** float(tok[2:])
    return float(tok)


def read_hand_gemvs():
    cases = []
    with open(os.path.join(GOLDEN, "hand_gemv_1x8x128.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            p = line.split()
            name, K = p[0], int(p[1])
            words = [int(t, 16) for t in p[2:4] if t != "-"]
            scale_tok, x_tok = p[4], p[5]
            expected = [float(t) for t in p[6:]]
            cases.append((name, K, words, scale_tok, x_tok, expected))
    return cases


def build_hand_case(K, words, scale_tok, x_tok):
    N, G = 8, 128
    qw = np.zeros((N, K // 8), np.uint32)
    for g, w in enumerate(words):
        qw[:, g * 16:(g + 1) * 16] = w
    sc = np.zeros((N, K // G), np.uint16)
    for n in range(N):
        toks = scale_tok.split(",")
        for g in range(K // G):
            sc[n, g] = np.float16(_parse_scale(toks[g], n)).view(np.uint16)
    if x_tok == "ones":
        x = np.full((1, K), 0x3C00, np.uint16)
    else:
        k = int(x_tok.split("_")[1])
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3C00
    return qw, sc, x


def pin_hand_gemvs(L):
    for name, K, words, scale_tok, x_tok, expected in read_hand_gemvs():
        qw, sc, x = build_hand_case(K, words, scale_tok, x_tok)
        y = oracle.gemv(qw, sc, x, 128, L)
        assert y[0].tolist() == expected, (name, x_tok, y[0].tolist(), expected)
        # the row-sampled entry point gives the same numbers
        yr = oracle.gemv_rows(qw, sc, x, np.array([7, 0, 3]), 128, L)
        assert yr[0].tolist() == [expected[7], expected[0], expected[3]]


# --------------------------------------------------------------------------- quantiser

def pin_quantizer_properties(L, N=64, K=1024, seed=0):
    """On Normal(0, 0.02) weights: s = fp16_RN(fp32(max|w| / 7)) (checked with
    numpy's fp32 division and float16 rounding), q in [-8, 7], every group has
    a |q| = 7, and |w - q s| <= s / 2 for every element."""
    w = synth.weights(N, K, seed).numpy()
    qw, sc = oracle.quantize(w, 128, L)
    G = 128
    wg = w.reshape(N, K // G, G)
    amax = np.abs(wg).max(axis=2).astype(np.float32)
    s_want = (amax / np.float32(7.0)).astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(sc, s_want)
    q = oracle.unpack(qw, L).astype(np.int64).reshape(N, K // G, G)
    assert q.min() >= -8 and q.max() <= 7
    assert np.all(np.abs(q).max(axis=2) == 7)
    s = sc.view(np.float16).astype(np.float64)[:, :, None]
    err = np.abs(wg.astype(np.float64) - q * s)
    assert np.all(err <= s / 2.0)


def pin_quantizer_exact_recovery(L, seed=3):
    """W built as q * s (each group holding a +-7) quantises back to exactly
    (q, s): pins the scale formula, the rounding and the packing round trip."""
    rng = np.random.default_rng(seed)
    N, K, G = 16, 512, 128
    q = rng.integers(-7, 8, (N, K))
    q = q.reshape(N, K // G, G)
    q[:, :, 5] = np.where(rng.random((N, K // G)) < 0.5, 7, -7)
    q = q.reshape(N, K)
    s = np.exp2(rng.integers(-12, 0, (N, K // G))) * rng.integers(1024, 2048, (N, K // G)) / 1024.0
    s = s.astype(np.float16).astype(np.float64)
    w = (q * np.repeat(s, G, axis=1)).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), q * np.repeat(s, G, axis=1))  # exact in fp32
    qw, sc = oracle.quantize(w, G, L)
    assert np.array_equal(sc.view(np.float16).astype(np.float64), s)
    assert np.array_equal(oracle.unpack(qw, L).astype(np.int64), q)


def pin_quantizer_rounding_ties(L):
    """w / s exactly at a half-integer rounds away from zero."""
    G = 128
    w = np.zeros((1, G), np.float32)
    w[0, 0] = 7.0            # max -> s = 1
    w[0, 1] = 2.5            # -> 3
    w[0, 2] = -2.5           # -> -3
    w[0, 3] = 0.5            # -> 1
    w[0, 4] = -0.5           # -> -1
    w[0, 5] = 2.4999998      # -> 2
    w[0, 6] = -6.5           # -> -7
    qw, sc = oracle.quantize(w, G, L)
    assert int(sc[0, 0]) == 0x3C00
    q = oracle.unpack(qw, L)[0, :7].tolist()
    assert q == [7, 3, -3, 1, -1, 2, -7], q


def pin_quantizer_zero_group(L):
    w = np.zeros((2, 256), np.float32)
    w[1, 200] = -0.25
    qw, sc = oracle.quantize(w, 128, L)
    assert sc.tolist() == [[0, 0], [0, int(np.float16(0.25 / 7).view(np.uint16))]]
    q = oracle.unpack(qw, L)
    assert np.count_nonzero(q) == 1 and q[1, 200] == -7


def pin_quantizer_errors(L):
    w = np.zeros((1, 128), np.float32)
    w[0, 3] = np.inf
    try:
        oracle.quantize(w, 128, L)
        raise AssertionError("non-finite input accepted")
    except oracle.OracleError as e:
        assert "status 2" in str(e)
    w[0, 3] = 7.0 * 65520.0
    try:
        oracle.quantize(w, 128, L)
        raise AssertionError("scale overflow accepted")
    except oracle.OracleError as e:
        assert "status 3" in str(e)
    w[0, 3] = 7.0 * 65504.0  # largest finite scale
    qw, sc = oracle.quantize(w, 128, L)
    assert int(sc[0, 0]) == 0x7BFF


# --------------------------------------------------------------------------- GEMV

def pin_gemv_vs_numpy_matmul(L):
    """Brute force on small shapes: the oracle GEMV equals numpy's float64
    matmul of x and the dense w_hat built from (q, s), to double rounding."""
    for seed, (M, N, K) in enumerate([(1, 1, 128), (3, 3, 256), (16, 8, 128), (5, 13, 384),
                                      (16, 17, 1024)]):
        rng = np.random.default_rng(100 + seed)
        G = 128
        q = np.clip(rng.integers(-8, 8, (N, K)), -7, 7)
        q.reshape(N, K // G, G)[:, :, 7] = 7
        s = (rng.integers(1024, 2048, (N, K // G)) / 1024.0) * np.exp2(rng.integers(-10, -3, (N, K // G)))
        s = s.astype(np.float16).astype(np.float64)
        w_hat = q * np.repeat(s, G, axis=1)
        qw, sc = oracle.quantize(w_hat.astype(np.float32), G, L)
        x = rng.standard_normal((M, K)).astype(np.float16)
        y = oracle.gemv(qw, sc, x.view(np.uint16), G, L)
        y_np = x.astype(np.float64) @ w_hat.T
        scale = np.abs(x.astype(np.float64)) @ np.abs(w_hat).T
        assert np.all(np.abs(y - y_np) <= 4 * K * 2.0 ** -53 * scale + 1e-300), (M, N, K)
        # dequant agrees with the dense matrix, rounded to fp16
        dq = oracle.dequant(qw, sc, G, L)
        assert np.array_equal(dq, w_hat.astype(np.float16).view(np.uint16))


def pin_gemv_m_consistency(L):
    """A GEMV over M activation rows is M GEMVs over one row each (bitwise)."""
    w = synth.weights(24, 256, 7).numpy()
    qw, sc = oracle.quantize(w, 128, L)
    x = synth.activations(6, 256, 7).numpy().view(np.uint16)
    y = oracle.gemv(qw, sc, x, 128, L)
    for m in range(6):
        assert np.array_equal(y[m], oracle.gemv(qw, sc, x[m], 128, L)[0])


def pin_gemv_fused_equals_separate(L):
    """[gate; up] stacked along N gives [y_gate, y_up] (the fused gate+up GEMV)."""
    wg = synth.weights(16, 256, 11).numpy()
    wu = synth.weights(16, 256, 12).numpy()
    qg, sg = oracle.quantize(wg, 128, L)
    qu, su = oracle.quantize(wu, 128, L)
    x = synth.activations(2, 256, 11).numpy().view(np.uint16)
    y = oracle.gemv(np.vstack([qg, qu]), np.vstack([sg, su]), x, 128, L)
    assert np.array_equal(y, np.hstack([oracle.gemv(qg, sg, x, 128, L), oracle.gemv(qu, su, x, 128, L)]))


def pin_silu_closed_forms(L):
    """silu(v) = v sigmoid(v): silu(0) = 0; silu(v) - silu(-v) = v (because
    sigmoid(v) + sigmoid(-v) = 1); silu tends to v for large positive v and to
    0 for large negative v; it is positive for v > 0 and negative for v < 0;
    its minimum lies at v = -1.27846... where the derivative
    sigmoid(v) (1 + v (1 - sigmoid(v))) vanishes, so silu there is below both
    neighbours."""
    assert oracle.silu(0.0, L) == 0.0
    for v in (1e-3, 0.5, 1.0, 2.75, 7.0, 13.5):
        assert abs((oracle.silu(v, L) - oracle.silu(-v, L)) - v) <= 1e-15 * max(1.0, v)
        assert oracle.silu(v, L) > 0.0 > oracle.silu(-v, L)
    assert abs(oracle.silu(40.0, L) - 40.0) < 1e-12
    assert abs(oracle.silu(-40.0, L)) < 1e-12
    vmin = -1.2784645427610738  # the minimum: sigmoid(v)(1 + v(1 - sigmoid(v))) = 0
    assert oracle.silu(vmin, L) < oracle.silu(vmin - 0.01, L)
    assert oracle.silu(vmin, L) < oracle.silu(vmin + 0.01, L)


def pin_swiglu_vs_numpy(L):
    """h = fp16_RN(silu(g) u) against numpy float64 arithmetic rounded by
    numpy's float16 conversion, on random and special fp16 inputs; u = 1 and
    a large g give h = g exactly, g = 0 gives 0."""
    rng = np.random.default_rng(7)
    g = rng.standard_normal(20000).astype(np.float16)
    u = (rng.standard_normal(20000) * 2).astype(np.float16)
    g[:6] = np.array([0.0, -0.0, 30.0, -30.0, 1e-4, 65504.0], dtype=np.float16)
    u[:6] = np.array([1.0, 1.0, 1.0, 1.0, 3.0, 1.0], dtype=np.float16)
    h = oracle.swiglu(g.view(np.uint16), u.view(np.uint16), L).view(np.float16)
    gd, ud = g.astype(np.float64), u.astype(np.float64)
    with np.errstate(over="ignore"):
        want = (gd / (1.0 + np.exp(-gd)) * ud).astype(np.float16)
    assert np.array_equal(h.view(np.uint16), want.view(np.uint16))
    assert h[2] == np.float16(30.0) and h[0] == 0.0


def _attn_inputs(seed, H, Hkv, T, D=128, t_stride=None):
    rng = np.random.default_rng(seed)
    t_stride = T if t_stride is None else t_stride
    q = rng.standard_normal((H, D)).astype(np.float16).view(np.uint16)
    k = rng.standard_normal((Hkv, t_stride, D)).astype(np.float16).view(np.uint16)
    v = rng.standard_normal((Hkv, t_stride, D)).astype(np.float16).view(np.uint16)
    return q, k, v


def pin_attn_single_key(L):
    """T = 1: every softmax weight is 1, so o_h is exactly the value row of
    the KV head its group reads (h / 7 for 28 query heads over 4 KV heads)."""
    q, k, v = _attn_inputs(1, 28, 4, 1)
    o = oracle.attn_decode(q, k, v, L=L)
    vd = v.view(np.float16).astype(np.float64)
    for h in range(28):
        assert np.array_equal(o[h], vd[h // 7, 0]), h


def pin_attn_two_keys_scale(L):
    """T = 2 with q = e0, k0 = 8 e0, k1 = 0 (D = 128): the scores are
    8 / sqrt(128) = 1/sqrt(2) and 0, so p0 is the logistic function of
    1/sqrt(2) and o = p0 v0 + (1 - p0) v1."""
    D = 128
    q = np.zeros((1, D), np.float16)
    q[0, 0] = 1.0
    k = np.zeros((1, 2, D), np.float16)
    k[0, 0, 0] = 8.0
    v = np.random.default_rng(2).standard_normal((1, 2, D)).astype(np.float16)
    o = oracle.attn_decode(q.view(np.uint16), k.view(np.uint16), v.view(np.uint16), L=L)
    p0 = 1.0 / (1.0 + math.exp(-1.0 / math.sqrt(2.0)))
    vd = v.astype(np.float64)
    assert np.allclose(o[0], p0 * vd[0, 0] + (1.0 - p0) * vd[0, 1], rtol=0, atol=1e-13)


def pin_attn_uniform_and_constant(L):
    """Identical keys give uniform weights, so o is the mean of the value
    rows; identical value rows give o equal to that row whatever q is."""
    q, k, v = _attn_inputs(3, 4, 2, 9)
    k[:, :, :] = k[:, :1, :]
    o = oracle.attn_decode(q, k, v, L=L)
    vd = v.view(np.float16).astype(np.float64)
    for h in range(4):
        assert np.allclose(o[h], vd[h // 2].mean(axis=0), rtol=0, atol=1e-13)
    q, k, v = _attn_inputs(4, 4, 2, 9)
    v[:, :, :] = v[:, :1, :]
    o = oracle.attn_decode(q, k, v, L=L)
    vd = v.view(np.float16).astype(np.float64)
    for h in range(4):
        assert np.allclose(o[h], vd[h // 2, 0], rtol=0, atol=1e-13)


def pin_attn_permutation_and_dominance(L):
    """Permuting the (key, value) pairs together leaves o unchanged; a key
    with a score far above the others takes all the weight."""
    q, k, v = _attn_inputs(5, 7, 1, 33)
    o = oracle.attn_decode(q, k, v, L=L)
    perm = np.random.default_rng(5).permutation(33)
    o2 = oracle.attn_decode(q, k[:, perm].copy(), v[:, perm].copy(), L=L)
    assert np.allclose(o, o2, rtol=0, atol=1e-12)
    qd = q.view(np.float16)
    k2 = k.view(np.float16).copy()
    k2[0, 17] = (qd[0] * 8).astype(np.float16)  # score of key 17 for head 0: ~ 8 |q|^2 / sqrt(D)
    o3 = oracle.attn_decode(q, k2.view(np.uint16), v, L=L)
    assert np.allclose(o3[0], v.view(np.float16)[0, 17].astype(np.float64), rtol=0, atol=1e-9)


def pin_attn_stride_and_prefix(L):
    """Keys at t >= T are never read (poisoned with NaN there), and a cache
    of T keys inside a larger stride gives the same o as the compact one."""
    q, k, v = _attn_inputs(6, 8, 2, 24, t_stride=40)
    k[:, 24:] = np.float16(np.nan).view(np.uint16)
    v[:, 24:] = np.float16(np.nan).view(np.uint16)
    o = oracle.attn_decode(q, k, v, T=24, L=L)
    o2 = oracle.attn_decode(q, k[:, :24].copy(), v[:, :24].copy(), L=L)
    assert np.isfinite(o).all() and np.array_equal(o, o2)


def _a8_reference(x_u16: np.ndarray):
    """Block-64 int8 quantisation of one fp16 row with numpy: FP32 division
    and product (IEEE single, as the definition states), rounding to nearest
    with ties to even (numpy's rint)."""
    x = x_u16.view(np.float16).astype(np.float32).reshape(-1, 64)
    amax = np.abs(x).max(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = np.where(amax > 0, amax / np.float32(127.0), np.float32(0.0)).astype(np.float32)
        inv = np.where(amax > 0, np.float32(127.0) / amax, np.float32(0.0)).astype(np.float32)
    p = (x * inv[:, None]).astype(np.float32)
    q = np.rint(p).astype(np.int8)
    return q.reshape(-1), s


def pin_a8_quantize_vs_numpy(L):
    """Codes and scales equal a numpy restatement bit for bit; every code of a
    nonzero block is within half a step of x / s, and the block maximum maps
    to +-127."""
    rng = np.random.default_rng(21)
    x = (rng.standard_normal(64 * 40) * np.repeat(rng.uniform(0.01, 30, 40), 64)).astype(np.float16)
    xq, s = oracle.quantize_act_a8(x.view(np.uint16), L)
    rq, rs = _a8_reference(x.view(np.uint16))
    assert np.array_equal(xq, rq) and np.array_equal(s.view(np.uint32), rs.view(np.uint32))
    xb = x.astype(np.float64).reshape(-1, 64)
    err = np.abs(xb - xq.reshape(-1, 64) * s[:, None].astype(np.float64))
    assert (err <= s[:, None] * (0.5 + 1e-6)).all()
    assert (np.abs(xq.reshape(-1, 64)).max(axis=1) == 127).all()


def pin_a8_ties_and_zero_block(L):
    """With block maximum 127 the scale is 1: ties go to even (2.5 -> 2,
    -2.5 -> -2, 3.5 -> 4, -0.5 -> 0), integers map to themselves; an all-zero
    block has scale 0 and codes 0."""
    x = np.zeros(128, np.float16)
    x[0], x[1], x[2], x[3], x[4], x[5] = 127.0, 2.5, -2.5, 7.0, -0.5, 3.5
    xq, s = oracle.quantize_act_a8(x.view(np.uint16), L)
    assert s[0] == 1.0 and list(xq[:6]) == [127, 2, -2, 7, 0, 4]
    assert s[1] == 0.0 and not xq[64:].any()


def pin_a8_gemv_vs_numpy_and_exact_case(L):
    """The W4A8 GEMV equals sum_b s_w s_b (q . xq) from numpy integer matmuls
    per block; with activations that quantise exactly (integers, block
    maximum 127) it equals the W4A16 GEMV."""
    w = synth.weights(12, 384, 23).numpy()
    qw, sc = oracle.quantize(w, 128, L)
    x = synth.activations(3, 384, 23).numpy().view(np.uint16)
    y = oracle.gemv_w4a8(qw, sc, x, 128, L)
    q = oracle.unpack(qw, L).astype(np.int64)
    sw = sc.view(np.float16).astype(np.float64)
    for m in range(3):
        xq, sx = _a8_reference(x[m])
        ref = np.zeros(12)
        for b in range(6):
            isum = q[:, 64 * b:64 * b + 64] @ xq[64 * b:64 * b + 64].astype(np.int64)
            ref += isum * sw[:, b // 2] * np.float64(sx[b])
        assert np.allclose(y[m], ref, rtol=1e-13, atol=1e-13)
    xi = np.random.default_rng(24).integers(-126, 127, (2, 384)).astype(np.float16)
    xi[:, ::64] = 127.0
    y8 = oracle.gemv_w4a8(qw, sc, xi.view(np.uint16), 128, L)
    assert np.array_equal(y8, oracle.gemv(qw, sc, xi.view(np.uint16), 128, L))


def _q4k_block(d, dmin, sc, mn, qs=None):
    """One 144-byte Q4_K block from its parts: d, dmin (float, stored fp16),
    eight 6-bit scales and minima (packed here into the 12 bytes the
    decoding reads back: j < 4 in the low 6 bits of bytes j and j + 4, j >= 4
    split into bytes j + 4 (low nibble: scale, high: minimum) and the top two
    bits of bytes j - 4 (scale) and j (minimum)), 128 code bytes."""
    b = np.zeros(144, np.uint8)
    b[0:2] = np.frombuffer(np.array([d], np.float16).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.array([dmin], np.float16).tobytes(), np.uint8)
    p = np.zeros(12, np.int64)
    for j in range(4):
        p[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        p[j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)
        p[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    b[4:16] = p.astype(np.uint8)
    if qs is not None:
        b[16:] = qs
    return b


def pin_q4k_scales_and_minima(L):
    """With d = dmin = 1: all-zero codes give w = -m_j on sub-block j, codes
    of 1 give sc_j - m_j, for random 6-bit scales and minima (every bit of
    the packing exercised)."""
    rng = np.random.default_rng(31)
    for _ in range(4):
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        w0 = oracle.q4k_dequant(_q4k_block(1.0, 1.0, sc, mn), 1, 256, L)[0]
        w1 = oracle.q4k_dequant(_q4k_block(1.0, 1.0, sc, mn, np.full(128, 0x11, np.uint8)), 1, 256, L)[0]
        for j in range(8):
            assert (w0[32 * j:32 * j + 32] == -mn[j]).all(), j
            assert (w1[32 * j:32 * j + 32] == sc[j] - mn[j]).all(), j


def pin_q4k_element_order(L):
    """Single nibbles land at the documented weights: low nibble of code byte
    5 -> weight 5, its high nibble -> weight 37, high nibble of byte 64 + 9
    (chunk 2) -> weight 128 + 32 + 9; scales 1..8 tell the sub-blocks apart."""
    qs = np.zeros(128, np.uint8)
    qs[5] = 0x73
    qs[64 + 9] = 0x20
    sc = np.arange(1, 9)
    w = oracle.q4k_dequant(_q4k_block(1.0, 0.0, sc, np.zeros(8, np.int64), qs), 1, 256, L)[0]
    want = np.zeros(256, np.float32)
    want[5] = 3 * 1
    want[37] = 7 * 2
    want[169] = 2 * 6
    assert np.array_equal(w, want)


def pin_q4k_fp32_and_gemv(L):
    """On random blocks the FP32 dequantisation is within three roundings of
    the exact weights (read back as GEMV columns through one-hot
    activations), and the GEMV equals x . w within the FP32 rounding of w."""
    rng = np.random.default_rng(33)
    N, K = 4, 512
    b = rng.integers(0, 256, (N * 2, 144)).astype(np.uint8)
    for i in range(N * 2):
        b[i, 0:2] = np.frombuffer(np.array([rng.uniform(1e-3, 0.05)], np.float16).tobytes(), np.uint8)
        b[i, 2:4] = np.frombuffer(np.array([rng.uniform(1e-3, 0.05)], np.float16).tobytes(), np.uint8)
    w32 = oracle.q4k_dequant(b.reshape(-1), N, K, L).astype(np.float64)
    eye = np.eye(K, dtype=np.float16)[::37]
    cols = oracle.q4k_gemv(b.reshape(-1), eye.view(np.uint16), N, K, L)  # rows = exact w[:, k]
    exact = cols.T
    assert (np.abs(w32[:, ::37] - exact) <= 4 * np.spacing(np.abs(exact).astype(np.float32)) + 1e-12).all()
    x = rng.standard_normal((2, K)).astype(np.float16)
    y = oracle.q4k_gemv(b.reshape(-1), x.view(np.uint16), N, K, L)
    ref = x.astype(np.float64) @ w32.T
    assert np.allclose(y, ref, rtol=0, atol=1e-5 * np.abs(x).sum())



# --------------------------------------------------------------------------- tolerance machinery
#
# Every GPU parity test is checked against the GEMV bound (per activation row m,
# max_n |y - y_ref| <= 2e-3 ||x_m||_2 max_n ||w_hat_n||_2 + 1e-3, and the
# relative L2 error over the whole output <= 1e-3) and by the attention bound
# (per query head, max_d |o - o_ref| <= 2e-3 max|v| + 1e-5 over the keys t < T
# of the KV head it reads).  These pins fix the functions that evaluate them
# (the exact weights behind the row norms, the norms, both checkers) to values
# worked out by hand, so that a mistake in any of them cannot loosen every
# parity test at once.  They take O, the module providing the Python-level
# functions, so that planted mistakes in those functions can be checked too.

def _hand_two_group_matrix():
    """N = 3, K = 256: group 0 of every row holds 16 words 0x76543210 (q = 0..7)
    at scale 2^-n, group 1 holds 16 words 0x89ABCDEF (q = -1..-8) at scale
    2^-(n+4).  Returns (qweight, scales, dense exact w_hat from the hand-decoded
    golden words)."""
    words = dict(read_hand_words())
    qa, qb = np.array(words[0x76543210], np.float64), np.array(words[0x89ABCDEF], np.float64)
    N, K = 3, 256
    qw = np.zeros((N, K // 8), np.uint32)
    qw[:, :16] = 0x76543210
    qw[:, 16:] = 0x89ABCDEF
    sc = np.zeros((N, 2), np.uint16)
    dense = np.zeros((N, K))
    for n in range(N):
        sc[n] = np.array([2.0 ** -n, 2.0 ** -(n + 4)], np.float16).view(np.uint16)
        dense[n, :128] = np.tile(qa, 16) * 2.0 ** -n
        dense[n, 128:] = np.tile(qb, 16) * 2.0 ** -(n + 4)
    return qw, sc, dense


def pin_dequant_f64_hand(L, O=oracle):
    """The exact weights behind the row norms: element by element equal to
    the hand-decoded words times their group scale, on a 3 x 256 matrix whose
    rows and groups all differ (a transposed index or a wrong group scale
    moves values)."""
    qw, sc, dense = _hand_two_group_matrix()
    got = O.dequant_f64(qw, sc, 128, L)
    assert got.shape == dense.shape and np.array_equal(got, dense)


def pin_row_norms_closed_form(L, O=oracle):
    """||w_hat_n||_2 in closed form.  16 words 0x76543210 at s = 1: q = 0..7
    sixteen times, sum q^2 = 16 * 140 = 2240.  The two-group matrix: row n
    has 16 * 140 * 4^-n from group 0 and 16 * 204 * 4^-(n+4) from group 1,
    so ||w_hat_n||^2 = 4^-n (2240 + 3264 / 256) = 2252.75 * 4^-n, and the norm
    is sqrt(2252.75) 2^-n (both sums are exact, and a power of 4 leaves the
    square root exact)."""
    one = O.row_norms(np.full((1, 16), 0x76543210, np.uint32), np.array([[0x3C00]], np.uint16), 128, L)
    assert one.shape == (1,) and one[0] == math.sqrt(2240.0)
    qw, sc, _ = _hand_two_group_matrix()
    got = O.row_norms(qw, sc, 128, L)
    want = np.array([math.sqrt(2252.75) * 2.0 ** -n for n in range(3)])
    assert got.shape == (3,) and np.array_equal(got, want)


def pin_check_gemv_abs_bound(L, O=oracle):
    """The per-row absolute bound, with slope 2^-9 and floor 2^-10 so that
    every bound is exact: x rows of norm 1, 2 and 5 ([1,0,0,0], [1,1,1,1],
    [0,0,3,4]) and max row norm 4 give bounds 2^-7 + 2^-10 = 0.0087890625,
    2^-6 + 2^-10 = 0.0166015625 and 20 2^-9 + 2^-10 = 0.0400390625.  An error
    exactly at a row's bound passes; one unit in the last place above it
    fails; a larger row's bound planted in a smaller row fails; a NaN
    fails."""
    x = np.array([[1, 0, 0, 0], [1, 1, 1, 1], [0, 0, 3, 4]], np.float64)
    bounds = [0.0087890625, 0.0166015625, 0.0400390625]
    y_ref = np.zeros((3, 5))

    def run(row, col, err):
        y = y_ref.copy()
        y[row, col] = err
        return O.check_gemv(y, y_ref, x, 4.0, rel_l2=np.inf, abs_slope=2.0 ** -9, abs_floor=2.0 ** -10)

    for m in range(3):
        assert run(m, 2, bounds[m])["ok"], m
        assert run(m, 2, -bounds[m])["ok"], m
        assert not run(m, 2, np.nextafter(bounds[m], np.inf))["ok"], m
    assert not run(0, 4, bounds[2])["ok"]
    assert not run(1, 0, bounds[2])["ok"]
    assert run(2, 0, bounds[0])["ok"]
    # every row at its own bound at once
    y = np.array([[bounds[0], 0, 0, 0, 0], [0, -bounds[1], 0, 0, 0], [0, 0, 0, 0, bounds[2]]])
    assert O.check_gemv(y, y_ref, x, 4.0, rel_l2=np.inf, abs_slope=2.0 ** -9, abs_floor=2.0 ** -10)["ok"]
    y[1, 3] = np.nan
    assert not O.check_gemv(y, y_ref, x, 4.0, rel_l2=np.inf, abs_slope=2.0 ** -9,
                            abs_floor=2.0 ** -10)["ok"]
    # the default constants: ||x|| = 3 ([1, 2, 2]), max row norm 5:
    # 2e-3 * 3 * 5 + 1e-3 = 0.031 (y_ref of norm 100 keeps the L2 test loose)
    x1 = np.array([[1.0, 2.0, 2.0]])
    y_ref1 = np.array([[100.0, 0.0]])
    assert O.check_gemv(np.array([[100.0, 0.0309]]), y_ref1, x1, 5.0)["ok"]
    assert not O.check_gemv(np.array([[100.0, 0.0311]]), y_ref1, x1, 5.0)["ok"]


def pin_check_gemv_rel_l2(L, O=oracle):
    """The relative L2 bound over the whole [M][N] output.  y_ref has norm
    1024 (one entry), the planted error norm 1, so the relative error is
    exactly 2^-10: it passes at rel_l2 = 2^-10 and fails one unit in the last
    place above; the error may sit in another activation row (the norm is over
    the whole output, not per row).  With the default 1e-3: 0.999 over a
    reference of norm 1000 passes, 1.001 fails."""
    x = np.array([[4096.0], [4096.0]])  # abs bound far away
    y_ref = np.array([[1024.0, 0.0], [0.0, 0.0]])
    for (r, c) in ((0, 1), (1, 0), (1, 1)):
        y = y_ref.copy()
        y[r, c] = 1.0
        assert O.check_gemv(y, y_ref, x, 1.0, rel_l2=2.0 ** -10)["ok"], (r, c)
        y[r, c] = np.nextafter(1.0, 2.0)
        assert not O.check_gemv(y, y_ref, x, 1.0, rel_l2=2.0 ** -10)["ok"], (r, c)
    # two errors of norm 2^-1/2 each combine in quadrature to 1 (not 2^1/2 or 2^-1/2)
    y = y_ref.copy()
    y[0, 1] = y[1, 1] = math.sqrt(0.5)
    rep = O.check_gemv(y, y_ref, x, 1.0, rel_l2=2.0 ** -10)
    assert abs(rep["rel_l2"] - 2.0 ** -10) <= 2.0 ** -60
    x1 = np.array([[1000.0]])
    y_ref1 = np.array([[1000.0, 0.0]])
    assert O.check_gemv(np.array([[1000.0, 0.999]]), y_ref1, x1, 1000.0)["ok"]
    assert not O.check_gemv(np.array([[1000.0, 1.001]]), y_ref1, x1, 1000.0)["ok"]


def pin_check_attn_bound(L, O=oracle):
    """The attention bound: 4 query heads over 2 KV heads (heads 0, 1 read
    KV head 0; heads 2, 3 read KV head 1), T = 3 keys of a stride of 5, whose
    rows past T hold 1000 (never part of the bound).  max|v| is 2 for KV head
    0 and 8 for KV head 1, so with slope 2^-8 and floor 2^-12 the bounds are
    2^-7 + 2^-12 and 2^-5 + 2^-12.  An error at a head's bound passes, one
    unit in the last place above fails, KV head 1's bound planted in head 1
    fails and KV head 0's in head 2 passes.  With the default constants and
    max|v| = 1 the bound is 2e-3 + 1e-5 = 0.00201."""
    D = 4
    v = np.zeros((2, 5, D), np.float16)
    v[0, 1, 2] = -2.0
    v[0, 0, 0] = 1.5
    v[1, 2, 3] = 8.0
    v[1, 0, 1] = -7.5
    v[:, 3:, :] = 1000.0
    v = v.view(np.uint16)
    o_ref = np.zeros((4, D))
    b0, b1 = 2.0 ** -7 + 2.0 ** -12, 2.0 ** -5 + 2.0 ** -12

    def run(h, d, err):
        o = o_ref.copy()
        o[h, d] = err
        return O.check_attn(o, o_ref, v, 4, 3, slope=2.0 ** -8, floor=2.0 ** -12)

    for h, b in ((0, b0), (1, b0), (2, b1), (3, b1)):
        assert run(h, 1, b)["ok"] and run(h, 3, -b)["ok"], h
        assert not run(h, 1, np.nextafter(b, np.inf))["ok"], h
    assert not run(1, 0, b1)["ok"]
    assert run(2, 0, b0)["ok"]
    o = o_ref.copy()
    o[3, 2] = np.nan
    assert not O.check_attn(o, o_ref, v, 4, 3, slope=2.0 ** -8, floor=2.0 ** -12)["ok"]
    v1 = np.ones((1, 2, D), np.float16).view(np.uint16)
    o_ref1 = np.zeros((2, D))
    assert O.check_attn(np.full((2, D), 0.002), o_ref1, v1, 2, 2)["ok"]
    assert not O.check_attn(np.full((2, D), 0.00202), o_ref1, v1, 2, 2)["ok"]


ALL_PINS = [
    pin_half_to_double_exhaustive, pin_half_roundtrip, pin_half_midpoints_ties_to_even,
    pin_half_overflow_and_specials, pin_half_vs_numpy_random, pin_hand_words,
    pin_dequant_half_scale, pin_hand_gemvs, pin_quantizer_properties,
    pin_quantizer_exact_recovery, pin_quantizer_rounding_ties, pin_quantizer_zero_group,
    pin_quantizer_errors, pin_gemv_vs_numpy_matmul, pin_gemv_m_consistency,
    pin_gemv_fused_equals_separate, pin_silu_closed_forms, pin_swiglu_vs_numpy,
    pin_attn_single_key, pin_attn_two_keys_scale, pin_attn_uniform_and_constant,
    pin_attn_permutation_and_dominance, pin_attn_stride_and_prefix,
    pin_a8_quantize_vs_numpy, pin_a8_ties_and_zero_block, pin_a8_gemv_vs_numpy_and_exact_case,
    pin_q4k_scales_and_minima, pin_q4k_element_order, pin_q4k_fp32_and_gemv,
]


# The pins of the tolerance machinery (they also take the Python-level module).
CHECK_PINS = [
    pin_dequant_f64_hand, pin_row_norms_closed_form, pin_check_gemv_abs_bound,
    pin_check_gemv_rel_l2, pin_check_attn_bound,
]


def failing_pins(L, O=oracle) -> list[str]:
    """Names of the pins that fail (or crash) against oracle library L, with
    the Python-level functions of module O."""
    bad = []
    for pin in ALL_PINS + CHECK_PINS:
        try:
            if pin in CHECK_PINS:
                pin(L, O)
            else:
                pin(L)
        except Exception as e:  # noqa: BLE001 -- a crash is a failure too
            bad.append(f"{pin.__name__}: {type(e).__name__}")
    return bad
