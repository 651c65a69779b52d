"""Run by tests/test_gpu_checked_build.py in a child process with
W4A16_LIBRARY=checked: the entry points on the index-checked build of the
library, each result against the oracle, then the device status word (no
index check may have failed).  Prints one JSON line."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import int4_weight_only_gemv_gb300 as w4  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_helpers import Case, to_np_u16  # noqa: E402

report = {"lib": w4.LIB_PATH, "fail": []}
dev = torch.device("cuda", 0)
w4.lib()
w4.w4a16_device_status(clear=True)


def note(name, ok):
    if not ok:
        report["fail"].append(name)


# GEMV kernels: M = 1 (warp-per-row kernel for a small 300 x 1024, task
# kernel, K split at 19456; CUDA-core rows kernel past K = 28672), M = 3, 5, 9, 16 (tensor cores: an odd group count at
# K = 640 takes the half-range box, K = 32768 a cluster of more than 8 CTAs),
# ragged N
for (M, N, K) in ((1, 300, 1024), (1, 1000, 3584), (1, 37, 19456), (1, 153, 18944), (1, 64, 32768), (3, 333, 1024),
                  (4, 50, 640), (9, 100, 3584), (16, 777, 2048), (5, 64, 32768)):
    c = Case(N, K, M, seed=300 + M + N)
    note(f"packed {M}x{N}x{K}", c.packed_equal())
    note(f"gemv {M}x{N}x{K}", c.check(c.gemv())["ok"])
# dequant
c = Case(64, 1024, 1, seed=7)
dq = to_np_u16(w4.w4a16_dequant(c.qw, c.sc))
note("dequant", np.array_equal(dq, oracle.dequant(c.qw_ref, c.sc_ref)))
# a two-layer sequence with and without SwiGLU, small shapes
h, kv, ffn, n = 256, 128, 512, 2
layers = []
for l in range(n):
    lw = {}
    for pj, name in enumerate(synth.PROJ_NAMES):
        NN, KK = {"q": (h, h), "k": (kv, h), "v": (kv, h), "o": (h, h), "gate": (ffn, h), "up": (ffn, h),
                  "down": (h, ffn)}[name]
        lw[name] = w4.w4a16_quantize(synth.weights(NN, KK, 91000 + 8 * l + pj).to(dev))
    layers.append(lw)
for swiglu in (False, True):
    io = {"x": synth.activations(n, h, 91999).view(n, 1, h).to(dev)}
    for name, width in (("y_q", h), ("y_k", kv), ("y_v", kv), ("y_o", h), ("y_gu", 2 * ffn), ("y_down", h)):
        io[name] = torch.full((n, 1, width), float("nan"), dtype=torch.float16, device=dev)
    seq = w4.LayerSeq(layers, io, 1, h, kv, ffn, swiglu=swiglu)
    seq.run()
    seq.sync()
    note(f"layer_seq swiglu={swiglu} written", not any(torch.isnan(io[k]).any().item() for k in io if k != "x"))
    y = w4.w4a16_gemv(*layers[1]["q"], io["x"][1])
    note(f"layer_seq swiglu={swiglu} q", torch.equal(y.view(torch.int16), io["y_q"][1].view(torch.int16)))
    seq.close()
# decode attention
g = torch.Generator().manual_seed(3)
q = torch.randn((28, 128), generator=g).half()
k = torch.randn((4, 300, 128), generator=g).half()
v = torch.randn((4, 300, 128), generator=g).half()
o = w4.w4a16_attn_decode(q.to(dev), k.to(dev), v.to(dev)).double().cpu().numpy()
u16 = [t.view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
note("attention", oracle.check_attn(o, oracle.attn_decode(*u16), u16[2], 28, 300)["ok"])
# W4A8
c = Case(500, 3584, 1, seed=17)
y = w4.w4a16_gemv_a8(c.qw, c.sc, c.x_dev).double().cpu().numpy()
y_ref = oracle.gemv_w4a8(c.qw_ref, c.sc_ref, c.x_u16)
note("w4a8", oracle.check_gemv(y, y_ref, c.x_f64, c.max_row_norm())["ok"])
torch.cuda.synchronize()
report["status"] = w4.w4a16_device_status(clear=True)
print(json.dumps(report))
