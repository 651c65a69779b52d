"""Shared helpers of the GPU parity tests.

Inputs come from synth (drawn on the CPU); the expected values come only from
the oracle.  The GPU side quantises with its own kernel; parity of the packed
weights is checked bit for bit before any GEMV is compared.
"""
from __future__ import annotations

import numpy as np
import torch

import int4_weight_only_gemv_gb300 as w4
import oracle
import synth


def to_np_u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def to_np_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_torch_i32(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int32)).to(dev)


def to_torch_f16(a_u16: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.float16).to(dev)


class Case:
    """One weight matrix + activations, quantised by the oracle (CPU) and by
    the GPU kernel, with the packed results checked identical."""

    def __init__(self, N, K, M, seed, dev="cuda", w_cpu=None, x_cpu=None):
        self.N, self.K, self.M = N, K, M
        w = synth.weights(N, K, seed) if w_cpu is None else w_cpu
        x = synth.activations(M, K, seed) if x_cpu is None else x_cpu
        self.w_np = w.numpy()
        self.x_u16 = x.view(torch.int16).numpy().view(np.uint16)
        self.x_f64 = x.to(torch.float64).numpy()
        self.qw_ref, self.sc_ref = oracle.quantize(self.w_np)
        self.w_dev = w.to(dev)
        self.x_dev = x.to(dev)
        self.qw, self.sc = w4.w4a16_quantize(self.w_dev)
        torch.cuda.synchronize()

    def packed_equal(self) -> bool:
        return (np.array_equal(to_np_u32(self.qw), self.qw_ref)
                and np.array_equal(to_np_u16(self.sc), self.sc_ref))

    def max_row_norm(self, rows=None) -> float:
        qw, sc = self.qw_ref, self.sc_ref
        if rows is not None:
            qw, sc = qw[rows], sc[rows]
        return float(oracle.row_norms(qw, sc).max())

    def gemv(self, x_dev=None, y=None):
        return w4.w4a16_gemv(self.qw, self.sc, self.x_dev if x_dev is None else x_dev, y)

    def check(self, y_dev, rows=None, x_u16=None, x_f64=None):
        """Oracle tolerance check of y (all rows, or the sampled `rows`)."""
        x_u16 = self.x_u16 if x_u16 is None else x_u16
        x_f64 = self.x_f64 if x_f64 is None else x_f64
        y = y_dev.detach().to(torch.float64).cpu().numpy()
        if rows is None:
            y_ref = oracle.gemv(self.qw_ref, self.sc_ref, x_u16)
        else:
            y_ref = oracle.gemv_rows(self.qw_ref, self.sc_ref, x_u16, rows)
            y = y[:, rows]
        rep = oracle.check_gemv(y, y_ref, x_f64, self.max_row_norm())
        return rep


def sample_rows(N: int, count: int, seed: int = 0) -> np.ndarray:
    """First, last, ragged-tail and random rows."""
    rng = np.random.default_rng(seed)
    fixed = {0, 1, N - 1, N - 2, N // 2, N - 17 if N > 17 else 0}
    rest = rng.choice(N, size=min(count, N), replace=False)
    return np.array(sorted(fixed | set(int(r) for r in rest)), np.int64)
