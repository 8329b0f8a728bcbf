"""Shared helpers for the GPU parity tests: move numpy arrays to the device,
quantise seeded inputs with the oracle, and run the tolerance check."""
import numpy as np
import torch

import oracle
import synth


def dev():
    return torch.device("cuda:0")


def to_dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(a).to(dev())


def scalar(v):
    return torch.tensor([float(v)], dtype=torch.float32, device=dev())


class Operand:
    """A quantised operand: host copies (for the oracle) and device copies."""

    def __init__(self, bf16_bits):
        self.q, self.sf, self.g = oracle.quantize(bf16_bits)
        self.rows, self.K = bf16_bits.shape
        self.dq, self.dsf, self.dg = to_dev(self.q), to_dev(self.sf), scalar(self.g)


def dense_case(M, N, K, seed, x_std=1.0, x_out=0.0, w_std=1.0):
    x, w = synth.dense_inputs(M, N, K, seed, x_std, x_out, w_std)
    return Operand(x), Operand(w)


def check_gemm(y_dev, A, B, rows=None, cols=None):
    """Compares y (device bf16 [M, N]) with the oracle on the chosen rows/cols."""
    M, N, K = A.rows, B.rows, A.K
    yr, ad = oracle.gemm(A.q, A.sf, A.g, B.q, B.sf, B.g, M, N, K, rows=rows, cols=cols)
    y = y_dev.float().cpu().numpy()
    if rows is not None:
        y = y[np.asarray(rows)]
    if cols is not None:
        y = y[:, np.asarray(cols)]
    ok, worst = oracle.within_tolerance(y, yr, ad)
    if not ok:
        err = np.abs(y - yr) > 4e-3 * np.abs(yr) + 1e-5 * ad
        bad_r, bad_c = np.nonzero(err)
        raise AssertionError(
            f"parity failed: worst ratio {worst:.3g}, {err.sum()} of {err.size} bad; "
            f"bad rows {np.unique(bad_r)[:12]} bad cols {np.unique(bad_c)[:12]}; "
            f"sample gpu {y[bad_r[0], bad_c[0]]} ref {yr[bad_r[0], bad_c[0]]}")
    return worst
