"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module draws random numbers and lays out routing structure only; it holds
none of the NVFP4 arithmetic (no quantisation, no scale layout, no GEMM).

Generator (counter-based, so any element can be drawn independently):
  * draw i of stream `seed` is SplitMix64's output for state
    seed * 2^32 + (i + 1) * 0x9E3779B97F4A7C15 (mod 2^64), i.e. SplitMix64's
    published finaliser applied to its Weyl sequence;
  * a uniform in (0, 1] is ((z >> 11) + 1) * 2^-53;
  * element e of a normal tensor uses draws 3e, 3e+1 (Box-Muller, cosine
    branch, in float64) and 3e+2 (the outlier coin: with probability p the
    value is multiplied by the outlier factor);
  * float64 -> float32 (round to nearest) -> bfloat16 (round to nearest even on
    the float32 bits).

Workloads (the shapes of the NVFP4 linear-layer and MoE decode workloads on the
reference pages): x ~ N(0,1) with 0.1% outliers x20, W ~ N(0, 0.02), and MoE
routing of each token to 8 distinct experts drawn uniformly (partial
Fisher-Yates), rows sorted by expert.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.c")
_LIB = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles the C form of the generator (same definition, OpenMP for speed)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-shared", "-fPIC", "-o",
            _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _c():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.syn_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_void_p]
            L.syn_uniform.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_void_p]
            _lib = L
    return _lib


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of stream `seed` as uint64."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        z = np.uint64((seed << 32) & 0xFFFFFFFFFFFFFFFF) + idx * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, start: int, count: int) -> np.ndarray:
    """Uniforms in (0, 1] as float64 (draws start .. start+count-1 of stream `seed`)."""
    out = np.empty(count, dtype=np.float64)
    _c().syn_uniform(seed, start, count, out.ctypes.data)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even. Finite inputs only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, std: float = 1.0, outlier_p: float = 0.0,
                outlier_mult: float = 20.0) -> np.ndarray:
    """Seeded N(0, std^2) tensor with optional outliers, as bf16 bit patterns (uint16)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    _c().syn_normal_bf16(seed, 0, n, std, outlier_p, outlier_mult, out.ctypes.data)
    return out.reshape(shape)


def route_topk(n_tokens: int, n_experts: int, topk: int, seed: int, zipf_s: float = 0.0):
    """Each token picks `topk` distinct experts.

    zipf_s == 0: uniformly (partial Fisher-Yates on the token's draws).
    zipf_s > 0: skewed; expert e has popularity (e + 1) ** -zipf_s and the token draws
    without replacement in proportion to the popularity of the experts it has not
    picked yet (one uniform draw per pick, inverse CDF over the remaining experts in
    index order).

    Returns (token_of_row, expert_of_row, expert_offsets): the routed rows sorted
    by expert (ties by token), and offsets[E+1] with rows offsets[e]..offsets[e+1]
    belonging to expert e.
    """
    u = uniform01(seed, 0, n_tokens * topk).reshape(n_tokens, topk)
    choice = np.empty((n_tokens, topk), dtype=np.int64)
    if zipf_s == 0.0:
        for t in range(n_tokens):
            perm = np.arange(n_experts)
            for j in range(topk):
                r = j + min(int(u[t, j] * (n_experts - j)), n_experts - j - 1)
                perm[j], perm[r] = perm[r], perm[j]
            choice[t] = perm[:topk]
    else:
        pop = (np.arange(n_experts, dtype=np.float64) + 1.0) ** (-zipf_s)
        for t in range(n_tokens):
            w = pop.copy()
            for j in range(topk):
                cdf = np.cumsum(w)
                e = int(np.searchsorted(cdf, u[t, j] * cdf[-1], side="right"))
                e = min(e, n_experts - 1)
                while w[e] == 0.0:  # a draw at a removed expert's edge: next remaining one
                    e -= 1
                choice[t, j] = e
                w[e] = 0.0
    tok = np.repeat(np.arange(n_tokens), topk)
    exp = choice.reshape(-1)
    order = np.lexsort((tok, exp))
    tok, exp = tok[order], exp[order]
    counts = np.bincount(exp, minlength=n_experts)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    return tok.astype(np.int64), exp.astype(np.int64), offsets


# Workload recipes (shapes from the NVFP4 linear-layer and MoE decode pages).
WORKLOADS = {
    "tiny": dict(M=128, N=128, K=256, x_std=1.0, x_outlier=0.0, w_std=1.0, seed=0),
    "square": dict(M=8192, N=8192, K=8192, x_std=1.0, x_outlier=1e-3, w_std=0.02, seed=1),
    "decode": dict(M=(1, 16, 32), N=8192, K=8192, x_std=1.0, x_outlier=1e-3, w_std=0.02, seed=2),
    "moe": dict(tokens=512, experts=256, topk=8, N=4096, K=6144, x_std=1.0, w_std=0.02, seed=3),
    "prefill": dict(M=4096, N=28672, K=8192, x_std=1.0, x_outlier=1e-3, w_std=0.02, seed=4),
}


def dense_inputs(M: int, N: int, K: int, seed: int, x_std=1.0, x_outlier=0.0, w_std=1.0):
    """bf16 bit patterns for x [M,K] (stream 2*seed) and W [N,K] (stream 2*seed+1)."""
    x = normal_bf16((M, K), 2 * seed, x_std, x_outlier)
    w = normal_bf16((N, K), 2 * seed + 1, w_std)
    return x, w


def moe_tokens(tokens: int, experts: int, topk: int, K: int, seed: int, x_std=1.0, zipf_s=0.0):
    """Routed token activations, gathered into expert-sorted rows.

    Returns (a_rows [tokens*topk, K] bf16 bits, offsets[E+1], token_of_row).
    """
    tok, _, offsets = route_topk(tokens, experts, topk, 1000 + seed, zipf_s)
    x = normal_bf16((tokens, K), 2 * seed, x_std)
    return x[tok], offsets, tok


def moe_expert_weight(e: int, N: int, K: int, seed: int, w_std=0.02) -> np.ndarray:
    """Expert e's weight [N, K] as bf16 bits (its own stream, so experts can be drawn one by one)."""
    return normal_bf16((N, K), 100000 + 1000 * seed + e, w_std)
