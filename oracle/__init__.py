"""NVFP4 oracle (test infrastructure only).

A plain CPU statement of the NVFP4 path, in C (nvfp4_oracle.c: float64 and
exact 128-bit integer arithmetic, float32 only where the quantisation recipe
fixes float32), wrapped here with ctypes and numpy. Only tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg use it; the library
never does, and the two share no code.

What is computed, and from which passage, is stated in nvfp4_oracle.c's header.
Every function here is pinned by a CPU test against something other than
itself (format tables, brute-force enumeration, exact integer arithmetic,
library routines, closed forms); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available). Returns the .so path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-shared",
            "-fPIC", "-o", _LIB_PATH + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.nvo_e2m1_value.restype = ctypes.c_double
            L.nvo_e2m1_value.argtypes = [ctypes.c_int]
            L.nvo_e4m3_value.restype = ctypes.c_double
            L.nvo_e4m3_value.argtypes = [ctypes.c_int]
            L.nvo_e2m1_encode.restype = ctypes.c_int
            L.nvo_e2m1_encode.argtypes = [ctypes.c_float]
            L.nvo_e4m3_encode.restype = ctypes.c_int
            L.nvo_e4m3_encode.argtypes = [ctypes.c_float]
            L.nvo_e2m1_encode_n.argtypes = [_f32p, ctypes.c_int64, _u8p]
            L.nvo_e4m3_encode_n.argtypes = [_f32p, ctypes.c_int64, _u8p]
            L.nvo_scale_bytes.restype = ctypes.c_int64
            L.nvo_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.nvo_sf_offset.restype = ctypes.c_int64
            L.nvo_sf_offset.argtypes = [ctypes.c_int64] * 3
            L.nvo_sf_unswizzle.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
            L.nvo_sf_swizzle.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
            L.nvo_amax_bf16.restype = ctypes.c_float
            L.nvo_amax_bf16.argtypes = [_u16p, ctypes.c_int64]
            L.nvo_global_scale.restype = ctypes.c_float
            L.nvo_global_scale.argtypes = [ctypes.c_float]
            L.nvo_quantize.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                       _u8p, _u8p]
            L.nvo_dequantize.argtypes = [_u8p, _u8p, ctypes.c_float, ctypes.c_int64,
                                         ctypes.c_int64, _f64p]
            L.nvo_gemm_f64.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, ctypes.c_float,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       _i64p, ctypes.c_int64, _i64p, ctypes.c_int64,
                                       _f64p, _f64p]
            L.nvo_gemm_exact.restype = ctypes.c_int
            L.nvo_gemm_exact.argtypes = [_u8p, _u8p, _u8p, _u8p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, _i64p, _u64p]
            L.nvo_grouped_gemm_f64.restype = ctypes.c_int
            L.nvo_grouped_gemm_f64.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, _f32p,
                                               _i32p, ctypes.c_int32, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, _i64p,
                                               ctypes.c_int64, _i64p, ctypes.c_int64,
                                               _f64p, _f64p]
            L.nvo_num_threads.restype = ctypes.c_int
            L.nvo_prune_pairs.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, _u16p, _u8p]
            L.nvo_meta_tiled_bytes.restype = ctypes.c_int64
            L.nvo_meta_tiled_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.nvo_meta_offset.restype = ctypes.c_int64
            L.nvo_meta_offset.argtypes = [ctypes.c_int64] * 3
            L.nvo_meta_tile.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
            L.nvo_meta_untile.argtypes = [_u8p, ctypes.c_int64, ctypes.c_int64, _u8p]
            L.nvo_scale_bytes_bs.restype = ctypes.c_int64
            L.nvo_scale_bytes_bs.argtypes = [ctypes.c_int64] * 3
            L.nvo_quantize_b32.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_float,
                                           _u8p, _u8p]
            L.nvo_sparse_gemm_f64.argtypes = [_u8p, _u8p, ctypes.c_float, _u8p, _u8p, _u8p, ctypes.c_float,
                                              ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                              _i64p, ctypes.c_int64, _i64p, ctypes.c_int64,
                                              _f64p, _f64p]
            _lib = L
    return _lib


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(t)


def _opt_idx(idx):
    if idx is None:
        return None, 0, None
    arr = np.ascontiguousarray(idx, dtype=np.int64)
    return arr, len(arr), _p(arr, _i64p)


# ---- formats -----------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return lib().nvo_e2m1_value(int(code))


def e4m3_value(code: int) -> float:
    return lib().nvo_e4m3_value(int(code))


def e2m1_encode(v: float) -> int:
    return lib().nvo_e2m1_encode(float(v))


def e4m3_encode(t: float) -> int:
    return lib().nvo_e4m3_encode(float(t))


def e2m1_encode_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, dtype=np.uint8)
    lib().nvo_e2m1_encode_n(_p(v, _f32p), v.size, _p(out, _u8p))
    return out


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.zeros(v.shape, dtype=np.uint8)
    lib().nvo_e4m3_encode_n(_p(v, _f32p), v.size, _p(out, _u8p))
    return out


def scale_bytes(rows: int, K: int) -> int:
    return int(lib().nvo_scale_bytes(rows, K))


def sf_offset(r: int, c: int, K: int) -> int:
    return int(lib().nvo_sf_offset(r, c, K))


def sf_unswizzle(sf: np.ndarray, rows: int, K: int) -> np.ndarray:
    lin = np.zeros((rows, K // 16), dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    lib().nvo_sf_unswizzle(_p(sf, _u8p), rows, K, _p(lin, _u8p))
    return lin


def sf_swizzle(lin: np.ndarray, rows: int, K: int) -> np.ndarray:
    sf = np.zeros(scale_bytes(rows, K), dtype=np.uint8)
    lin = np.ascontiguousarray(lin, dtype=np.uint8)
    lib().nvo_sf_swizzle(_p(lin, _u8p), rows, K, _p(sf, _u8p))
    return sf


# ---- quantisation --------------------------------------------------------------

def amax(x_bf16: np.ndarray) -> float:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    return float(np.float32(lib().nvo_amax_bf16(_p(x, _u16p), x.size)))


def global_scale(amax_value: float) -> np.float32:
    return np.float32(lib().nvo_global_scale(float(amax_value)))


def quantize(x_bf16: np.ndarray, g=None):
    """bf16 bits [M, K] -> (q [M, K/2] u8, sf swizzled u8, g float32)."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    M, K = x.shape
    if g is None:
        g = global_scale(amax(x))
    q = np.zeros((M, K // 2), dtype=np.uint8)
    sf = np.zeros(scale_bytes(M, K), dtype=np.uint8)
    lib().nvo_quantize(_p(x, _u16p), M, K, float(g), _p(q, _u8p), _p(sf, _u8p))
    return q, sf, np.float32(g)


def dequantize(q: np.ndarray, sf: np.ndarray, g: float, rows: int, K: int) -> np.ndarray:
    out = np.zeros((rows, K), dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    sf = np.ascontiguousarray(sf, dtype=np.uint8)
    lib().nvo_dequantize(_p(q, _u8p), _p(sf, _u8p), float(g), rows, K, _p(out, _f64p))
    return out


# ---- GEMM ------------------------------------------------------------------------

def gemm(a, sfa, ga, b, sfb, gb, M, N, K, rows=None, cols=None):
    """float64 y [nr, nc] and the tolerance magnitude term sum_k |x^ w^| (same shape)."""
    a, sfa, b, sfb = (np.ascontiguousarray(t, dtype=np.uint8) for t in (a, sfa, b, sfb))
    r_arr, nr, r_ptr = _opt_idx(rows)
    c_arr, nc, c_ptr = _opt_idx(cols)
    nr = M if rows is None else nr
    nc = N if cols is None else nc
    y = np.zeros((nr, nc), dtype=np.float64)
    ad = np.zeros((nr, nc), dtype=np.float64)
    lib().nvo_gemm_f64(_p(a, _u8p), _p(sfa, _u8p), float(ga), _p(b, _u8p), _p(sfb, _u8p),
                       float(gb), M, N, K, r_ptr, nr, c_ptr, nc, _p(y, _f64p), _p(ad, _f64p))
    return y, ad


def gemm_exact(a, sfa, b, sfb, M, N, K):
    """Exact integer sums S [M, N] (Python ints); the real dot product is S * 2^-20."""
    a, sfa, b, sfb = (np.ascontiguousarray(t, dtype=np.uint8) for t in (a, sfa, b, sfb))
    hi = np.zeros((M, N), dtype=np.int64)
    lo = np.zeros((M, N), dtype=np.uint64)
    nan = lib().nvo_gemm_exact(_p(a, _u8p), _p(sfa, _u8p), _p(b, _u8p), _p(sfb, _u8p), M, N, K,
                               _p(hi, _i64p), _p(lo, _u64p))
    if nan:
        raise ValueError("NaN scale code in exact GEMM input")
    return [[(int(hi[i, j]) << 64) + int(lo[i, j]) for j in range(N)] for i in range(M)]


def grouped_gemm(a, sfa, ga, b, sfb, gb, offsets, E, M_total, N, K, rows=None, cols=None):
    a, sfa, b, sfb = (np.ascontiguousarray(t, dtype=np.uint8) for t in (a, sfa, b, sfb))
    gb = np.ascontiguousarray(gb, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    r_arr, nr, r_ptr = _opt_idx(rows)
    c_arr, nc, c_ptr = _opt_idx(cols)
    nr = M_total if rows is None else nr
    nc = N if cols is None else nc
    y = np.zeros((nr, nc), dtype=np.float64)
    ad = np.zeros((nr, nc), dtype=np.float64)
    bad = lib().nvo_grouped_gemm_f64(_p(a, _u8p), _p(sfa, _u8p), float(ga), _p(b, _u8p),
                                     _p(sfb, _u8p), _p(gb, _f32p), _p(off, _i32p), E, M_total,
                                     N, K, r_ptr, nr, c_ptr, nc, _p(y, _f64p), _p(ad, _f64p))
    if bad:
        raise ValueError("malformed expert offsets")
    return y, ad


def silu(v: np.ndarray) -> np.ndarray:
    """SiLU (swish with beta = 1), float64: v * sigmoid(v) = v / (1 + exp(-v))."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def grouped_gemm_swiglu(a, sfa, ga, b_gu, sfb_gu, gb, offsets, E, M_total, N_gu, K, rows=None, cols=None):
    """MoE gate/up projection with the SwiGLU product fused after it.

    Each expert's weight b_gu[e] holds 2I = N_gu rows interleaved row by row: row 2c is
    gate row c, row 2c + 1 is up row c (a layout convention of the library; the pages
    name the fused gate+up projection, "The Moment of Synthesis", Reasoning, but give no
    layout). gate and up are the grouped GEMM's float64 outputs for those rows and
    y[t, c] = silu(gate[t, c]) * up[t, c], c in [0, I). `cols` selects output columns c.
    Returns (y, gate, up, absdot_gate, absdot_up).
    """
    I = N_gu // 2
    c = np.arange(I) if cols is None else np.asarray(cols, dtype=np.int64)
    gate, ad_g = grouped_gemm(a, sfa, ga, b_gu, sfb_gu, gb, offsets, E, M_total, N_gu, K, rows=rows, cols=2 * c)
    up, ad_u = grouped_gemm(a, sfa, ga, b_gu, sfb_gu, gb, offsets, E, M_total, N_gu, K, rows=rows, cols=2 * c + 1)
    return silu(gate) * up, gate, up, ad_g, ad_u


def within_tolerance_swiglu(y_gpu, gate, up, ad_g, ad_u, rel: float = 4e-3, absk: float = 1e-5):
    """Tolerance of the fused output, propagated from the GEMM tolerance of each factor.

    The GPU's gate g' and up u' lie within tg, tu (the GEMM bounds rel*|v| + absk*sum_k|x^ w^|)
    of the exact g, u. silu is Lipschitz with constant max|silu'| = 1.0998... < 1.1, so
    |silu(g')u' - silu(g)u| <= |silu(g') - silu(g)| |u'| + |silu(g)| |u' - u|
                             <= 1.1 tg (|u| + tu) + |silu(g)| tu =: B.
    The GPU returns silu(g')u' (1 + eta) with |eta| <= 2^-8 (one bf16 rounding, 2^-9, plus the
    fp32 activation's few ulps), and |silu(g')u'| <= |y| + B, so the error is at most
    (1 + 2^-8) B + 2^-8 |y|, y = silu(g) u. Returns (ok, worst ratio).
    """
    y_ref = silu(gate) * up
    tg = rel * np.abs(gate) + absk * ad_g
    tu = rel * np.abs(up) + absk * ad_u
    b = 1.1 * tg * (np.abs(up) + tu) + np.abs(silu(gate)) * tu
    bound = (1.0 + 2.0 ** -8) * b + 2.0 ** -8 * np.abs(y_ref)
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(err <= bound)), worst


def within_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, absdot: np.ndarray,
                     rel: float = 4e-3, absk: float = 1e-5):
    """Per-element |y_gpu - y_ref| <= rel*|y_ref| + absk*sum_k|x^ w^|; returns (ok, worst ratio)."""
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - y_ref)
    bound = rel * np.abs(y_ref) + absk * absdot
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(ratio)) if ratio.size else 0.0
    return bool(np.all(err <= bound)), worst


# ---- pair-wise 2:4 sparsity ---------------------------------------------------------

def prune_pairs(w_bits: np.ndarray):
    """Pair-wise 2:4 pruning and compression of a bf16 [N, K] weight (K % 8 == 0): per
    group of 8 K elements the two pairs with the largest |w_2j| + |w_2j+1| are kept (ties
    to the lower pair index). Returns (c bf16 bits [N, K/2], meta [N, K/16] u8), meta
    nibble per group = i0 | i1 << 2 of the kept pair indices, group 2b in the low nibble."""
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    N, K = w.shape
    c = np.empty((N, K // 2), dtype=np.uint16)
    meta = np.empty((N, K // 16), dtype=np.uint8)
    lib().nvo_prune_pairs(_p(w, _u16p), N, K, _p(c, _u16p), _p(meta, _u8p))
    return c, meta


def meta_tiled_bytes(N: int, K: int) -> int:
    return int(lib().nvo_meta_tiled_bytes(N, K))


def meta_offset(n: int, b: int, K: int) -> int:
    return int(lib().nvo_meta_offset(n, b, K))


def meta_tile(meta: np.ndarray, N: int, K: int) -> np.ndarray:
    """Linear [N, K/16] metadata -> the tiled layout (4096-byte tile per 128 rows x 512 K)."""
    lin = np.ascontiguousarray(meta, dtype=np.uint8)
    out = np.empty(meta_tiled_bytes(N, K), dtype=np.uint8)
    lib().nvo_meta_tile(_p(lin, _u8p), N, K, _p(out, _u8p))
    return out


def meta_untile(tiled: np.ndarray, N: int, K: int) -> np.ndarray:
    t = np.ascontiguousarray(tiled, dtype=np.uint8)
    out = np.empty((N, K // 16), dtype=np.uint8)
    lib().nvo_meta_untile(_p(t, _u8p), N, K, _p(out, _u8p))
    return out


def sf_unswizzle_bs(sf: np.ndarray, rows: int, K: int, bs: int) -> np.ndarray:
    """Tiled scale tensor with `bs`-element blocks -> linear [rows, K/bs] (numpy restatement
    of the tile formula with K/bs scale columns)."""
    kc = K // bs
    kc4 = (kc + 3) // 4
    r = np.arange(rows)[:, None]
    c = np.arange(kc)[None, :]
    off = ((r // 128) * kc4 + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    return np.asarray(sf)[off]


def sf_swizzle_bs(lin: np.ndarray, rows: int, K: int, bs: int) -> np.ndarray:
    kc = K // bs
    kc4 = (kc + 3) // 4
    r = np.arange(rows)[:, None]
    c = np.arange(kc)[None, :]
    off = ((r // 128) * kc4 + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)
    out = np.zeros((rows + 127) // 128 * 128 * kc4 * 4, dtype=np.uint8)
    out[off] = lin
    return out


def scale_bytes_b32(rows: int, K: int) -> int:
    return int(lib().nvo_scale_bytes_bs(rows, K, 32))


def quantize_b32(x_bits: np.ndarray, g_fixed=None):
    """The quantisation recipe with 32-element blocks (the dense operand of the sparse GEMM).
    Returns (q [M, K/2], sf tiled over K/32 columns, g)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x.shape
    g = np.float32(global_scale(amax(x))) if g_fixed is None else np.float32(g_fixed)
    q = np.empty((M, K // 2), dtype=np.uint8)
    sf = np.empty(scale_bytes_b32(M, K), dtype=np.uint8)
    lib().nvo_quantize_b32(_p(x, _u16p), M, K, float(g), _p(q, _u8p), _p(sf, _u8p))
    return q, sf, g


def sparse_quantize_weight(w_bits: np.ndarray):
    """Prune, compress and quantise a bf16 weight [N, K]: returns (cq [N, K/4] u8 codes of
    the compressed values, csf their tiled 16-block scales over K/2, g, meta [N, K/16])."""
    c, meta = prune_pairs(w_bits)
    cq, csf, g = quantize(c)
    return cq, csf, g, meta


def sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, M: int, N: int, K: int, rows=None, cols=None):
    """y = x . W^T in float64 with x in 32-element blocks and W pair-wise 2:4 sparse
    (compressed codes cq, scales csf, metadata meta [N, K/16]); returns (y, absdot)."""
    r_arr, nr, r_ptr = _opt_idx(rows)
    c_arr, nc, c_ptr = _opt_idx(cols)
    nr = M if rows is None else nr
    nc = N if cols is None else nc
    y = np.zeros((nr, nc), dtype=np.float64)
    ad = np.zeros((nr, nc), dtype=np.float64)
    xq, xsf, cq, csf, meta = (np.ascontiguousarray(a, dtype=np.uint8) for a in (xq, xsf, cq, csf, meta))
    lib().nvo_sparse_gemm_f64(_p(xq, _u8p), _p(xsf, _u8p), float(gx), _p(cq, _u8p), _p(csf, _u8p),
                              _p(meta, _u8p), float(gw), M, N, K, r_ptr, nr, c_ptr, nc,
                              _p(y, _f64p), _p(ad, _f64p))
    return y, ad


def grouped_sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, offsets, E: int, M_total: int, N: int, K: int,
                        rows=None, cols=None):
    """Grouped (MoE) form of sparse_gemm: rows offsets[e] .. offsets[e+1]-1 of x (32-element
    blocks, sorted by expert) use expert e's compressed weight cq[e], csf[e], meta[e] (linear
    [N, K/16]) and global scale gw[e]. Returns (y, absdot) over the selected rows/cols."""
    off = np.asarray(offsets, dtype=np.int64)
    if off[0] != 0 or off[-1] != M_total or np.any(np.diff(off) < 0):
        raise ValueError("malformed expert offsets")
    sel = np.arange(M_total) if rows is None else np.asarray(rows, dtype=np.int64)
    nc = N if cols is None else len(cols)
    y = np.zeros((len(sel), nc), dtype=np.float64)
    ad = np.zeros((len(sel), nc), dtype=np.float64)
    for e in range(E):
        pick = np.nonzero((sel >= off[e]) & (sel < off[e + 1]))[0]
        if pick.size == 0:
            continue
        ye, ade = sparse_gemm(xq, xsf, gx, cq[e], csf[e], meta[e], gw[e], M_total, N, K, rows=sel[pick], cols=cols)
        y[pick] = ye
        ad[pick] = ade
    return y, ad


def num_threads() -> int:
    return int(lib().nvo_num_threads())
