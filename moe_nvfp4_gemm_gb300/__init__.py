"""Thin Python binding of the NVFP4 C ABI (include/nvfp4.h).

Argument marshalling only: every entry point takes torch CUDA tensors, passes
their data pointers and the current CUDA stream to the function of the same
name in libnvfp4.so, and raises on a non-zero status. All arithmetic runs in
the library's kernels; there is no fallback of any kind. Output tensors and
workspaces are allocated here with torch (the library itself never allocates).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libnvfp4.so")

NVFP4_TUNE_DENSE_BN = 1
NVFP4_TUNE_DENSE_GRID = 2
NVFP4_TUNE_STREAM_MAX_M = 3
NVFP4_TUNE_STREAM_SPLIT = 4
NVFP4_TUNE_STREAM_STAGES = 5
NVFP4_TUNE_GROUPED_GRID = 6
NVFP4_TUNE_GROUPED_STAGES = 7
NVFP4_TUNE_DENSE_KERNEL = 8
NVFP4_TUNE_PDL = 9
NVFP4_TUNE_WEIGHT_L2 = 10
NVFP4_TUNE_DENSE_RASTER = 11
NVFP4_TUNE_WATCHDOG_US = 12
NVFP4_TUNE_TEST_WITHHOLD_STAGE = 13
NVFP4_TUNE_STREAM_L2_PREFETCH = 14
NVFP4_TUNE_GROUPED_TILE_ROWS = 15

STATUS = {0: "NVFP4_OK", -1: "NVFP4_ERR_INVALID_ARG", -2: "NVFP4_ERR_UNSUPPORTED_SHAPE",
          -3: "NVFP4_ERR_ALIGNMENT", -4: "NVFP4_ERR_ARCH", -5: "NVFP4_ERR_CUDA",
          -6: "NVFP4_ERR_WORKSPACE", -7: "NVFP4_ERR_TIMEOUT", -8: "NVFP4_ERR_BAD_OFFSETS"}

EXPORTS = ["nvfp4_status_string", "nvfp4_scale_bytes", "nvfp4_amax_workspace_bytes", "nvfp4_amax",
           "nvfp4_quantize", "nvfp4_gemm_workspace_bytes", "nvfp4_gemm", "nvfp4_gemm_quantize_out",
           "nvfp4_grouped_gemm_workspace_bytes", "nvfp4_grouped_gemm", "nvfp4_grouped_gemm_gather",
           "nvfp4_grouped_gemm_gather_workspace_bytes",
           "nvfp4_grouped_gemm_swiglu",
           "nvfp4_grouped_gemm_noalloc",
           "nvfp4_encode_e2m1",
           "nvfp4_encode_e4m3", "nvfp4_tune", "nvfp4_last_launch_count",
           "nvfp4_sparse_meta_bytes", "nvfp4_scale_bytes_b32", "nvfp4_prune_pairs", "nvfp4_quantize_b32",
           "nvfp4_sparse_gemm", "nvfp4_grouped_sparse_gemm", "nvfp4_gemm_batched",
           "nvfp4_grouped_gemm_swiglu_quantize_out"]


class NVFP4Error(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t

NVFP4_MAX_BATCH = 8


class GemmProblem(ctypes.Structure):
    """One problem of nvfp4_gemm_batched (the C struct nvfp4_gemm_problem)."""
    _fields_ = [("a", ctypes.c_void_p), ("sfa", ctypes.c_void_p), ("ga", ctypes.c_void_p),
                ("b", ctypes.c_void_p), ("sfb", ctypes.c_void_p), ("gb", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


def lib():
    """The loaded libnvfp4.so; raises if it was not built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"NVFP4 CUDA library missing at {LIB_PATH}: run "
                                  "`python -c 'import __graft_entry__ as g; g.build()'` first")
            L = ctypes.CDLL(LIB_PATH)
            L.nvfp4_status_string.restype = ctypes.c_char_p
            L.nvfp4_status_string.argtypes = [ctypes.c_int]
            L.nvfp4_scale_bytes.restype = _i64
            L.nvfp4_scale_bytes.argtypes = [_i64, _i64]
            L.nvfp4_amax_workspace_bytes.restype = _sz
            L.nvfp4_amax_workspace_bytes.argtypes = [_i64]
            L.nvfp4_amax.argtypes = [_vp, _i64, _vp, _vp, _vp, _sz, _vp]
            L.nvfp4_quantize.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp]
            L.nvfp4_gemm_workspace_bytes.restype = _sz
            L.nvfp4_gemm_workspace_bytes.argtypes = [_i64, _i64, _i64]
            L.nvfp4_gemm.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _sz,
                                     _vp, _vp]
            L.nvfp4_gemm_quantize_out.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                                  _i64, _vp, _vp]
            L.nvfp4_grouped_gemm_workspace_bytes.restype = _sz
            L.nvfp4_grouped_gemm_workspace_bytes.argtypes = [_i32, _i64, _i64, _i64]
            L.nvfp4_grouped_gemm.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64,
                                             _i64, _vp, _vp, _sz, _vp, _vp]
            L.nvfp4_grouped_gemm_gather_workspace_bytes.restype = _sz
            L.nvfp4_grouped_gemm_gather_workspace_bytes.argtypes = [_i32, _i64, _i64, _i64]
            L.nvfp4_grouped_gemm_gather.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64,
                                                    _i64, _i64, _vp, _vp, _sz, _vp, _vp]
            L.nvfp4_grouped_gemm_swiglu.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64,
                                                    _i64, _vp, _vp, _sz, _vp, _vp]
            L.nvfp4_grouped_gemm_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64,
                                                     _i64, _i64, _vp, _vp, _vp]
            L.nvfp4_encode_e2m1.argtypes = [_vp, _i64, _vp, _vp]
            L.nvfp4_encode_e4m3.argtypes = [_vp, _i64, _vp, _vp]
            L.nvfp4_tune.argtypes = [ctypes.c_int, ctypes.c_int]
            L.nvfp4_sparse_meta_bytes.restype = _i64
            L.nvfp4_sparse_meta_bytes.argtypes = [_i64, _i64]
            L.nvfp4_scale_bytes_b32.restype = _i64
            L.nvfp4_scale_bytes_b32.argtypes = [_i64, _i64]
            L.nvfp4_prune_pairs.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp]
            L.nvfp4_quantize_b32.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp]
            L.nvfp4_sparse_gemm.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp]
            L.nvfp4_grouped_sparse_gemm.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64,
                                                    _i64, _vp, _vp, _sz, _vp, _vp]
            L.nvfp4_gemm_batched.argtypes = [_vp, _i32, _i64, _vp, _vp]
            L.nvfp4_grouped_gemm_swiglu_quantize_out.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64,
                                                                 _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp, _vp]
            L.nvfp4_last_launch_count.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn, rc):
    if rc != 0:
        raise NVFP4Error(fn, rc)


def _cuda(t, dtype, name):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous CUDA tensor of {dtype}")
    return t


def nvfp4_scale_bytes(rows: int, K: int) -> int:
    return int(lib().nvfp4_scale_bytes(rows, K))


def nvfp4_tune(key: int, value: int) -> None:
    _check("nvfp4_tune", lib().nvfp4_tune(key, value))


def nvfp4_last_launch_count() -> int:
    return int(lib().nvfp4_last_launch_count())


def nvfp4_amax_workspace_bytes(n: int) -> int:
    return int(lib().nvfp4_amax_workspace_bytes(n))


def nvfp4_gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(lib().nvfp4_gemm_workspace_bytes(M, N, K))


def nvfp4_status_string(status: int) -> str:
    return lib().nvfp4_status_string(status).decode()


def nvfp4_amax(x: torch.Tensor, amax_out=None, g_out=None, workspace=None, stream=None):
    """Returns (amax, g) as 1-element fp32 CUDA tensors; g = amax / 2688 (1 if amax == 0)."""
    _cuda(x, torch.bfloat16, "x")
    dev = x.device
    amax_out = torch.empty(1, dtype=torch.float32, device=dev) if amax_out is None else amax_out
    g_out = torch.empty(1, dtype=torch.float32, device=dev) if g_out is None else g_out
    nbytes = int(lib().nvfp4_amax_workspace_bytes(x.numel()))
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _check("nvfp4_amax", lib().nvfp4_amax(_ptr(x), x.numel(), _ptr(amax_out), _ptr(g_out),
                                          _ptr(workspace), workspace.numel(), _stream(stream)))
    return amax_out, g_out


def nvfp4_quantize(x: torch.Tensor, global_scale: torch.Tensor, q_out=None, sf_out=None, stream=None):
    """bf16 [M, K] -> (q u8 [M, K/2], sf u8 [nvfp4_scale_bytes(M, K)])."""
    _cuda(x, torch.bfloat16, "x")
    _cuda(global_scale, torch.float32, "global_scale")
    M, K = x.shape
    q_out = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device) if q_out is None else q_out
    sf_out = (torch.empty(nvfp4_scale_bytes(M, K), dtype=torch.uint8, device=x.device)
              if sf_out is None else sf_out)
    _check("nvfp4_quantize", lib().nvfp4_quantize(_ptr(x), M, K, _ptr(global_scale), _ptr(q_out),
                                                  _ptr(sf_out), _stream(stream)))
    return q_out, sf_out


def nvfp4_gemm(a, sfa, ga, b, sfb, gb, M: int, N: int, K: int, y=None, dev_status=None,
               stream=None):
    """y = x @ W^T in bf16 [M, N] from packed NVFP4 operands (see include/nvfp4.h)."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=a.device) if y is None else y
    ws_bytes = int(lib().nvfp4_gemm_workspace_bytes(M, N, K))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=a.device) if ws_bytes else None
    _check("nvfp4_gemm", lib().nvfp4_gemm(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb),
                                          _ptr(y), M, N, K, _ptr(ws), ws_bytes, _ptr(dev_status),
                                          _stream(stream)))
    return y


def nvfp4_grouped_gemm_workspace_bytes(E: int, M_total: int, N: int, K: int) -> int:
    return int(lib().nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K))


def nvfp4_gemm_quantize_out(a, sfa, ga, b, sfb, gb, g_out, M: int, N: int, K: int, q_out=None, sf_out=None,
                            dev_status=None, stream=None):
    """y = x . W^T as nvfp4_gemm, emitted as NVFP4 with global scale g_out: returns
    (codes uint8 [M, N/2], tiled scales uint8 [nvfp4_scale_bytes(M, N)])."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
        _cuda(t, torch.uint8, n)
    for t, n in ((ga, "ga"), (gb, "gb"), (g_out, "g_out")):
        _cuda(t, torch.float32, n)
    if q_out is None:
        q_out = torch.empty((M, N // 2), dtype=torch.uint8, device=a.device)
    if sf_out is None:
        sf_out = torch.empty(nvfp4_scale_bytes(M, N), dtype=torch.uint8, device=a.device)
    _check("nvfp4_gemm_quantize_out",
           lib().nvfp4_gemm_quantize_out(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb), _ptr(g_out),
                                         _ptr(q_out), _ptr(sf_out), M, N, K, _ptr(dev_status), _stream(stream)))
    return q_out, sf_out


def nvfp4_grouped_gemm(a, sfa, ga, b, sfb, gb, expert_offsets, E: int, M_total: int, N: int,
                       K: int, y=None, workspace=None, dev_status=None, stream=None):
    """Per-expert y[rows of e] = x[rows of e] @ W_e^T, rows sorted by expert (bf16 [M_total, N])."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    _cuda(expert_offsets, torch.int32, "expert_offsets")
    y = torch.empty((M_total, N), dtype=torch.bfloat16, device=a.device) if y is None else y
    ws_bytes = nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=a.device)
    _check("nvfp4_grouped_gemm",
           lib().nvfp4_grouped_gemm(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb),
                                    _ptr(expert_offsets), E, M_total, N, K, _ptr(y),
                                    _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                    _stream(stream)))
    return y


def nvfp4_grouped_gemm_gather(a_tok, sfa_tok, ga, b, sfb, gb, expert_offsets, row_token, E: int, T: int,
                              M_total: int, N: int, K: int, y=None, workspace=None, dev_status=None, stream=None):
    """Grouped GEMM over routed rows r (sorted by expert) that read token row row_token[r] of
    the T-row activations a_tok: bf16 [M_total, N] in routed-row order. The default
    workspace has room for the rows to be copied out ahead of the GEMM; one of
    nvfp4_grouped_gemm_workspace_bytes bytes makes the GEMM's load stage gather them."""
    for t, n in ((a_tok, "a_tok"), (sfa_tok, "sfa_tok"), (b, "b"), (sfb, "sfb")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    _cuda(expert_offsets, torch.int32, "expert_offsets")
    _cuda(row_token, torch.int32, "row_token")
    y = torch.empty((M_total, N), dtype=torch.bfloat16, device=a_tok.device) if y is None else y
    ws_bytes = nvfp4_grouped_gemm_gather_workspace_bytes(E, M_total, N, K)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=a_tok.device)
    _check("nvfp4_grouped_gemm_gather",
           lib().nvfp4_grouped_gemm_gather(_ptr(a_tok), _ptr(sfa_tok), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb),
                                           _ptr(expert_offsets), _ptr(row_token), E, T, M_total, N, K, _ptr(y),
                                           _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)))
    return y


def nvfp4_grouped_gemm_gather_workspace_bytes(E: int, M_total: int, N: int, K: int) -> int:
    return int(lib().nvfp4_grouped_gemm_gather_workspace_bytes(E, M_total, N, K))


def nvfp4_grouped_gemm_swiglu(a, sfa, ga, b_gu, sfb_gu, gb, expert_offsets, E: int, M_total: int, N_gu: int,
                              K: int, y=None, workspace=None, dev_status=None, stream=None):
    """Gate/up projection with fused SwiGLU: b_gu interleaves gate and up rows (row 2c gate c,
    2c + 1 up c); returns y[m, c] = silu(gate) * up as bf16 [M_total, N_gu // 2]."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b_gu, "b_gu"), (sfb_gu, "sfb_gu")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    _cuda(expert_offsets, torch.int32, "expert_offsets")
    y = torch.empty((M_total, N_gu // 2), dtype=torch.bfloat16, device=a.device) if y is None else y
    ws_bytes = nvfp4_grouped_gemm_workspace_bytes(E, M_total, N_gu, K)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=a.device)
    _check("nvfp4_grouped_gemm_swiglu",
           lib().nvfp4_grouped_gemm_swiglu(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b_gu), _ptr(sfb_gu), _ptr(gb),
                                           _ptr(expert_offsets), E, M_total, N_gu, K, _ptr(y),
                                           _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                           _stream(stream)))
    return y


NVFP4_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def nvfp4_grouped_gemm_noalloc(a, sfa, ga, b, sfb, gb, expert_offsets, E: int, M_total: int, N: int,
                               K: int, y=None, dev_status=None, stream=None):
    """nvfp4_grouped_gemm without a workspace argument: the library's built-in scratch is used.

    For callers that cannot allocate device memory where they run the MoE layer (runtimes
    with a fixed memory budget and no allocator). Only `y` is allocated here when not given.
    """
    for t, n in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    _cuda(expert_offsets, torch.int32, "expert_offsets")
    y = torch.empty((M_total, N), dtype=torch.bfloat16, device=a.device) if y is None else y
    _check("nvfp4_grouped_gemm_noalloc",
           lib().nvfp4_grouped_gemm_noalloc(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b), _ptr(sfb), _ptr(gb),
                                            _ptr(expert_offsets), E, M_total, N, K, _ptr(y),
                                            _ptr(dev_status), _stream(stream)))
    return y


def nvfp4_sparse_meta_bytes(N: int, K: int) -> int:
    return int(lib().nvfp4_sparse_meta_bytes(N, K))


def nvfp4_scale_bytes_b32(rows: int, K: int) -> int:
    return int(lib().nvfp4_scale_bytes_b32(rows, K))


def nvfp4_prune_pairs(w: torch.Tensor, c_out=None, meta_out=None, stream=None):
    """Pair-wise 2:4 pruning + compression of a bf16 weight [N, K]: returns (c bf16 [N, K/2],
    tiled metadata uint8 [nvfp4_sparse_meta_bytes(N, K)])."""
    _cuda(w, torch.bfloat16, "w")
    N, K = w.shape
    c_out = torch.empty((N, K // 2), dtype=torch.bfloat16, device=w.device) if c_out is None else c_out
    meta_out = (torch.empty(nvfp4_sparse_meta_bytes(N, K), dtype=torch.uint8, device=w.device)
                if meta_out is None else meta_out)
    _check("nvfp4_prune_pairs", lib().nvfp4_prune_pairs(_ptr(w), N, K, _ptr(c_out), _ptr(meta_out),
                                                        _stream(stream)))
    return c_out, meta_out


def nvfp4_quantize_b32(x: torch.Tensor, global_scale: torch.Tensor, q_out=None, sf_out=None, stream=None):
    """bf16 [M, K] -> NVFP4 with 32-element blocks: (q u8 [M, K/2], sf u8 [nvfp4_scale_bytes_b32(M, K)])."""
    _cuda(x, torch.bfloat16, "x")
    _cuda(global_scale, torch.float32, "global_scale")
    M, K = x.shape
    q_out = torch.empty((M, K // 2), dtype=torch.uint8, device=x.device) if q_out is None else q_out
    sf_out = (torch.empty(nvfp4_scale_bytes_b32(M, K), dtype=torch.uint8, device=x.device)
              if sf_out is None else sf_out)
    _check("nvfp4_quantize_b32", lib().nvfp4_quantize_b32(_ptr(x), M, K, _ptr(global_scale), _ptr(q_out),
                                                          _ptr(sf_out), _stream(stream)))
    return q_out, sf_out


def nvfp4_grouped_gemm_swiglu_quantize_out(a, sfa, ga, b_gu, sfb_gu, gb, expert_offsets, E: int, M_total: int,
                                           N_gu: int, K: int, g_out, q_out=None, sf_out=None, workspace=None,
                                           dev_status=None, stream=None):
    """Gate/up projection with SwiGLU emitting NVFP4 with the global scale g_out: returns
    (codes u8 [M_total, N_gu // 4], tiled scales u8 [nvfp4_scale_bytes(M_total, N_gu // 2)])."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b_gu, "b_gu"), (sfb_gu, "sfb_gu")):
        _cuda(t, torch.uint8, n)
    for t, n in ((ga, "ga"), (gb, "gb"), (g_out, "g_out")):
        _cuda(t, torch.float32, n)
    dev = a.device
    q_out = torch.empty((M_total, N_gu // 4), dtype=torch.uint8, device=dev) if q_out is None else q_out
    sf_out = (torch.empty(nvfp4_scale_bytes(M_total, N_gu // 2), dtype=torch.uint8, device=dev)
              if sf_out is None else sf_out)
    ws_bytes = int(lib().nvfp4_grouped_gemm_workspace_bytes(E, M_total, N_gu, K))
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    _check("nvfp4_grouped_gemm_swiglu_quantize_out",
           lib().nvfp4_grouped_gemm_swiglu_quantize_out(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b_gu), _ptr(sfb_gu),
                                                        _ptr(gb), _ptr(expert_offsets), E, M_total, N_gu, K,
                                                        _ptr(g_out), _ptr(q_out), _ptr(sf_out), _ptr(workspace),
                                                        workspace.numel(), _ptr(dev_status), _stream(stream)))
    return q_out, sf_out


def nvfp4_gemm_batched(problems, M: int, dev_status=None, stream=None):
    """Several decode-M GEMMs in one launch. problems: sequence of (a, sfa, ga, b, sfb, gb, y)
    tuples of CUDA tensors (y bf16 [M, N], preallocated); N and K come from b and a."""
    arr = (GemmProblem * max(1, len(problems)))()
    for i, (a, sfa, ga, b, sfb, gb, y) in enumerate(problems):
        for t, n in ((a, "a"), (sfa, "sfa"), (b, "b"), (sfb, "sfb")):
            _cuda(t, torch.uint8, n)
        _cuda(ga, torch.float32, "ga")
        _cuda(gb, torch.float32, "gb")
        _cuda(y, torch.bfloat16, "y")
        arr[i] = GemmProblem(a.data_ptr(), sfa.data_ptr(), ga.data_ptr(), b.data_ptr(), sfb.data_ptr(),
                             gb.data_ptr(), y.data_ptr(), b.shape[0], 2 * b.shape[1])
    _check("nvfp4_gemm_batched", lib().nvfp4_gemm_batched(ctypes.cast(arr, ctypes.c_void_p), len(problems), M,
                                                          _ptr(dev_status), _stream(stream)))


def nvfp4_sparse_gemm(a, sfa, ga, b_c, sfb_c, meta, gb, M: int, N: int, K: int, y=None, dev_status=None,
                      stream=None):
    """y = x @ W^T, W pair-wise 2:4 sparse (compressed codes b_c [N, K/4], scales sfb_c, tiled meta),
    x in 32-element blocks; bf16 [M, N]."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b_c, "b_c"), (sfb_c, "sfb_c"), (meta, "meta")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    y = torch.empty((M, N), dtype=torch.bfloat16, device=a.device) if y is None else y
    _check("nvfp4_sparse_gemm", lib().nvfp4_sparse_gemm(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b_c), _ptr(sfb_c),
                                                        _ptr(meta), _ptr(gb), _ptr(y), M, N, K, _ptr(dev_status),
                                                        _stream(stream)))
    return y


def nvfp4_grouped_sparse_gemm(a, sfa, ga, b_c, sfb_c, meta, gb, expert_offsets, E: int, M_total: int, N: int,
                              K: int, y=None, workspace=None, dev_status=None, stream=None):
    """Grouped form of nvfp4_sparse_gemm over pair-wise 2:4 sparse experts; bf16 [M_total, N]."""
    for t, n in ((a, "a"), (sfa, "sfa"), (b_c, "b_c"), (sfb_c, "sfb_c"), (meta, "meta")):
        _cuda(t, torch.uint8, n)
    _cuda(ga, torch.float32, "ga")
    _cuda(gb, torch.float32, "gb")
    _cuda(expert_offsets, torch.int32, "expert_offsets")
    y = torch.empty((M_total, N), dtype=torch.bfloat16, device=a.device) if y is None else y
    if workspace is None:
        workspace = torch.empty(max(1, nvfp4_grouped_gemm_workspace_bytes(E, M_total, N, K)), dtype=torch.uint8,
                                device=a.device)
    _check("nvfp4_grouped_sparse_gemm",
           lib().nvfp4_grouped_sparse_gemm(_ptr(a), _ptr(sfa), _ptr(ga), _ptr(b_c), _ptr(sfb_c), _ptr(meta),
                                           _ptr(gb), _ptr(expert_offsets), E, M_total, N, K, _ptr(y),
                                           _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream)))
    return y


def nvfp4_encode_e2m1(v: torch.Tensor, stream=None) -> torch.Tensor:
    _cuda(v, torch.float32, "v")
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check("nvfp4_encode_e2m1", lib().nvfp4_encode_e2m1(_ptr(v), v.numel(), _ptr(out), _stream(stream)))
    return out


def nvfp4_encode_e4m3(v: torch.Tensor, stream=None) -> torch.Tensor:
    _cuda(v, torch.float32, "v")
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    _check("nvfp4_encode_e4m3", lib().nvfp4_encode_e4m3(_ptr(v), v.numel(), _ptr(out), _stream(stream)))
    return out
