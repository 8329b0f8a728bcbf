"""CPU checks of the C ABI: the library builds, loads without a GPU, exports every
symbol include/nvfp4.h declares, and rejects bad arguments on the host before
touching the device (no compute calls here)."""
import ctypes
import os
import re

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_nvfp4_gemm_gb300 import build
    path = build.build()
    import moe_nvfp4_gemm_gb300 as m
    return m.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    import moe_nvfp4_gemm_gb300 as m
    assert sorted(m.EXPORTS) == names


def test_status_strings(lib):
    for code, name in [(0, b"NVFP4_OK"), (-2, b"NVFP4_ERR_UNSUPPORTED_SHAPE"),
                       (-8, b"NVFP4_ERR_BAD_OFFSETS"), (5, b"NVFP4_UNKNOWN_STATUS")]:
        assert lib.nvfp4_status_string(code) == name


def test_scale_bytes_matches_oracle(lib):
    for rows, K in [(1, 64), (128, 256), (130, 8192), (4096, 6144), (0, 64)]:
        assert lib.nvfp4_scale_bytes(rows, K) == oracle.scale_bytes(rows, K)
    assert lib.nvfp4_scale_bytes(-1, 64) == 0


P = ctypes.c_void_p


def _gemm(lib, M, N, K, a=16, y=16):
    return lib.nvfp4_gemm(P(a), P(16), P(16), P(16), P(16), P(16), P(y), M, N, K, None, 0, None, None)


def test_gemm_host_validation(lib):
    assert _gemm(lib, 0, 128, 256) == 0                 # empty M: nothing to do
    assert _gemm(lib, 4, 128, 100) == -2                # K % 64
    assert _gemm(lib, 4, 12, 256) == -2                 # N % 8
    assert _gemm(lib, -1, 128, 256) == -1
    assert _gemm(lib, 4, 0, 256) == -1
    assert _gemm(lib, 4, 128, 256, a=0) == -1            # null operand
    assert _gemm(lib, 4, 128, 256, a=24) == -3           # misaligned operand
    assert _gemm(lib, 4, 128, 256, y=40) == -3           # misaligned output
    assert _gemm(lib, 1 << 31, 128, 256) == -2           # size limit


def test_grouped_host_validation(lib):
    g = lambda E, Mt, ws, wsb, off=16: lib.nvfp4_grouped_gemm(
        P(16), P(16), P(16), P(16), P(16), P(16), P(off), E, Mt, 128, 256, P(16), P(ws), wsb, None, None)
    need = lib.nvfp4_grouped_gemm_workspace_bytes(4, 100, 128, 256)
    assert need > 0
    assert g(0, 100, 256, need) == -1                   # no experts
    assert g(4, 0, 256, need) == 0                      # no rows
    assert g(4, 100, 0, need) == -6                     # missing workspace
    assert g(4, 100, 256, need - 1) == -6               # short workspace
    assert g(4, 100, 272, need) == -3                   # workspace not 256-byte aligned
    assert g(4, 100, 256, need, off=0) == -1            # null offsets
    assert g(4, (1 << 30) + 1, 256, 1 << 62) == -2      # more routed rows than 32-bit indexing allows


def test_quantize_and_amax_host_validation(lib):
    q = lambda M, K, x=16: lib.nvfp4_quantize(P(x), M, K, P(16), P(16), P(16), None)
    assert q(0, 64) == 0
    assert q(4, 48) == -2
    assert q(4, 64, x=0) == -1
    assert q(4, 64, x=8) == -3
    assert lib.nvfp4_amax(P(16), 100, P(16), P(16), None, 0, None) == -6
    assert lib.nvfp4_amax(P(8), 100, P(16), P(16), P(16), 4096, None) == -3


def test_gather_workspace_holds_the_routed_rows(lib):
    for E, Mt, N, K in [(256, 4096, 4096, 6144), (3, 17, 128, 64), (1, 1, 8, 64)]:
        plain = lib.nvfp4_grouped_gemm_workspace_bytes(E, Mt, N, K)
        assert lib.nvfp4_grouped_gemm_gather_workspace_bytes(E, Mt, N, K) == (plain + 255) // 256 * 256 + Mt * K // 2
    assert lib.nvfp4_grouped_gemm_gather_workspace_bytes(0, 16, 128, 64) == 0


def test_tune_rejects_bad_values(lib):
    assert lib.nvfp4_tune(1, 200) == -1
    assert lib.nvfp4_tune(4, 9) == -1
    assert lib.nvfp4_tune(99, 1) == -1
    assert lib.nvfp4_tune(1, 0) == 0
    assert lib.nvfp4_tune(10, 2) == -1   # weight L2 residency: 0 streamed, 1 kept
    assert lib.nvfp4_tune(10, -1) == -1
    assert lib.nvfp4_tune(10, 1) == 0
    assert lib.nvfp4_tune(10, 0) == 0
    assert lib.nvfp4_tune(14, -2) == -1  # decode L2 prefetch: -1 none, 0 all, k blocks
    assert lib.nvfp4_tune(14, -1) == 0
    assert lib.nvfp4_tune(14, 5) == 0
    assert lib.nvfp4_tune(14, 0) == 0
    assert lib.nvfp4_tune(15, 96) == -1  # grouped token tile rows: 0 (128), 64 or 128
    assert lib.nvfp4_tune(15, 64) == 0
    assert lib.nvfp4_tune(15, 0) == 0


def test_sparse_sizes_match_oracle(lib):
    for rows, K in [(1, 128), (128, 512), (130, 8192), (4096, 6144), (0, 128)]:
        assert lib.nvfp4_scale_bytes_b32(rows, K) == oracle.scale_bytes_b32(rows, K)
        assert lib.nvfp4_sparse_meta_bytes(rows, K) == oracle.meta_tiled_bytes(rows, K)
    assert lib.nvfp4_sparse_meta_bytes(-1, 128) == 0 and lib.nvfp4_scale_bytes_b32(4, -1) == 0


def test_sparse_host_validation(lib):
    sg = lambda M, N, K, a=16, meta=16: lib.nvfp4_sparse_gemm(P(a), P(16), P(16), P(16), P(16), P(meta), P(16),
                                                              P(16), M, N, K, None, None)
    assert sg(0, 128, 256) == 0                  # empty M
    assert sg(4, 128, 192) == -2                 # K % 128
    assert sg(4, 12, 256) == -2                  # N % 8
    assert sg(4, 128, 256, meta=0) == -1         # null metadata
    assert sg(4, 128, 256, a=24) == -3           # misaligned operand
    pr = lambda N, K, w=16: lib.nvfp4_prune_pairs(P(w), N, K, P(16), P(16), None)
    assert pr(0, 128) == 0 and pr(4, 64) == -2 and pr(4, 128, w=0) == -1 and pr(4, 128, w=8) == -3
    qb = lambda M, K, x=16: lib.nvfp4_quantize_b32(P(x), M, K, P(16), P(16), P(16), None)
    assert qb(0, 128) == 0 and qb(4, 64) == -2 and qb(4, 128, x=0) == -1 and qb(4, 128, x=24) == -3


def _batched(lib, problems, count, M):
    import moe_nvfp4_gemm_gb300 as m
    arr = (m.GemmProblem * max(1, len(problems)))(*problems)
    return lib.nvfp4_gemm_batched(ctypes.cast(arr, P), count, M, None, None)


def test_gemm_batched_host_validation(lib):
    import moe_nvfp4_gemm_gb300 as m
    ok = m.GemmProblem(16, 16, 16, 16, 16, 16, 16, 256, 512)
    assert lib.nvfp4_gemm_batched(None, 1, 4, None, None) == -1   # no problems
    assert _batched(lib, [ok], 0, 4) == -1                         # count out of range
    assert _batched(lib, [ok] * 9, 9, 4) == -1
    assert _batched(lib, [ok], 1, -1) == -1                        # negative M
    assert _batched(lib, [ok], 1, 129) == -2                       # above the decode range
    assert _batched(lib, [ok], 1, 0) == 0                          # empty M: nothing to do
    assert _batched(lib, [ok, m.GemmProblem(16, 16, 16, 16, 16, 16, 16, 256, 100)], 2, 4) == -2  # K % 64
    assert _batched(lib, [ok, m.GemmProblem(16, 16, 16, 0, 16, 16, 16, 256, 512)], 2, 4) == -1   # null b
    assert _batched(lib, [ok, m.GemmProblem(16, 16, 16, 24, 16, 16, 16, 256, 512)], 2, 4) == -3  # misaligned b


def test_grouped_swiglu_quantize_out_host_validation(lib):
    def call(N_gu, q=16, M=8):
        return lib.nvfp4_grouped_gemm_swiglu_quantize_out(P(16), P(16), P(16), P(16), P(16), P(16), P(16), 2, M, N_gu,
                                                          256, P(16), P(q), P(16), P(256), 1 << 20, None, None)
    assert call(136) == -2           # N_gu not a multiple of 128
    assert call(256, q=0) == -1      # no code output
    assert call(256, M=0) == 0       # no routed rows: nothing to do
