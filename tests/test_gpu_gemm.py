"""GPU parity of the dense NVFP4 GEMM (tile kernel and weight-streaming kernel)
against the oracle, element by element, through the C ABI.

Tolerance (per element): |y - y_ref| <= 4e-3 |y_ref| + 1e-5 sum_k |x^_k w^_k|.
"""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
import oracle
import synth
from tests.helpers import Operand, check_gemm, dense_case, dev, scalar, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    yield
    for key in range(1, 16):
        m.nvfp4_tune(key, 0)


def _run(A, B, status=None):
    y = m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, A.rows, B.rows, A.K, dev_status=status)
    torch.cuda.synchronize()
    return y


def test_tiny_workload_both_kernels():
    # 128 x 128 x 256, x and W ~ N(0, 1), seed 0
    A, B = dense_case(128, 128, 256, 0)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, -1)
    check_gemm(_run(A, B), A, B)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, 128)
    check_gemm(_run(A, B), A, B)


TILE_KERNELS = [(1, 128), (1, 256), (2, 0)]  # (single-CTA, BN) and the CTA-pair 256 x 256 kernel


@pytest.mark.parametrize("kernel,bn", TILE_KERNELS)
@pytest.mark.parametrize("M,N,K", [
    (256, 256, 256), (300, 264, 320), (129, 512, 1024), (1000, 136, 576), (384, 768, 2048),
    (520, 1032, 1344)])
def test_tile_kernel_shapes(kernel, bn, M, N, K):
    A, B = dense_case(M, N, K, 11, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, -1)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_KERNEL, kernel)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_BN, bn)
    check_gemm(_run(A, B), A, B)


@pytest.mark.parametrize("kernel,grid", [(1, 3), (2, 6)])
def test_tile_kernel_persistent_loop_small_grid(kernel, grid):
    # fewer CTAs than tiles: every CTA walks several tiles through the TMEM handoff
    A, B = dense_case(640, 1024, 512, 12, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, -1)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_KERNEL, kernel)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_GRID, grid)
    check_gemm(_run(A, B), A, B)


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("raster", [-1, 3, 64])
def test_tile_kernel_raster_orders(kernel, raster):
    # every tile order (n fastest, bands of 3 m-blocks with a ragged last band, one band)
    # visits each output tile exactly once
    A, B = dense_case(1800, 1288, 512, 17, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, -1)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_KERNEL, kernel)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_GRID, 10)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_RASTER, raster)
    check_gemm(_run(A, B), A, B)


@pytest.mark.parametrize("split", [1, 2, 4, 8])
@pytest.mark.parametrize("M,N,K", [(1, 256, 2048), (16, 384, 2048), (32, 128, 4096), (77, 264, 1088),
                                   (128, 512, 512)])
def test_stream_kernel_shapes(split, M, N, K):
    A, B = dense_case(M, N, K, 13, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, split)
    check_gemm(_run(A, B), A, B)


def test_identity_gives_exact_weights():
    K = 256
    M, N = 128, 256
    codes = np.zeros((M, K), dtype=np.uint8)
    codes[np.arange(M), np.arange(M)] = 0x2
    A = Operand(synth.f32_to_bf16_bits(np.eye(M, K, dtype=np.float32)))
    B = Operand(synth.normal_bf16((N, K), 5, 0.02))
    for max_m, kernel in ((-1, 1), (-1, 2), (128, 0)):
        m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, max_m)
        m.nvfp4_tune(m.NVFP4_TUNE_DENSE_KERNEL, kernel)
        y = _run(A, B)
        ref, _ = oracle.gemm(A.q, A.sf, A.g, B.q, B.sf, B.g, M, N, K)
        ref_bf16 = synth.f32_to_bf16_bits(ref.astype(np.float32))
        got = y.view(torch.int16).cpu().numpy().view(np.uint16)
        # ref values are short dyadics (exact in fp32), so bf16 rounding is unique
        assert np.array_equal(got, ref_bf16)


@pytest.mark.parametrize("M", [1, 16, 32])
def test_decode_workload_full_size(M):
    # N = K = 8192, x ~ N(0,1) + 0.1% x20, W ~ N(0, 0.02); all rows, sampled columns
    A, B = dense_case(M, 8192, 8192, 2, 1.0, 1e-3, 0.02)
    y = _run(A, B)
    cols = np.random.default_rng(M).choice(8192, 512, replace=False)
    check_gemm(y, A, B, cols=cols)


def _every_tile_sample(M, N, seed):
    """Rows: one random row in every 32-row group (each TMEM lane quarter of each CTA of
    every 256-row tile, random lanes); columns: one random column in every 64-column group
    (each column half of every 256-column tile and both 64-column store boxes in it)."""
    rng = np.random.default_rng(seed)
    rows = np.arange(0, M, 32) + rng.integers(0, 32, (M + 31) // 32)
    cols = np.arange(0, N, 64) + rng.integers(0, 64, (N + 63) // 64)
    rows = np.unique(np.concatenate([np.minimum(rows, M - 1), [0, M - 1]]))
    cols = np.unique(np.concatenate([np.minimum(cols, N - 1), [0, N - 1]]))
    return rows, cols


def test_square_workload_sampled():
    # M = N = K = 8192 in the benchmark's launch configuration; a sample that reaches every
    # 256 x 256 tile, every epilogue warp's rows and every output store box
    A, B = dense_case(8192, 8192, 8192, 1, 1.0, 1e-3, 0.02)
    y = _run(A, B)
    rows, cols = _every_tile_sample(8192, 8192, 0)
    check_gemm(y, A, B, rows=rows, cols=cols)
    # properties at full size: finite everywhere
    assert torch.isfinite(y.float()).all()


def test_prefill_workload_sampled():
    # prefill GEMM in the benchmark's configuration: x 4096 x 8192 (N(0,1) + 0.1% x20, seed 8)
    # against W 28672 x 8192 (N(0, 0.02), seed 9); 1792 tiles of 256 x 256, 23.6 per CTA pair;
    # the sample reaches every tile, epilogue warp and store box
    A = Operand(synth.normal_bf16((4096, 8192), 8, 1.0, 1e-3))
    B = Operand(synth.normal_bf16((28672, 8192), 9, 0.02))
    y = _run(A, B)
    rows, cols = _every_tile_sample(4096, 28672, 4)
    check_gemm(y, A, B, rows=rows, cols=cols)
    assert torch.isfinite(y.float()).all()


# The smallest shapes the library accepts: K of one to three 64-element MMA steps (one
# partial 256-element stage), N below one 128-row weight tile or one 64-column store box.
SMALL_K = [64, 128, 192]
SMALL_N = [8, 16, 72, 120]


@pytest.mark.parametrize("K", SMALL_K)
@pytest.mark.parametrize("N", SMALL_N)
@pytest.mark.parametrize("kernel,bn", TILE_KERNELS)
@pytest.mark.parametrize("M", [1, 16, 200])
def test_tile_kernels_smallest_shapes(M, kernel, bn, N, K):
    A, B = dense_case(M, N, K, 15, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, -1)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_KERNEL, kernel)
    m.nvfp4_tune(m.NVFP4_TUNE_DENSE_BN, bn)
    check_gemm(_run(A, B), A, B)


@pytest.mark.parametrize("K", SMALL_K)
@pytest.mark.parametrize("N", SMALL_N)
@pytest.mark.parametrize("M,split", [(1, 0), (16, 0), (16, 3), (77, 1)])
def test_stream_kernel_smallest_shapes(M, split, N, K):
    A, B = dense_case(M, N, K, 16, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, split)
    check_gemm(_run(A, B), A, B)


@pytest.mark.parametrize("M,N,K,max_m", [
    (256, 512, 65536, -1),    # CTA-pair kernel, 256 K blocks per tile
    (32, 384, 131072, 128),   # streaming kernel, split-K clusters over 512 K blocks
    (128, 256, 32768, 128),   # the largest M the streaming kernel takes
])
def test_long_k_sampled(M, N, K, max_m):
    A, B = dense_case(M, N, K, 14, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, max_m)
    y = _run(A, B)
    cols = np.random.default_rng(K).choice(N, 48, replace=False)
    check_gemm(y, A, B, cols=cols)


def test_status_untouched_on_success():
    A, B = dense_case(64, 128, 256, 3)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    _run(A, B, st)
    assert st.item() == 0


def test_empty_m_is_noop():
    A, B = dense_case(1, 128, 256, 4)
    y = torch.full((0, 128), 7.0, dtype=torch.bfloat16, device=dev())
    m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, 0, 128, 256, y=y)


@pytest.mark.parametrize("M,split", [(1, 0), (16, 4), (77, 1)])
def test_weights_kept_in_l2_give_identical_results(M, split):
    # the weight loads' L2 priority (evict_first or evict_last) changes no arithmetic
    A, B = dense_case(M, 384, 2048, 33, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, split)
    streamed = _run(A, B).clone()
    m.nvfp4_tune(m.NVFP4_TUNE_WEIGHT_L2, 1)
    kept = _run(A, B)
    assert torch.equal(kept.view(torch.int16), streamed.view(torch.int16))
    check_gemm(kept, A, B)


@pytest.mark.parametrize("prefetch", [0, 3, -1])
def test_l2_prefetch_sees_weights_the_previous_kernel_wrote(prefetch):
    # A decode call prefetches its weight slice into L2 before it waits for the previous
    # kernel in the stream (0: all of it, the default; 3: three K blocks; -1: none). Here the
    # previous kernel is the quantiser writing the call's weights into the same buffers,
    # alternating between two matrices inside one CUDA graph: each call must see the matrix
    # quantised just before it, bit for bit as outside the graph.
    M, N, K = 16, 512, 2048
    x1, w1 = synth.dense_inputs(M, N, K, 51, 1.0, 1e-3, 0.02)
    _, w2 = synth.dense_inputs(M, N, K, 52, 1.0, 1e-3, 0.02)
    A, B1, B2 = Operand(x1), Operand(w1), Operand(w2)
    wdev = [to_dev(w1), to_dev(w2)]
    gs = [B1.dg, B2.dg]
    wq = torch.empty_like(B1.dq)
    sfw = torch.empty_like(B1.dsf)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_L2_PREFETCH, prefetch)

    def step(j, out):
        m.nvfp4_quantize(wdev[j], gs[j], q_out=wq, sf_out=sfw)
        m.nvfp4_gemm(A.dq, A.dsf, A.dg, wq, sfw, gs[j], M, N, K, y=out)

    refs = []
    for j in range(2):
        r = torch.empty((M, N), dtype=torch.bfloat16, device=dev())
        step(j, r)
        torch.cuda.synchronize()
        assert torch.equal(wq, (B1, B2)[j].dq) and torch.equal(sfw, (B1, B2)[j].dsf)
        refs.append(r)
    check_gemm(refs[0], A, B1)
    check_gemm(refs[1], A, B2)
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device=dev()) for _ in range(8)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i, o in enumerate(outs):
            step(i % 2, o)
    g.replay()
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o.view(torch.int16), refs[i % 2].view(torch.int16)), i


@pytest.mark.parametrize("pdl", [1, 2, -1])
def test_programmatic_dependent_launch_keeps_stream_order(pdl):
    # Back-to-back decode calls with programmatic dependent launch inside one CUDA graph
    # (1: weights requested before the dependency wait, 2: set-up overlap only, the
    # default; -1: plain stream order),
    # alternating between two problems: (1) each writing its own output must produce the
    # problem's own result; (2) all writing the same output, the last call's result must
    # win (every output write is ordered after the previous call's completion).
    A1, B1 = dense_case(16, 512, 1024, 31, 1.0, 1e-3, 0.02)
    A2, B2 = dense_case(16, 512, 1024, 32, 1.0, 1e-3, 0.02)
    m.nvfp4_tune(m.NVFP4_TUNE_PDL, -1)
    ref1 = _run(A1, B1).clone()
    ref2 = _run(A2, B2).clone()
    m.nvfp4_tune(m.NVFP4_TUNE_PDL, pdl)
    calls = [(A1, B1), (A2, B2)] * 4 + [(A1, B1)]
    outs = [torch.empty_like(ref1) for _ in calls]
    y = torch.empty_like(ref1)
    gemm = lambda A, B, out: m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, 16, 512, 1024, y=out)
    for A, B in calls[:2]:  # warm up outside capture
        gemm(A, B, y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for (A, B), o in zip(calls, outs):
            gemm(A, B, o)
        for A, B in calls:
            gemm(A, B, y)
    y.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, ref1 if i % 2 == 0 else ref2), i
    assert torch.equal(y, ref1)
