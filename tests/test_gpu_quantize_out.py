"""GPU check of the GEMM whose epilogue emits NVFP4 (nvfp4_gemm_quantize_out): its
codes and tiled scales must equal the oracle's quantisation of the bf16 values the
plain GEMM returns for the same operands, bit for bit, and those values must agree
with the oracle's GEMM within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
import oracle
from tests.helpers import check_gemm, dense_case, dev, scalar

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_MAX_M, -1)  # the plain GEMM takes the same CTA-pair kernel
    yield
    for key in range(1, 16):
        m.nvfp4_tune(key, 0)


def _bits(y):
    return y.cpu().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,N,K,g_mode", [
    (256, 256, 256, "amax"),
    (300, 320, 512, "amax"),       # ragged rows (scale padding rows 300..383 zero), N not a multiple of 256
    (129, 1024, 1024, "pow2"),     # power-of-two global scale
    (520, 576, 1344, "small"),     # small global scale: many blocks saturate at 448 / 6
    (64, 192, 256, "amax"),        # fewer rows than one tile
])
def test_quantized_output_equals_quantize_of_plain_output(M, N, K, g_mode):
    A, B = dense_case(M, N, K, 51, 1.0, 1e-3, 0.05)
    y = m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, M, N, K)
    torch.cuda.synchronize()
    check_gemm(y, A, B)
    yb = _bits(y)
    if g_mode == "amax":
        g = oracle.global_scale(oracle.amax(yb))
    elif g_mode == "pow2":
        g = np.float32(2.0 ** -7)
    else:
        g = np.float32(oracle.global_scale(oracle.amax(yb)) / 64)
    q_ref, sf_ref, _ = oracle.quantize(yb, np.float32(g))
    q, sf = m.nvfp4_gemm_quantize_out(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, scalar(np.float32(g)), M, N, K)
    torch.cuda.synchronize()
    qg, sfg = q.cpu().numpy(), sf.cpu().numpy()
    bad = np.argwhere(qg != q_ref)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"
    assert np.array_equal(sfg, sf_ref)


def test_quantized_output_rejects_n_not_multiple_of_64():
    A, B = dense_case(128, 136, 256, 52)
    with pytest.raises(m.NVFP4Error):
        m.nvfp4_gemm_quantize_out(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, scalar(np.float32(1.0)), 128, 136, 256)


def test_chained_layers_keep_stream_order():
    # layer 1 emits NVFP4 that layer 2 reads as its activations, back to back in one CUDA
    # graph (both launches overlap their set-up with the previous kernel): the result must
    # equal the same chain run with a synchronisation between the layers, and writing the
    # same output twice must leave the last call's values
    A, B1 = dense_case(512, 512, 1024, 53, 1.0, 1e-3, 0.05)
    _, B2 = dense_case(512, 768, 512, 54, 1.0, 1e-3, 0.05)
    g1 = scalar(np.float32(2.0 ** -5))
    q1, sf1 = m.nvfp4_gemm_quantize_out(A.dq, A.dsf, A.dg, B1.dq, B1.dsf, B1.dg, g1, 512, 512, 1024)
    torch.cuda.synchronize()
    ref = m.nvfp4_gemm(q1, sf1, g1, B2.dq, B2.dsf, B2.dg, 512, 768, 512).clone()
    torch.cuda.synchronize()
    q = torch.empty_like(q1)
    sf = torch.empty_like(sf1)
    y = torch.empty_like(ref)
    y_other = torch.empty_like(ref)
    y_mid = torch.empty((512, 512), dtype=torch.bfloat16, device=dev())

    def chain():
        m.nvfp4_gemm_quantize_out(A.dq, A.dsf, A.dg, B1.dq, B1.dsf, B1.dg, g1, 512, 512, 1024, q_out=q, sf_out=sf)
        m.nvfp4_gemm(q, sf, g1, B2.dq, B2.dsf, B2.dg, 512, 768, 512, y=y_other)  # overwritten next
        m.nvfp4_gemm(A.dq, A.dsf, A.dg, B1.dq, B1.dsf, B1.dg, 512, 512, 1024, y=y_mid)
        m.nvfp4_gemm(q, sf, g1, B2.dq, B2.dsf, B2.dg, 512, 768, 512, y=y)

    chain()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    q.zero_()
    y.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(q, q1) and torch.equal(sf, sf1)
    assert torch.equal(y, ref)
