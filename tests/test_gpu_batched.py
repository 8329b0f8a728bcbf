"""GPU parity of the batched decode GEMM (nvfp4_gemm_batched): several independent
problems sharing M, each with its own operands, N and K, in one launch. Every problem's
output is compared with the oracle's GEMM of that problem, element by element:
|y - y_ref| <= 4e-3 |y_ref| + 1e-5 sum_k |x^_k w^_k| ("NVFP4 linear layer", kernelindex,
operation header: y = x @ W^T per problem)."""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
from tests.helpers import Operand, check_gemm, dev
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    yield
    for key in range(1, 16):
        m.nvfp4_tune(key, 0)


def _problems(M, shapes, seed):
    out = []
    for i, (N, K) in enumerate(shapes):
        x, w = synth.dense_inputs(M, N, K, seed + i, 1.0, 1e-3, 0.02)
        out.append((Operand(x), Operand(w)))
    return out


def _run(M, probs, status=None):
    ys = [torch.full((M, B.rows), float("nan"), dtype=torch.bfloat16, device=dev()) for _, B in probs]
    m.nvfp4_gemm_batched([(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, y) for (A, B), y in zip(probs, ys)], M,
                         dev_status=status)
    torch.cuda.synchronize()
    return ys


MIXED = [(256, 512), (136, 1088), (512, 2048), (8, 64), (1032, 192)]


@pytest.mark.parametrize("M", [1, 5, 16, 33, 128])
def test_batched_mixed_shapes_match_oracle(M):
    # N from one partial 128-row weight tile to several with a ragged last one, K from one
    # partial stage to several; every output element is written (the outputs start as NaN)
    probs = _problems(M, MIXED, 100)
    for (A, B), y in zip(probs, _run(M, probs)):
        check_gemm(y, A, B)


@pytest.mark.parametrize("split", [1, 2, 4])
def test_batched_equals_single_calls_with_the_same_split(split):
    # the same kernel body on the same tiles: bit for bit what single calls give when both
    # use one split-K cluster size
    M = 16
    probs = _problems(M, [(384, 1024), (128, 2048), (640, 512)], 200)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, split)
    ys = _run(M, probs)
    for (A, B), y in zip(probs, ys):
        y1 = m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, M, B.rows, A.K)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y1.view(torch.int16))
        check_gemm(y, A, B)


def test_batched_eight_problems_and_status_untouched():
    M = 32
    probs = _problems(M, [(512 + 128 * i, 1024 + 256 * (i % 3)) for i in range(m.NVFP4_MAX_BATCH)], 300)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    for (A, B), y in zip(probs, _run(M, probs, st)):
        check_gemm(y, A, B)
    assert st.item() == 0


def test_batched_rejects_bad_batches():
    M = 4
    (A, B), = _problems(M, [(128, 256)], 400)
    y = torch.empty((M, 128), dtype=torch.bfloat16, device=dev())
    one = (A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, y)
    with pytest.raises(m.NVFP4Error) as e:
        m.nvfp4_gemm_batched([one] * (m.NVFP4_MAX_BATCH + 1), M)
    assert e.value.status == -1
    with pytest.raises(m.NVFP4Error) as e:
        m.nvfp4_gemm_batched([one], 129)
    assert e.value.status == -2


def test_batched_decode_workload_sampled():
    # four N = K = 8192 problems at M = 16 (the decode workload's shape), sampled on
    # every 128-row weight tile's first and last rows
    M, SQ = 16, 8192
    probs = _problems(M, [(SQ, SQ)] * 4, 500)
    cols = np.unique(np.concatenate([np.arange(0, SQ, 128), np.arange(127, SQ, 128)]))
    for (A, B), y in zip(probs, _run(M, probs)):
        check_gemm(y, A, B, cols=cols)


@pytest.mark.parametrize("pdl", [1, 2, -1])
def test_batched_launches_keep_stream_order(pdl):
    # Back-to-back batched launches inside one CUDA graph (1: weights requested before the
    # launch dependency, 2: set-up overlap only, the default; -1: plain stream order),
    # alternating between two sets of problems that all write the same outputs: every
    # output write is ordered after the previous launch's, so the last launch's results win,
    # and a launch writing its own outputs gets exactly its own results.
    M = 16
    p1 = _problems(M, [(256, 1024), (384, 512)], 600)
    p2 = _problems(M, [(256, 1024), (384, 512)], 700)
    m.nvfp4_tune(m.NVFP4_TUNE_PDL, -1)
    r1 = [y.clone() for y in _run(M, p1)]
    r2 = [y.clone() for y in _run(M, p2)]
    m.nvfp4_tune(m.NVFP4_TUNE_PDL, pdl)
    shared = [torch.empty_like(r) for r in r1]
    own = [[torch.empty_like(r) for r in r1] for _ in range(5)]

    def launch(probs, ys):
        m.nvfp4_gemm_batched([(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, y) for (A, B), y in zip(probs, ys)], M)

    sets = [p1, p2, p1, p2, p1]
    for probs in sets[:2]:  # warm up outside capture
        launch(probs, shared)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for probs, ys in zip(sets, own):
            launch(probs, ys)
        for probs in sets:
            launch(probs, shared)
    for y in shared:
        y.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for i, ys in enumerate(own):
        ref = r1 if i % 2 == 0 else r2
        for y, r in zip(ys, ref):
            assert torch.equal(y.view(torch.int16), r.view(torch.int16)), i
    for y, r in zip(shared, r1):
        assert torch.equal(y.view(torch.int16), r.view(torch.int16))
