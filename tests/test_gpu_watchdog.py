"""The timeout path of the GEMM kernels, made to run out on purpose without faulting
anything: with a short watchdog limit (NVFP4_TUNE_WATCHDOG_US) the first CTA of the kernel
withholds one pipeline stage's loads (NVFP4_TUNE_TEST_WITHHOLD_STAGE), so that stage's
barrier never completes. Every wait is bounded: the CTA gives up, stops its other roles,
frees its tensor memory and writes NVFP4_ERR_TIMEOUT to dev_status, and its cluster peers
leave through their own bounded waits. The next ordinary call on the same context must
then produce the oracle's result."""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
from tests.helpers import check_gemm, dense_case, dev
from tests.test_gpu_grouped import Grouped

pytestmark = pytest.mark.gpu

TIMEOUT = -7
LIMIT_US = 20_000  # 20 ms


@pytest.fixture(autouse=True)
def _reset_tuning():
    yield
    for key in range(1, 16):
        m.nvfp4_tune(key, 0)
    torch.cuda.synchronize()


def _timed_out_then_recovers(run, check, stage):
    m.nvfp4_tune(m.NVFP4_TUNE_WATCHDOG_US, LIMIT_US)
    m.nvfp4_tune(m.NVFP4_TUNE_TEST_WITHHOLD_STAGE, stage)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    run(st)
    torch.cuda.synchronize()
    assert st.item() == TIMEOUT, f"expected NVFP4_ERR_TIMEOUT, got {st.item()}"
    m.nvfp4_tune(m.NVFP4_TUNE_TEST_WITHHOLD_STAGE, 0)
    st.zero_()
    y = run(st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check(y)


# (kernel selection, M): the single-CTA tile kernel, the CTA-pair kernel, the weight-streaming
# kernel alone and in split-K clusters of 4 (whose owners wait for every peer's partials);
# the sparse variant of the streaming kernel and the grouped kernel below
DENSE_FAMILIES = {
    "tile_single_cta": (dict(STREAM_MAX_M=-1, DENSE_KERNEL=1), 256),
    "tile_cta_pair": (dict(STREAM_MAX_M=-1, DENSE_KERNEL=2), 256),
    "stream_split1": (dict(STREAM_SPLIT=1), 16),
    "stream_split4": (dict(STREAM_SPLIT=4), 16),
}


@pytest.mark.parametrize("family", list(DENSE_FAMILIES))
@pytest.mark.parametrize("stage", [1, 2])
def test_dense_kernels_time_out_cleanly_and_recover(family, stage):
    tune, M = DENSE_FAMILIES[family]
    A, B = dense_case(M, 512, 2048, 41, 1.0, 1e-3, 0.02)

    def run(st):
        for k, v in tune.items():
            m.nvfp4_tune(getattr(m, "NVFP4_TUNE_" + k), v)
        return m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, M, 512, 2048, dev_status=st)

    _timed_out_then_recovers(run, lambda y: check_gemm(y, A, B), stage)


@pytest.mark.parametrize("stage", [1, 2])
def test_sparse_kernel_times_out_cleanly_and_recovers(stage):
    from tests.test_gpu_sparse import Sparse
    g = Sparse(16, 256, 4096, 44)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, 4)
    _timed_out_then_recovers(lambda st: g.run(status=st), g.check, stage)


@pytest.mark.parametrize("stage", [1, 3])
def test_grouped_kernel_times_out_cleanly_and_recovers(stage):
    g = Grouped((20, 0, 70, 5), 256, 1024, 42)
    _timed_out_then_recovers(lambda st: g.run(status=st), g.check, stage)


@pytest.mark.parametrize("stage", [1, 2])
def test_batched_kernel_times_out_cleanly_and_recovers(stage):
    # the first CTA of every problem in the launch withholds the stage (a problem with fewer
    # stages per CTA withholds nothing); split-K clusters of 4
    from tests.test_gpu_batched import _problems
    M = 16
    probs = _problems(M, [(512, 2048), (256, 1024)], 45)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, 4)

    def run(st):
        ys = [torch.empty((M, B.rows), dtype=torch.bfloat16, device=dev()) for _, B in probs]
        m.nvfp4_gemm_batched([(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, y) for (A, B), y in zip(probs, ys)], M,
                             dev_status=st)
        return ys

    def check(ys):
        for (A, B), y in zip(probs, ys):
            check_gemm(y, A, B)

    _timed_out_then_recovers(run, check, stage)


def test_default_limit_is_restored():
    # with the hook off and the limit back at its default an ordinary call succeeds
    A, B = dense_case(128, 256, 512, 43)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    y = m.nvfp4_gemm(A.dq, A.dsf, A.dg, B.dq, B.dsf, B.dg, 128, 256, 512, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    check_gemm(y, A, B)
