"""The allocation-free grouped GEMM (nvfp4_grouped_gemm_noalloc).

It serves callers that cannot allocate device memory where they run the MoE layer
(runtimes with a fixed memory budget and no allocator, plugins that must not use the
host program's allocator): instead of a caller-provided workspace it uses a fixed
scratch array built into the library. These checks call it through the C ABI twice
in a row, on two different problems so that the second call runs on the scratch the
first one left behind. Both entry points run the same kernels on the same inputs, so
each result must equal the ordinary entry point's bit for bit; it must also lie
within the oracle's GEMM tolerance |y - y_ref| <= 4e-3 |y_ref| + 1e-5 sum_k |x^_k w^_k|.
This file is named to be collected last so that a run stopping at the first failure
has run everything else; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
import oracle
import synth
from tests.helpers import dev, scalar, to_dev

pytestmark = pytest.mark.gpu


def _problem(counts, N, K, seed):
    E = len(counts)
    off = np.zeros(E + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    Mt = int(off[-1])
    qa, sfa, ga = oracle.quantize(synth.normal_bf16((Mt, K), 2 * seed, 1.0))
    qs, ss, gs = zip(*[oracle.quantize(synth.moe_expert_weight(e, N, K, seed)) for e in range(E)])
    host = dict(qa=qa, sfa=sfa, ga=ga, qb=np.stack(qs), sfb=np.stack(ss), gb=np.array(gs, np.float32),
                off=off, E=E, Mt=Mt, N=N, K=K)
    devs = (to_dev(qa), to_dev(sfa), scalar(ga), to_dev(host["qb"]), to_dev(host["sfb"]),
            to_dev(host["gb"]), to_dev(off))
    return host, devs


def _close(y, y_ref, absdot):
    err = np.abs(y - y_ref)
    return bool(np.all(err <= 4e-3 * np.abs(y_ref) + 1e-5 * absdot))


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    problems = [_problem((9, 0, 70, 1, 33), 384, 768, 41), _problem((2, 130, 17), 256, 1088, 42)]
    for host, devs in problems:
        E, Mt, N, K = host["E"], host["Mt"], host["N"], host["K"]
        st = torch.zeros(1, dtype=torch.int32, device=dev())
        y_noalloc = m.nvfp4_grouped_gemm_noalloc(*devs, E, Mt, N, K, dev_status=st)
        y_ws = m.nvfp4_grouped_gemm(*devs, E, Mt, N, K)
        torch.cuda.synchronize()
        assert st.item() == 0
        yr, ad = oracle.grouped_gemm(host["qa"], host["sfa"], host["ga"], host["qb"], host["sfb"],
                                     host["gb"], host["off"], E, Mt, N, K)
        assert torch.equal(y_noalloc.view(torch.int16), y_ws.view(torch.int16)), \
            "allocation-free result differs from the workspace entry point"
        assert _close(y_noalloc.float().cpu().numpy(), yr, ad), "allocation-free result outside the oracle tolerance"


def test_noalloc_rejects_problems_larger_than_its_scratch():
    E, Mt, N, K = 256, 4096, 4096, 65536  # needs far more than the 16 MiB scratch
    need = m.nvfp4_grouped_gemm_workspace_bytes(E, Mt, N, K)
    assert need > m.NVFP4_NOALLOC_SCRATCH_BYTES
    t = torch.zeros(16, dtype=torch.uint8, device=dev())
    g = torch.ones(1, dtype=torch.float32, device=dev())
    off = torch.zeros(E + 1, dtype=torch.int32, device=dev())
    y = torch.empty(16, dtype=torch.bfloat16, device=dev())
    with pytest.raises(m.NVFP4Error) as ei:
        m.nvfp4_grouped_gemm_noalloc(t, t, g, t, t, g, off, E, Mt, N, K, y=y)
    assert ei.value.status == -6  # NVFP4_ERR_WORKSPACE
