"""The second half of the fused MoE step, through the C ABI: the gate/up projection with
SwiGLU fused into its epilogue, the global amax and block quantisation of its bf16 output
on the GPU, then the down-projection grouped GEMM over the same routing ("The Moment of
Synthesis", magik.net, Reasoning: a fused 2048 x 2 gate+up projection feeding a K = 2048
down projection). Each link is checked against the oracle: the SwiGLU output within its
propagated tolerance, the quantised codes and scales bit for bit (the oracle's quantiser
applied to the GPU's own bf16 output), the down projection within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
import oracle
import synth
from tests.helpers import scalar, to_dev

pytestmark = pytest.mark.gpu


def _experts(E, N, K, seed):
    qs, ss, gs = zip(*[oracle.quantize(synth.moe_expert_weight(e, N, K, seed)) for e in range(E)])
    return np.stack(qs), np.stack(ss), np.array(gs, np.float32)


def _chain(a_rows, off, N_gu, K, N_down, seed, rows=None, cols=None):
    E = len(off) - 1
    Mt = int(off[-1])
    I = N_gu // 2
    qa, sfa, ga = oracle.quantize(a_rows)
    qgu, sgu, ggu = _experts(E, N_gu, K, seed)
    qdn, sdn, gdn = _experts(E, N_down, I, seed + 50)
    off_d = to_dev(off.astype(np.int32))
    # 1. gate/up projection with SwiGLU in the epilogue
    y_act = m.nvfp4_grouped_gemm_swiglu(to_dev(qa), to_dev(sfa), scalar(ga), to_dev(qgu), to_dev(sgu),
                                        to_dev(ggu), off_d, E, Mt, N_gu, K)
    # 2. global amax and block quantisation of the activation on the GPU
    amax, g_act = m.nvfp4_amax(y_act)
    q_act, sf_act = m.nvfp4_quantize(y_act, g_act)
    # 3. down projection over the same routing, K = I
    y_down = m.nvfp4_grouped_gemm(q_act, sf_act, g_act, to_dev(qdn), to_dev(sdn), to_dev(gdn), off_d, E, Mt,
                                  N_down, I)
    torch.cuda.synchronize()

    act_bits = y_act.view(torch.int16).cpu().numpy().view(np.uint16)
    r = np.arange(Mt) if rows is None else np.asarray(rows)
    c_act = np.arange(I) if cols is None else np.asarray(cols) % I
    yr, gate, up, adg, adu = oracle.grouped_gemm_swiglu(qa, sfa, ga, qgu, sgu, ggu, off, E, Mt, N_gu, K,
                                                        rows=r, cols=c_act)
    ok, worst = oracle.within_tolerance_swiglu(synth.bf16_bits_to_f32(act_bits[np.ix_(r, c_act)]), gate, up,
                                               adg, adu)
    assert ok, f"SwiGLU output outside tolerance: worst ratio {worst}"
    q_o, sf_o, g_o = oracle.quantize(act_bits)
    assert np.float32(g_act.item()) == g_o
    assert np.array_equal(q_act.cpu().numpy(), q_o) and np.array_equal(sf_act.cpu().numpy(), sf_o)
    c_dn = np.arange(N_down) if cols is None else np.asarray(cols)
    yd, ad = oracle.grouped_gemm(q_o, sf_o, g_o, qdn, sdn, gdn, off, E, Mt, N_down, I, rows=r, cols=c_dn)
    ok, worst = oracle.within_tolerance(y_down.float().cpu().numpy()[np.ix_(r, c_dn)], yd, ad)
    assert ok, f"down projection outside tolerance: worst ratio {worst}"


@pytest.mark.parametrize("counts,N_gu,K,N_down", [
    ((5, 0, 17, 64, 65, 3), 512, 512, 384),   # ragged counts, an empty expert, K_down = 256
    ((40, 130), 128, 1024, 136),             # K_down = 64 (one MMA step), N_down not a multiple of 128
])
def test_moe_gate_up_swiglu_quantize_down_chain(counts, N_gu, K, N_down):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    a_rows = synth.normal_bf16((int(off[-1]), K), 71, 1.0, 1e-3)
    _chain(a_rows, off, N_gu, K, N_down, 72)


def test_moe_down_projection_workload_shape_sampled():
    # the MoE workload's routing (512 tokens top-8 over 256 experts, 4096 rows): gate/up
    # K = 6144, N_gu = 4096 (I = 2048), then the down projection K = 2048 -> N = 6144
    a_rows, off, _ = synth.moe_tokens(512, 256, 8, 6144, 3)
    rng = np.random.default_rng(9)
    rows = np.concatenate([[0, int(off[-1]) - 1], rng.choice(int(off[-1]), 22, replace=False)])
    cols = np.concatenate([[0, 2047, 2048, 6143], rng.choice(6144, 36, replace=False)])
    _chain(a_rows, off, 4096, 6144, 6144, 3, rows=rows, cols=cols)
