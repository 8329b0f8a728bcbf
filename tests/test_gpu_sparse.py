"""GPU parity of the pair-wise 2:4 sparse NVFP4 path against the oracle, through the C ABI:
pruning + compression and the 32-element-block quantiser bit for bit, the sparse GEMM
(tcgen05.mma.sp) within |y - y_ref| <= 4e-3 |y_ref| + 1e-5 sum_k |x^_k w^_k|."""
import numpy as np
import pytest
import torch

import moe_nvfp4_gemm_gb300 as m
import oracle
import synth
from tests.helpers import dev, scalar, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_tuning():
    yield
    for key in range(1, 16):
        m.nvfp4_tune(key, 0)


@pytest.mark.parametrize("N,K,std,seed", [(128, 512, 0.02, 1), (200, 640, 1.0, 2), (5, 128, 3.0, 3),
                                          (300, 1536, 0.5, 4)])
def test_prune_pairs_bit_exact(N, K, std, seed):
    wb = synth.normal_bf16((N, K), 50 + seed, std, 1e-2)
    c, meta = m.nvfp4_prune_pairs(to_dev(wb))
    torch.cuda.synchronize()
    c_o, meta_o = oracle.prune_pairs(wb)
    assert np.array_equal(c.view(torch.int16).cpu().numpy().view(np.uint16), c_o)
    assert np.array_equal(meta.cpu().numpy(), oracle.meta_tile(meta_o, N, K))


def test_prune_pairs_ties_bit_exact():
    rng = np.random.default_rng(9)
    vals = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, -3.0], dtype=np.float32)
    wb = synth.f32_to_bf16_bits(rng.choice(vals, size=(64, 1024)).astype(np.float32))
    c, meta = m.nvfp4_prune_pairs(to_dev(wb))
    torch.cuda.synchronize()
    c_o, meta_o = oracle.prune_pairs(wb)
    assert np.array_equal(c.view(torch.int16).cpu().numpy().view(np.uint16), c_o)
    assert np.array_equal(meta.cpu().numpy(), oracle.meta_tile(meta_o, 64, 1024))


@pytest.mark.parametrize("M,K,seed", [(128, 256, 0), (1, 128, 1), (333, 1152, 2), (4096, 8192, 3)])
def test_quantize_b32_bit_exact(M, K, seed):
    xb = synth.normal_bf16((M, K), 60 + seed, 1.0, 1e-3)
    x = to_dev(xb)
    amax, g = m.nvfp4_amax(x)
    q, sf = m.nvfp4_quantize_b32(x, g)
    torch.cuda.synchronize()
    qo, sfo, go = oracle.quantize_b32(xb)
    assert np.float32(g.item()) == go
    assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(sf.cpu().numpy(), sfo)


class Sparse:
    """Host operands from the oracle (so the GEMM is tested on its own) and device copies."""

    def __init__(self, M, N, K, seed, x_std=1.0, w_std=0.02):
        xb = synth.normal_bf16((M, K), 2 * seed, x_std, 1e-3)
        wb = synth.normal_bf16((N, K), 2 * seed + 1, w_std)
        self.M, self.N, self.K = M, N, K
        self.xq, self.xsf, self.gx = oracle.quantize_b32(xb)
        self.cq, self.csf, self.gw, self.meta = oracle.sparse_quantize_weight(wb)
        self.d = (to_dev(self.xq), to_dev(self.xsf), scalar(self.gx), to_dev(self.cq), to_dev(self.csf),
                  to_dev(oracle.meta_tile(self.meta, N, K)), scalar(self.gw))

    def run(self, status=None):
        y = m.nvfp4_sparse_gemm(*self.d, self.M, self.N, self.K, dev_status=status)
        torch.cuda.synchronize()
        return y

    def check(self, y, rows=None, cols=None):
        yr, ad = oracle.sparse_gemm(self.xq, self.xsf, self.gx, self.cq, self.csf, self.meta, self.gw,
                                    self.M, self.N, self.K, rows=rows, cols=cols)
        yg = y.float().cpu().numpy()
        if rows is not None:
            yg = yg[np.asarray(rows)]
        if cols is not None:
            yg = yg[:, np.asarray(cols)]
        ok, worst = oracle.within_tolerance(yg, yr, ad)
        assert ok, f"sparse parity failed: worst ratio {worst}"


@pytest.mark.parametrize("M,N,K", [(1, 128, 512), (16, 264, 1024), (77, 128, 640), (128, 384, 2048),
                                   (200, 136, 512), (3, 8, 128), (32, 512, 4096)])
def test_sparse_gemm_matches_oracle(M, N, K):
    g = Sparse(M, N, K, 70)
    g.check(g.run())


@pytest.mark.parametrize("split", [1, 2, 4, 8])
def test_sparse_gemm_split_k(split):
    g = Sparse(16, 256, 4096, 71)
    m.nvfp4_tune(m.NVFP4_TUNE_STREAM_SPLIT, split)
    g.check(g.run())


def test_sparse_gemm_status_untouched():
    g = Sparse(16, 128, 512, 72)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    g.check(g.run(st))
    assert st.item() == 0


def test_sparse_chain_on_the_gpu():
    # every step on the GPU: prune the bf16 weight, quantise its compressed values, quantise
    # the activations in 32-element blocks, multiply; checked against the oracle's chain
    M, N, K = 16, 384, 2048
    xb = synth.normal_bf16((M, K), 73, 1.0, 1e-3)
    wb = synth.normal_bf16((N, K), 74, 0.02)
    x, w = to_dev(xb), to_dev(wb)
    c, meta = m.nvfp4_prune_pairs(w)
    _, gw = m.nvfp4_amax(c)
    cq, csf = m.nvfp4_quantize(c, gw)
    _, gx = m.nvfp4_amax(x)
    xq, xsf = m.nvfp4_quantize_b32(x, gx)
    y = m.nvfp4_sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, M, N, K)
    torch.cuda.synchronize()
    cq_o, csf_o, gw_o, meta_o = oracle.sparse_quantize_weight(wb)
    xq_o, xsf_o, gx_o = oracle.quantize_b32(xb)
    assert np.array_equal(cq.cpu().numpy(), cq_o) and np.array_equal(csf.cpu().numpy(), csf_o)
    assert np.array_equal(xq.cpu().numpy(), xq_o) and np.array_equal(xsf.cpu().numpy(), xsf_o)
    assert np.float32(gw.item()) == gw_o and np.float32(gx.item()) == gx_o
    yr, ad = oracle.sparse_gemm(xq_o, xsf_o, gx_o, cq_o, csf_o, meta_o, gw_o, M, N, K)
    ok, worst = oracle.within_tolerance(y.float().cpu().numpy(), yr, ad)
    assert ok, worst


@pytest.mark.parametrize("M", [1, 16, 32])
def test_sparse_decode_full_size_sampled(M):
    # the decode workload's shape, N = K = 8192, x ~ N(0,1) + 0.1% x20, W ~ N(0, 0.02) pruned
    g = Sparse(M, 8192, 8192, 2)
    y = g.run()
    rng = np.random.default_rng(M)
    cols = np.concatenate([[0, 127, 128, 8191], rng.choice(8192, 252, replace=False)])
    g.check(y, cols=cols)


class GroupedSparse:
    def __init__(self, counts, N, K, seed, a_rows=None, w=None):
        E = len(counts)
        self.E, self.N, self.K = E, N, K
        self.off = np.zeros(E + 1, dtype=np.int32)
        self.off[1:] = np.cumsum(counts)
        self.Mt = int(self.off[-1])
        if a_rows is None:
            a_rows = synth.normal_bf16((max(self.Mt, 1), K), 2 * seed, 1.0)[: self.Mt]
        if w is None:
            w = lambda e: synth.moe_expert_weight(e, N, K, seed)
        self.xq, self.xsf, self.gx = oracle.quantize_b32(a_rows)
        ws = [oracle.sparse_quantize_weight(w(e)) for e in range(E)]
        self.cq = np.stack([t[0] for t in ws])
        self.csf = np.stack([t[1] for t in ws])
        self.gw = np.array([t[2] for t in ws], np.float32)
        self.meta = np.stack([t[3] for t in ws])
        self.meta_t = np.stack([oracle.meta_tile(self.meta[e], N, K) for e in range(E)])

    def run(self, status=None, offsets=None):
        off = self.off if offsets is None else offsets
        y = m.nvfp4_grouped_sparse_gemm(to_dev(self.xq), to_dev(self.xsf), scalar(self.gx), to_dev(self.cq),
                                        to_dev(self.csf), to_dev(self.meta_t), to_dev(self.gw), to_dev(off), self.E,
                                        self.Mt, self.N, self.K, dev_status=status)
        torch.cuda.synchronize()
        return y

    def check(self, y, rows=None, cols=None):
        yr, ad = oracle.grouped_sparse_gemm(self.xq, self.xsf, self.gx, self.cq, self.csf, self.meta, self.gw,
                                            self.off, self.E, self.Mt, self.N, self.K, rows=rows, cols=cols)
        yg = y.float().cpu().numpy()
        if rows is not None:
            yg = yg[np.asarray(rows)]
        if cols is not None:
            yg = yg[:, np.asarray(cols)]
        ok, worst = oracle.within_tolerance(yg, yr, ad)
        assert ok, f"grouped sparse parity failed: worst ratio {worst}"


@pytest.mark.parametrize("tile_rows", [0, 64])
@pytest.mark.parametrize("counts,N,K", [
    ((3, 0, 17, 1, 0, 9), 256, 512),
    ((64, 65, 63, 1, 127, 128, 129, 0), 136, 1024),
    ((0, 300, 0), 128, 640),
    ((5,), 8, 128),
])
def test_grouped_sparse_matches_oracle(counts, N, K, tile_rows):
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_TILE_ROWS, tile_rows)
    g = GroupedSparse(counts, N, K, 91)
    g.check(g.run())


def test_grouped_sparse_bad_offsets_reported():
    g = GroupedSparse((4, 4), 128, 512, 92)
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    g.run(status=st, offsets=np.array([0, 5, 4], dtype=np.int32))
    assert st.item() == -8


def test_grouped_sparse_moe_workload_sampled():
    # the MoE workload with pair-wise 2:4 sparse experts: 256 experts, 512 tokens top-8
    # (4096 routed rows), K = 6144, N = 4096
    a_rows, off, _ = synth.moe_tokens(512, 256, 8, 6144, 3)
    g = GroupedSparse(tuple(np.diff(off)), 4096, 6144, 3, a_rows=a_rows,
                      w=lambda e: synth.moe_expert_weight(e, 4096, 6144, 3))
    y = g.run()
    rng = np.random.default_rng(13)
    rows = np.concatenate([[0, g.Mt - 1], rng.choice(g.Mt, 22, replace=False)])
    cols = np.concatenate([[0, 127, 128, 4095], rng.choice(4096, 36, replace=False)])
    g.check(y, rows=rows, cols=cols)
