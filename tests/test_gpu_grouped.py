"""GPU parity of the grouped (MoE) NVFP4 GEMM against the oracle, through the C ABI."""
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


class Grouped:
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
        self.qa, self.sfa, self.ga = oracle.quantize(a_rows) if self.Mt else (None, None, 1.0)
        sfb_bytes = oracle.scale_bytes(N, K)
        self.qb = np.empty((E, N, K // 2), dtype=np.uint8)
        self.sfb = np.empty((E, sfb_bytes), dtype=np.uint8)
        self.gb = np.empty(E, dtype=np.float32)
        for e in range(E):
            self.qb[e], self.sfb[e], self.gb[e] = oracle.quantize(w(e))

    def run(self, status=None, offsets=None):
        off = self.off if offsets is None else offsets
        y = m.nvfp4_grouped_gemm(to_dev(self.qa), to_dev(self.sfa), scalar(self.ga), to_dev(self.qb),
                                 to_dev(self.sfb), to_dev(self.gb), to_dev(off), self.E, self.Mt,
                                 self.N, self.K, dev_status=status)
        torch.cuda.synchronize()
        return y

    def run_swiglu(self):
        y = m.nvfp4_grouped_gemm_swiglu(to_dev(self.qa), to_dev(self.sfa), scalar(self.ga), to_dev(self.qb),
                                        to_dev(self.sfb), to_dev(self.gb), to_dev(self.off), self.E, self.Mt,
                                        self.N, self.K)
        torch.cuda.synchronize()
        return y

    def check_swiglu(self, y, rows=None, cols=None):
        yr, gate, up, adg, adu = oracle.grouped_gemm_swiglu(self.qa, self.sfa, self.ga, self.qb, self.sfb,
                                                            self.gb, self.off, self.E, self.Mt, self.N, self.K,
                                                            rows=rows, cols=cols)
        yg = y.float().cpu().numpy()
        if rows is not None:
            yg = yg[np.asarray(rows)]
        if cols is not None:
            yg = yg[:, np.asarray(cols)]
        ok, worst = oracle.within_tolerance_swiglu(yg, gate, up, adg, adu)
        assert ok, f"swiglu parity failed: worst ratio {worst}"

    def check(self, y, rows=None, cols=None):
        yr, ad = oracle.grouped_gemm(self.qa, self.sfa, self.ga, self.qb, self.sfb, self.gb, self.off,
                                     self.E, self.Mt, self.N, self.K, rows=rows, cols=cols)
        yg = y.float().cpu().numpy()
        if rows is not None:
            yg = yg[np.asarray(rows)]
        if cols is not None:
            yg = yg[:, np.asarray(cols)]
        ok, worst = oracle.within_tolerance(yg, yr, ad)
        assert ok, f"grouped parity failed: worst ratio {worst}"


@pytest.mark.parametrize("tile_rows", [0, 64])
@pytest.mark.parametrize("counts", [
    (3, 0, 17, 1, 0, 9),                 # ragged, empty experts
    (64, 65, 63, 1, 127, 128, 129, 0),   # tile-boundary counts
    (255, 256, 0, 257, 1),               # several 128-row tiles per expert, ragged last tiles
    (0, 0, 300, 0),                      # one expert owns every row
    (5,),                                # single expert
])
def test_grouped_ragged_counts(counts, tile_rows):
    # token tiles of up to 128 rows (0: the default) or 64
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_TILE_ROWS, tile_rows)
    g = Grouped(counts, 256, 512, 21)
    g.check(g.run())


def test_grouped_tile_rows_change_no_result():
    # 64- or 128-row token tiles cut the same rows into different MMAs (N = 64 or 128
    # token columns); every output element is the same K-ordered sum either way
    g = Grouped((200, 0, 64, 129, 5, 300), 384, 1088, 27)
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_TILE_ROWS, 64)
    y64 = g.run().clone()
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_TILE_ROWS, 128)
    y128 = g.run()
    assert torch.equal(y64.view(torch.int16), y128.view(torch.int16))
    g.check(y128)


def test_grouped_many_experts():
    # more experts than the preparation kernel has threads: each thread scans a run of
    # experts' tile counts (empty experts among them)
    rng = np.random.default_rng(25)
    counts = tuple(int(c) for c in rng.integers(0, 4, size=600))
    g = Grouped(counts, 128, 256, 25)
    g.check(g.run())


@pytest.mark.parametrize("K", [64, 128, 192])
@pytest.mark.parametrize("N", [8, 16, 72, 120])
def test_grouped_smallest_shapes(N, K):
    # N below one 128-row weight tile (the tile's box then also covers the next experts'
    # rows, whose outputs are never stored) and K of one partial 256-element stage
    g = Grouped((3, 0, 17, 1, 70), N, K, 26)
    g.check(g.run())


def test_grouped_ragged_n_and_k():
    g = Grouped((10, 40, 0, 7), 136, 1088, 22)
    g.check(g.run())


def test_grouped_weights_kept_in_l2_identical():
    g = Grouped((10, 40, 0, 7, 70), 256, 1024, 24)
    streamed = g.run().clone()
    m.nvfp4_tune(m.NVFP4_TUNE_WEIGHT_L2, 1)
    kept = g.run()
    assert torch.equal(kept.view(torch.int16), streamed.view(torch.int16))
    g.check(kept)


def test_grouped_small_persistent_grid_and_stages():
    g = Grouped((33, 2, 70, 16, 16), 384, 768, 23)
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_GRID, 5)
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_STAGES, 2)
    g.check(g.run())


def test_grouped_moe_workload_sampled():
    # 256 experts, 512 tokens routed top-8 uniformly (~16 rows / expert), K = 6144, N = 4096
    a_rows, off, tok = synth.moe_tokens(512, 256, 8, 6144, 3)
    counts = np.diff(off)
    g = Grouped(tuple(counts), 4096, 6144, 3, a_rows=a_rows,
                w=lambda e: synth.moe_expert_weight(e, 4096, 6144, 3))
    assert np.array_equal(g.off, off)
    y = g.run()
    rng = np.random.default_rng(1)
    rows = np.concatenate([[0, g.Mt - 1], rng.choice(g.Mt, 30, replace=False)])
    cols = np.concatenate([[0, 4095], rng.choice(4096, 62, replace=False)])
    g.check(y, rows=rows, cols=cols)


def test_grouped_moe_skewed_routing_sampled():
    # Zipf(1) expert popularity: expert 0 takes ~400 of the 4096 rows (7 token tiles),
    # the tail experts one or two rows; K = 6144, N = 4096 as in the MoE workload
    a_rows, off, tok = synth.moe_tokens(512, 256, 8, 6144, 3, zipf_s=1.0)
    counts = np.diff(off)
    assert counts.max() > 300
    g = Grouped(tuple(counts), 4096, 6144, 3, a_rows=a_rows,
                w=lambda e: synth.moe_expert_weight(e, 4096, 6144, 3))
    y = g.run()
    rng = np.random.default_rng(2)
    heavy = np.arange(off[0], off[1])  # every 64-row token tile of the heaviest expert
    rows = np.concatenate([heavy[[0, 63, 64, 127, 128, len(heavy) - 1]], [g.Mt - 1],
                           rng.choice(g.Mt, 24, replace=False)])
    cols = np.concatenate([[0, 127, 128, 4095], rng.choice(4096, 44, replace=False)])
    g.check(y, rows=rows, cols=cols)


def test_grouped_bad_offsets_reported_and_output_untouched():
    g = Grouped((4, 4, 4), 128, 256, 24)
    bad = g.off.copy()
    bad[1], bad[2] = bad[2], bad[1]
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    y = torch.full((g.Mt, g.N), 3.0, dtype=torch.bfloat16, device=dev())
    m.nvfp4_grouped_gemm(to_dev(g.qa), to_dev(g.sfa), scalar(g.ga), to_dev(g.qb), to_dev(g.sfb),
                         to_dev(g.gb), to_dev(bad), g.E, g.Mt, g.N, g.K, y=y, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == -8
    assert (y.float() == 3.0).all()
    bad = g.off.copy()
    bad[-1] -= 1
    st.zero_()
    m.nvfp4_grouped_gemm(to_dev(g.qa), to_dev(g.sfa), scalar(g.ga), to_dev(g.qb), to_dev(g.sfb),
                         to_dev(g.gb), to_dev(bad), g.E, g.Mt, g.N, g.K, y=y, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == -8


@pytest.mark.parametrize("tile_rows", [0, 64])
@pytest.mark.parametrize("counts,N_gu,K", [
    ((3, 0, 17, 1, 0, 9), 256, 512),           # ragged, empty experts
    ((64, 65, 1, 127, 0), 136, 1088),          # tile-boundary counts, N_gu not a multiple of 128
    ((0, 300, 0), 512, 256),                   # one expert, several token tiles
])
def test_grouped_swiglu_matches_oracle(counts, N_gu, K, tile_rows):
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_TILE_ROWS, tile_rows)
    g = Grouped(counts, N_gu, K, 31)
    y = g.run_swiglu()
    assert tuple(y.shape) == (g.Mt, N_gu // 2)
    g.check_swiglu(y)


def test_grouped_swiglu_is_silu_of_even_rows_times_odd_rows_of_the_plain_gemm():
    # the fused epilogue against the unfused grouped GEMM's own output (same kernel path,
    # same accumulators): silu(y[:, 0::2]) * y[:, 1::2] up to the bf16 rounding of y
    g = Grouped((12, 40, 0, 70), 384, 768, 32)
    y_plain = g.run().float()
    y_fused = g.run_swiglu().float()
    gate, up = y_plain[:, 0::2].double(), y_plain[:, 1::2].double()
    ref = gate / (1 + torch.exp(-gate)) * up
    err = (y_fused.double() - ref).abs()
    assert (err <= 2 ** -6 * ref.abs() + 1e-3 * ref.abs().max()).all()


def test_grouped_swiglu_moe_workload_sampled():
    # gate+up of the MoE workload: 256 experts, 512 tokens top-8, K = 6144, N_gu = 4096 (I = 2048)
    a_rows, off, tok = synth.moe_tokens(512, 256, 8, 6144, 3)
    counts = np.diff(off)
    g = Grouped(tuple(counts), 4096, 6144, 3, a_rows=a_rows,
                w=lambda e: synth.moe_expert_weight(e, 4096, 6144, 3))
    y = g.run_swiglu()
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0, g.Mt - 1], rng.choice(g.Mt, 30, replace=False)])
    cols = np.concatenate([[0, 63, 64, 2047], rng.choice(2048, 40, replace=False)])
    g.check_swiglu(y, rows=rows, cols=cols)



def _gathered(qa_tok, sfa_tok, T, K, row_token):
    """The routed-row operands a plain grouped GEMM would take: packed rows and block
    scales gathered by token (blocks run along K, so gathering commutes with quantising)."""
    Mt = len(row_token)
    qa = np.ascontiguousarray(qa_tok[row_token])
    sfa = oracle.sf_swizzle(oracle.sf_unswizzle(sfa_tok, T, K)[row_token], Mt, K)
    return qa, sfa


def _gather_ws(copy, E, Mt, N, K):
    """None: the binding's default workspace (rows copied out ahead of the GEMM); else one
    of the plain grouped size, which makes the GEMM's load stage gather the rows."""
    if copy:
        return None
    return torch.empty(m.nvfp4_grouped_gemm_workspace_bytes(E, Mt, N, K), dtype=torch.uint8, device=dev())


@pytest.mark.parametrize("copy", [True, False])
@pytest.mark.parametrize("T,counts,N,K", [
    (37, (3, 0, 17, 1, 0, 9), 256, 512),
    (200, (64, 65, 1, 70, 0), 136, 1088),
    (300, (130, 0, 255, 2), 256, 512),     # 128-row tiles: all four token indices per lane
    (5, (40,), 256, 256),                  # more routed rows than tokens: tokens repeat
])
def test_grouped_gather_matches_gathered_plain_and_oracle(T, counts, N, K, copy):
    rng = np.random.default_rng(T)
    Mt = int(sum(counts))
    row_token = rng.integers(0, T, size=Mt).astype(np.int32)
    qa_tok, sfa_tok, ga = oracle.quantize(synth.normal_bf16((T, K), 61, 1.0, 1e-3))
    qa, sfa = _gathered(qa_tok, sfa_tok, T, K, row_token)
    g = Grouped(counts, N, K, 62)
    g.qa, g.sfa, g.ga = qa, sfa, ga
    y_plain = g.run()
    y = m.nvfp4_grouped_gemm_gather(to_dev(qa_tok), to_dev(sfa_tok), scalar(ga), to_dev(g.qb), to_dev(g.sfb),
                                    to_dev(g.gb), to_dev(g.off), to_dev(row_token), g.E, T, Mt, N, K,
                                    workspace=_gather_ws(copy, g.E, Mt, N, K))
    torch.cuda.synchronize()
    assert torch.equal(y, y_plain)
    g.check(y)


@pytest.mark.parametrize("copy", [True, False])
def test_grouped_gather_moe_workload(copy):
    # 512 tokens quantised once, routed top-8 over 256 experts (4096 rows), K = 6144, N = 4096
    T, K, N = 512, 6144, 4096
    tok, _, off = synth.route_topk(T, 256, 8, 1003)
    qa_tok, sfa_tok, ga = oracle.quantize(synth.normal_bf16((T, K), 6, 1.0))
    qa, sfa = _gathered(qa_tok, sfa_tok, T, K, tok.astype(np.int64))
    counts = np.diff(off)
    gg = Grouped(tuple(counts), N, K, 3, a_rows=synth.normal_bf16((int(off[-1]), K), 6, 1.0),
                 w=lambda e: synth.moe_expert_weight(e, N, K, 3))
    gg.qa, gg.sfa, gg.ga = qa, sfa, ga
    y_plain = gg.run()
    y = m.nvfp4_grouped_gemm_gather(to_dev(qa_tok), to_dev(sfa_tok), scalar(ga), to_dev(gg.qb), to_dev(gg.sfb),
                                    to_dev(gg.gb), to_dev(gg.off), to_dev(tok.astype(np.int32)), 256, T,
                                    int(off[-1]), N, K, workspace=_gather_ws(copy, 256, int(off[-1]), N, K))
    torch.cuda.synchronize()
    assert torch.equal(y, y_plain)
    rng = np.random.default_rng(5)
    rows = np.concatenate([[0, gg.Mt - 1], rng.choice(gg.Mt, 20, replace=False)])
    cols = np.concatenate([[0, 4095], rng.choice(4096, 30, replace=False)])
    gg.check(y, rows=rows, cols=cols)


@pytest.mark.parametrize("copy", [True, False])
def test_grouped_gather_bad_token_index_reported(copy):
    T, K, N = 16, 256, 128
    qa_tok, sfa_tok, ga = oracle.quantize(synth.normal_bf16((T, K), 63, 1.0))
    g = Grouped((4, 4), N, K, 64)
    row_token = np.array([0, 1, 2, 3, 4, 5, 16, 7], dtype=np.int32)  # 16 is out of range
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    m.nvfp4_grouped_gemm_gather(to_dev(qa_tok), to_dev(sfa_tok), scalar(ga), to_dev(g.qb), to_dev(g.sfb),
                                to_dev(g.gb), to_dev(g.off), to_dev(row_token), g.E, T, 8, N, K, dev_status=st,
                                workspace=_gather_ws(copy, g.E, 8, N, K))
    torch.cuda.synchronize()
    assert st.item() == -8


def _swiglu_then_quantize(g, g_out):
    """The unfused reference on the GPU: the plain SwiGLU epilogue's bf16 output, then the
    stand-alone quantiser with the same global scale."""
    y = g.run_swiglu()
    q, sf = m.nvfp4_quantize(y, g_out)
    torch.cuda.synchronize()
    return y, q, sf


def _fused(g, g_out, status=None):
    M, N_gu = g.Mt, g.N
    q = torch.full((M, N_gu // 4), 0xAB, dtype=torch.uint8, device=dev())
    sf = torch.full((m.nvfp4_scale_bytes(M, N_gu // 2),), 0xAB, dtype=torch.uint8, device=dev())
    m.nvfp4_grouped_gemm_swiglu_quantize_out(to_dev(g.qa), to_dev(g.sfa), scalar(g.ga), to_dev(g.qb), to_dev(g.sfb),
                                             to_dev(g.gb), to_dev(g.off), g.E, g.Mt, g.N, g.K, g_out, q_out=q,
                                             sf_out=sf, dev_status=status)
    torch.cuda.synchronize()
    return q, sf


@pytest.mark.parametrize("tile_rows", [0, 64])
@pytest.mark.parametrize("counts,N_gu,K", [
    ((3, 0, 17, 1, 0, 9), 256, 512),           # ragged, empty experts, 30 rows (scale padding rows)
    ((64, 65, 1, 127, 0, 200), 384, 1088),     # tile boundaries, several 32-token chunks
    ((0, 300, 0), 128, 256),                   # one expert, several token tiles, one weight tile
])
def test_grouped_swiglu_quantize_out_equals_quantised_swiglu(counts, N_gu, K, tile_rows):
    # Codes and tiled scales (padding rows included, from garbage-filled outputs) equal the
    # stand-alone quantiser applied to the plain SwiGLU epilogue's bf16 output, bit for bit;
    # those codes also equal the oracle's quantiser on the same bf16 values, and the bf16
    # values are within the SwiGLU tolerance of the oracle.
    m.nvfp4_tune(m.NVFP4_TUNE_GROUPED_TILE_ROWS, tile_rows)
    g = Grouped(counts, N_gu, K, 33)
    y0 = g.run_swiglu()
    _, g_out = m.nvfp4_amax(y0)
    y, q_ref, sf_ref = _swiglu_then_quantize(g, g_out)
    q, sf = _fused(g, g_out)
    assert torch.equal(q, q_ref)
    assert torch.equal(sf, sf_ref)
    yb = y.view(torch.int16).cpu().numpy().view(np.uint16)
    qo, sfo, _ = oracle.quantize(yb, float(g_out.item()))
    assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(sf.cpu().numpy(), sfo)
    g.check_swiglu(y)


def test_grouped_swiglu_quantize_out_moe_workload():
    # gate+up of the MoE workload (256 experts, 512 tokens top-8, K = 6144, N_gu = 4096),
    # every output row: fused codes and scales against the unfused path on the GPU
    a_rows, off, tok = synth.moe_tokens(512, 256, 8, 6144, 3)
    g = Grouped(tuple(np.diff(off)), 4096, 6144, 3, a_rows=a_rows,
                w=lambda e: synth.moe_expert_weight(e, 4096, 6144, 3))
    y0 = g.run_swiglu()
    _, g_out = m.nvfp4_amax(y0)
    _, q_ref, sf_ref = _swiglu_then_quantize(g, g_out)
    q, sf = _fused(g, g_out)
    assert torch.equal(q, q_ref)
    assert torch.equal(sf, sf_ref)


def test_grouped_swiglu_quantize_out_rejects_and_reports():
    g = Grouped((4, 4), 256, 256, 34)
    g_out = torch.ones(1, dtype=torch.float32, device=dev())
    bad = Grouped((4, 4), 136, 256, 34)  # N_gu not a multiple of 128
    with pytest.raises(m.NVFP4Error) as e:
        _fused(bad, g_out)
    assert e.value.status == -2
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    g.off = np.array([0, 5, 4], dtype=np.int32)  # decreasing offsets
    _fused(g, g_out, status=st)
    assert st.item() == -8


@pytest.mark.parametrize("g_value", [1e-30, 3e-36, 1e30])
def test_grouped_swiglu_quantize_out_extreme_global_scales(g_value):
    # global scales at and beyond the fast division's guard (the quantiser's IEEE-division
    # fallback, saturating and all-zero codes): still nvfp4_quantize of the SwiGLU output
    g = Grouped((7, 0, 40, 130), 256, 512, 35)
    g_out = torch.tensor([g_value], dtype=torch.float32, device=dev())
    _, q_ref, sf_ref = _swiglu_then_quantize(g, g_out)
    q, sf = _fused(g, g_out)
    assert torch.equal(q, q_ref)
    assert torch.equal(sf, sf_ref)
