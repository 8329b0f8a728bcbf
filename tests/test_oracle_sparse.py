"""Pins for the oracle's pair-wise 2:4 sparse path (CPU only).

Independent references: a brute-force top-2 pair selection in numpy, the tiled
metadata layout's bijection, the 16-element-block quantiser (already pinned) for
the 32-element-block one, the dense GEMM oracle (already pinned) on operands
decompressed here in numpy, and exact rational arithmetic on a tiny case decoded
through the golden E2M1 list and torch's float8_e4m3fn.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
import synth

E2M1 = [0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6]


def _tie_heavy_weights(N, K, seed):
    rng = np.random.default_rng(seed)
    vals = np.array([0.0, -0.0, 0.5, -0.5, 1.0, -1.0, 2.0, 3.0], dtype=np.float32)
    w = rng.choice(vals, size=(N, K)).astype(np.float32)
    mask = rng.random((N, K)) < 0.3
    w[mask] = rng.normal(0, 1, int(mask.sum())).astype(np.float32)
    return synth.f32_to_bf16_bits(w)


def _brute_prune(wb):
    w = synth.bf16_bits_to_f32(wb)
    N, K = w.shape
    c = np.empty((N, K // 2), dtype=np.uint16)
    meta = np.zeros((N, K // 16), dtype=np.uint8)
    for n in range(N):
        for g in range(K // 8):
            sc = [np.float32(abs(w[n, 8 * g + 2 * j])) + np.float32(abs(w[n, 8 * g + 2 * j + 1])) for j in range(4)]
            keep = sorted(sorted(range(4), key=lambda j: (-sc[j], j))[:2])
            for h, j in enumerate(keep):
                c[n, 4 * g + 2 * h] = wb[n, 8 * g + 2 * j]
                c[n, 4 * g + 2 * h + 1] = wb[n, 8 * g + 2 * j + 1]
            meta[n, g // 2] |= (keep[0] | keep[1] << 2) << (4 * (g % 2))
    return c, meta


def test_prune_pairs_matches_brute_force_with_ties():
    for seed, (N, K) in enumerate([(7, 64), (16, 256), (3, 1024)]):
        wb = _tie_heavy_weights(N, K, seed)
        c, meta = oracle.prune_pairs(wb)
        c2, meta2 = _brute_prune(wb)
        assert np.array_equal(c, c2) and np.array_equal(meta, meta2)


def test_prune_pairs_keeps_the_two_largest_pairs_and_decompresses():
    wb = synth.normal_bf16((32, 512), 5, 1.0, 1e-2)
    w = synth.bf16_bits_to_f32(wb)
    c, meta = oracle.prune_pairs(wb)
    cv = synth.bf16_bits_to_f32(c)
    for n in range(32):
        for g in range(64):
            nib = int(meta[n, g // 2] >> (4 * (g % 2))) & 15
            i0, i1 = nib & 3, nib >> 2
            assert i0 < i1
            sc = np.abs(w[n, 8 * g:8 * g + 8]).reshape(4, 2).sum(axis=1)
            dropped = [j for j in range(4) if j not in (i0, i1)]
            assert min(sc[i0], sc[i1]) >= max(sc[dropped])
            assert np.array_equal(cv[n, 4 * g:4 * g + 2], w[n, 8 * g + 2 * i0:8 * g + 2 * i0 + 2])
            assert np.array_equal(cv[n, 4 * g + 2:4 * g + 4], w[n, 8 * g + 2 * i1:8 * g + 2 * i1 + 2])


def test_meta_tiling_is_a_bijection_with_zero_padding():
    for N, K in [(128, 512), (200, 1536), (5, 128)]:
        rng = np.random.default_rng(N + K)
        lin = rng.integers(0, 256, size=(N, K // 16), dtype=np.uint8)
        t = oracle.meta_tile(lin, N, K)
        assert t.size == (N + 127) // 128 * ((K + 511) // 512) * 4096
        assert np.array_equal(oracle.meta_untile(t, N, K), lin)
        offs = np.array([oracle.meta_offset(n, b, K) for n in range(N) for b in range(K // 16)])
        assert len(np.unique(offs)) == offs.size and offs.max() < t.size
        mask = np.ones(t.size, bool)
        mask[offs] = False
        assert not t[mask].any()
    # within a tile: rows in groups of 8, each row's 32 bytes as two 16-byte halves
    assert oracle.meta_offset(0, 0, 512) == 0 and oracle.meta_offset(1, 0, 512) == 16
    assert oracle.meta_offset(0, 16, 512) == 128 and oracle.meta_offset(8, 0, 512) == 256
    assert oracle.meta_offset(0, 32, 1024) == 4096 and oracle.meta_offset(128, 0, 1024) == 2 * 4096


def test_quantize_b32_is_the_16_block_recipe_on_32_blocks():
    # the 32-block scale depends only on the block's amax: it equals the 16-block scale of
    # the half that holds the maximum, and that half's codes are the 16-block codes
    xb = synth.normal_bf16((40, 512), 6, 1.0, 1e-2)
    q32, sf32, g = oracle.quantize_b32(xb)
    q16, sf16, g16 = oracle.quantize(xb, g)
    assert g16 == g
    s32 = oracle.sf_unswizzle_bs(sf32, 40, 512, 32)
    s16 = oracle.sf_unswizzle(sf16, 40, 512)
    x = np.abs(synth.bf16_bits_to_f32(xb))
    for r in range(40):
        for c in range(16):
            h = int(x[r, 32 * c + 16:32 * c + 32].max() > x[r, 32 * c:32 * c + 16].max())
            assert s32[r, c] == s16[r, 2 * c + h]
            sl = slice(16 * c + 8 * h, 16 * c + 8 * h + 8)
            assert np.array_equal(q32[r, sl], q16[r, sl])
    # both halves sharing the amax: identical to the 16-block quantiser everywhere
    x2 = synth.bf16_bits_to_f32(xb).copy()
    for c in range(16):
        blk = x2[:, 32 * c:32 * c + 32]
        m = np.abs(blk).max(axis=1)
        blk[:, 0] = m
        blk[:, 16] = -m
    xb2 = synth.f32_to_bf16_bits(x2)
    q32, sf32, g = oracle.quantize_b32(xb2)
    q16, sf16, _ = oracle.quantize(xb2, g)
    assert np.array_equal(q32, q16)
    assert np.array_equal(np.repeat(oracle.sf_unswizzle_bs(sf32, 40, 512, 32), 2, axis=1),
                          oracle.sf_unswizzle(sf16, 40, 512))


def _decompress(cq, csf, meta, N, K):
    """Dense codes [N, K/2] (pruned positions code 0) and 16-block logical scales."""
    codes_st = np.empty((N, K // 2), dtype=np.uint8)
    codes_st[:, 0::2] = cq & 15
    codes_st[:, 1::2] = cq >> 4
    codes = np.zeros((N, K), dtype=np.uint8)
    for g in range(K // 8):
        nib = (meta[:, g // 2].astype(np.int64) >> (4 * (g % 2))) & 15
        for h, idx in enumerate((nib & 3, nib >> 2)):
            for e in range(2):
                codes[np.arange(N), 8 * g + 2 * idx + e] = codes_st[:, 4 * g + 2 * h + e]
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    s_st = oracle.sf_unswizzle(csf, N, K // 2)          # one scale per 16 stored = 32 logical
    return q, oracle.sf_swizzle(np.repeat(s_st, 2, axis=1), N, K)


def test_sparse_gemm_equals_dense_oracle_on_decompressed_operands():
    M, N, K = 9, 21, 1024
    xb = synth.normal_bf16((M, K), 7, 1.0, 1e-2)
    wb = synth.normal_bf16((N, K), 8, 0.02)
    xq, xsf, gx = oracle.quantize_b32(xb)
    cq, csf, gw, meta = oracle.sparse_quantize_weight(wb)
    y, ad = oracle.sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, M, N, K)
    wq, wsf = _decompress(cq, csf, meta, N, K)
    x16 = oracle.sf_swizzle(np.repeat(oracle.sf_unswizzle_bs(xsf, M, K, 32), 2, axis=1), M, K)
    yd, add = oracle.gemm(xq, x16, gx, wq, wsf, gw, M, N, K)
    assert np.array_equal(y, yd) and np.array_equal(ad, add)
    ys, _ = oracle.sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, M, N, K, rows=[8, 0], cols=[3, 20, 0])
    assert np.array_equal(ys, y[np.ix_([8, 0], [3, 20, 0])])


def test_sparse_gemm_exact_on_a_tiny_case():
    # M = N = 1, K = 128 decoded by hand: golden E2M1 list, torch float8_e4m3fn, Fractions
    rng = np.random.default_rng(11)
    K = 128
    xq = rng.integers(0, 256, size=(1, K // 2), dtype=np.uint8)
    cq = rng.integers(0, 256, size=(1, K // 4), dtype=np.uint8)
    xs = rng.integers(0x20, 0x48, size=(1, K // 32), dtype=np.uint8)
    cs = rng.integers(0x20, 0x48, size=(1, K // 32), dtype=np.uint8)
    nibs = rng.choice([0x4, 0x8, 0xC, 0x9, 0xD, 0xE], size=K // 8)
    meta = np.array([[nibs[2 * b] | nibs[2 * b + 1] << 4 for b in range(K // 16)]], dtype=np.uint8)
    xsf = oracle.sf_swizzle_bs(xs, 1, K, 32)
    csf = oracle.sf_swizzle(cs, 1, K // 2)
    gx, gw = np.float32(0.375), np.float32(1.25)
    y, _ = oracle.sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, 1, 1, K)
    f8 = lambda b: Fraction(float(torch.tensor([int(b)], dtype=torch.uint8).view(torch.float8_e4m3fn).float()))
    xv = [Fraction(E2M1[(xq[0, k // 2] >> (4 * (k % 2))) & 15]) * f8(xs[0, k // 32]) for k in range(K)]
    total = Fraction(0)
    for g in range(K // 8):
        pairs = (int(nibs[g]) & 3, int(nibs[g]) >> 2)
        for h in range(2):
            for e in range(2):
                st = 4 * g + 2 * h + e
                wv = Fraction(E2M1[(cq[0, st // 2] >> (4 * (st % 2))) & 15]) * f8(cs[0, st // 16])
                total += xv[8 * g + 2 * pairs[h] + e] * wv
    expect = total * Fraction(float(gx)) * Fraction(float(gw))
    assert abs(Fraction(float(y[0, 0])) - expect) <= abs(expect) * Fraction(1, 2 ** 50)


def test_grouped_sparse_gemm_is_per_expert_sparse_gemm_and_matches_dense_grouped():
    E, N, K = 4, 40, 512
    counts = np.array([5, 0, 17, 3])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    Mt = int(off[-1])
    xq, xsf, gx = oracle.quantize_b32(synth.normal_bf16((Mt, K), 81, 1.0, 1e-2))
    ws = [oracle.sparse_quantize_weight(synth.moe_expert_weight(e, N, K, 82)) for e in range(E)]
    cq = np.stack([w[0] for w in ws])
    csf = np.stack([w[1] for w in ws])
    gw = np.array([w[2] for w in ws], np.float32)
    meta = np.stack([w[3] for w in ws])
    y, ad = oracle.grouped_sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, off, E, Mt, N, K)
    for e in range(E):
        r = np.arange(off[e], off[e + 1])
        if r.size:
            ye, _ = oracle.sparse_gemm(xq, xsf, gx, cq[e], csf[e], meta[e], gw[e], Mt, N, K, rows=r)
            assert np.array_equal(y[r], ye)
    # the dense grouped oracle on operands decompressed here
    dq, dsf = zip(*[_decompress(cq[e], csf[e], meta[e], N, K) for e in range(E)])
    x16 = oracle.sf_swizzle(np.repeat(oracle.sf_unswizzle_bs(xsf, Mt, K, 32), 2, axis=1), Mt, K)
    yd, add = oracle.grouped_gemm(xq, x16, gx, np.stack(dq), np.stack(dsf), gw, off, E, Mt, N, K)
    assert np.array_equal(y, yd) and np.array_equal(ad, add)
    ys, _ = oracle.grouped_sparse_gemm(xq, xsf, gx, cq, csf, meta, gw, off, E, Mt, N, K, rows=[24, 0, 6],
                                       cols=[39, 1])
    assert np.array_equal(ys, y[np.ix_([24, 0, 6], [39, 1])])
