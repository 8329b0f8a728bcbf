"""Pins for the oracle's float64 GEMM and grouped GEMM (CPU only).

Independent references: exact 128-bit integer sums (checked with Python
integers), a numpy matmul of operands decoded through torch's float8_e4m3fn and
the golden E2M1 table, identity / one-hot / all-ones closed forms, brute-force
enumeration of every code pair at M = N = 1, K = 16, and per-expert dense calls.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


def _decode_independent(q, sf, rows, K):
    """Decode with the golden E2M1 list and torch's E4M3 conversion (not the oracle)."""
    codes = np.empty((rows, K), dtype=np.int64)
    codes[:, 0::2] = q & 15
    codes[:, 1::2] = q >> 4
    lin = oracle.sf_unswizzle(sf, rows, K)
    s = torch.from_numpy(lin.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return E2M1[codes] * np.repeat(s, 16, axis=1)


def _rand_operands(M, N, K, seed, lo=0x28, hi=0x48):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sfa = oracle.sf_swizzle(rng.integers(lo, hi, size=(M, K // 16), dtype=np.uint8), M, K)
    sfb = oracle.sf_swizzle(rng.integers(lo, hi, size=(N, K // 16), dtype=np.uint8), N, K)
    return a, sfa, b, sfb


def test_gemm_matches_numpy_matmul_of_independent_decode():
    M, N, K = 37, 50, 320
    a, sfa, b, sfb = _rand_operands(M, N, K, 1)
    ga, gb = np.float32(0.37), np.float32(1.9)
    y, ad = oracle.gemm(a, sfa, ga, b, sfb, gb, M, N, K)
    A = _decode_independent(a, sfa, M, K)
    B = _decode_independent(b, sfb, N, K)
    ref = (A @ B.T) * float(ga) * float(gb)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())
    assert np.allclose(ad, np.abs(A) @ np.abs(B).T * abs(float(ga) * float(gb)), rtol=1e-12)


def test_gemm_f64_agrees_with_exact_integer_sum():
    M, N, K = 9, 11, 1024
    a, sfa, b, sfb = _rand_operands(M, N, K, 2, lo=0x01, hi=0x7E)
    y, ad = oracle.gemm(a, sfa, 1.0, b, sfb, 1.0, M, N, K)
    S = oracle.gemm_exact(a, sfa, b, sfb, M, N, K)
    for i in range(M):
        for j in range(N):
            exact = Fraction(S[i][j], 1 << 20)
            # float64 summation of K exact products: |err| <= K * 2^-53 * sum|p|
            bound = Fraction(K) * Fraction(1, 1 << 53) * Fraction(ad[i, j]) * 2
            assert abs(Fraction(y[i, j]) - exact) <= bound


def test_gemm_identity_returns_weights():
    K = 128
    M = K
    N = 24
    codes = np.zeros((M, K), dtype=np.uint8)
    codes[np.arange(M), np.arange(M)] = 0x2  # 1.0
    a = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sfa = oracle.sf_swizzle(np.full((M, K // 16), 0x38, dtype=np.uint8), M, K)  # 1.0
    _, _, b, sfb = _rand_operands(1, N, K, 3)
    gb = np.float32(0.5)
    y, _ = oracle.gemm(a, sfa, 1.0, b, sfb, gb, M, N, K)
    W = _decode_independent(b, sfb, N, K) * 0.5
    assert np.array_equal(y, W.T)


def test_gemm_one_hot_selects_entries():
    M, N, K = 8, 8, 256
    _, _, b, sfb = _rand_operands(1, N, K, 4)
    rng = np.random.default_rng(5)
    cols = rng.integers(0, K, size=M)
    codes = np.zeros((M, K), dtype=np.uint8)
    codes[np.arange(M), cols] = 0x4  # 2.0
    a = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sfa = oracle.sf_swizzle(np.full((M, K // 16), 0x30, dtype=np.uint8), M, K)  # 0.5
    y, _ = oracle.gemm(a, sfa, 1.0, b, sfb, 1.0, M, N, K)
    W = _decode_independent(b, sfb, N, K)
    assert np.array_equal(y, W[:, cols].T * 1.0)


def test_gemm_all_ones_closed_form():
    M, N, K = 5, 7, 512
    a = np.full((M, K // 2), 0x22, dtype=np.uint8)
    b = np.full((N, K // 2), 0x22, dtype=np.uint8)
    sfa = oracle.sf_swizzle(np.full((M, K // 16), 0x40, dtype=np.uint8), M, K)  # 2.0
    sfb = oracle.sf_swizzle(np.full((N, K // 16), 0x31, dtype=np.uint8), N, K)  # 0.5625
    ga, gb = np.float32(0.75), np.float32(3.0)
    y, ad = oracle.gemm(a, sfa, ga, b, sfb, gb, M, N, K)
    assert (y == K * 2.0 * 0.5625 * 0.75 * 3.0).all()
    assert (ad == y).all()


def test_gemm_brute_force_every_code_pair():
    K = 16
    for sa_code, sb_code in [(0x38, 0x38), (0x01, 0x7E), (0x45, 0x2B)]:
        sa, sb = oracle.e4m3_value(sa_code), oracle.e4m3_value(sb_code)
        sfa = oracle.sf_swizzle(np.array([[sa_code]], dtype=np.uint8), 1, K)
        sfb = oracle.sf_swizzle(np.array([[sb_code]], dtype=np.uint8), 1, K)
        for ca in range(16):
            for cb in range(16):
                for slot in (0, 7, 15):
                    ac = np.zeros(K, dtype=np.uint8)
                    bc = np.zeros(K, dtype=np.uint8)
                    ac[slot], bc[slot] = ca, cb
                    a = (ac[0::2] | (ac[1::2] << 4)).astype(np.uint8)[None]
                    b = (bc[0::2] | (bc[1::2] << 4)).astype(np.uint8)[None]
                    y, _ = oracle.gemm(a, sfa, 1.0, b, sfb, 1.0, 1, 1, K)
                    assert y[0, 0] == E2M1[ca] * E2M1[cb] * sa * sb


def test_gemm_row_and_column_sampling_matches_full():
    M, N, K = 40, 30, 256
    a, sfa, b, sfb = _rand_operands(M, N, K, 6)
    y, ad = oracle.gemm(a, sfa, 0.5, b, sfb, 2.0, M, N, K)
    rows, cols = [3, 39, 0], [29, 1]
    ys, ads = oracle.gemm(a, sfa, 0.5, b, sfb, 2.0, M, N, K, rows=rows, cols=cols)
    assert np.array_equal(ys, y[np.ix_(rows, cols)])
    assert np.array_equal(ads, ad[np.ix_(rows, cols)])


def _grouped_case(E=6, N=48, K=128, counts=(3, 0, 17, 1, 0, 9), seed=7):
    rng = np.random.default_rng(seed)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    Mt = int(offsets[-1])
    a = rng.integers(0, 256, size=(Mt, K // 2), dtype=np.uint8)
    sfa = oracle.sf_swizzle(rng.integers(0x28, 0x48, size=(Mt, K // 16), dtype=np.uint8), Mt, K)
    b = rng.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    sfb = np.stack([oracle.sf_swizzle(rng.integers(0x28, 0x48, size=(N, K // 16),
                                                   dtype=np.uint8), N, K) for _ in range(E)])
    gb = rng.uniform(0.5, 2, size=E).astype(np.float32)
    return a, sfa, b, sfb, gb, offsets, E, Mt, N, K


def test_grouped_equals_per_expert_dense_calls():
    a, sfa, b, sfb, gb, off, E, Mt, N, K = _grouped_case()
    ga = np.float32(0.8)
    y, ad = oracle.grouped_gemm(a, sfa, ga, b, sfb, gb, off, E, Mt, N, K)
    A = _decode_independent(a, sfa, Mt, K)
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        W = _decode_independent(b[e], sfb[e], N, K)
        ref = (A[r0:r1] @ W.T) * float(ga) * float(gb[e])
        assert np.allclose(y[r0:r1], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_grouped_row_sampling_and_permutation_invariance():
    a, sfa, b, sfb, gb, off, E, Mt, N, K = _grouped_case()
    y, _ = oracle.grouped_gemm(a, sfa, 1.0, b, sfb, gb, off, E, Mt, N, K)
    rows = [29, 0, 12, 3]
    ys, _ = oracle.grouped_gemm(a, sfa, 1.0, b, sfb, gb, off, E, Mt, N, K, rows=rows)
    assert np.array_equal(ys, y[rows])
    # permuting rows inside an expert's slice permutes the outputs the same way
    perm = np.arange(Mt)
    perm[3:20] = perm[3:20][::-1]  # expert 2 owns rows 3..19
    lin = oracle.sf_unswizzle(sfa, Mt, K)[perm]
    yp, _ = oracle.grouped_gemm(a[perm].copy(), oracle.sf_swizzle(lin, Mt, K), 1.0, b, sfb, gb,
                                off, E, Mt, N, K)
    assert np.array_equal(yp, y[perm])


def test_grouped_rejects_malformed_offsets():
    a, sfa, b, sfb, gb, off, E, Mt, N, K = _grouped_case()
    bad = off.copy()
    bad[2], bad[3] = bad[3], bad[2]
    with pytest.raises(ValueError):
        oracle.grouped_gemm(a, sfa, 1.0, b, sfb, gb, bad, E, Mt, N, K)
    bad = off.copy()
    bad[-1] -= 1
    with pytest.raises(ValueError):
        oracle.grouped_gemm(a, sfa, 1.0, b, sfb, gb, bad, E, Mt, N, K)


def test_tolerance_helper():
    ref = np.array([1.0, -2.0, 0.0])
    ad = np.array([10.0, 10.0, 10.0])
    ok, worst = oracle.within_tolerance(ref + np.array([4e-3 + 1e-4, 0, 0]), ref, ad)
    assert ok and worst <= 1.0
    ok, worst = oracle.within_tolerance(ref + np.array([4e-3 + 2e-4, 0, 0]), ref, ad)
    assert not ok and worst > 1.0


def test_synth_generator_is_seeded_and_shaped():
    x1 = synth.normal_bf16((64, 64), 3, 1.0, 1e-3)
    x2 = synth.normal_bf16((64, 64), 3, 1.0, 1e-3)
    assert np.array_equal(x1, x2)
    v = synth.bf16_bits_to_f32(synth.normal_bf16((512, 512), 4, 0.02))
    assert abs(v.std() - 0.02) < 1e-3 and abs(v.mean()) < 1e-3
    tok, exp, off = synth.route_topk(512, 256, 8, 1)
    assert off[-1] == 4096 and (np.diff(off) >= 0).all()
    for t in range(512):
        assert len(set(exp[tok == t])) == 8


def test_skewed_routing_is_seeded_distinct_and_zipf_ordered():
    tok, exp, off = synth.route_topk(512, 256, 8, 1003, 1.0)
    tok2, exp2, off2 = synth.route_topk(512, 256, 8, 1003, 1.0)
    assert np.array_equal(exp, exp2) and np.array_equal(off, off2)
    assert off[-1] == 4096 and (np.diff(off) >= 0).all()
    for t in range(512):
        assert len(set(exp[tok == t])) == 8
    c = np.diff(off)
    # popularity (e + 1)^-1: expert 0 is picked by most tokens, counts fall with the index
    assert c[0] > 0.6 * 512 and c[0] > c[1] > c[4] > c[32] and c[:8].sum() > c[128:].sum()
    # a token's first pick follows the popularity law: P(e) = (1/(e+1)) / H_256
    first = np.array([exp[tok == t].min() for t in range(512)])
    assert (first == 0).mean() > 0.3
    # uniform routing is the zipf_s = 0 case, unchanged
    tu, eu, ou = synth.route_topk(512, 256, 8, 1003)
    tz, ez, oz = synth.route_topk(512, 256, 8, 1003, 0.0)
    assert np.array_equal(eu, ez) and np.diff(ou).max() < 40


def test_skewed_routing_single_draw_law():
    # topk = 1: each token's expert is the inverse CDF of its draw over (e + 1)^-s
    tok, exp, off = synth.route_topk(20000, 16, 1, 77, 2.0)
    pop = (np.arange(16) + 1.0) ** -2.0
    expect = pop / pop.sum() * 20000
    got = np.diff(off)
    assert np.all(np.abs(got - expect) < 5 * np.sqrt(expect) + 2)


def test_silu_against_library_and_identities():
    special = pytest.importorskip("scipy.special")
    v = np.concatenate([np.linspace(-40, 40, 4001), [0.0, 1e-300, -1e-300, 700.0, -700.0]])
    s = oracle.silu(v)
    assert np.allclose(s, v * special.expit(v), rtol=1e-15, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(oracle.silu(v) - oracle.silu(-v), v, rtol=1e-14, atol=1e-14)  # silu(v) - silu(-v) = v


def test_swiglu_oracle_is_interleaved_grouped_gemm_then_silu_times_up():
    special = pytest.importorskip("scipy.special")
    E, N_gu, K = 3, 48, 128
    counts = np.array([5, 0, 7])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    Mt = int(off[-1])
    qa, sfa, ga = oracle.quantize(synth.normal_bf16((Mt, K), 41, 1.0))
    sfb_bytes = oracle.scale_bytes(N_gu, K)
    qb = np.empty((E, N_gu, K // 2), dtype=np.uint8)
    sfb = np.empty((E, sfb_bytes), dtype=np.uint8)
    gb = np.empty(E, dtype=np.float32)
    for e in range(E):
        qb[e], sfb[e], gb[e] = oracle.quantize(synth.normal_bf16((N_gu, K), 42 + e, 0.5))
    full, _ = oracle.grouped_gemm(qa, sfa, ga, qb, sfb, gb, off, E, Mt, N_gu, K)
    y, gate, up, adg, adu = oracle.grouped_gemm_swiglu(qa, sfa, ga, qb, sfb, gb, off, E, Mt, N_gu, K)
    assert np.array_equal(gate, full[:, 0::2]) and np.array_equal(up, full[:, 1::2])
    assert np.allclose(y, gate * special.expit(gate) * up, rtol=1e-14, atol=1e-300)
    # the gate is the even row: swapping the roles gives a different product here
    assert not np.allclose(y, up * special.expit(up) * gate)
    cols = np.array([0, 7, 23])
    ys, gs, us, _, _ = oracle.grouped_gemm_swiglu(qa, sfa, ga, qb, sfb, gb, off, E, Mt, N_gu, K, cols=cols)
    assert np.array_equal(ys, y[:, cols])


def test_swiglu_tolerance_bound_edges():
    gate = np.array([2.0, -3.0, 0.0, 10.0])
    up = np.array([1.5, 0.25, 4.0, -2.0])
    adg = np.array([50.0, 10.0, 100.0, 5.0])
    adu = np.array([20.0, 30.0, 1.0, 7.0])
    y = oracle.silu(gate) * up
    tg = 4e-3 * np.abs(gate) + 1e-5 * adg
    tu = 4e-3 * np.abs(up) + 1e-5 * adu
    bound = 1.1 * tg * (np.abs(up) + tu) + np.abs(oracle.silu(gate)) * tu + 2.0 ** -8 * np.abs(y)
    ok, worst = oracle.within_tolerance_swiglu(y + 0.999 * bound, gate, up, adg, adu)
    assert ok and worst < 1.0
    ok, worst = oracle.within_tolerance_swiglu(y - 1.001 * bound, gate, up, adg, adu)
    assert not ok and worst > 1.0
