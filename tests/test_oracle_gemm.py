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


def _bf16_round(v):
    """float64 -> nearest bf16 value (ties to even), through float32 as the GPU does."""
    b = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def _worst_gpu_outputs(gate, up, adg, adu, rel=4e-3, absk=1e-5):
    """Outputs a GPU within the GEMM tolerance could return: gate and up moved to every
    corner of their tolerance boxes (shrunk by 2^-20 so that float32 stays inside), the
    activation in float32, then either the bf16 rounding or a worst-case 2^-9 relative
    error pushed away from the exact product."""
    tg = rel * np.abs(gate) + absk * adg
    tu = rel * np.abs(up) + absk * adu
    y = oracle.silu(gate) * up
    outs = []
    for sg in (-1.0, 1.0):
        for su in (-1.0, 1.0):
            g1 = np.float32(gate + sg * tg * (1 - 2.0 ** -20))
            u1 = np.float32(up + su * tu * (1 - 2.0 ** -20))
            act = np.float32(g1 / (np.float32(1) + np.float32(np.exp(-g1.astype(np.float64)))))
            prod = (act * u1).astype(np.float64)
            outs.append(_bf16_round(prod))
            away = np.sign(prod - y)
            outs.append(prod * (1 + away * np.sign(prod) * 2.0 ** -9))
    return outs


def test_silu_lipschitz_constant_below_1_1():
    # silu'(v) = s(v) (1 + v (1 - s(v))), s the logistic function: its maximum (at v ~ 2.3994)
    # is the Lipschitz constant the SwiGLU tolerance takes as 1.1
    special = pytest.importorskip("scipy.special")
    v = np.linspace(-60.0, 60.0, 1_200_001)
    s = special.expit(v)
    d = s * (1 + v * (1 - s))
    assert 1.0997 < d.max() < 1.1 and abs(v[d.argmax()] - 2.3994) < 1e-3
    assert d.min() > -0.1  # the steepest descent (near v = -2.4) is far smaller in magnitude
    # the oracle's silu has that derivative (central differences)
    h = 1e-6
    fd = (oracle.silu(v[::997] + h) - oracle.silu(v[::997] - h)) / (2 * h)
    assert np.allclose(fd, d[::997], atol=1e-8)


def test_swiglu_tolerance_holds_for_every_output_within_the_gemm_bounds():
    # soundness: any gate/up within their GEMM tolerances, activated in fp32 and rounded to
    # bf16 (or off by a full 2^-9 the other way), passes the propagated bound
    rng = np.random.default_rng(7)
    n = 200_000
    gate = rng.normal(0, 3, n) * rng.choice([1e-3, 1, 4], n)
    up = rng.normal(0, 3, n) * rng.choice([1e-3, 1, 4], n)
    adg = np.abs(rng.normal(0, 1, n)) * rng.choice([0, 10, 1e3, 5e4], n)
    adu = np.abs(rng.normal(0, 1, n)) * rng.choice([0, 10, 1e3, 5e4], n)
    for y in _worst_gpu_outputs(gate, up, adg, adu):
        ok, worst = oracle.within_tolerance_swiglu(y, gate, up, adg, adu)
        assert ok, worst


@pytest.mark.parametrize("gate,up,adg,adu,term", [
    (2.15, 1.0, 49_000.0, 0.0, "slope of silu times |u|"),   # g' spans the steepest stretch
    (5.0, 0.1, 0.0, 49_960.0, "|silu(g)| times t_u"),
    (1.9, 0.0, 99_240.0, 1e5, "slope times t_g t_u"),           # y = 0: all error from both bounds
])
def test_swiglu_tolerance_is_tight(gate, up, adg, adu, term):
    # in each regime one part of the bound dominates and a GPU result at a corner of the
    # tolerance boxes uses at least 95 % of it, so dropping or shrinking that part (or the
    # Lipschitz constant) makes these corner outputs fail the check above
    g, u, ag, au = (np.array([v]) for v in (gate, up, adg, adu))
    ratios = [oracle.within_tolerance_swiglu(y, g, u, ag, au)[1] for y in _worst_gpu_outputs(g, u, ag, au)]
    assert 0.95 <= max(ratios) <= 1.0, (term, ratios)
