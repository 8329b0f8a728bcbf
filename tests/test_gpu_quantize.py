"""GPU parity of the quantisation path (amax, global scale, block quantiser,
device encoders) against the oracle: bit-exact, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests.helpers import dev, to_dev

pytestmark = pytest.mark.gpu
m = pytest.importorskip("moe_nvfp4_gemm_gb300")


def test_encode_e2m1_exhaustive_decision_range():
    lo = int(np.float32(0.125).view(np.uint32))
    hi = int(np.float32(16.0).view(np.uint32))
    bits = np.arange(lo, hi, dtype=np.uint32)
    v = bits.view(np.float32)
    for sign in (1, -1):
        vv = (v * sign).astype(np.float32)
        got = m.nvfp4_encode_e2m1(to_dev(vv)).cpu().numpy()
        assert np.array_equal(got, oracle.e2m1_encode_array(vv))


def test_encode_e2m1_random_bit_patterns():
    rng = np.random.default_rng(1)
    v = rng.integers(0, 2**32, size=1 << 22, dtype=np.uint64).astype(np.uint32).view(np.float32)
    v = np.ascontiguousarray(v[np.isfinite(v)])
    got = m.nvfp4_encode_e2m1(to_dev(v)).cpu().numpy()
    assert np.array_equal(got, oracle.e2m1_encode_array(v))


def test_encode_e4m3_matches_oracle():
    # every float32 in [2^-12, 512) plus neighbourhoods of every rounding midpoint
    lo = int(np.float32(2.0 ** -12).view(np.uint32))
    hi = int(np.float32(512.0).view(np.uint32))
    v = np.arange(lo, hi, 7, dtype=np.uint32).view(np.float32)
    mids = []
    for c in range(0, 0x7E):
        mb = int(np.float32((oracle.e4m3_value(c) + oracle.e4m3_value(c + 1)) / 2).view(np.uint32))
        mids.append(np.arange(mb - 64, mb + 65, dtype=np.uint32))
    v = np.concatenate([v, np.concatenate(mids).view(np.float32), np.float32([0, 448, 464, 1e30])])
    got = m.nvfp4_encode_e4m3(to_dev(v)).cpu().numpy()
    assert np.array_equal(got, oracle.e4m3_encode_array(v))


def _quantize_and_compare(xb, g_fixed=None):
    x = to_dev(xb)
    amax, g = m.nvfp4_amax(x)
    if g_fixed is not None:
        g = torch.tensor([g_fixed], dtype=torch.float32, device=dev())
    # outputs start as garbage: every code byte and every scale byte, the padding rows'
    # included (written 0), must be written
    M, K = xb.shape
    q = torch.full((M, K // 2), 0xAB, dtype=torch.uint8, device=dev())
    sf = torch.full((m.nvfp4_scale_bytes(M, K),), 0xAB, dtype=torch.uint8, device=dev())
    m.nvfp4_quantize(x, g, q_out=q, sf_out=sf)
    qo, sfo, go = oracle.quantize(xb, g_fixed)
    torch.cuda.synchronize()
    assert np.float32(amax.item()) == np.float32(oracle.amax(xb))
    assert np.float32(g.item()) == go
    qg, sfg = q.cpu().numpy(), sf.cpu().numpy()
    bad = np.argwhere(qg != qo)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"
    assert np.array_equal(sfg, sfo)


@pytest.mark.parametrize("M,K,seed,std,out", [
    (128, 256, 0, 1.0, 0.0),       # the tiny workload's x
    (1, 64, 1, 1.0, 0.0),          # single row, single scale tile column
    (200, 512, 2, 0.02, 1e-3),     # ragged row tile
    (333, 1088, 3, 3.0, 1e-2),     # ragged rows, K not a multiple of 256
])
def test_quantize_bit_exact(M, K, seed, std, out):
    _quantize_and_compare(synth.normal_bf16((M, K), seed, std, out))


@pytest.mark.parametrize("M,K", [(1000, 64 * 37), (4096 + 7, 1024 + 64), (129, 64)])
def test_quantize_ragged_edges_bit_exact(M, K):
    # K not a multiple of 256 (partial last CTA column group), rows not a multiple of 128,
    # a single 64-column group
    _quantize_and_compare(synth.normal_bf16((M, K), 9, 0.5, 1e-3))


def test_quantize_adversarial_blocks():
    K = 256
    rows = []
    # ties of the E2M1 grid after division by a power-of-two block scale
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2, dtype=np.float32)
    rows.append(np.concatenate([ties, -ties] * 8))
    rows.append(np.zeros(K, dtype=np.float32))                       # all-zero blocks
    one = np.zeros(K, dtype=np.float32)
    one[::16] = np.float32(3.0)                                       # single nonzero per block
    rows.append(one)
    rows.append(np.full(K, 1e30, dtype=np.float32))                   # saturating blocks
    tiny = np.zeros(K, dtype=np.float32)
    tiny[::7] = np.float32(1e-30)                                     # scale underflows to 0
    rows.append(tiny)
    rows.append(np.where(np.arange(K) % 2 == 0, -1e-6, 2.0).astype(np.float32))  # -0 codes
    x = np.stack(rows)
    xb = synth.f32_to_bf16_bits(x)
    # a power-of-two global scale keeps every block scale exact (ties stay ties)
    _quantize_and_compare(xb, np.float32(2.0 ** -6))
    _quantize_and_compare(xb)


def test_quantize_prefill_size_bit_exact():
    # the prefill workload's activations: 4096 x 8192 bf16, N(0,1) + 0.1% outliers x20
    xb = synth.normal_bf16((4096, 8192), 8, 1.0, 1e-3)
    _quantize_and_compare(xb)


@pytest.mark.parametrize("g", [1e-30, 3e-36, 1e30, 2.5e35])
def test_quantize_extreme_global_scales_bit_exact(g):
    # block scales (amax / 6) / g far above 448 (saturate) or far below the smallest E4M3
    # subnormal (all codes zero): the quotients leave the fast path's exact range
    xb = synth.normal_bf16((256, 512), 10, 1.0, 1e-2)
    _quantize_and_compare(xb, np.float32(g))


@pytest.mark.parametrize("n", [1, 7, 9, 2047, 8 * 1024 * 37 + 5, 33554432 + 3])
def test_amax_any_length_bit_exact(n):
    # every CTA sweeps one contiguous range of 16-byte vectors; the last CTA also takes the
    # elements past the last whole vector. The largest |x| sits in the scalar tail, at a
    # range boundary and at the start in turn.
    xb = synth.normal_bf16((n,), 71, 1.0, 1e-3)
    big = np.array([0x4480], dtype=np.uint16)  # 1024.0, above every drawn value
    for pos in {n - 1, (n // 8) * 8 - 1 if n >= 8 else 0, 0}:
        xi = xb.copy()
        xi[pos] = big[0] | (0x8000 if pos % 2 else 0)  # either sign
        amax, g = m.nvfp4_amax(to_dev(xi))
        torch.cuda.synchronize()
        assert np.float32(amax.item()) == np.float32(oracle.amax(xi)) == np.float32(1024.0)
        assert np.float32(g.item()) == oracle.global_scale(oracle.amax(xi))


def test_amax_zero_tensor_gives_unit_scale():
    x = torch.zeros(1000, dtype=torch.bfloat16, device=dev())
    amax, g = m.nvfp4_amax(x)
    assert amax.item() == 0.0 and g.item() == 1.0


def test_quantize_quotients_near_every_rounding_boundary():
    # Per block: a random global scale g and block maximum, then elements whose quotients
    # x / (E4M3(s) g) fall within a few ulps of every E2M1 rounding threshold (0.25, 0.75,
    # 1.25, 1.75, 2.5, 3.5, 5) and the saturation point 6, with both signs. The quantiser
    # must round each of them exactly as the oracle's float32 division does.
    rng = np.random.default_rng(77)
    rows = 256
    K = 1024
    x = np.zeros((rows, K), dtype=np.float32)
    g = np.float32(rng.uniform(1e-3, 2.0))
    thresholds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], dtype=np.float32)
    for r in range(rows):
        for b in range(K // 16):
            amax = np.float32(rng.uniform(0.5, 3000.0) * g)
            t = np.float32(np.float32(amax / np.float32(6.0)) / g)
            s = oracle.e4m3_encode(min(float(t), 448.0))
            d = np.float32(np.float32(oracle.e4m3_value(s)) * g)
            thr = rng.choice(thresholds, size=15)
            jitter = rng.integers(-3, 4, size=15).astype(np.float64)
            vals = thr.astype(np.float64) * float(d) * (1.0 + jitter * 2.0 ** -9)
            vals *= rng.choice([-1.0, 1.0], size=15)
            blk = np.concatenate([[amax], vals]).astype(np.float32)
            x[r, b * 16:(b + 1) * 16] = blk
    xb = synth.f32_to_bf16_bits(x)
    _quantize_and_compare(xb, g)


def _global_scales_for_division_sweep():
    rng = np.random.default_rng(2024)
    g = list(np.float32(2.0 ** rng.uniform(-60.0, 60.0, 320)))
    g += [np.float32(v) for v in (2.0 ** -10, 1.0, 2.0 ** 10, 1.0 / 2688, 20.0 / 2688, 0.08 / 2688)]
    # the fast path's guard edges: block scales d = E4M3(s) g landing around 1e-30 and 1e30
    for s in (1, 8, 56, 100, 126):
        v = oracle.e4m3_value(s)
        for edge in (1e-30, 1e30):
            c = np.float32(edge / v)
            g += [c, np.nextafter(c, np.float32(0)), np.nextafter(c, np.float32(np.inf))]
    g += [np.float32(v) for v in (1e-30, 1e30, 1e-36, 1e36)]
    return [x for x in g if np.isfinite(x) and x > 0]


def _blocks_for_every_quotient(g):
    """For each E4M3 scale code s a block maximum A (the largest bf16 at or below
    6 g E4M3(s)), then every bf16 magnitude in [A / 64, A] with both signs (the
    quotients from 0.09 to 6.x, where the E2M1 code can change), 15 per block after
    a leading +-A, plus a few smaller values down to subnormals and zero."""
    rng = np.random.default_rng(int(np.float32(g).view(np.uint32)))
    blocks = []
    for s in range(1, 127):
        a64 = 6.0 * float(g) * oracle.e4m3_value(s)
        if not a64 < 3.0e38:  # beyond bf16's finite range
            continue
        a = np.float32(a64)
        a_bits = int(a.view(np.uint32)) >> 16  # round down to bf16
        if a_bits == 0 or a_bits >= 0x7F80:
            continue
        lo = np.float32(float(synth.bf16_bits_to_f32(np.array([a_bits], np.uint16))[0]) / 64.0)
        lo_bits = max(1, (int(lo.view(np.uint32)) + 0xFFFF) >> 16)
        mags = np.arange(lo_bits, a_bits + 1, dtype=np.uint32)
        small = rng.integers(0, max(lo_bits, 2), 24, dtype=np.uint32)
        vals = np.concatenate([mags, mags | 0x8000, small, small | 0x8000]).astype(np.uint16)
        rng.shuffle(vals)
        n = (len(vals) + 14) // 15
        vals = np.concatenate([vals, np.zeros(n * 15 - len(vals), np.uint16)]).reshape(n, 15)
        lead = np.where(rng.random(n) < 0.5, a_bits, a_bits | 0x8000).astype(np.uint16)
        blocks.append(np.concatenate([lead[:, None], vals], axis=1))
    return np.concatenate(blocks) if blocks else np.zeros((0, 16), np.uint16)


def test_quantize_division_exact_for_every_bf16_quotient():
    # The quantiser divides without a division instruction (reciprocal + two fma
    # corrections, correctly rounded by Markstein's theorem inside a guarded range, IEEE
    # division outside it). Over 350 global scales (random over 2^+-60 and the guard's
    # edges) and every E4M3 block scale, every bf16 element whose quotient can decide an
    # E2M1 code is quantised and compared with the oracle's IEEE division, bit for bit.
    K = 2048
    per_row = K // 16
    mismatches = 0
    for g in _global_scales_for_division_sweep():
        blk = _blocks_for_every_quotient(g)
        if len(blk) == 0:
            continue
        rows = (len(blk) + per_row - 1) // per_row
        xb = np.zeros((rows * per_row, 16), np.uint16)
        xb[:len(blk)] = blk
        xb = xb.reshape(rows, K)
        x = to_dev(xb)
        gd = torch.tensor([float(g)], dtype=torch.float32, device=dev())
        q, sf = m.nvfp4_quantize(x, gd)
        qo, sfo, _ = oracle.quantize(xb, np.float32(g))
        qg, sfg = q.cpu().numpy(), sf.cpu().numpy()
        bad = int((qg != qo).sum() + (sfg != sfo).sum())
        assert bad == 0, f"g = {float(g)!r}: {bad} code or scale bytes differ"
        mismatches += bad
    assert mismatches == 0
