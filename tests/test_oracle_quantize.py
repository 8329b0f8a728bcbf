"""Pins for the oracle's quantisation recipe (CPU only).

The recipe (a reading: the pages name the formats but no recipe) is
  g = amax / 2688, s = E4M3((amax_block / 6) / g), q = E2M1(x / (E4M3(s) * g)).
Independent checks: a numpy/torch restatement per block, idempotence for
power-of-two global scales, single-nonzero / all-zero / saturating blocks.
"""
import numpy as np
import torch

import oracle
import synth


def _f32(bits):
    return synth.bf16_bits_to_f32(bits)


def _nearest_e2m1(v):
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[..., None] - mags)
    best = d.min(axis=-1, keepdims=True)
    idx = np.arange(8)
    tied = d == best
    even = np.where(tied & (idx % 2 == 0), idx, 99).min(axis=-1)
    anyp = np.where(tied, idx, 99).min(axis=-1)
    code = np.where(even < 99, even, anyp)
    code = np.where(a > 6, 7, code)
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def _restated_quantize(x_bits, g):
    """The recipe restated with numpy float32 ops and torch's E4M3 conversion."""
    x = _f32(x_bits)
    M, K = x.shape
    blk = x.reshape(M, K // 16, 16)
    amax = np.abs(blk).max(axis=-1).astype(np.float32)
    t = (amax / np.float32(6.0)) / np.float32(g)
    t = np.minimum(t, np.float32(448.0))  # saturating reading
    s = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    dec = torch.from_numpy(s.copy()).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    d = (dec * np.float32(g)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        v = (blk / d[..., None]).astype(np.float32)
    codes = _nearest_e2m1(v)
    codes[s == 0] = 0
    codes = codes.reshape(M, K)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return q, s


def test_amax_and_global_scale():
    x = synth.normal_bf16((64, 256), 11, 1.0, 1e-2)
    assert oracle.amax(x) == float(np.abs(_f32(x)).max())
    assert oracle.global_scale(2688.0) == np.float32(1.0)
    assert oracle.global_scale(0.0) == np.float32(1.0)
    assert oracle.global_scale(5.0) == np.float32(5.0) / np.float32(2688.0)


def test_quantize_matches_restatement_on_random_inputs():
    for seed, (M, K), std, out in [(0, (128, 256), 1.0, 0.0), (5, (200, 512), 0.02, 1e-3),
                                   (9, (33, 1024), 3.0, 1e-2)]:
        x = synth.normal_bf16((M, K), seed, std, out)
        q, sf, g = oracle.quantize(x)
        q2, s2 = _restated_quantize(x, g)
        assert np.array_equal(q, q2)
        assert np.array_equal(oracle.sf_unswizzle(sf, M, K), s2)


def test_quantize_idempotent_for_power_of_two_global_scale():
    rng = np.random.default_rng(2)
    M, K = 64, 256
    codes = rng.integers(0, 16, size=(M, K), dtype=np.uint8)
    # make each block's largest magnitude exactly 6 so the block scale is recovered
    codes[:, ::16] = 7
    scales = rng.integers(0x20, 0x60, size=(M, K // 16), dtype=np.uint8)
    q = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    sf = oracle.sf_swizzle(scales, M, K)
    g = np.float32(0.25)
    xhat = oracle.dequantize(q, sf, g, M, K)
    xb = synth.f32_to_bf16_bits(xhat.astype(np.float32))
    assert np.array_equal(_f32(xb).astype(np.float64), xhat)  # exactly representable in bf16
    q2, sf2, _ = oracle.quantize(xb, g)
    assert np.array_equal(q2, q)
    assert np.array_equal(sf2, sf)


def test_single_nonzero_block_maps_to_six():
    K = 64
    x = np.zeros((1, K), dtype=np.float32)
    x[0, 5] = -3.0
    x[0, 16 + 9] = 1.5
    g = np.float32(2.0 ** -6)
    q, sf, _ = oracle.quantize(synth.f32_to_bf16_bits(x), g)
    s = oracle.sf_unswizzle(sf, 1, K)[0]
    # (3 / 6) / 2^-6 = 32 and (1.5 / 6) / 2^-6 = 16 are exact E4M3 values
    assert oracle.e4m3_value(int(s[0])) == 32.0 and oracle.e4m3_value(int(s[1])) == 16.0
    assert q[0, 2] == 0xF0  # element 5 (odd -> high nibble) is -6
    assert q[0, 12] == 0x70  # element 25 (odd) is +6
    assert s[2] == 0 and s[3] == 0
    q[0, 2] = 0
    q[0, 12] = 0
    assert not q.any()


def test_all_zero_block_and_saturation():
    K = 32
    x = np.zeros((2, K), dtype=np.float32)
    x[1, :16] = 1000.0
    x[1, 16:] = -1e-30  # underflows to scale code 0 -> all-zero codes
    g = np.float32(2.0 ** -8)
    q, sf, _ = oracle.quantize(synth.f32_to_bf16_bits(x), g)
    s = oracle.sf_unswizzle(sf, 2, K)
    assert s[0, 0] == 0 and s[0, 1] == 0 and not q[0].any()
    assert s[1, 0] == 0x7E  # (1000/6)/2^-8 = 42666 saturates to 448
    assert (q[1, :8] == 0x77).all()  # 1000 / (448 * 2^-8) = 571 saturates to 6
    assert s[1, 1] == 0 and not q[1, 8:].any()


def test_global_scale_makes_tensor_max_land_on_448_times_six():
    x = synth.normal_bf16((128, 256), 21, 1.0, 1e-3)
    q, sf, g = oracle.quantize(x)
    s = oracle.sf_unswizzle(sf, 128, 256)
    assert s.max() == 0x7E  # the block holding the tensor's amax gets scale 448


def test_row_gather_commutes_with_quantisation():
    # Blocks run along K, so quantising gathered rows (with the same global scale) gives
    # exactly the gathered codes and scales of the quantised tensor; the routed-row path
    # (tokens quantised once, rows gathered by token) depends on this.
    T, K = 40, 320
    x = synth.normal_bf16((T, K), 71, 1.0, 1e-2)
    g = oracle.global_scale(oracle.amax(x))
    rows = np.random.default_rng(72).integers(0, T, size=97)  # repeats and omissions
    q_all, sf_all, _ = oracle.quantize(x, g)
    q_sel, sf_sel, _ = oracle.quantize(np.ascontiguousarray(x[rows]), g)
    assert np.array_equal(q_sel, q_all[rows])
    lin_all = oracle.sf_unswizzle(sf_all, T, K)
    lin_sel = oracle.sf_unswizzle(sf_sel, len(rows), K)
    assert np.array_equal(lin_sel, lin_all[rows])
