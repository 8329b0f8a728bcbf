"""Pins for the oracle's format functions (CPU only).

Each check compares the oracle against something other than itself: the
hand-listed golden tables, torch's float8_e4m3fn conversions (a library
routine), and a vectorised brute-force nearest-value search written here.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    rows = []
    with open(os.path.join(GOLD, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_e2m1_table_matches_golden():
    for code, val in _read("e2m1_values.txt"):
        v = oracle.e2m1_value(int(code))
        assert v == float(val)
        assert math.copysign(1.0, v) == math.copysign(1.0, float(val))


def test_e4m3_landmarks_match_golden():
    for code, val in _read("e4m3_points.txt"):
        v = oracle.e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(v)
        else:
            assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))


def test_e4m3_all_codes_match_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]


def test_e4m3_decode_encode_roundtrip_every_finite_code():
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(v):
            continue
        assert oracle.e4m3_encode(v) == c


def test_e2m1_decode_encode_roundtrip():
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_value(c)) == c


def test_e2m1_rounding_golden():
    for v, code in _read("e2m1_rounding.txt"):
        assert oracle.e2m1_encode(float(v)) == int(code), v


def _brute_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest E2M1 magnitude by exhaustive distance, ties to even code, sign kept."""
    mags = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - mags[None, :])
    best = d.min(axis=1, keepdims=True)
    tied = d == best
    idx = np.arange(8)[None, :]
    # prefer the lowest even index among the nearest, else the nearest index
    even_pick = np.where(tied & (idx % 2 == 0), idx, 99).min(axis=1)
    any_pick = np.where(tied, idx, 99).min(axis=1)
    code = np.where(even_pick < 99, even_pick, any_pick)
    code = np.where(a > 6.0, 7, code)
    return (code | (np.signbit(v).astype(np.int64) << 3)).astype(np.uint8)


def test_e2m1_encode_exhaustive_over_decision_range():
    # every float32 in [2^-3, 2^4) (all rounding decisions happen there), both signs
    lo = np.float32(0.125).view(np.uint32)
    hi = np.float32(16.0).view(np.uint32)
    step = 1 << 22
    for s in range(int(lo), int(hi), step):
        bits = np.arange(s, min(s + step, int(hi)), dtype=np.uint32)
        v = bits.view(np.float32)
        assert np.array_equal(oracle.e2m1_encode_array(v), _brute_e2m1(v))
        assert np.array_equal(oracle.e2m1_encode_array(-v), _brute_e2m1(-v))


def test_e2m1_encode_small_and_large_values():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    assert np.array_equal(oracle.e2m1_encode_array(v), _brute_e2m1(v))


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_in_range():
    # all float32 in [2^-12, 448]: torch's conversion is round-to-nearest-even there
    mids = []
    for c in range(0, 0x7E):
        a, b = oracle.e4m3_value(c), oracle.e4m3_value(c + 1)
        m = np.float32((a + b) / 2)
        mb = int(m.view(np.uint32))
        mids.append(np.arange(mb - 64, mb + 65, dtype=np.uint32))
    v = np.concatenate(mids).view(np.float32)
    rng = np.random.default_rng(3)
    v = np.concatenate([v, rng.uniform(0, 448, 1 << 18).astype(np.float32),
                        np.exp2(rng.uniform(-14, 8.8, 1 << 18)).astype(np.float32)])
    v = v[(v >= 0) & (v <= 448)]
    assert np.array_equal(oracle.e4m3_encode_array(v), _torch_e4m3(v))


def test_e4m3_encode_saturates_and_underflows():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # half the smallest subnormal: tie -> even (0)
    assert oracle.e4m3_encode(np.nextafter(np.float32(2.0 ** -10), np.float32(1))) == 0x01
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02  # tie between 1 and 2 -> even
    assert oracle.e4m3_encode(0.0) == 0x00


def test_scale_layout_is_a_bijection_with_tile_structure():
    for rows, K in [(1, 64), (128, 256), (130, 192), (300, 1024)]:
        kc = K // 16
        n = oracle.scale_bytes(rows, K)
        assert n == ((rows + 127) // 128) * 128 * (((kc + 3) // 4) * 4)
        offs = np.array([[oracle.sf_offset(r, c, K) for c in range(kc)] for r in range(rows)])
        assert len(np.unique(offs)) == rows * kc and offs.max() < n and offs.min() >= 0
        # each 512-byte block holds exactly one 128-row x 4-column tile
        for r in range(rows):
            for c in range(kc):
                blk = offs[r, c] // 512
                assert blk == (r // 128) * ((kc + 3) // 4) + c // 4
        # neighbouring scale columns are adjacent bytes; rows r, r+1 are 16 bytes
        # apart within a 32-row group; rows r, r+32 are 4 bytes apart
        if kc >= 2:
            assert offs[0, 1] - offs[0, 0] == 1
        if rows >= 33:
            assert offs[1, 0] - offs[0, 0] == 16 and offs[32, 0] - offs[0, 0] == 4
    lin = np.random.default_rng(1).integers(0, 256, size=(200, 48), dtype=np.uint8)
    sw = oracle.sf_swizzle(lin, 200, 768)
    assert np.array_equal(oracle.sf_unswizzle(sw, 200, 768), lin)
    # padding bytes are zero
    mask = np.ones(sw.size, dtype=bool)
    for r in range(200):
        for c in range(48):
            mask[oracle.sf_offset(r, c, 768)] = False
    assert not sw[mask].any()
