"""Pins for the fp8 (E4M3) cache oracle.

The codec is written from the format's definition; it is pinned here by
values the definition fixes (largest finite 448, smallest subnormal 2^-9,
1.0 = 0x38, the NaN pattern), by torch's own float8_e4m3fn conversion (an
independent implementation) on every representable value and on many
random in-range values including exact midpoints, and by the
round-to-nearest-even rule on midpoints.  The scale rule and the
row quantiser are pinned by their error bound (half an E4M3 step of the
scaled value) and by the saturation of the largest element to exactly 448.
"""

import numpy as np
import pytest
import torch

from oracle.fp8_cache import (E4M3_MAX, dequantize_row, e4m3_to_float, e4m3_to_float_array, float_to_e4m3,
                              float_to_e4m3_array, gather_dequantized, quantize_row, quantize_rows,
                              reshape_and_cache_fp8)


def test_definition_values():
    assert e4m3_to_float(0x7E) == 448.0 and e4m3_to_float(0xFE) == -448.0
    assert e4m3_to_float(0x01) == 2.0 ** -9
    assert e4m3_to_float(0x08) == 2.0 ** -6            # smallest normal
    assert e4m3_to_float(0x38) == 1.0
    assert np.isnan(e4m3_to_float(0x7F)) and np.isnan(e4m3_to_float(0xFF))
    assert float_to_e4m3(448.0) == 0x7E and float_to_e4m3(1e9) == 0x7E and float_to_e4m3(-1e9) == 0xFE
    assert float_to_e4m3(1.0) == 0x38 and float_to_e4m3(0.0) == 0x00


def test_decode_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    theirs = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([e4m3_to_float(c) for c in range(256)])
    nan = np.isnan(theirs)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ours[~nan], theirs[~nan])


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    vals = np.array([e4m3_to_float(c) for c in range(256) if c not in (0x7F, 0xFF)])
    mids = (np.sort(vals)[:-1] + np.sort(vals)[1:]) / 2           # exact ties
    x = np.concatenate([vals, mids, rng.standard_normal(20000) * 40, rng.uniform(-448, 448, 20000),
                        rng.standard_normal(5000) * 1e-3]).astype(np.float32)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = float_to_e4m3_array(x)
    # torch keeps the sign of zero; so does the oracle
    assert np.array_equal(ours, theirs)
    assert np.array_equal(ours[:500], np.array([float_to_e4m3(v) for v in x[:500]], dtype=np.uint8))


def test_ties_go_to_even():
    # 1.0 = 0x38 and 1.125 = 0x39: the midpoint rounds to the even code 0x38;
    # 1.125 and 1.25 (0x3A): the midpoint rounds to 0x3A
    assert float_to_e4m3(1.0625) == 0x38
    assert float_to_e4m3(1.1875) == 0x3A
    assert float_to_e4m3(2.0 ** -10) == 0x00            # half the smallest subnormal
    assert float_to_e4m3(3 * 2.0 ** -10) == 0x02        # between 0x01 and 0x02: even
    # 448 + half a step would round up to a value past 448: saturates
    assert float_to_e4m3(464.0) == 0x7E


def test_round_trip_of_every_finite_code():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = e4m3_to_float(c)
        got = float_to_e4m3(v)
        assert got == c or (v == 0 and got in (0x00, 0x80))


def test_row_quantiser_bound_and_saturation():
    rng = np.random.default_rng(1)
    for scale_in in (1e-3, 0.5, 1.0, 30.0):
        row = (rng.standard_normal(128) * scale_in).astype(np.float32)
        codes, s = quantize_row(row)
        assert s == np.float32(np.max(np.abs(row))) / np.float32(448)
        assert abs(e4m3_to_float(codes[np.argmax(np.abs(row))])) == 448.0
        deq = dequantize_row(codes, s)
        # |x / s - code| is at most half the E4M3 step at that magnitude (1/16 relative) ...
        rel = np.abs(deq - row.astype(np.float64)) / np.maximum(np.abs(row.astype(np.float64)), 2.0 ** -6 * s)
        assert np.all(rel <= 1.0 / 16 + 1e-6)
    codes, s = quantize_row(np.zeros(64, dtype=np.float32))
    assert s == 1.0 and not codes.any()
    batch = (rng.standard_normal((3, 5, 64)) * 2).astype(np.float32)
    c2, s2 = quantize_rows(batch)
    for i in range(3):
        for j in range(5):
            c1, s1 = quantize_row(batch[i, j])
            assert np.array_equal(c1, c2[i, j]) and s1 == s2[i, j]
    assert np.array_equal(e4m3_to_float_array(c2[0, 0]), np.array([e4m3_to_float(c) for c in c2[0, 0]]))


def test_quantised_scatter_and_gather():
    rng = np.random.default_rng(2)
    nb, bs, hkv, d = 6, 4, 2, 16
    kc = np.zeros((nb, bs, hkv, d), np.uint8)
    vc = np.zeros_like(kc)
    ks = np.full((nb, hkv, bs), np.nan, np.float32)
    vs = np.full_like(ks, np.nan)
    k = rng.standard_normal((7, hkv, d)).astype(np.float32)
    v = rng.standard_normal((7, hkv, d)).astype(np.float32)
    table = [4, 1]
    slots = [table[p // bs] * bs + p % bs for p in range(6)] + [-1]
    reshape_and_cache_fp8(k, v, kc, vc, ks, vs, slots)
    assert np.isnan(ks[0]).all() and np.isnan(ks[1, :, 2:]).all()     # untouched
    got = gather_dequantized(kc, ks, table, 6)
    for t in range(6):
        for h in range(hkv):
            c, s = quantize_row(k[t, h])
            assert np.array_equal(got[t, h], dequantize_row(c, s))
    with pytest.raises(ValueError):
        reshape_and_cache_fp8(k, v, kc, vc, ks, vs, [nb * bs])
    assert E4M3_MAX == 448.0
