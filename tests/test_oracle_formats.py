"""Oracle number formats pinned to library routines and brute force.

E4M3FN decode: torch.float8_e4m3fn (a library dtype) over all 256 codes.
E4M3FN encode: brute-force nearest-even search over that library table for
every fp16 input, every midpoint +-1 ulp and random fp32; the library cast
for in-range values; saturation at 448 for finite overflow and infinities.
fp16 decode: numpy's float16 over all 65,536 patterns.
"""
import numpy as np
import pytest
import torch

import oracle


def lib_table():
    return (torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
            .to(torch.float64).numpy())


def test_e4m3_decode_table_matches_library():
    ours = oracle.e4m3_decode_table()
    ref = lib_table()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_half_decode_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    ours = np.array([oracle.half_to_double(b) for b in range(0, 65536, 1)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def brute_force_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 value by exhaustive search over the library table,
    ties to the even code; sign kept (incl. -0); NaN -> NaN."""
    t = lib_table()
    pos_codes = np.arange(0, 0x7F)  # 0x00..0x7E, finite, non-negative
    vals = t[pos_codes]
    x = np.asarray(x, np.float32).astype(np.float64)
    # Above the largest finite value every |x| has the same nearest value
    # (448); clipping at 896 keeps that answer and keeps the float64
    # distances exact for huge inputs.
    a = np.minimum(np.abs(x), 896.0)
    d = np.abs(a[:, None] - vals[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    # prefer even codes among ties
    even = cand & (pos_codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    code = pos_codes[pick].astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    code = np.where(np.isnan(x), (code & 0x80) | 0x7F, code).astype(np.uint8)
    return code


def test_encoder_all_fp16_inputs_brute_force():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16).astype(np.float32)
    fin = np.isfinite(x)
    ours = oracle.e4m3_encode_array(x)
    ref = brute_force_encode(x[fin])
    assert np.array_equal(ours[fin], ref)
    # infinities saturate to +-448
    inf = np.isinf(x)
    assert set(ours[inf & (x > 0)]) == {0x7E} and set(ours[inf & (x < 0)]) == {0xFE}
    nan = np.isnan(x)
    assert set(ours[nan] & 0x7F) == {0x7F}


def test_encoder_midpoints_and_neighbours():
    t = lib_table()
    vals = t[0:0x7F]
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (vals[:-1] + vals[1:]) / 2)  # exact
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(0))
    beyond = np.array([448, 456, 463.99997, 464, 464.00003, 479.9, 480, 500, 1e6,
                       3.4e38], np.float32)
    xs = np.concatenate([mids, up, dn, beyond])
    xs = np.concatenate([xs, -xs])
    assert np.array_equal(oracle.e4m3_encode_array(xs), brute_force_encode(xs))


def test_encoder_random_fp32_brute_force():
    rng = np.random.Generator(np.random.PCG64(11))
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * np.float32(50),
        (rng.standard_normal(50000) * 2.0 ** rng.integers(-20, 10, 50000)).astype(np.float32),
        rng.uniform(-2 ** -8, 2 ** -8, 50000).astype(np.float32),
    ])
    assert np.array_equal(oracle.e4m3_encode_array(x), brute_force_encode(x))


def test_encoder_agrees_with_library_cast_in_range():
    rng = np.random.Generator(np.random.PCG64(12))
    x = (rng.standard_normal(200000) * 100).astype(np.float32)
    x = x[np.abs(x) < 464]  # the library cast turns overflow into NaN
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode_array(x), ref)


def test_encode_decode_round_trip_and_monotone():
    t = oracle.e4m3_decode_table()
    finite = [c for c in range(256) if not np.isnan(t[c])]
    assert len(finite) == 254
    for c in finite:
        assert oracle.e4m3_from_float(np.float32(t[c])) == c
    xs = np.linspace(-500, 500, 20001, dtype=np.float32)
    dec = t[oracle.e4m3_encode_array(xs)]
    assert np.all(np.diff(dec) >= 0)


@pytest.mark.parametrize("scale", [1.0, 0.0123, 3.7e-3, 448.0 / 5.25])
def test_quantize_is_fp32_divide_then_one_rounding(scale):
    rng = np.random.Generator(np.random.PCG64(13))
    v = rng.standard_normal(100000).astype(np.float32) * np.float32(2.0)
    s = np.float32(scale)
    x = v / s  # numpy float32 IEEE division
    ours = oracle.quantize_array(v, s)
    assert np.array_equal(ours, brute_force_encode(x))
    fin = np.abs(x) < 464
    ref = torch.from_numpy(x[fin]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours[fin], ref)


def test_quantize_fp16_input_widens_exactly():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    v16 = bits.view(np.float16)
    v16 = v16[np.isfinite(v16)]
    s = np.float32(0.031)
    ours = oracle.quantize_array(v16, s)
    assert np.array_equal(ours, brute_force_encode(v16.astype(np.float32) / s))
