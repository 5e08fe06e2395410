"""Pins of the oracle's E4M3 and bf16 codecs against the format definitions,
brute force and a library implementation (torch's CPU float8/bfloat16 casts)."""
import numpy as np
import torch

from oracle import (bf16_decode, bf16_encode, e4m3_decode, e4m3_encode,
                    e4m3_encode_bruteforce)


def test_e4m3_decode_closed_forms():
    # OCP E4M3FN: bias 7, 3 mantissa bits, no infinities, one NaN pattern per sign.
    d = e4m3_decode(np.arange(256, dtype=np.uint8))
    assert d[0x00] == 0.0 and np.signbit(d[0x80])
    assert d[0x01] == 2.0 ** -9            # smallest subnormal
    assert d[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert d[0x08] == 2.0 ** -6            # smallest normal
    assert d[0x38] == 1.0 and d[0x40] == 2.0 and d[0x3C] == 1.5
    assert d[0x7E] == 448.0 and d[0xFE] == -448.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.array_equal(d[0x80:0xFF], -d[0x00:0x7F])


def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    ours = e4m3_decode(np.arange(256, dtype=np.uint8))
    same = (ref == ours) | (np.isnan(ref) & np.isnan(ours))
    assert same.all()


def test_e4m3_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bf16_decode(bits)
    return v[~np.isnan(v)]


def test_e4m3_encode_matches_torch_on_every_bf16_in_range():
    # torch's cast is round-to-nearest-even without saturation: compare where it
    # cannot overflow (|v| <= 464, the tie between 448 and the NaN slot).
    v = _all_bf16_values()
    v = v[np.abs(v) <= 464.0]
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(v), ref)


def test_e4m3_encode_matches_bruteforce():
    rng = np.random.default_rng(0)
    vals = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2                       # exact ties
    pts = np.concatenate([
        vals, -vals, mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9),
        [0.0, -0.0, 1e-9, -1e-9, 2.0 ** -10, -2.0 ** -10, 448.0, 449.0, 463.9, 464.0,
         465.0, 1e6, -1e6, np.inf, -np.inf],
        rng.standard_normal(400) * 50, rng.standard_normal(200) * 0.01,
    ])
    assert np.array_equal(e4m3_encode(pts), e4m3_encode_bruteforce(pts))


def test_e4m3_encode_saturation_and_signed_zero():
    got = e4m3_encode(np.array([500.0, 1e30, np.inf, -500.0, -np.inf, -0.0, -1e-12, 0.0]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x80, 0x80, 0x00]
    assert e4m3_encode(np.array([np.nan]))[0] == 0x7F


def test_bf16_encode_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(100000) * 10.0 ** rng.integers(-20, 20, 100000),
                        [0.0, -0.0, 1.0, -1.0, 3.0e38]]).astype(np.float32)
    # add exact bf16 midpoints (ties) and their neighbours
    base = torch.from_numpy(rng.standard_normal(1000).astype(np.float32)).to(torch.bfloat16)
    b = base.view(torch.int16).numpy().astype(np.uint16).astype(np.uint32)
    mid = ((b << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, mid, np.nextafter(mid, np.float32(np.inf)),
                        np.nextafter(mid, np.float32(-np.inf))])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(bf16_encode(x.astype(np.float64)), ref)


def test_bf16_encode_rounds_float64_once():
    # 1 + 2^-8 is the exact midpoint between bf16 1.0 and 1.0078125 -> even (1.0);
    # 1 + 2^-8 + 2^-40 is above it and must round up even though float32 would
    # first round it back to the midpoint.
    got = bf16_encode(np.array([1 + 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -40, 1 + 3 * 2.0 ** -8]))
    assert list(bf16_decode(got)) == [1.0, 1.0078125, 1.015625]


def test_bf16_decode_is_exact():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = bf16_decode(bits)
    ok = ~np.isnan(v)
    assert np.array_equal(bf16_encode(v[ok]), bits[ok])
