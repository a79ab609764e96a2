"""Pins for the oracle's E4M3 / UE8M0 codecs (CPU only).

The codec is pinned to PyTorch's own CPU float8_e4m3fn casts (an independent
library implementation of the same OCP format) exhaustively, and to the
ties-to-even rule at every midpoint.
"""
import numpy as np
import pytest
import torch

from oracle.e4m3 import e4m3_decode, e4m3_encode, ue8m0_to_float, E4M3_MAX


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_all_codes():
    ours = e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = _torch_decode_all()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))
    assert np.nanmax(ours) == E4M3_MAX == 448.0
    assert set(np.flatnonzero(nan)) == {0x7F, 0xFF}


def test_encode_decode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(e4m3_encode(e4m3_decode(codes)), codes)


def _all_finite_bf16_as_f32():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    v = bits.view(torch.bfloat16).to(torch.float32)
    return v[torch.isfinite(v)]


@pytest.mark.parametrize("shift", list(range(-140, 130, 7)) + [0, 1, -1, 2, -2, -6, -9, -10])
def test_encode_matches_torch_on_all_bf16_times_power_of_two(shift):
    """Every finite bf16 value times 2^shift that lies within E4M3's range is
    cast by the oracle exactly as torch casts it."""
    v = _all_finite_bf16_as_f32().to(torch.float64) * (2.0 ** shift)
    v = v[(v.abs() <= E4M3_MAX) & (v.abs() < 3.4e38)]
    v32 = v.to(torch.float32)
    exact = v32.to(torch.float64) == v                   # keep values float32 holds exactly
    v, v32 = v[exact], v32[exact]
    assert v.numel() > 0
    ref = v32.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = e4m3_encode(v.numpy())
    bad = np.flatnonzero(ours != ref)
    assert bad.size == 0, (v.numpy()[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_ties_round_to_even_at_every_midpoint():
    vals = e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8))    # 0 .. 448 ascending
    assert np.all(np.diff(vals) > 0)
    mids = (vals[:-1] + vals[1:]) / 2.0
    got = e4m3_encode(mids)
    lo = np.arange(0x00, 0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    assert np.array_equal(e4m3_encode(-mids), want | 0x80)


def test_signed_zero_and_underflow():
    assert e4m3_encode(np.array([0.0]))[0] == 0x00
    assert e4m3_encode(np.array([-0.0]))[0] == 0x80
    # below half the smallest subnormal (2^-9) rounds to a signed zero
    assert e4m3_encode(np.array([2.0 ** -11]))[0] == 0x00
    assert e4m3_encode(np.array([-(2.0 ** -11)]))[0] == 0x80
    # exactly half of 2^-9 is a tie between 0 (even) and 2^-9 (odd) -> 0
    assert e4m3_encode(np.array([2.0 ** -10]))[0] == 0x00
    assert e4m3_encode(np.array([1.5 * 2.0 ** -10]))[0] == 0x01


def test_saturation_above_448():
    assert e4m3_encode(np.array([480.0, 1e6, -1e6])).tolist() == [0x7E, 0x7E, 0xFE]


def test_ue8m0_values():
    b = np.arange(255)
    assert np.array_equal(ue8m0_to_float(b), np.ldexp(1.0, b - 127))
    assert ue8m0_to_float(127) == 1.0
    assert np.isnan(ue8m0_to_float(255))
