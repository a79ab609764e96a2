"""Pins for the oracle's column-block quantiser (CPU only).

The scale exponent is pinned to an integer rule on float32 bit patterns (a
different method from the oracle's frexp) and to its defining inequality; the
whole quantiser is pinned to a brute-force nearest-value search in exact
rational arithmetic on small inputs, and to the E4M3 round-trip error bounds.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from grouped_fp8_weight_gb300 import workloads
from oracle.e4m3 import e4m3_decode
from oracle.quant import quant_colblock, scale_exponent


def _exp_from_f32_bits(amax_f32: np.ndarray) -> np.ndarray:
    """448 = 1.75 * 2^8, so for amax = f 2^q (f in [1, 2)):
    ceil(log2(amax/448)) = q - 8 + (f > 1.75); subnormal or zero -> clamp."""
    bits = amax_f32.astype(np.float32).view(np.uint32).astype(np.int64)
    ef = (bits >> 23) & 0xFF
    mant = bits & 0x7FFFFF
    e = (ef - 127) - 8 + (mant > 0x600000)
    e = np.where(ef == 0, -127, e)
    return np.clip(e, -127, 127)


def test_scale_exponent_matches_bit_rule():
    rng = np.random.default_rng(1)
    amax = np.concatenate([
        np.abs(rng.standard_normal(20000)).astype(np.float32),
        np.ldexp(np.float32(1.75), np.arange(-126, 128)).astype(np.float32),
        np.nextafter(np.ldexp(np.float32(1.75), np.arange(-126, 127)).astype(np.float32),
                     np.float32(np.inf)),
        np.ldexp(np.float32(1.0), np.arange(-149, 128)).astype(np.float32),
        np.array([0.0, 448.0, 449.0, 447.9, 3.3895e38, 1e-40, 2.0 ** -119, 2.0 ** -120],
                 dtype=np.float32),
    ])
    assert np.array_equal(scale_exponent(amax.astype(np.float64)), _exp_from_f32_bits(amax))


def test_scale_exponent_defining_inequality():
    rng = np.random.default_rng(2)
    amax = np.ldexp(rng.uniform(1, 2, 5000), rng.integers(-100, 100, 5000))
    e = scale_exponent(amax)
    r = amax / 448.0
    assert np.all(np.ldexp(1.0, e) >= r)
    assert np.all(np.ldexp(1.0, e - 1) < r)


def test_scale_exponent_edge_values():
    assert scale_exponent(np.array([448.0]))[0] == 0
    assert scale_exponent(np.array([448.0 * (1 + 2 ** -20)]))[0] == 1
    assert scale_exponent(np.array([224.0]))[0] == -1
    assert scale_exponent(np.array([0.0]))[0] == -127
    assert scale_exponent(np.array([1e-45]))[0] == -127
    assert scale_exponent(np.array([3.3895e38]))[0] == 120


_E4M3_CODES = [(Fraction(float(v)), c) for c, v in
               enumerate(e4m3_decode(np.arange(256, dtype=np.uint8)))
               if np.isfinite(v)]


def _brute_quant_value(y: Fraction, negative: bool) -> int:
    """Nearest E4M3 code of the given sign to y; ties go to the even code."""
    cands = [(v, c) for v, c in _E4M3_CODES if bool(c & 0x80) == negative]
    return min(cands, key=lambda vc: (abs(vc[0] - y), vc[1] & 1))[1]


def _brute_quant(x: np.ndarray, gran_k: int):
    T, C = x.shape
    q = np.zeros((T, C), dtype=np.uint8)
    sf = np.zeros((T // gran_k, C), dtype=np.uint8)
    for kb in range(T // gran_k):
        for c in range(C):
            rows = range(kb * gran_k, (kb + 1) * gran_k)
            amax = max(abs(Fraction(float(x[k, c]))) for k in rows)
            e = -127                      # smallest e with amax <= 448 * 2^e
            while e < 127 and amax > 448 * Fraction(2) ** e:
                e += 1
            sf[kb, c] = e + 127
            for k in rows:
                y = Fraction(float(x[k, c])) / Fraction(2) ** e
                q[k, c] = _brute_quant_value(y, bool(np.signbit(x[k, c])))
    return q, sf


@pytest.mark.parametrize("gran_k", [32, 128])
def test_quant_matches_brute_force_small(gran_k):
    x = workloads.randn((256, 6), seed=11, dtype=torch.bfloat16).float().numpy()
    x[:, 1] *= 1e-30          # tiny column
    x[:, 2] = 0.0             # zero column
    x[5, 2] = -0.0
    x[:, 3] *= 1e20           # huge column
    x[:40, 4] = -1e-40        # negative subnormals in one block
    q, sf = quant_colblock(x, gran_k)
    qb, sfb = _brute_quant(x, gran_k)
    assert np.array_equal(sf, sfb)
    assert np.array_equal(q, qb)


@pytest.mark.parametrize("gran_k", [32, 128])
def test_quant_roundtrip_bounds(gran_k):
    x = workloads.randn((1024, 96), seed=3).numpy().astype(np.float64)
    x[:, :8] *= 1e-3
    q, sf = quant_colblock(x, gran_k)
    e = sf.astype(np.int64) - 127
    scale = np.ldexp(1.0, np.repeat(e, gran_k, axis=0))
    y = e4m3_decode(q) * scale
    xs = x / scale
    normal = np.abs(xs) >= 2.0 ** -6
    assert np.all(np.abs(y - x)[normal] <= 2.0 ** -4 * np.abs(x)[normal])
    assert np.all(np.abs(y - x)[~normal] <= 2.0 ** -10 * scale[~normal])
    # The scale is tight: each block's largest element lands in (224, 448].
    blk_max = np.abs(xs).reshape(-1, gran_k, x.shape[1]).max(axis=1)
    assert np.all((blk_max > 224) & (blk_max <= 448))


def test_channel_layout_is_transpose_of_token_layout():
    x = workloads.randn((384, 48), seed=5).numpy()
    q_t, sf_t = quant_colblock(x, 128, "token")
    q_c, sf_c = quant_colblock(x, 128, "channel")
    assert q_c.shape == (48, 384)
    assert np.array_equal(q_c, q_t.T)
    assert np.array_equal(sf_c, sf_t)


def test_quant_rejects_bad_arguments():
    with pytest.raises(ValueError):
        quant_colblock(np.zeros((100, 4)), 128)
    with pytest.raises(ValueError):
        quant_colblock(np.zeros((128, 4)), 64)
