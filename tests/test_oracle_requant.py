"""Pins for the oracle's re-quantisation of stored FP8 activations and its MoE
token layout (CPU only).

Pinned against: a brute-force nearest-code search in exact rational arithmetic
(the forward 1 x 128 cast), torch's own E4M3 decoding times exact powers of
two (dequantisation), a closed form (stored tiles that already share one scale
per column block re-quantise to themselves), the exact power-of-two shift of
all scales, a Python loop (row gather), and invariants of the composed cast
(token permutations inside a block, padding rows).  The last test plants
mistakes in copies of the oracle and checks that these pins catch them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.quant as Q
from grouped_fp8_weight_gb300 import workloads
from oracle.e4m3 import e4m3_decode

_E4M3_CODES = [(Fraction(float(v)), c) for c, v in
               enumerate(e4m3_decode(np.arange(256, dtype=np.uint8)))
               if np.isfinite(v)]


def _nearest_code(y: Fraction, negative: bool) -> int:
    cands = [(v, c) for v, c in _E4M3_CODES if bool(c & 0x80) == negative]
    return min(cands, key=lambda vc: (abs(vc[0] - y), vc[1] & 1))[1]


def _brute_rowtile(x):
    """Per token and 128-channel tile: the smallest e with amax <= 448 * 2^e,
    then each value's nearest E4M3 code at that scale (ties to even)."""
    T, C = x.shape
    q = np.zeros((T, C), dtype=np.uint8)
    sf = np.zeros((T, C // 128), dtype=np.uint8)
    for t in range(T):
        for g in range(C // 128):
            cols = range(128 * g, 128 * g + 128)
            amax = max(abs(Fraction(float(x[t, c]))) for c in cols)
            e = -127
            while e < 127 and amax > 448 * Fraction(2) ** e:
                e += 1
            sf[t, g] = e + 127
            for c in cols:
                y = Fraction(float(x[t, c])) / Fraction(2) ** e
                q[t, c] = _nearest_code(y, bool(np.signbit(x[t, c])))
    return q, sf


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C              # no NaN codes
    return c


def test_rowtile_quant_matches_brute_force():
    x = workloads.randn((6, 256), seed=21, dtype=torch.bfloat16).float().numpy()
    x[1] *= 1e-30                 # tiny token
    x[2, :128] = 0.0              # zero tile
    x[3, 128:] *= 1e20            # huge tile
    x[4, :64] = -1e-40            # subnormals
    q, sf = Q.quant_rowtile(x)
    qb, sfb = _brute_rowtile(x)
    assert np.array_equal(sf, sfb)
    assert np.array_equal(q, qb)


def _check_dequant(mod) -> bool:
    """dequant_rowtile against torch's E4M3 decoding times 2^(b - 127) taken
    in exact rational arithmetic, over every scale byte 0..254."""
    rng = np.random.default_rng(3)
    T, C = 255, 256
    q = _rand_codes(rng, (T, C))
    sf = np.stack([np.full(C // 128, b, dtype=np.uint8) for b in range(255)])
    sf[::2, 1] = rng.integers(0, 255, size=(T + 1) // 2)   # the two tiles differ
    got = mod.dequant_rowtile(q, sf)
    dec = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    for t in range(0, T, 7):
        for c in list(range(0, C, 37)) + [127, 128, 255]:
            want = Fraction(float(dec[t, c])) * Fraction(2) ** (int(sf[t, c // 128]) - 127)
            if Fraction(float(got[t, c])) != want:
                return False
    return True


def test_dequant_matches_torch_decode_times_exact_scale():
    assert _check_dequant(Q)


def _check_identity(mod) -> bool:
    """Stored tiles whose scale is the same for all 128 tokens of a block, with
    a code in (224, 448] in every column block, are already a valid 128 x 1
    quantisation: re-quantising returns the same codes and scale bytes."""
    rng = np.random.default_rng(5)
    T, C = 512, 384
    q = _rand_codes(rng, (T, C))
    q[::128] = rng.choice(np.array([0x78, 0x7A, 0x7E, 0xF8, 0xFE], dtype=np.uint8),
                          size=(T // 128, C))       # |v| in {256, 320, 448}
    b = rng.integers(20, 235, size=(T // 128, C // 128)).astype(np.uint8)
    sf_row = np.repeat(b, 128, axis=0)               # constant down each block
    q2, sf2 = mod.requant_colblock(q, sf_row, 128)
    return bool(np.array_equal(q2, q) and np.array_equal(sf2, np.repeat(b, 128, axis=1)))


def test_requant_of_uniform_tiles_is_identity():
    assert _check_identity(Q)


def _check_shift(mod) -> bool:
    """Scaling every stored tile by 2^d scales every block by 2^d: the scale
    bytes move by d and the codes do not change."""
    x = workloads.randn((256, 256), seed=8).numpy()
    x[:, 5] *= 1e-3
    q, sf = Q.quant_rowtile(x)
    q0, s0 = mod.requant_colblock(q, sf, 128)
    for d in (-9, 3, 17):
        q1, s1 = mod.requant_colblock(q, (sf.astype(np.int64) + d).astype(np.uint8), 128)
        if not (np.array_equal(q1, q0)
                and np.array_equal(s1.astype(np.int64), s0.astype(np.int64) + d)):
            return False
    return True


def test_requant_scale_shift():
    assert _check_shift(Q)


@pytest.mark.parametrize("gran_k", [128, 32])
def test_requant_error_bounds(gran_k):
    """The re-quantised value is within E4M3 rounding of the dequantised
    stored value, and each block's scale is tight."""
    x = workloads.randn((512, 384), seed=9).numpy()
    x[:, :16] *= 1e-4
    q, sf = Q.quant_rowtile(x)
    x1 = Q.dequant_rowtile(q, sf)
    q2, sf2 = Q.requant_colblock(q, sf, gran_k)
    scale = np.ldexp(1.0, np.repeat(sf2.astype(np.int64) - 127, gran_k, axis=0))
    y = e4m3_decode(q2) * scale
    xs = x1 / scale
    normal = np.abs(xs) >= 2.0 ** -6
    assert np.all(np.abs(y - x1)[normal] <= 2.0 ** -4 * np.abs(x1)[normal])
    assert np.all(np.abs(y - x1)[~normal] <= 2.0 ** -10 * scale[~normal])
    blk = np.abs(xs).reshape(-1, gran_k, x.shape[1]).max(axis=1)
    assert np.all((blk > 224) & (blk <= 448))


def test_channel_layout_is_transpose():
    x = workloads.randn((256, 256), seed=10).numpy()
    q, sf = Q.quant_rowtile(x)
    qt, st = Q.requant_colblock(q, sf, 128, "token")
    qc, sc = Q.requant_colblock(q, sf, 128, "channel")
    assert np.array_equal(qc, qt.T) and np.array_equal(sc, st)


def test_gather_rows_matches_loop():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((37, 5))
    src = rng.integers(-1, 37, size=64)
    got = Q.gather_rows(x, src)
    for i, s in enumerate(src):
        assert np.array_equal(got[i], x[s] if s >= 0 else np.zeros(5))
    with pytest.raises(ValueError):
        Q.gather_rows(x, np.array([0, 37]))
    with pytest.raises(ValueError):
        Q.gather_rows(x, np.array([-2]))


def test_moe_layout_cast_invariants():
    """A token permutation inside each 128-token block permutes the codes and
    keeps the scales; padding rows give code 0 and leave a block's scale as
    the data rows alone set it."""
    rng = np.random.default_rng(12)
    x = workloads.randn((300, 128), seed=13, dtype=torch.bfloat16).float().numpy()
    src = rng.permutation(300)[:256]
    q, sf = Q.moe_layout_cast(x, src)
    perm = np.concatenate([128 * b + rng.permutation(128) for b in range(2)])
    q2, sf2 = Q.moe_layout_cast(x, src[perm])
    assert np.array_equal(sf2, sf) and np.array_equal(q2, q[perm])
    # first block: 100 data rows then 28 padding rows
    src_pad = np.concatenate([src[:100], -np.ones(28, dtype=np.int64), src[128:]])
    q3, sf3 = Q.moe_layout_cast(x, src_pad)
    assert np.all(q3[100:128] == 0)
    q4, sf4 = Q.quant_colblock(x[src[:100]][np.r_[np.arange(100), np.zeros(28, int)]], 128)
    assert np.array_equal(sf3[0], sf4[0]) and np.array_equal(q3[:100], q4[:100])
    # the FP8 source form equals the float form on the dequantised values
    qs, ss = Q.quant_rowtile(x)
    a = Q.moe_layout_cast(qs, src_pad, sf_row=ss)
    b = Q.moe_layout_cast(Q.dequant_rowtile(qs, ss), src_pad)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_argument_checks():
    with pytest.raises(ValueError):
        Q.quant_rowtile(np.zeros((4, 100)))
    with pytest.raises(ValueError):
        Q.dequant_rowtile(np.zeros((4, 128), np.uint8), np.zeros((4, 2), np.uint8))


# --- planted mistakes: each mutant must fail at least one pin ---------------

class _Mut:
    """A copy of the oracle's re-quantisation with one function replaced."""

    def __init__(self, dequant):
        self.dequant_rowtile = dequant

    def requant_colblock(self, q, sf_row, gran_k=128, layout="token"):
        return Q.quant_colblock(self.dequant_rowtile(q, sf_row), gran_k, layout)


def _all_pins(mod) -> bool:
    return _check_dequant(mod) and _check_identity(mod) and _check_shift(mod)


def test_planted_mistakes_are_caught():
    from oracle.e4m3 import ue8m0_to_float
    assert _all_pins(_Mut(Q.dequant_rowtile))

    def group_of_64(q, sf):            # tile width read as 64
        idx = np.minimum(np.arange(q.shape[1]) // 64, sf.shape[1] - 1)
        return e4m3_decode(q) * ue8m0_to_float(sf[:, idx])
    assert not _all_pins(_Mut(group_of_64))

    def bias_126(q, sf):               # UE8M0 bias off by one
        return Q.dequant_rowtile(q, sf) * 2.0
    assert not _all_pins(_Mut(bias_126))

    def no_sign(q, sf):                # sign bit dropped
        return np.abs(Q.dequant_rowtile(q, sf))
    assert not _all_pins(_Mut(no_sign))

    def next_token(q, sf):             # scale of the next token
        return e4m3_decode(q) * np.repeat(ue8m0_to_float(np.roll(sf, -1, axis=0)), 128, axis=1)
    assert not _all_pins(_Mut(next_token))

    def codes_only(q, sf):             # scales ignored
        return e4m3_decode(q)
    assert not _all_pins(_Mut(codes_only))


def test_moe_layout_plan_matches_stable_sort():
    """The plan against a construction from numpy's stable argsort of the
    routing entries by expert (a library sort)."""
    rng = np.random.default_rng(14)
    T, topk, G = 300, 3, 7
    idx = rng.integers(-1, G, size=(T, topk))
    ks, src, pair = Q.moe_layout_plan(idx, G)
    flat = idx.reshape(-1)
    order = np.argsort(np.where(flat < 0, G, flat), kind="stable")
    want_pair = []
    for e in range(G):
        sel = order[flat[order] == e]
        want_pair += list(sel) + [-1] * ((-len(sel)) % 128)
    want_pair = np.array(want_pair)
    assert np.array_equal(pair, want_pair)
    assert np.array_equal(src, np.where(want_pair >= 0, want_pair // topk, -1))
    assert np.array_equal(ks, [len(pair[sum(ks[:e]):sum(ks[:e + 1])]) for e in range(G)])
    counts = np.bincount(flat[flat >= 0], minlength=G)
    assert np.array_equal(ks, -(-counts // 128) * 128)
    with pytest.raises(ValueError):
        Q.moe_layout_plan(np.array([[G]]), G)
