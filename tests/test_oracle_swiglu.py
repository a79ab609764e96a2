"""Pins for the oracle's SwiGLU backward (CPU only): central differences of
the forward (the mathematics of a derivative), the identity
silu'(g) + silu'(-g) = 1 (silu(g) - silu(-g) = g), closed forms at g = 0 and in
the tails, linearity in u and da; planted mistakes are each caught."""
import numpy as np
import pytest

import oracle.swiglu as S


def _fwd(g, u):
    return g * S.sigmoid(g) * u


def _check_derivatives(mod) -> bool:
    rng = np.random.default_rng(1)
    T, I = 64, 48
    g = rng.standard_normal((T, I)) * 3
    u = rng.standard_normal((T, I))
    da = rng.standard_normal((T, I))
    dh, a = mod.swiglu_backward(np.concatenate([g, u], axis=1), da)
    eps = 1e-5
    dg_fd = da * (_fwd(g + eps, u) - _fwd(g - eps, u)) / (2 * eps)
    du_fd = da * (_fwd(g, u + 1.0) - _fwd(g, u))            # a is linear in u
    ok = np.allclose(dh[:, :I], dg_fd, rtol=1e-7, atol=1e-9)
    ok &= np.allclose(dh[:, I:], du_fd, rtol=1e-12, atol=1e-14)
    ok &= np.allclose(a, _fwd(g, u), rtol=1e-15, atol=0)
    return bool(ok)


def _check_symmetry(mod) -> bool:
    g = np.linspace(-30, 30, 601)[:, None]
    one = np.ones_like(g)
    dp, _ = mod.swiglu_backward(np.concatenate([g, one], axis=1), one)
    dn, _ = mod.swiglu_backward(np.concatenate([-g, one], axis=1), one)
    return bool(np.allclose(dp[:, :1] + dn[:, :1], 1.0, rtol=0, atol=1e-14))


def _check_closed_forms(mod) -> bool:
    h = np.array([[0.0, 2.0], [60.0, 3.0], [-60.0, 5.0]])
    da = np.array([[4.0], [2.0], [7.0]])
    dh, a = mod.swiglu_backward(h, da)
    ok = np.allclose(dh[0], [0.5 * 4 * 2, 0.0])          # sigma(0) = 1/2, silu(0) = 0
    ok &= np.allclose(dh[1], [2 * 3, 2 * 60.0])           # sigma -> 1: silu' -> 1
    ok &= np.allclose(dh[2], [0.0, 0.0], atol=1e-20)      # sigma -> 0
    ok &= np.allclose(a[:, 0], [0.0, 180.0, 0.0], atol=1e-20)
    return bool(ok)


def test_derivatives():
    assert _check_derivatives(S)


def test_symmetry():
    assert _check_symmetry(S)


def test_closed_forms():
    assert _check_closed_forms(S)


def test_extreme_inputs_stay_finite():
    big = 3.0e38
    dh, a = S.swiglu_backward(np.array([[big, -big, 1.0, 1.0]]), np.array([[1.0, 1.0]]))
    assert np.all(np.isfinite(dh)) and np.all(np.isfinite(a))


def test_cast_is_quant_of_values():
    from oracle.quant import quant_colblock
    rng = np.random.default_rng(2)
    h = rng.standard_normal((256, 64))
    da = rng.standard_normal((256, 32))
    dh, a, (q, sf), (qa, sfa) = S.swiglu_backward_cast(h, da)
    q2, sf2 = quant_colblock(dh)
    assert np.array_equal(q, q2) and np.array_equal(sf, sf2)
    with pytest.raises(ValueError):
        S.swiglu_backward(np.zeros((4, 3)), np.zeros((4, 1)))


class _Mut:
    def __init__(self, fn):
        self.swiglu_backward = fn


def _all(mod):
    return _check_derivatives(mod) and _check_symmetry(mod) and _check_closed_forms(mod)


def test_planted_mistakes_are_caught():
    assert _all(S)

    def no_second_term(h, da):             # silu' taken as sigma
        I = h.shape[1] // 2
        g, u = h[:, :I], h[:, I:]
        s = S.sigmoid(g)
        return np.concatenate([da * u * s, da * g * s], axis=1), g * s * u
    assert not _all(_Mut(no_second_term))

    def halves_swapped(h, da):             # [up | gate] read as [gate | up]
        I = h.shape[1] // 2
        return S.swiglu_backward(np.concatenate([h[:, I:], h[:, :I]], axis=1), da)
    assert not _all(_Mut(halves_swapped))

    def sign_flip(h, da):                  # sigma(-g) for sigma(g)
        I = h.shape[1] // 2
        g, u = h[:, :I], h[:, I:]
        s = S.sigmoid(-g)
        return (np.concatenate([da * u * s * (1 + g * (1 - s)), da * g * s], axis=1), g * s * u)
    assert not _all(_Mut(sign_flip))

    def outputs_swapped(h, da):            # [du | dg]
        dh, a = S.swiglu_backward(h, da)
        I = h.shape[1] // 2
        return np.concatenate([dh[:, I:], dh[:, :I]], axis=1), a
    assert not _all(_Mut(outputs_swapped))
