"""Pins for the oracle's M-grouped data-gradient GEMM (CPU only).

Pinned against: exact rational arithmetic on tiny shapes (brute force); the
weight-gradient oracle (pinned on its own in test_oracle_wgrad.py) on
transposed operands, since dy_e W_e = (dy_e^T)^T W_e is a K-grouped product
with K = h_out; a dense product computed by torch from torch's own FP8
decoding (G = 1); closed forms that expose a transposed weight, a transposed
scale index or a wrong expert; and the invariants of the grouping
(permutation of experts, a split of K, empty experts).  The last test plants
mistakes in copies of the oracle and checks that the pins catch them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.dgrad as DG
import oracle.wgrad as W
from oracle.e4m3 import e4m3_decode


def _rand_fp8(rng, *shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C            # no NaN codes
    return c


def _rand_sf(rng, *shape, lo=110, hi=140):
    return rng.integers(lo, hi, size=shape).astype(np.uint8)


def _case(rng, ms, K, N, g):
    sm, G = sum(ms), len(ms)
    return (_rand_fp8(rng, sm, K), _rand_sf(rng, sm, K // g),
            _rand_fp8(rng, G, K, N), _rand_sf(rng, G, K // g, N))


def _exact(a, sfa, w, sfw, ms, g):
    """Brute force: exact rational sum per element."""
    av, wv = e4m3_decode(a), e4m3_decode(w)
    K, N = w.shape[1], w.shape[2]
    out = np.zeros((a.shape[0], N))
    off = W.expert_offsets(ms)
    for e in range(len(ms)):
        for t in range(off[e], off[e + 1]):
            for n in range(N):
                s = Fraction(0)
                for k in range(K):
                    s += (Fraction(float(av[t, k])) * Fraction(2) ** (int(sfa[t, k // g]) - 127)
                          * Fraction(float(wv[e, k, n]))
                          * Fraction(2) ** (int(sfw[e, k // g, n]) - 127))
                out[t, n] = float(s)
    return out


@pytest.mark.parametrize("g,ms,K", [(32, [2, 0, 3], 64), (128, [1, 2], 256), (32, [0, 0], 32)])
def test_matches_exact_rational_sum(g, ms, K):
    rng = np.random.default_rng(11)
    a, sfa, w, sfw = _case(rng, ms, K, 5, g)
    D, S = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, g)
    assert D.shape == (sum(ms), 5)
    ref = _exact(a, sfa, w, sfw, ms, g)
    assert np.all(np.abs(D - ref) <= 1e-13 * S + 1e-300)


@pytest.mark.parametrize("g", [32, 128])
def test_equals_weight_gradient_oracle_on_transposed_operands(g):
    """dy_e W_e is the K-grouped product with A = dy_e^T [K, M_e] (its scales
    per column per g rows of K: sfa_e^T) and B = W_e [K, N]."""
    rng = np.random.default_rng(12)
    ms, K, N = [128, 0, 256, 128], 384, 48
    a, sfa, w, sfw = _case(rng, ms, K, N, g)
    D, S = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, g)
    off = W.expert_offsets(ms)
    for e in range(len(ms)):
        if ms[e] == 0:
            continue
        r0, r1 = off[e], off[e + 1]
        De, Se = W.kgrouped_fp8_wgrad(np.ascontiguousarray(a[r0:r1].T),
                                      np.ascontiguousarray(sfa[r0:r1].T),
                                      w[e], sfw[e], [K], g)
        assert np.all(np.abs(D[r0:r1] - De[0]) <= 1e-13 * Se[0])
        assert np.allclose(S[r0:r1], Se[0], rtol=1e-13, atol=0)


def test_single_expert_equals_dense_product_from_torch_decode():
    rng = np.random.default_rng(13)
    M, K, N, g = 40, 256, 24, 128
    a, sfa, w, sfw = _case(rng, [M], K, N, g)
    D, _ = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, [M], g)

    def deq(codes, sf, dim):
        v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
        s = torch.from_numpy(sf.astype(np.int64) - 127).repeat_interleave(g, dim=dim)
        return torch.ldexp(v, s.to(torch.float64))

    ref = (deq(a, sfa, 1) @ deq(w[0], sfw[0], 0)).numpy()
    assert np.allclose(D, ref, rtol=1e-13, atol=0)


def test_closed_form_exposes_transposes_and_expert_choice():
    """dy all 1.0 (code 0x38) with scale 2^(t mod 3) per row: row t of expert e
    is 2^(t mod 3) times the column sums of expert e's dequantised weight."""
    rng = np.random.default_rng(14)
    ms, K, N, g = [3, 0, 4, 2], 64, 6, 32
    G, sm = len(ms), sum(ms)
    a = np.full((sm, K), 0x38, np.uint8)
    sfa = np.repeat((127 + np.arange(sm) % 3)[:, None], K // g, axis=1).astype(np.uint8)
    w = _rand_fp8(rng, G, K, N)
    sfw = _rand_sf(rng, G, K // g, N)
    D, _ = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, g)
    off = W.expert_offsets(ms)
    for e in range(G):
        wd = e4m3_decode(w[e]) * 2.0 ** (np.repeat(sfw[e].astype(np.int64), g, axis=0) - 127)
        for t in range(off[e], off[e + 1]):
            assert np.allclose(D[t], 2.0 ** (t % 3) * wd.sum(axis=0), rtol=1e-14, atol=0)


def test_closed_form_one_hot_selects_weight_rows():
    """dy[t, k] = [k == t mod K]: row t is row (t mod K) of W_e, scaled."""
    rng = np.random.default_rng(15)
    ms, K, N, g = [40, 24], 32, 8, 32
    sm = sum(ms)
    a = np.zeros((sm, K), np.uint8)
    a[np.arange(sm), np.arange(sm) % K] = 0x38
    sfa = np.full((sm, 1), 127, np.uint8)
    w = _rand_fp8(rng, 2, K, N)
    sfw = np.full((2, 1, N), 127, np.uint8)
    D, _ = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, g)
    wv = e4m3_decode(w)
    for t in range(sm):
        e = 0 if t < ms[0] else 1
        assert np.array_equal(D[t], wv[e, t % K])


def test_permutation_and_split_invariance():
    rng = np.random.default_rng(16)
    ms, K, N, g = [256, 0, 128, 384], 256, 20, 128
    a, sfa, w, sfw = _case(rng, ms, K, N, g)
    D, S = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, g)
    off = W.expert_offsets(ms)
    perm = [2, 0, 3, 1]
    pa = np.concatenate([a[off[e]:off[e + 1]] for e in perm])
    psa = np.concatenate([sfa[off[e]:off[e + 1]] for e in perm])
    Dp, _ = DG.mgrouped_fp8_dgrad(pa, psa, w[perm], sfw[perm], [ms[e] for e in perm], g)
    poff = W.expert_offsets([ms[e] for e in perm])
    for i, e in enumerate(perm):
        assert np.array_equal(Dp[poff[i]:poff[i + 1]], D[off[e]:off[e + 1]])
    # K split in two halves (whole scale blocks): the two products add up
    h = K // 2
    D1, _ = DG.mgrouped_fp8_dgrad(np.ascontiguousarray(a[:, :h]), sfa[:, :h // g], w[:, :h],
                                  sfw[:, :h // g], ms, g)
    D2, _ = DG.mgrouped_fp8_dgrad(np.ascontiguousarray(a[:, h:]), sfa[:, h // g:], w[:, h:],
                                  sfw[:, h // g:], ms, g)
    assert np.all(np.abs(D1 + D2 - D) <= 1e-13 * S)


def test_sampled_rows_equal_full():
    rng = np.random.default_rng(17)
    ms, K, N, g = [64, 0, 96, 32], 128, 12, 32
    a, sfa, w, sfw = _case(rng, ms, K, N, g)
    D, S = DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, ms, g)
    rows = [0, 63, 64, 100, 159, 160, 191]
    Dr, Sr = DG.mgrouped_fp8_dgrad_rows(a, sfa, w, sfw, ms, rows, g)
    assert np.array_equal(Dr, D[rows])
    assert np.array_equal(Sr, S[rows])


def test_shape_checks():
    a = np.zeros((256, 128), np.uint8)
    sfa = np.full((256, 1), 127, np.uint8)
    w = np.zeros((2, 128, 16), np.uint8)
    sfw = np.full((2, 1, 16), 127, np.uint8)
    with pytest.raises(ValueError):
        DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, [128, 64], 128)     # sum mismatch
    with pytest.raises(ValueError):
        DG.mgrouped_fp8_dgrad(a, sfa, w, sfw, [256], 128)         # G mismatch
    with pytest.raises(ValueError):
        DG.mgrouped_fp8_dgrad(a[:, :96], sfa, w[:, :96], sfw, [128, 128], 128)   # K % g


# --- planted mistakes: each mutant must fail at least one pin ---------------

def _pins_pass(fn) -> bool:
    rng = np.random.default_rng(18)
    ms, K, N, g = [2, 0, 3], 64, 4, 32
    a, sfa, w, sfw = _case(rng, ms, K, N, g)
    D, S = fn(a, sfa, w, sfw, ms, g)
    ref = _exact(a, sfa, w, sfw, ms, g)
    return bool(np.all(np.abs(D - ref) <= 1e-13 * S + 1e-300))


def test_planted_mistakes_are_caught(monkeypatch):
    assert _pins_pass(DG.mgrouped_fp8_dgrad)
    real = DG.mgrouped_fp8_dgrad

    # 1. each weight column given its neighbour's scale
    def deq_w_t(codes, sf, gran_k):
        v = e4m3_decode(codes)
        sfv = np.roll(np.asarray(sf), 1, axis=1)
        return v * 2.0 ** (sfv[np.arange(v.shape[0]) // gran_k].astype(np.int64) - 127)
    monkeypatch.setattr(DG, "dequant_weight", deq_w_t)
    assert not _pins_pass(DG.mgrouped_fp8_dgrad)
    monkeypatch.undo()

    # 2. the next expert's weight
    def next_expert(a, sfa, w, sfw, ms, g):
        return real(a, sfa, np.roll(w, -1, axis=0), np.roll(sfw, -1, axis=0), ms, g)
    assert not _pins_pass(next_expert)

    # 3. dy's scale of the neighbouring block
    def shifted_sfa(a, sfa, w, sfw, ms, g):
        return real(a, sfa, w, sfw, ms, g) if sfa.shape[1] < 2 else \
            real(a, np.roll(sfa, 1, axis=1), w, sfw, ms, g)
    assert not _pins_pass(shifted_sfa)

    # 4. weight transposed within each K x N block (K == N rows only): use the
    #    block's first N rows as columns
    def w_transposed(a, sfa, w, sfw, ms, g):
        wt = w.copy()
        n = min(w.shape[1], w.shape[2])
        wt[:, :n, :n] = np.swapaxes(w[:, :n, :n], 1, 2)
        return real(a, sfa, wt, sfw, ms, g)
    assert not _pins_pass(w_transposed)

    # 5. last k-block of the contraction dropped
    def dropped(a, sfa, w, sfw, ms, g):
        a2 = a.copy()
        a2[:, -g:] = 0
        return real(a2, sfa, w, sfw, ms, g)
    assert not _pins_pass(dropped)
