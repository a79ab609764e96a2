"""Pins for the oracle's K-grouped weight-gradient GEMM (CPU only).

Pinned against: exact rational arithmetic on tiny shapes (brute force), a
dense A^T B computed by torch from torch's own FP8 decoding (G = 1), closed
forms that expose transposed or shifted operands, and the invariants of the
grouped sum (empty groups, splitting a group, permuting experts).  The last
tests plant mistakes in a copy of the oracle and check that the pins catch
them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle.wgrad as W
from grouped_fp8_weight_gb300 import workloads
from oracle.e4m3 import e4m3_decode


def _rand_fp8(rng, rows, cols):
    c = rng.integers(0, 256, size=(rows, cols)).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3C            # no NaN codes
    return c


def _rand_sf(rng, blocks, cols, lo=110, hi=140):
    return rng.integers(lo, hi, size=(blocks, cols)).astype(np.uint8)


def _exact_fp8(a, sfa, b, sfb, ks, g, c=None):
    """Brute force: exact rational sum per element."""
    G, M, N = len(ks), a.shape[1], b.shape[1]
    av = e4m3_decode(a)
    bv = e4m3_decode(b)
    out = np.zeros((G, M, N))
    off = 0
    for e in range(G):
        for m in range(M):
            for n in range(N):
                s = Fraction(0) if c is None else Fraction(float(c[e, m, n]))
                for k in range(off, off + ks[e]):
                    s += (Fraction(float(av[k, m])) * Fraction(2) ** (int(sfa[k // g, m]) - 127)
                          * Fraction(float(bv[k, n])) * Fraction(2) ** (int(sfb[k // g, n]) - 127))
                out[e, m, n] = float(s)
        off += ks[e]
    return out


@pytest.mark.parametrize("g,ks", [(128, [128, 0, 256]), (32, [64, 32, 0, 96]), (128, [0, 0])])
def test_fp8_matches_exact_rational_sum(g, ks):
    rng = np.random.default_rng(7)
    sk, M, N = sum(ks), 5, 6
    a, b = _rand_fp8(rng, sk, M), _rand_fp8(rng, sk, N)
    sfa, sfb = _rand_sf(rng, sk // g, M), _rand_sf(rng, sk // g, N)
    c = rng.standard_normal((len(ks), M, N))
    for cc in (None, c):
        D, S = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g, cc)
        ref = _exact_fp8(a, sfa, b, sfb, ks, g, cc)
        assert np.all(np.abs(D - ref) <= 1e-13 * (S + (0 if cc is None else np.abs(cc))) + 1e-300)


def test_bf16_matches_exact_rational_sum():
    ks = [3, 0, 7, 1]
    sk, M, N = sum(ks), 4, 3
    a = workloads.randn((sk, M), 21, torch.bfloat16).float().numpy()
    b = workloads.randn((sk, N), 22, torch.bfloat16).float().numpy()
    c = workloads.randn((len(ks), M, N), 23).numpy()
    D, S = W.kgrouped_bf16_wgrad(a, b, ks, c)
    off = W.expert_offsets(ks)
    for e in range(len(ks)):
        for m in range(M):
            for n in range(N):
                s = Fraction(float(c[e, m, n])) + sum(
                    (Fraction(float(a[k, m])) * Fraction(float(b[k, n]))
                     for k in range(off[e], off[e + 1])), Fraction(0))
                assert abs(D[e, m, n] - float(s)) <= 1e-14 * (S[e, m, n] + abs(c[e, m, n]))


def test_single_group_equals_dense_product_from_torch_decode():
    """G = 1: D = A^T B on values decoded by torch's float8_e4m3fn cast."""
    rng = np.random.default_rng(3)
    sk, M, N, g = 384, 24, 40, 128
    a, b = _rand_fp8(rng, sk, M), _rand_fp8(rng, sk, N)
    sfa, sfb = _rand_sf(rng, sk // g, M), _rand_sf(rng, sk // g, N)
    D, _ = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, [sk], g)

    def deq(codes, sf):
        v = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64)
        s = torch.from_numpy(sf.astype(np.int64) - 127).repeat_interleave(g, dim=0)
        return torch.ldexp(v, s.to(torch.float64))

    ref = (deq(a, sfa).T @ deq(b, sfb)).numpy()
    assert np.allclose(D[0], ref, rtol=1e-13, atol=0)


def test_closed_form_block_scales_and_counts():
    """A, B all 1.0 (code 0x38): D[e, m, n] = sum over the expert's blocks of
    2^(sfa[kb, m] - 127 + sfb[kb, n] - 127)."""
    g, ks, M, N = 128, [256, 0, 128, 384], 3, 4
    sk = sum(ks)
    a = np.full((sk, M), 0x38, np.uint8)
    b = np.full((sk, N), 0x38, np.uint8)
    kb = np.arange(sk // g)
    sfa = (127 + kb[:, None] + np.arange(M)[None, :]).astype(np.uint8)
    sfb = (127 - kb[:, None] + 2 * np.arange(N)[None, :]).astype(np.uint8)
    D, S = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g)
    off = W.expert_offsets(ks)
    for e in range(len(ks)):
        blocks = range(off[e] // g, off[e + 1] // g)
        want = np.array([[sum(g * 2.0 ** (m + 2 * n) for _ in blocks) for n in range(N)]
                         for m in range(M)])
        # 2^(kb + m) * 2^(-kb + 2n) = 2^(m + 2n) per token
        assert np.array_equal(D[e], want)
        assert np.array_equal(S[e], want)


def test_closed_form_one_hot_exposes_transpose():
    """A[k, m] = [m == k mod M] so D[e, m, n] = sum_{k in e, k mod M == m} B[k, n]."""
    g, ks, M, N = 32, [64, 96], 8, 8
    sk = sum(ks)
    a = np.zeros((sk, M), np.uint8)
    a[np.arange(sk), np.arange(sk) % M] = 0x38
    rng = np.random.default_rng(9)
    b = _rand_fp8(rng, sk, N)
    sfa = np.full((sk // g, M), 127, np.uint8)
    sfb = np.full((sk // g, N), 127, np.uint8)
    D, _ = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g)
    bv = e4m3_decode(b)
    off = W.expert_offsets(ks)
    for e in range(2):
        for m in range(M):
            rows = [k for k in range(off[e], off[e + 1]) if k % M == m]
            assert np.allclose(D[e, m], bv[rows].sum(axis=0), rtol=1e-15, atol=0)


def test_empty_groups_keep_accumulator_bitwise():
    rng = np.random.default_rng(4)
    ks, M, N, g = [0, 128, 0], 16, 16, 128
    a, b = _rand_fp8(rng, 128, M), _rand_fp8(rng, 128, N)
    sfa, sfb = _rand_sf(rng, 1, M), _rand_sf(rng, 1, N)
    c = rng.standard_normal((3, M, N)).astype(np.float32)
    D, S = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g, c)
    assert np.array_equal(D[0], c[0].astype(np.float64))
    assert np.array_equal(D[2], c[2].astype(np.float64))
    assert not S[0].any() and not S[2].any()
    D0, _ = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g, None)
    assert not D0[0].any() and not D0[2].any()


def test_split_invariance():
    rng = np.random.default_rng(5)
    g, M, N = 128, 12, 20
    a, b = _rand_fp8(rng, 512, M), _rand_fp8(rng, 512, N)
    sfa, sfb = _rand_sf(rng, 4, M), _rand_sf(rng, 4, N)
    D1, S1 = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, [128, 384], g)
    D2, _ = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, [128, 256, 128], g)
    assert np.all(np.abs(D2[1] + D2[2] - D1[1]) <= 1e-13 * S1[1])
    assert np.array_equal(D2[0], D1[0])


def test_permutation_equivariance():
    rng = np.random.default_rng(6)
    g, M, N = 128, 10, 14
    ks = [256, 0, 128, 384]
    off = W.expert_offsets(ks)
    a, b = _rand_fp8(rng, sum(ks), M), _rand_fp8(rng, sum(ks), N)
    sfa, sfb = _rand_sf(rng, sum(ks) // g, M), _rand_sf(rng, sum(ks) // g, N)
    D, _ = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g)
    perm = [2, 0, 3, 1]
    sl = lambda x, e, gg=1: x[off[e] // gg:off[e + 1] // gg]
    pa = np.concatenate([sl(a, e) for e in perm])
    pb = np.concatenate([sl(b, e) for e in perm])
    psa = np.concatenate([sl(sfa, e, g) for e in perm])
    psb = np.concatenate([sl(sfb, e, g) for e in perm])
    Dp, _ = W.kgrouped_fp8_wgrad(pa, psa, pb, psb, [ks[e] for e in perm], g)
    for i, e in enumerate(perm):
        assert np.array_equal(Dp[i], D[e])


def test_sampled_rows_equal_full():
    rng = np.random.default_rng(8)
    g, ks, M, N = 32, [64, 0, 96], 20, 12
    a, b = _rand_fp8(rng, sum(ks), M), _rand_fp8(rng, sum(ks), N)
    sfa, sfb = _rand_sf(rng, sum(ks) // g, M), _rand_sf(rng, sum(ks) // g, N)
    c = rng.standard_normal((3, M, N))
    D, S = W.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g, c)
    rows = [0, 7, 19]
    part = W.kgrouped_fp8_wgrad_rows(a, sfa, b, sfb, ks, rows, g, c)
    for e in range(3):
        assert np.array_equal(part[e][0], D[e][rows])
        assert np.array_equal(part[e][1], S[e][rows])
    a16 = workloads.randn((sum(ks), M), 1, torch.bfloat16).float().numpy()
    b16 = workloads.randn((sum(ks), N), 2, torch.bfloat16).float().numpy()
    D, S = W.kgrouped_bf16_wgrad(a16, b16, ks, c)
    part = W.kgrouped_bf16_wgrad_rows(a16, b16, ks, rows, c)
    for e in range(3):
        assert np.array_equal(part[e][0], D[e][rows])


def test_shape_checks():
    a = np.zeros((256, 4), np.uint8)
    sf = np.full((2, 4), 127, np.uint8)
    with pytest.raises(ValueError):
        W.kgrouped_fp8_wgrad(a, sf, a, sf, [128, 64], 128)      # sum mismatch
    with pytest.raises(ValueError):
        W.kgrouped_fp8_wgrad(a, sf, a, sf, [192, 64], 128)      # not whole blocks
    with pytest.raises(ValueError):
        W.kgrouped_bf16_wgrad(np.zeros((5, 2)), np.zeros((5, 2)), [6, -1])


# --- planted mistakes: each mutant must fail at least one pin ---------------

def _pins_pass(mod) -> bool:
    """Re-run the brute-force and one-hot pins against a (possibly mutated)
    oracle module; True if all hold."""
    rng = np.random.default_rng(7)
    g, ks, M, N = 32, [64, 0, 96], 6, 6
    sk = sum(ks)
    a, b = _rand_fp8(rng, sk, M), _rand_fp8(rng, sk, N)
    sfa, sfb = _rand_sf(rng, sk // g, M), _rand_sf(rng, sk // g, N)
    D, S = mod.kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g)
    ref = _exact_fp8(a, sfa, b, sfb, ks, g)
    return bool(np.all(np.abs(D - ref) <= 1e-13 * S + 1e-300))


def test_planted_mistakes_are_caught(monkeypatch):
    import oracle.e4m3 as E
    assert _pins_pass(W)
    orig_deq = W.dequant_colblock

    # 1. scale taken from the next block (wrong index)
    def deq_shift(codes, sf, gran_k, rows=None):
        k0, k1 = (0, codes.shape[0]) if rows is None else rows
        v = E.e4m3_decode(np.asarray(codes)[k0:k1])
        blk = np.minimum(np.arange(k0, k1) // gran_k + 1, np.asarray(sf).shape[0] - 1)
        return v * E.ue8m0_to_float(np.asarray(sf)[blk])
    monkeypatch.setattr(W, "dequant_colblock", deq_shift)
    assert not _pins_pass(W)

    # 2. sign dropped in decoding
    def deq_abs(codes, sf, gran_k, rows=None):
        return np.abs(orig_deq(codes, sf, gran_k, rows))
    monkeypatch.setattr(W, "dequant_colblock", deq_abs)
    assert not _pins_pass(W)

    # 3. scale exponent bias off by one
    def deq_bias(codes, sf, gran_k, rows=None):
        return orig_deq(codes, sf, gran_k, rows) * 2.0
    monkeypatch.setattr(W, "dequant_colblock", deq_bias)
    assert not _pins_pass(W)
    monkeypatch.setattr(W, "dequant_colblock", orig_deq)

    # 4. operands swapped (computes B^T A, i.e. D transposed for M == N)
    real = W.kgrouped_fp8_wgrad

    class Swapped:
        @staticmethod
        def kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g, c=None):
            D, S = real(b, sfb, a, sfa, ks, g, c)
            return D, S
    assert not _pins_pass(Swapped)

    # 5. last token of each expert dropped
    class Dropped:
        @staticmethod
        def kgrouped_fp8_wgrad(a, sfa, b, sfb, ks, g, c=None):
            a2 = a.copy()
            off = W.expert_offsets(ks)
            for e in range(len(ks)):
                if ks[e]:
                    a2[off[e + 1] - 1] = 0
            return real(a2, sfa, b, sfb, ks, g, c)
    assert not _pins_pass(Dropped)
