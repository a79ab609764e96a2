"""The C-ABI boundary on the host: the library loads, exports every symbol
the header declares, and rejects bad arguments with the documented status
before touching the device (so these run without a GPU)."""
import ctypes
import os
import re

import pytest

from grouped_fp8_weight_gb300 import binding as B
from grouped_fp8_weight_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dg_wgrad.h")


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return B.lib()


def _declared():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"^\S.*?\b(dg_[a-z0-9_]+)\s*\(", txt, re.M)))


def test_header_declares_the_api():
    assert _declared() == sorted(B.SIGNATURES)


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name
    assert L.dg_version() == 100


FAKE = 0x10000          # aligned, never dereferenced: validation fails first
MIS = 0x10008           # 8-byte aligned only


def _ks(v):
    return (ctypes.c_int * max(1, len(v)))(*v)


def _fp8(L, **kw):
    a = dict(a=FAKE, sfa=FAKE, b=FAKE, sfb=FAKE, d=FAKE, dt=B.DG_F32, c=None, G=2, M=128,
             N=256, sk=256, ks=[128, 128], ksd=FAKE, g=128)
    a.update(kw)
    return L.dg_k_grouped_fp8_wgrad(a["a"], a["sfa"], a["b"], a["sfb"], a["d"], a["dt"], a["c"],
                                    a["G"], a["M"], a["N"], a["sk"], _ks(a["ks"]), a["ksd"],
                                    a["g"], None)


@pytest.mark.parametrize("kw,why", [
    (dict(G=-1), "G = -1"),
    (dict(M=100), "multiples of 16"),
    (dict(N=0), "multiples of 16"),
    (dict(g=64), "gran_k = 64"),
    (dict(ks=[128, 64], sk=192), "not a multiple of 128"),
    (dict(ks=[128, -128], sk=0), "< 0"),
    (dict(sk=512), "!= sum_k"),
    (dict(dt=B.DG_BF16, c=FAKE), "accumulator needs FP32"),
    (dict(dt=7), "unknown output dtype"),
    (dict(a=MIS), "16-byte aligned"),
    (dict(sfb=None), "sfa and sfb"),
    (dict(d=None), "d must be"),
    (dict(c=MIS), "c must be"),
    (dict(ksd=None), "ks_host and ks_dev"),
    (dict(G=0, sk=128), "G = 0 but"),
])
def test_fp8_invalid_arguments(L, kw, why):
    assert _fp8(L, **kw) == B.DG_ERR_INVALID_ARG
    assert why in L.dg_last_error().decode()


def test_fp8_nt_invalid_arguments(L):
    st = L.dg_k_grouped_fp8_wgrad_nt(FAKE, FAKE, FAKE, FAKE, FAKE, B.DG_F32, None, 2, 128, 100,
                                     256, _ks([128, 128]), FAKE, 128, None)
    assert st == B.DG_ERR_INVALID_ARG
    assert "dg_k_grouped_fp8_wgrad_nt" in L.dg_last_error().decode()


def test_fp8_group_limit(L):
    ks = [0] * (B.DG_MAX_GROUPS + 1)
    assert _fp8(L, G=len(ks), ks=ks, sk=0) == B.DG_ERR_UNSUPPORTED


def test_fp8_empty_problem_is_ok_without_device(L):
    assert _fp8(L, G=0, sk=0) == B.DG_OK
    assert L.dg_last_error().decode() == ""


def test_noalloc_rejects_oversize_scale_records_without_device(L):
    """The allocation-free entry point keeps the packed scale records in a
    32 MiB static array: a problem needing more is refused before any CUDA
    call.  G = 8 experts of 16384 tokens at gran_k 32 on 4096 x 7168 needs
    (8 * 128 groups) x (32 + 64 records) x 512 B = 48 MiB."""
    ks = [16384] * 8
    st = L.dg_k_grouped_fp8_wgrad_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, B.DG_F32, None, 8, 4096,
                                          7168, sum(ks), _ks(ks), FAKE, 32, None)
    assert st == B.DG_ERR_UNSUPPORTED
    assert "packed scale factors need" in L.dg_last_error().decode()


def _dgrad(L, **kw):
    a = dict(a=FAKE, sfa=FAKE, w=FAKE, sfw=FAKE, d=FAKE, dt=B.DG_BF16, G=2, K=256, N=224,
             sm=384, ms=[128, 256], msd=FAKE, g=128)
    a.update(kw)
    return L.dg_m_grouped_fp8_dgrad(a["a"], a["sfa"], a["w"], a["sfw"], a["d"], a["dt"], a["G"],
                                    a["K"], a["N"], a["sm"], _ks(a["ms"]), a["msd"], a["g"], None)


@pytest.mark.parametrize("kw,why", [
    (dict(G=-1), "G = -1"),
    (dict(K=192), "K = 192 must be a positive multiple of 128"),
    (dict(K=0), "multiple of 128"),
    (dict(N=200), "N = 200 must be a positive multiple of 16"),
    (dict(g=64), "gran_k = 64"),
    (dict(dt=5), "unknown output dtype"),
    (dict(ms=[128, 64], sm=192), "not a multiple of 128"),
    (dict(ms=[512, -128]), "< 0"),
    (dict(sm=512), "!= sum_m"),
    (dict(msd=None), "ms_host and ms_dev"),
    (dict(G=0, sm=128), "G = 0 but"),
    (dict(a=MIS), "16-byte aligned"),
    (dict(sfw=None), "16-byte aligned"),
    (dict(d=None), "16-byte aligned"),
])
def test_dgrad_invalid_arguments(L, kw, why):
    assert _dgrad(L, **kw) == B.DG_ERR_INVALID_ARG
    assert "dg_m_grouped_fp8_dgrad" in L.dg_last_error().decode()
    assert why in L.dg_last_error().decode()


def test_dgrad_nt_invalid_arguments(L):
    st = L.dg_m_grouped_fp8_dgrad_nt(FAKE, FAKE, FAKE, FAKE, FAKE, B.DG_BF16, 2, 192, 224, 384,
                                     _ks([128, 256]), FAKE, 128, None)
    assert st == B.DG_ERR_INVALID_ARG
    assert "dg_m_grouped_fp8_dgrad_nt" in L.dg_last_error().decode()
    st = L.dg_m_grouped_fp8_dgrad_nt(FAKE, FAKE, FAKE, FAKE, FAKE, B.DG_BF16, 2, 256, 2 ** 30,
                                     384, _ks([128, 256]), FAKE, 128, None)
    assert st == B.DG_ERR_UNSUPPORTED      # G * N >= 2^31


def test_dgrad_limits_and_empty_problems_without_device(L):
    ms = [0] * (B.DG_MAX_GROUPS + 1)
    assert _dgrad(L, G=len(ms), ms=ms, sm=0) == B.DG_ERR_UNSUPPORTED
    assert _dgrad(L, G=2, K=2 ** 30, ms=[128, 256]) == B.DG_ERR_UNSUPPORTED   # G * K >= 2^31
    assert _dgrad(L, G=0, sm=0) == B.DG_OK
    # every expert empty: no rows to write, nothing enqueued
    assert _dgrad(L, ms=[0, 0], sm=0, a=None, w=None, d=None) == B.DG_OK
    assert L.dg_last_error().decode() == ""


def _bf16(L, **kw):
    a = dict(a=FAKE, b=FAKE, d=FAKE, dt=B.DG_F32, c=None, G=2, M=64, N=72, sk=7, ks=[3, 4],
             ksd=FAKE)
    a.update(kw)
    return L.dg_k_grouped_bf16_wgrad(a["a"], a["b"], a["d"], a["dt"], a["c"], a["G"], a["M"],
                                     a["N"], a["sk"], _ks(a["ks"]), a["ksd"], None)


@pytest.mark.parametrize("kw,why", [
    (dict(M=60), "multiples of 8"),
    (dict(ks=[3, 5]), "!= sum_k"),
    (dict(b=MIS), "16-byte aligned"),
    (dict(dt=B.DG_BF16, c=FAKE), "accumulator"),
])
def test_bf16_invalid_arguments(L, kw, why):
    assert _bf16(L, **kw) == B.DG_ERR_INVALID_ARG
    assert why in L.dg_last_error().decode()


def _quant(L, **kw):
    a = dict(x=FAKE, T=256, C=64, q=FAKE, sf=FAKE, lay=B.DG_TOKEN_MAJOR, g=128)
    a.update(kw)
    return L.dg_quant_transpose_fp8(a["x"], a["T"], a["C"], a["q"], a["sf"], a["lay"], a["g"],
                                    None)


@pytest.mark.parametrize("kw,why", [
    (dict(T=200), "multiple of gran_k"),
    (dict(T=-128), "multiple of gran_k"),
    (dict(C=24), "multiple of 16"),
    (dict(g=16), "gran_k = 16"),
    (dict(lay=5), "unknown layout"),
    (dict(q=MIS), "16-byte aligned"),
    (dict(sf=None), "16-byte aligned"),
])
def test_quant_invalid_arguments(L, kw, why):
    assert _quant(L, **kw) == B.DG_ERR_INVALID_ARG
    assert why in L.dg_last_error().decode()


def test_quant_zero_tokens_is_ok(L):
    assert _quant(L, T=0) == B.DG_OK


def _requant(L, **kw):
    a = dict(q_in=FAKE, sf_in=FAKE, T=256, C=256, q=FAKE, sf=FAKE, lay=B.DG_TOKEN_MAJOR, g=128)
    a.update(kw)
    return L.dg_requant_transpose_fp8(a["q_in"], a["sf_in"], a["T"], a["C"], a["q"], a["sf"],
                                      a["lay"], a["g"], None)


@pytest.mark.parametrize("kw,why", [
    (dict(C=64), "multiple of 128"),
    (dict(T=96), "multiple of gran_k"),
    (dict(sf_in=None), "sf_in is required"),
    (dict(q_in=MIS), "16-byte aligned"),
    (dict(g=64), "gran_k = 64"),
])
def test_requant_invalid_arguments(L, kw, why):
    assert _requant(L, **kw) == B.DG_ERR_INVALID_ARG
    assert why in L.dg_last_error().decode()


def _moe(L, **kw):
    a = dict(x=FAKE, x_sf=None, Ts=300, C=64, src=FAKE, T=256, q=FAKE, sf=FAKE,
             lay=B.DG_TOKEN_MAJOR, g=128)
    a.update(kw)
    return L.dg_quant_moe_layout_fp8(a["x"], a["x_sf"], a["Ts"], a["C"], a["src"], a["T"],
                                     a["q"], a["sf"], a["lay"], a["g"], None)


@pytest.mark.parametrize("kw,why", [
    (dict(src=None), "src_rows is required"),
    (dict(Ts=-1), "T_src < 0"),
    (dict(x_sf=FAKE), "multiple of 128"),          # FP8 source needs C % 128 == 0
    (dict(T=130), "multiple of gran_k"),
    (dict(src=MIS), "16-byte aligned"),
    (dict(Ts=2 ** 31), "T_src above"),
])
def test_moe_layout_invalid_arguments(L, kw, why):
    st = _moe(L, **kw)
    assert st in (B.DG_ERR_INVALID_ARG, B.DG_ERR_UNSUPPORTED)
    assert why in L.dg_last_error().decode()


def test_casts_zero_rows_are_ok(L):
    assert _requant(L, T=0, sf_in=None) == B.DG_OK
    assert _moe(L, T=0, src=None) == B.DG_OK


def _plan(L, **kw):
    a = dict(idx=FAKE, T=100, k=2, G=8, al=128, ks=FAKE, src=FAKE, pair=None, cap=200 + 8 * 127)
    a.update(kw)
    return L.dg_moe_layout_plan(a["idx"], a["T"], a["k"], a["G"], a["al"], a["ks"], a["src"],
                                a["pair"], a["cap"], None)


@pytest.mark.parametrize("kw,why,st", [
    (dict(cap=200 + 8 * 127 - 1), "cap = ", B.DG_ERR_INVALID_ARG),
    (dict(G=0), "G = 0", B.DG_ERR_INVALID_ARG),
    (dict(G=B.DG_MAX_GROUPS + 1, cap=10 ** 6), "G = 1025", B.DG_ERR_UNSUPPORTED),
    (dict(k=0), "topk = 0", B.DG_ERR_INVALID_ARG),
    (dict(al=0), "align = 0", B.DG_ERR_INVALID_ARG),
    (dict(src=MIS), "16-byte aligned", B.DG_ERR_INVALID_ARG),
    (dict(idx=None), "16-byte aligned", B.DG_ERR_INVALID_ARG),
    (dict(T=2 ** 30, k=2, cap=2 ** 32), "above 2^31", B.DG_ERR_UNSUPPORTED),
])
def test_moe_plan_invalid_arguments(L, kw, why, st):
    assert _plan(L, **kw) == st
    assert why in L.dg_last_error().decode()


def _sg(L, **kw):
    a = dict(h=FAKE, da=FAKE, T=256, I=64, q=FAKE, sf=FAKE, qa=None, sfa=None, g=128)
    a.update(kw)
    return L.dg_swiglu_backward_quant_fp8(a["h"], a["da"], a["T"], a["I"], a["q"], a["sf"],
                                          a["qa"], a["sfa"], a["g"], None)


@pytest.mark.parametrize("kw,why", [
    (dict(I=24), "multiple of 16"),
    (dict(T=100), "multiple of gran_k"),
    (dict(g=64), "gran_k = 64"),
    (dict(qa=FAKE), "go together"),
    (dict(da=MIS), "16-byte aligned"),
])
def test_swiglu_invalid_arguments(L, kw, why):
    assert _sg(L, **kw) == B.DG_ERR_INVALID_ARG
    assert why in L.dg_last_error().decode()


def test_binding_raises_when_library_missing(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(B, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()
