"""Bounded device waits: a wait that runs out ends the kernel early and is
reported, and the context stays usable.

Every mbarrier wait of the GEMM kernel gives up after the call's wait limit
(DG_WAIT_LIMIT_US / DG_WAIT_LIMIT_MS, read at each call).  With a limit of two
microseconds, the first wait of an epilogue for a tile of 128 k-blocks (tens
of microseconds of MMAs) runs out: the kernel sets its abort flag, every role
leaves its loop, copies in flight land (drain waits have a floor of two
seconds), tensor memory is freed, and the status record says DG_ERR_TIMEOUT.
No barrier is left unarrived on purpose and nothing faults; the next call at
the default limit must give the oracle's result.
"""
import numpy as np
import pytest
import torch

import grouped_fp8_weight_gb300 as dg
from grouped_fp8_weight_gb300 import binding, workloads
import oracle
from tests.gpu_helpers import assert_close, fp8_operands, to_dev

pytestmark = pytest.mark.gpu

KS = [16384, 4096, 0, 1024]     # 128, 32 and 8 k-blocks: tiles run for tens of microseconds
M, N = 512, 448


def _operands():
    sk = sum(KS)
    qa, sa, qb, sb = fp8_operands(workloads.randn((sk, M), 31).numpy(),
                                  workloads.randn((sk, N), 32).numpy())
    return (qa, sa, qb, sb), [to_dev(x) for x in (qa, sa, qb, sb)]


def _call(ops, d, c, ks_dev):
    dg.dg_k_grouped_fp8_wgrad(*ops, d, c, KS, ks_dev, 128)


def test_short_wait_limit_reports_timeout_and_next_call_is_exact(monkeypatch):
    host, ops = _operands()
    ks_dev = torch.tensor(KS, dtype=torch.int32, device="cuda")
    d = torch.zeros(len(KS), M, N, dtype=torch.float32, device="cuda")
    dg.dg_sync_check()                      # nothing pending before the test
    monkeypatch.setenv("DG_WAIT_LIMIT_US", "2")
    _call(ops, d, None, ks_dev)             # returns at once: the launch itself is fine
    with pytest.raises(binding.DGError) as ei:
        dg.dg_sync_check()
    assert ei.value.status == binding.DG_ERR_TIMEOUT
    assert "timed out" in str(ei.value)
    dg.dg_sync_check()                      # the record was read and cleared
    monkeypatch.delenv("DG_WAIT_LIMIT_US")
    d.fill_(float("nan"))
    _call(ops, d, None, ks_dev)
    dg.dg_sync_check()
    D, S = oracle.kgrouped_fp8_wgrad(*host, KS, 128)
    assert_close(d, D, S, what="after a timed-out call")


def test_short_wait_limit_in_place_then_recovery(monkeypatch):
    # In-place accumulation (TMA reduce-add): a call ended early leaves D
    # unspecified; D is reset and accumulated again at the default limit.
    # DG_DETERMINISTIC keeps each expert in one schedule entry, so its tiles
    # keep their 128 k-blocks (the K-split would cut them to 8).
    host, ops = _operands()
    ks_dev = torch.tensor(KS, dtype=torch.int32, device="cuda")
    c = workloads.randn((len(KS), M, N), 33)
    d = c.cuda()
    monkeypatch.setenv("DG_DETERMINISTIC", "1")
    monkeypatch.setenv("DG_WAIT_LIMIT_US", "2")
    _call(ops, d, d, ks_dev)
    with pytest.raises(binding.DGError) as ei:
        dg.dg_sync_check()
    assert ei.value.status == binding.DG_ERR_TIMEOUT
    monkeypatch.delenv("DG_WAIT_LIMIT_US")
    d.copy_(c)
    _call(ops, d, d, ks_dev)
    dg.dg_sync_check()
    D, S = oracle.kgrouped_fp8_wgrad(*host, KS, 128, c.numpy())
    assert_close(d, D, S, what="in place after a timed-out call")
    assert torch.equal(d[2].cpu(), c[2])    # the empty expert is untouched


def test_deterministic_in_place_is_bitwise_reproducible(monkeypatch):
    # Without DG_DETERMINISTIC the long expert is split along K and its parts
    # are added into D in a timing-dependent order; with it, every element is
    # added to once and two runs agree bit for bit (and with the oracle).
    host, ops = _operands()
    ks_dev = torch.tensor(KS, dtype=torch.int32, device="cuda")
    c = workloads.randn((len(KS), M, N), 34).cuda()
    monkeypatch.setenv("DG_DETERMINISTIC", "1")
    runs = []
    for _ in range(2):
        d = c.clone()
        _call(ops, d, d, ks_dev)
        dg.dg_sync_check()
        runs.append(d)
    assert torch.equal(runs[0], runs[1])
    D, S = oracle.kgrouped_fp8_wgrad(*host, KS, 128, c.cpu().numpy())
    assert_close(runs[0], D, S, what="deterministic in place")
