"""The bounded waits of the staging engines run out, report, and leave the
GPU usable.

The bulk and staged engines wait on mbarriers for their cp.async.bulk copies.
A test hook (A2AV_DEBUG_STARVE, read by a2av_create) arms one stage of one
CTA for 16 bytes more than its copies deliver, so that phase never
completes: the waiting warp gives up after about a second, records
A2AV_ERR_TIMEOUT, lets the copies it issued land, and returns.  Nothing
faults, traps or hangs; every copy issued still completes.  The test then
runs a normal exchange on a fresh handle in the same context and checks it.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests._gpu import exchange_checked

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()


@pytest.mark.parametrize("path", [a2av.PATH_BULK, a2av.PATH_STAGED])
def test_starved_stage_times_out_and_context_survives(monkeypatch, path):
    w = wl.cfg2(8 << 20)
    ins = [torch.from_numpy(b).cuda() for b in w.inputs]
    S = torch.from_numpy(w.splits).cuda()
    outs = [torch.empty(int(w.splits[:, p].sum()) * w.row_bytes, dtype=torch.uint8, device="cuda")
            for p in range(w.W)]
    so = torch.empty((w.W, 2, w.W), dtype=torch.int64, device="cuda")
    monkeypatch.setenv("A2AV_DEBUG_STARVE", "1")
    with a2av.A2av(w.W, path=path) as eng:
        monkeypatch.delenv("A2AV_DEBUG_STARVE")
        eng.run(ins, S, outs, so, w.row_bytes)
        assert eng.status() == a2av.ERR_TIMEOUT
        assert eng.last_launch()["path"] == path
    torch.cuda.synchronize()
    # the context is intact: a normal exchange right after is exact
    exchange_checked(w.inputs, w.splits, w.row_bytes, path=path, expect_path=path)
