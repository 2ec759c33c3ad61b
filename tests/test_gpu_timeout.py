"""The bounded waits of the staging engines and of the grid barriers run
out, report, and leave the GPU usable.

The bulk and staged engines wait on mbarriers for their cp.async.bulk copies.
A test hook (A2AV_DEBUG_STARVE=1, read by a2av_create) arms one stage of one
CTA for 16 bytes more than its copies deliver, so that phase never
completes: the waiting warp gives up after about a second, records
A2AV_ERR_TIMEOUT, lets the copies it issued land, and returns.  With
A2AV_DEBUG_STARVE=2 the one-launch dispatch and combine kernels wait at
their grid barrier for one CTA more than the grid holds.  Nothing faults,
traps or hangs; every copy issued still completes.  Each test then runs a
normal call on a fresh handle in the same context and checks it.
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
    """Both staging engines: the starved stage's wait gives up; before the
    CTA leaves, the bulk engine waits (bounded) on every stage it issued, and
    the staged engine's producer drains the stages it filled that no
    consumer took, so no cp.async.bulk write into shared memory is pending
    when the CTA exits."""
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


@pytest.mark.parametrize("rb,combine", [(8192, False), (14336, False), (512, True), (2048, True),
                                        (14336, True)])
def test_starved_gather_stage_times_out_and_context_survives(monkeypatch, rb, combine):
    """The same hook on the dispatch's cp.async.bulk gather (one-row rings)
    and on the combine's (lane-issued 16- or 8-row stages after its own
    checks and grid barrier; one-row rings): the first stage of the first warp never
    completes, the warp reports A2AV_ERR_TIMEOUT and waits (bounded) for the
    copies it issued; a normal dispatch on a fresh handle afterwards is
    exact."""
    from tests._gpu import dispatch_checked
    rng = np.random.default_rng(rb)
    W, K, n, m = 4, 3, 64, 2000  # 8000 items: past the one-kernel path
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, n, m).astype(np.int32) for _ in range(W)]
    key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.from_numpy(x).cuda() for x in src]
    d_key = [torch.from_numpy(x).cuda() for x in key]
    d_pos = [torch.empty(m, dtype=torch.int64, device="cuda") for _ in range(W)]
    out = [torch.empty(W * m * rb, dtype=torch.uint8, device="cuda") for _ in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    isp = torch.empty((W, W), dtype=torch.int64, device="cuda")
    items = [torch.empty(m * rb, dtype=torch.uint8, device="cuda") for _ in range(W)]
    if combine:
        with a2av.A2av(W) as eng:
            eng.dispatch(d_rows, d_src, d_key, K, out, so, d_pos, rb, in_splits=isp)
            assert eng.status() == a2av.OK
    monkeypatch.setenv("A2AV_DEBUG_STARVE", "1")
    with a2av.A2av(W) as eng:
        monkeypatch.delenv("A2AV_DEBUG_STARVE")
        if combine:
            eng.combine_items(out, isp, d_key, d_pos, K, items, rb)
        else:
            eng.dispatch(d_rows, d_src, d_key, K, out, so, d_pos, rb, in_splits=isp)
        assert eng.status() == a2av.ERR_TIMEOUT
        assert eng.last_dispatch()["copy_kernel"] == "dispatch_gather_kernel"
    torch.cuda.synchronize()
    dispatch_checked(K, rows, src, key, rb)


@pytest.mark.parametrize("rb,combine,kernel", [
    (8, False, "dispatch_order_kernel"),
    (13, True, "combine_order_kernel"),
    (1024, True, "dispatch_gather_kernel"),
])
def test_starved_grid_barrier_times_out_and_writes_nothing(monkeypatch, rb, combine, kernel):
    """A2AV_DEBUG_STARVE=2: the grid barrier of the one-launch dispatch, of
    the one-launch combine and of the combine's checking gather waits for one
    CTA more than the grid holds -- a count nothing completes.  Every CTA
    gives up after about a second and the run records A2AV_ERR_TIMEOUT; no
    output row and no position is written; a normal call on a fresh handle
    afterwards is exact."""
    from tests._gpu import dispatch_checked
    rng = np.random.default_rng(rb + 3)
    W, K, n, m = 4, 3, 64, 3000  # 12000 items: past the one-kernel path
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, n, m).astype(np.int32) for _ in range(W)]
    key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.from_numpy(x).cuda() for x in src]
    d_key = [torch.from_numpy(x).cuda() for x in key]
    d_pos = [torch.empty(m, dtype=torch.int64, device="cuda") for _ in range(W)]
    out = [torch.empty(W * m * rb, dtype=torch.uint8, device="cuda") for _ in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    isp = torch.empty((W, W), dtype=torch.int64, device="cuda")
    items = [torch.full((m * rb,), 0xEE, dtype=torch.uint8, device="cuda") for _ in range(W)]
    if combine:
        with a2av.A2av(W) as eng:
            eng.dispatch(d_rows, d_src, d_key, K, out, so, d_pos, rb, in_splits=isp)
            assert eng.status() == a2av.OK
    else:
        for t in out:
            t.fill_(0xEE)
        for p in d_pos:
            p.fill_(-1)
    monkeypatch.setenv("A2AV_DEBUG_STARVE", "2")
    with a2av.A2av(W) as eng:
        monkeypatch.delenv("A2AV_DEBUG_STARVE")
        if combine:
            eng.combine_items(out, isp, d_key, d_pos, K, items, rb)
        else:
            eng.dispatch(d_rows, d_src, d_key, K, out, so, d_pos, rb, in_splits=isp)
        assert eng.status() == a2av.ERR_TIMEOUT
        assert eng.last_dispatch()["copy_kernel"] == kernel
    torch.cuda.synchronize()
    if combine:
        assert all(bool((t == 0xEE).all()) for t in items), "a row was written"
    else:
        assert all(bool((t == 0xEE).all()) for t in out), "a row was written"
        assert all(bool((p == -1).all()) for p in d_pos), "a position was written"
    dispatch_checked(K, rows, src, key, rb)
