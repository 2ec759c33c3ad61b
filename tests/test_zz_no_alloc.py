"""The allocation-free entry point, a2av_run_noalloc, through the C ABI.

Some callers cannot call cudaMalloc: engines that fix all their device memory
at start-up, hosts that own the only allocator, latency paths that cannot
afford an allocation's device synchronisation.  For them the library offers
a2av_run_noalloc, which takes no handle and keeps its status word in a small
array compiled into the library.  These tests check that it produces exactly
what the handle-based a2av_run produces, and what the CPU oracle produces --
every output byte and out_splits_offsets -- on two calls in a row, that each
call starts from a cleared status word, and that it rejects a rank count
beyond its limit.

This file is collected last on purpose, so that a failure here stops a
``-x`` run only after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()
    a2av.load()


def _device_case(w):
    ins = [torch.from_numpy(b).cuda() for b in w.inputs]
    S = torch.from_numpy(w.splits).cuda()
    recv = [int(w.splits[:, p].sum()) * w.row_bytes for p in range(w.W)]
    return ins, S, recv


def _fresh_outputs(recv, W):
    outs = [torch.full((n + 64,), 0xEE, dtype=torch.uint8, device="cuda") for n in recv]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    return outs, so


def _ptrs(ts):
    return [t.data_ptr() if t.numel() else 0 for t in ts]


def _with_handle(w, ins, S, recv, engine=None):
    outs, so = _fresh_outputs(recv, w.W)
    with a2av.A2av(w.W) as eng:
        eng.run(ins, S, outs, so, w.row_bytes)
        assert eng.status() == a2av.OK
        if engine is not None:
            assert eng.last_launch()["path"] == engine
    return outs, so


def _without_alloc(w, ins, S, recv):
    outs, so = _fresh_outputs(recv, w.W)
    stream = torch.cuda.current_stream().cuda_stream
    rc, status = a2av.a2av_run_noalloc(w.W, 0, 0, _ptrs(ins), S.data_ptr(), _ptrs(outs),
                                       so.data_ptr(), w.row_bytes, stream)
    assert rc == a2av.OK, a2av.a2av_error_string(rc)
    assert status == a2av.OK
    return outs, so


def test_noalloc_matches_a2av_run_on_two_calls_in_a_row():
    # an aligned exchange, then one of 13-byte rows: the engine AUTO picks,
    # which is the bulk engine for the first and the staged engine for the
    # second (a2av_run on a handle reports it; the call without a handle
    # chooses the same way)
    cases = [(wl.cfg1(0), a2av.PATH_BULK), (wl.cfg4(2, rows=1 << 15), a2av.PATH_STAGED)]
    for w, engine in cases:
        ins, S, recv = _device_case(w)
        ref_outs, ref_so = _with_handle(w, ins, S, recv, engine)
        got_outs, got_so = _without_alloc(w, ins, S, recv)
        torch.cuda.synchronize()
        # the same bar as every other test of this library: bit-exact, against
        # the handle-based entry point and against the CPU oracle
        assert torch.equal(got_so, ref_so)
        for g, r in zip(got_outs, ref_outs):
            assert torch.equal(g, r)
        want, want_so = oracle.default().exchange(w.inputs, w.splits, w.row_bytes)
        assert np.array_equal(got_so.cpu().numpy(), want_so)
        for p, g in enumerate(got_outs):
            n = want[p].size
            got = g.cpu().numpy()
            assert np.array_equal(got[:n], want[p]) and np.all(got[n:] == 0xEE)


def test_each_call_starts_from_a_cleared_status_word():
    w = wl.cfg1(1)
    ins, S, recv = _device_case(w)
    outs, so = _fresh_outputs(recv, w.W)
    bad = S.clone()
    bad[0, 1] = -1
    stream = torch.cuda.current_stream().cuda_stream
    rc, status = a2av.a2av_run_noalloc(w.W, 0, 0, _ptrs(ins), bad.data_ptr(), _ptrs(outs),
                                       so.data_ptr(), w.row_bytes, stream)
    assert rc == a2av.OK and status == a2av.ERR_BAD_SPLITS
    torch.cuda.synchronize()
    assert bool((so == -7).all()) and all(bool((o == 0xEE).all()) for o in outs)
    # the next valid call reports OK and matches the handle-based entry point
    got_outs, got_so = _without_alloc(w, ins, S, recv)
    ref_outs, ref_so = _with_handle(w, ins, S, recv)
    assert torch.equal(got_so, ref_so)
    for g, r in zip(got_outs, ref_outs):
        assert torch.equal(g, r)


def test_noalloc_rejects_sizes_beyond_its_limit():
    dummy = [0] * 40
    assert a2av.a2av_run_noalloc(a2av.MAX_RANKS + 1, 0, 0, dummy, 8, dummy, 8, 16)[0] \
        == a2av.ERR_UNSUPPORTED
    assert a2av.a2av_run_noalloc(0, 0, 0, dummy, 8, dummy, 8, 16)[0] == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run_noalloc(2, 0, 0, dummy, 8, dummy, 8, 0)[0] == a2av.ERR_INVALID_ARG
