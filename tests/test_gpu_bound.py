"""Bound calls: arguments marshalled once, the launch re-enqueued on the same
buffers while the device data change between calls (new splits, new keys).
Every call is checked against the oracle."""
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


@pytest.mark.parametrize("rb", [13, 64])
def test_bound_run_follows_new_splits(rb):
    W, cap = 4, 1500
    rng = np.random.default_rng(rb)
    host = [rng.integers(0, 256, cap * rb, dtype=np.uint8) for _ in range(W)]
    d_in = [torch.from_numpy(b).cuda() for b in host]
    d_out = [torch.full((W * cap * rb,), 0xEE, dtype=torch.uint8, device="cuda") for _ in range(W)]
    S = torch.zeros((W, W), dtype=torch.int64, device="cuda")
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    side = torch.cuda.Stream()
    with a2av.A2av(W, in_capacity_rows=cap, out_capacity_rows=W * cap) as eng:
        call = eng.bind_run(d_in, S, d_out, so, rb)
        for trial in range(4):
            splits = np.stack([rng.multinomial(int(rng.integers(0, cap + 1)),
                                               rng.dirichlet([0.4] * W)) for _ in range(W)])
            S.copy_(torch.from_numpy(splits.astype(np.int64)))
            if trial % 2:
                side.wait_stream(torch.cuda.current_stream())
                call(stream=side)  # the same launch on another stream
                torch.cuda.current_stream().wait_stream(side)
            else:
                call()
            torch.cuda.synchronize()
            assert eng.status() == a2av.OK
            used = [b[: int(splits[r].sum()) * rb] for r, b in enumerate(host)]
            ref, ref_so = oracle.default().exchange(used, splits, rb)
            assert np.array_equal(so.cpu().numpy(), ref_so)
            for p in range(W):
                assert np.array_equal(d_out[p][: ref[p].size].cpu().numpy(), ref[p]), (trial, p)


def test_bound_run_multi_keyed_jagged_pair():
    w = wl.cfg5(6, batch=512)
    parts = [wl.cfg5_lengths(w), w]
    bufs = []
    for x in parts:
        bufs.append(([torch.from_numpy(b).cuda() for b in x.inputs],
                     torch.from_numpy(x.splits).cuda(),
                     [torch.empty(int(x.splits[:, p].sum()) * x.row_bytes, dtype=torch.uint8,
                                  device="cuda") for p in range(x.W)],
                     torch.empty((x.W, 2, x.W), dtype=torch.int64, device="cuda")))
    with a2av.A2av(w.W) as eng:
        call = eng.bind_run_multi([(*b, x.row_bytes) for b, x in zip(bufs, parts)])
        for _ in range(3):
            for b in bufs:
                for t in b[2]:
                    t.fill_(0xEE)
            call()
            torch.cuda.synchronize()
            assert eng.status() == a2av.OK
            for (_, _, outs, so), x in zip(bufs, parts):
                ref, ref_so = oracle.default().exchange(x.inputs, x.splits, x.row_bytes)
                assert np.array_equal(so.cpu().numpy(), ref_so)
                for p in range(x.W):
                    assert np.array_equal(outs[p].cpu().numpy(), ref[p])


@pytest.mark.parametrize("rb", [8, 1024])
def test_bound_dispatch_follows_new_keys(rb):
    W, K, n, m = 3, 4, 700, 2600
    rng = np.random.default_rng(rb + 1)
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.zeros(m, dtype=torch.int32, device="cuda") for _ in range(W)]
    d_key = [torch.zeros(m, dtype=torch.int32, device="cuda") for _ in range(W)]
    d_pos = [torch.empty(m, dtype=torch.int64, device="cuda") for _ in range(W)]
    d_out = [torch.empty(W * m * rb, dtype=torch.uint8, device="cuda") for _ in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    isp = torch.empty((W, W), dtype=torch.int64, device="cuda")
    with a2av.A2av(W) as eng:
        call = eng.bind_dispatch(d_rows, d_src, d_key, K, d_out, so, d_pos, rb, in_splits=isp)
        for trial in range(3):
            src = [rng.integers(0, n, m).astype(np.int32) for _ in range(W)]
            key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
            for r in range(W):
                d_src[r].copy_(torch.from_numpy(src[r]))
                d_key[r].copy_(torch.from_numpy(key[r]))
            call()
            torch.cuda.synchronize()
            assert eng.status() == a2av.OK
            ref, ref_so, ref_pos, ref_S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
            assert np.array_equal(so.cpu().numpy(), ref_so)
            assert np.array_equal(isp.cpu().numpy(), ref_S)
            for p in range(W):
                assert np.array_equal(d_out[p][: ref[p].size].cpu().numpy(), ref[p]), (trial, p)
            for r in range(W):
                assert np.array_equal(d_pos[r].cpu().numpy(), ref_pos[r])


def test_bound_calls_on_host_buffers_take_the_vector_engine():
    """The library, not the binding, routes host-resident buffers: a bound
    call on pinned host memory runs the vector engine and is exact."""
    import oracle
    w = wl.cfg1(5)
    W, rb = w.W, w.row_bytes
    ref, ref_so = oracle.default().exchange(w.inputs, w.splits, rb)
    host_in = [torch.from_numpy(b).pin_memory() for b in w.inputs]
    outs = [torch.full((r.size,), 0xEE, dtype=torch.uint8, device="cuda") for r in ref]
    S = torch.from_numpy(w.splits).cuda()
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    with a2av.A2av(W) as eng:
        eng.bind_run(host_in, S, outs, so, rb)()
        assert eng.status() == a2av.OK
        assert eng.last_launch()["path"] == a2av.PATH_VECTOR
    for p in range(W):
        assert np.array_equal(outs[p].cpu().numpy(), ref[p])
    assert np.array_equal(so.cpu().numpy(), ref_so)


