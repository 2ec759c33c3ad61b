"""GPU parity: the CUDA exchange against the CPU oracle, byte for byte.

Covers the five workloads (config 4 over its 16 seeds), all three copy engines,
random split matrices with empty, skewed, diagonal and single-chunk patterns,
row sizes from 1 B to 14336 B, misaligned buffer addresses, small and large
grids (few or many tiles per CTA), W from 1 to 32, streams and reuse.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from tests._gpu import exchange_checked

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")
VEC, BULK, AUTO, STAGED = a2av.PATH_VECTOR, a2av.PATH_BULK, a2av.PATH_AUTO, a2av.PATH_STAGED


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()
    a2av.load()


@pytest.mark.parametrize("path", [AUTO, VEC, STAGED])
def test_cfg1(path):
    w = wl.cfg1(0)
    exchange_checked(w.inputs, w.splits, w.row_bytes, path=path,
                     expect_path=BULK if path == AUTO else path)


@pytest.mark.parametrize("seed", range(16))
def test_cfg4_seeds(seed):
    w = wl.cfg4(seed)
    exchange_checked(w.inputs, w.splits, w.row_bytes, expect_path=STAGED)
    if seed < 4:
        exchange_checked(w.inputs, w.splits, w.row_bytes, path=VEC, expect_path=VEC)


@pytest.mark.parametrize("path", [AUTO, VEC])
def test_cfg5(path):
    w = wl.cfg5(0)
    exchange_checked(w.inputs, w.splits, w.row_bytes, path=path,
                     expect_path=STAGED if path == AUTO else VEC)


@pytest.mark.parametrize("path", [AUTO, VEC, STAGED])
def test_cfg3_full(path):
    w = wl.cfg3(0)
    exchange_checked(w.inputs, w.splits, w.row_bytes, path=path)


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_cfg3_seeds_small_grid(seed):
    w = wl.cfg3(seed, tokens=2048)
    exchange_checked(w.inputs, w.splits, w.row_bytes, ctas_per_sm=1)


@pytest.mark.parametrize("mib", [0.5, 1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("path", [AUTO, VEC, STAGED])
def test_cfg2_sweep_points(mib, path):
    w = wl.cfg2(int(mib * (1 << 20)))
    exchange_checked(w.inputs, w.splits, w.row_bytes, path=path)


ROW_BYTES = [1, 2, 3, 4, 7, 8, 13, 16, 17, 31, 48, 256, 14336]


@pytest.mark.parametrize("rb", ROW_BYTES)
def test_random_splits(rb):
    rng = np.random.default_rng(rb)
    modes = ["uniform", "skew", "sparse", "empty", "diag", "one"]
    for k, W in enumerate([1, 2, 3, 5, 8, 13, 32]):
        for mode in modes:
            max_rows = 3000 if rb <= 16 else (300 if rb <= 256 else 6)
            w = wl.random_case(1000 * rb + 10 * k + modes.index(mode), W, rb, max_rows, mode)
            in_mis = [int(rng.integers(0, 16)) for _ in range(W)]
            out_mis = [int(rng.integers(0, 16)) for _ in range(W)]
            path = [AUTO, VEC, STAGED][(k + modes.index(mode)) % 3]
            exchange_checked(w.inputs, w.splits, rb, path=path, in_mis=in_mis, out_mis=out_mis,
                             ctas_per_sm=int(rng.choice([0, 1, 2])))


@pytest.mark.parametrize("path", [VEC, BULK, STAGED])
def test_aligned_engines_agree(path):
    for W, rb in ((4, 16), (8, 32), (3, 4096), (32, 16)):
        w = wl.random_case(7 + W, W, rb, 500, "uniform")
        exchange_checked(w.inputs, w.splits, rb, path=path, expect_path=path)


def test_bulk_request_on_misaligned_falls_back_to_staged():
    w = wl.random_case(3, 4, 16, 100, "uniform")
    exchange_checked(w.inputs, w.splits, 16, path=BULK, in_mis=[0, 4, 0, 0], expect_path=STAGED)
    w = wl.random_case(4, 4, 24, 100, "uniform")
    exchange_checked(w.inputs, w.splits, 24, path=BULK, expect_path=STAGED)


@pytest.mark.parametrize("grid", [1, 2, 8, 32])
def test_grid_sizes(grid):
    # more CTAs than fit on the GPU at once, for every engine
    w = wl.cfg4(5, rows=1 << 16)
    for path in (AUTO, VEC):
        exchange_checked(w.inputs, w.splits, w.row_bytes, path=path, ctas_per_sm=grid)
    w = wl.cfg2(4 << 20)
    for path in (AUTO, VEC, STAGED):
        exchange_checked(w.inputs, w.splits, w.row_bytes, path=path, ctas_per_sm=grid)


def test_single_huge_chunk_and_tile_edges():
    # one chunk that is an exact multiple of the tile, one with a ragged tail
    for rows in (4096, 4097, 65536 + 3):
        S = np.zeros((4, 4), np.int64)
        S[2, 1] = rows
        inputs = [np.zeros(0, np.uint8)] * 4
        inputs[2] = np.random.default_rng(rows).integers(0, 256, rows * 16, dtype=np.uint8)
        for path in (AUTO, VEC, STAGED):
            exchange_checked(inputs, S, 16, path=path)


def test_side_stream_and_reuse():
    s = torch.cuda.Stream()
    eng = a2av.A2av(4)
    try:
        for seed in range(3):
            w = wl.cfg4(seed, rows=1 << 14, W=4)
            with torch.cuda.stream(s):
                exchange_checked(w.inputs, w.splits, w.row_bytes, stream=s, engine=eng)
    finally:
        eng.close()


def test_round_trip_restores_inputs():
    w = wl.cfg4(9, rows=1 << 15)
    W, rb = w.W, w.row_bytes
    eng = a2av.A2av(W)
    ins = [torch.from_numpy(b).cuda() for b in w.inputs]
    S = torch.from_numpy(w.splits).cuda()
    mid = [torch.empty(int(w.splits[:, p].sum()) * rb, dtype=torch.uint8, device="cuda")
           for p in range(W)]
    back = [torch.empty_like(t) for t in ins]
    so1 = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    so2 = torch.empty_like(so1)
    eng.run(ins, S, mid, so1, rb)
    eng.run(mid, S.t().contiguous(), back, so2, rb)
    assert eng.status() == a2av.OK
    eng.close()
    for r in range(W):
        assert torch.equal(back[r], ins[r])
    assert torch.equal(so2[:, 0, :], S)


def test_back_to_back_without_sync_keeps_stream_order():
    eng = a2av.A2av(2)
    a = torch.arange(64, dtype=torch.uint8, device="cuda")
    b = torch.arange(64, 128, dtype=torch.uint8, device="cuda")
    o = [torch.zeros(64, dtype=torch.uint8, device="cuda") for _ in range(2)]
    so = torch.empty((2, 2, 2), dtype=torch.int64, device="cuda")
    S1 = torch.tensor([[64, 0], [0, 64]], dtype=torch.int64, device="cuda")
    S2 = torch.tensor([[0, 64], [64, 0]], dtype=torch.int64, device="cuda")
    for _ in range(50):
        eng.run([a, b], S1, o, so, 1)
        eng.run([a, b], S2, o, so, 1)
    assert eng.status() == a2av.OK
    eng.close()
    assert torch.equal(o[0], b) and torch.equal(o[1], a)
    assert so[:, 0, :].tolist() == [[0, 64], [64, 0]]


def test_many_tiny_segments_per_tile():
    # W = 32 ranks, a few 1-byte or 13-byte rows per chunk: every tile holds
    # dozens of segments, each with its own granule overhang in the stage
    for rb in (1, 13):
        S = np.random.default_rng(rb).integers(0, 4, size=(32, 32)).astype(np.int64)
        inputs = [np.random.default_rng(100 + r).integers(0, 256, int(S[r].sum()) * rb,
                                                          dtype=np.uint8) for r in range(32)]
        mis = list(range(16)) * 2
        for path in (AUTO, VEC, STAGED):
            exchange_checked(inputs, S, rb, path=path, in_mis=mis, out_mis=mis[::-1])


@pytest.mark.parametrize("path", [AUTO, VEC, STAGED])
def test_combine_returns_every_row_home(path):
    from tests._gpu import combine_checked
    import oracle
    cases = [wl.cfg3(4, tokens=1024), wl.cfg4(3, rows=1 << 16), wl.cfg5(1, batch=1024),
             wl.random_case(21, 13, 7, 200, "skew"), wl.random_case(22, 32, 1, 50, "sparse")]
    for w in cases:
        mid, dso = oracle.default().exchange(w.inputs, w.splits, w.row_bytes)
        mis = [r % 16 for r in range(w.W)]
        back = combine_checked(mid, dso, w.row_bytes, path=path, in_mis=mis, out_mis=mis[::-1])
        for r in range(w.W):
            assert np.array_equal(back[r], w.inputs[r]), "combine(dispatch(x)) != x"


def test_dispatch_then_combine_on_device():
    # the GPU's own out_splits_offsets drives the GPU's reverse exchange
    w = wl.cfg3(5, tokens=2048)
    W, rb = w.W, w.row_bytes
    ins = [torch.from_numpy(b).cuda() for b in w.inputs]
    S = torch.from_numpy(w.splits).cuda()
    mid = [torch.empty(int(w.splits[:, p].sum()) * rb, dtype=torch.uint8, device="cuda")
           for p in range(W)]
    back = [torch.full_like(t, 0xEE) for t in ins]
    dso = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    cso = torch.empty_like(dso)
    with a2av.A2av(W) as eng:
        eng.run(ins, S, mid, dso, rb)
        eng.combine(mid, dso, back, cso, rb)
        assert eng.status() == a2av.OK
    for r in range(W):
        assert torch.equal(back[r], ins[r])
    assert torch.equal(cso[:, 0, :], S)


def test_pinned_host_buffers_zero_copy():
    # inputs and outputs in pinned host memory: the kernel reads and writes
    # them over the host link (the binding picks the vector engine)
    import oracle
    for w in (wl.cfg4(11, rows=1 << 14), wl.cfg1(2)):
        W, rb = w.W, w.row_bytes
        ref, ref_so = oracle.default().exchange(w.inputs, w.splits, rb)
        S = torch.from_numpy(w.splits).cuda()
        so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
        host_in = [torch.from_numpy(b).pin_memory() for b in w.inputs]
        dev_in = [t.cuda() for t in host_in]
        for ins in (host_in, dev_in):
            outs = [torch.full((r.size,), 0xEE, dtype=torch.uint8).pin_memory() for r in ref]
            with a2av.A2av(W) as eng:
                eng.run(ins, S, outs, so, rb)
                assert eng.status() == a2av.OK
                assert eng.last_launch()["path"] == VEC
                # the configured engine comes back for device-only calls
                d_outs = [torch.empty(r.size, dtype=torch.uint8, device="cuda") for r in ref]
                eng.run(dev_in, S, d_outs, so, rb)
                assert eng.last_launch()["path"] == (BULK if rb % 16 == 0 else STAGED)
            torch.cuda.synchronize()
            for p in range(W):
                assert np.array_equal(outs[p].numpy(), ref[p])
                assert np.array_equal(d_outs[p].cpu().numpy(), ref[p])
            assert np.array_equal(so.cpu().numpy(), ref_so)


@pytest.mark.parametrize("requested", [a2av.PATH_AUTO, a2av.PATH_BULK, a2av.PATH_STAGED])
def test_library_routes_host_buffers_to_the_vector_engine(requested):
    """Through the raw C ABI (no binding logic): whatever engine the handle
    asks for, a call with a pinned host buffer runs the vector engine (plain
    loads and stores reach host memory; cp.async.bulk is kept to device
    memory), and the next all-device call gets the requested engine back."""
    import oracle
    w = wl.cfg1(3)
    W, rb = w.W, w.row_bytes
    ref, ref_so = oracle.default().exchange(w.inputs, w.splits, rb)
    S = torch.from_numpy(w.splits).cuda()
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    host_in = [torch.from_numpy(b).pin_memory() for b in w.inputs]
    dev_in = [t.cuda() for t in host_in]
    outs = [torch.full((r.size,), 0xEE, dtype=torch.uint8, device="cuda") for r in ref]
    rc, h = a2av.a2av_create(W)
    assert rc == a2av.OK
    try:
        assert a2av.a2av_set_path(h, requested) == a2av.OK
        stream = torch.cuda.current_stream().cuda_stream
        ptrs = lambda ts: [t.data_ptr() for t in ts]  # noqa: E731
        mixed = [host_in[0]] + dev_in[1:]  # one host buffer is enough
        assert a2av.a2av_run(h, ptrs(mixed), S.data_ptr(), ptrs(outs), so.data_ptr(), rb,
                             stream) == a2av.OK
        assert a2av.a2av_status(h, stream) == (a2av.OK, a2av.OK)
        assert a2av.a2av_last_launch(h)[1] == a2av.PATH_VECTOR
        for p in range(W):
            assert np.array_equal(outs[p].cpu().numpy(), ref[p])
        assert np.array_equal(so.cpu().numpy(), ref_so)
        assert a2av.a2av_run(h, ptrs(dev_in), S.data_ptr(), ptrs(outs), so.data_ptr(), rb,
                             stream) == a2av.OK
        assert a2av.a2av_status(h, stream) == (a2av.OK, a2av.OK)
        want = a2av.PATH_BULK if requested in (a2av.PATH_AUTO, a2av.PATH_BULK) else requested
        assert a2av.a2av_last_launch(h)[1] == want
        for p in range(W):
            assert np.array_equal(outs[p].cpu().numpy(), ref[p])
    finally:
        a2av.a2av_destroy(h)


def test_dispatch_on_host_rows_uses_plain_loads():
    """The fused dispatch through the raw C ABI with the source rows in
    pinned host memory: the library copies them with plain loads and stores
    (no cp.async.bulk), and the result equals the oracle's."""
    import oracle
    w = wl.cfg3(4, tokens=96, hidden=512)
    K, rows, src, key = wl.dispatch_items(w)
    W, rb = w.W, w.row_bytes
    ref, ref_so, ref_pos, ref_S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    h_rows = [torch.from_numpy(r).pin_memory() for r in rows]
    d_src = [torch.from_numpy(s).cuda() for s in src]
    d_key = [torch.from_numpy(k).cuda() for k in key]
    d_pos = [torch.full((k.size,), -1, dtype=torch.int64, device="cuda") for k in key]
    d_out = [torch.full((r.size,), 0xEE, dtype=torch.uint8, device="cuda") for r in ref]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    isp = torch.full((W, W), -7, dtype=torch.int64, device="cuda")
    m = [k.size for k in key]
    nbytes = a2av.a2av_dispatch_workspace_bytes(W, K, max(m))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc, h = a2av.a2av_create(W)
    assert rc == a2av.OK
    try:
        stream = torch.cuda.current_stream().cuda_stream
        rc = a2av.a2av_dispatch(h, K, [t.data_ptr() for t in h_rows], [r.size // rb for r in rows],
                                [t.data_ptr() for t in d_src], [t.data_ptr() for t in d_key], m,
                                [t.data_ptr() for t in d_out], so.data_ptr(),
                                [t.data_ptr() for t in d_pos], isp.data_ptr(), rb, ws.data_ptr(),
                                nbytes, stream)
        assert rc == a2av.OK
        assert a2av.a2av_status(h, stream) == (a2av.OK, a2av.OK)
    finally:
        a2av.a2av_destroy(h)
    assert np.array_equal(so.cpu().numpy(), ref_so) and np.array_equal(isp.cpu().numpy(), ref_S)
    for r in range(W):
        assert np.array_equal(d_pos[r].cpu().numpy(), ref_pos[r])
    for p in range(W):
        assert np.array_equal(d_out[p].cpu().numpy(), ref[p])
