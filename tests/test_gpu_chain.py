"""Exchanges enqueued back to back with no host synchronisation between them.

Each launch uses programmatic dependent launch (unless A2AV_PDL=0 when the
handle is made): its CTAs may be scheduled while the previous kernel on the
stream still runs, and must wait on the device for that kernel's writes
before reading.  These chains make every exchange read what the previous
one wrote, so a missing wait shows up as wrong bytes.  Also the keyed-jagged
pair of a sparse embedding batch -- bag lengths and keys -- on one stream and
on two.
"""
import os

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


def _engine(W, path, pdl):
    saved = os.environ.get("A2AV_PDL")
    os.environ["A2AV_PDL"] = "1" if pdl else "0"
    try:
        return a2av.A2av(W, path=path)
    finally:
        if saved is None:
            del os.environ["A2AV_PDL"]
        else:
            os.environ["A2AV_PDL"] = saved


def _chain_splits(rng, W, rows0, steps):
    """Split matrices whose step k + 1 sends exactly the rows step k received."""
    rows, out = np.asarray(rows0), []
    for _ in range(steps):
        S = np.stack([rng.multinomial(int(rows[r]), rng.dirichlet([0.5] * W)) for r in range(W)])
        out.append(S.astype(np.int64))
        rows = S.sum(axis=0)
    return out


@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("path,rb", [(a2av.PATH_AUTO, 1024), (a2av.PATH_AUTO, 13),
                                     (a2av.PATH_VECTOR, 48)])
def test_dependent_exchanges_back_to_back(pdl, path, rb):
    W, steps = 4, 8
    rng = np.random.default_rng(rb + 7 * pdl)
    rows0 = rng.integers(500, 3000, W)
    splits = _chain_splits(rng, W, rows0, steps)
    cap = int(max(max(S.sum(axis=0).max(), S.sum(axis=1).max()) for S in splits))
    host = [rng.integers(0, 256, int(rows0[r]) * rb, dtype=np.uint8) for r in range(W)]
    bufs = [[torch.zeros(cap * rb, dtype=torch.uint8, device="cuda") for _ in range(W)]
            for _ in range(2)]
    for r in range(W):
        bufs[0][r][: host[r].size].copy_(torch.from_numpy(host[r]))
    d_splits = [torch.from_numpy(S).cuda() for S in splits]
    sos = [torch.empty((W, 2, W), dtype=torch.int64, device="cuda") for _ in range(steps)]
    eng = _engine(W, path, pdl)
    torch.cuda.synchronize()
    for k in range(steps):  # no synchronisation inside the chain
        eng.run(bufs[k % 2], d_splits[k], bufs[(k + 1) % 2], sos[k], rb)
    torch.cuda.synchronize()
    assert eng.status() == a2av.OK
    eng.close()
    o = oracle.default()
    cur = host
    for k in range(steps):
        cur, so = o.exchange(cur, splits[k], rb)
        assert np.array_equal(sos[k].cpu().numpy(), so), k
    got = bufs[steps % 2]
    for p in range(W):
        assert np.array_equal(got[p][: cur[p].size].cpu().numpy(), cur[p]), p


@pytest.mark.parametrize("pdl", [True, False])
def test_dispatch_then_combine_chain(pdl):
    """The fused dispatch, then the reverse exchange reading its outputs and
    its out_splits_offsets, then a second dispatch reusing the workspace --
    all on one stream, one synchronisation at the end."""
    w = wl.cfg3(5, tokens=1024, hidden=256)
    K, rows, src, key = wl.dispatch_items(w)
    W, rb = w.W, w.row_bytes
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.from_numpy(x).cuda() for x in src]
    d_key = [torch.from_numpy(x).cuda() for x in key]
    recv = [int(w.splits[:, p].sum()) * rb for p in range(W)]
    outs = [[torch.empty(n, dtype=torch.uint8, device="cuda") for n in recv] for _ in range(2)]
    sos = [torch.empty((W, 2, W), dtype=torch.int64, device="cuda") for _ in range(2)]
    pos = [[torch.empty(x.size, dtype=torch.int64, device="cuda") for x in key] for _ in range(2)]
    back = [torch.empty(int(w.splits[r].sum()) * rb, dtype=torch.uint8, device="cuda")
            for r in range(W)]
    back_so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    eng = _engine(W, a2av.PATH_AUTO, pdl)
    torch.cuda.synchronize()
    eng.dispatch(d_rows, d_src, d_key, K, outs[0], sos[0], pos[0], rb)
    eng.combine(outs[0], sos[0], back, back_so, rb)
    eng.dispatch(d_rows, d_src, d_key, K, outs[1], sos[1], pos[1], rb)
    torch.cuda.synchronize()
    assert eng.status() == a2av.OK
    eng.close()
    ref, ref_so, ref_pos, _ = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    for j in range(2):
        assert np.array_equal(sos[j].cpu().numpy(), ref_so)
        for p in range(W):
            assert np.array_equal(outs[j][p].cpu().numpy(), ref[p]), (j, p)
        for r in range(W):
            assert np.array_equal(pos[j][r].cpu().numpy(), ref_pos[r]), (j, r)
    for r in range(W):  # combine returns the rows in key order: the generator's grouped input
        assert np.array_equal(back[r].cpu().numpy(), w.inputs[r]), r


@pytest.mark.parametrize("two_streams", [False, True])
def test_keyed_jagged_lengths_and_keys(two_streams):
    w = wl.cfg5(2, batch=1024)
    lw = wl.cfg5_lengths(w)
    W = w.W
    parts = [lw, w]
    dev = []
    for x in parts:
        d_in = [torch.from_numpy(b).cuda() for b in x.inputs]
        d_out = [torch.full((int(x.splits[:, p].sum()) * x.row_bytes,), 0xEE, dtype=torch.uint8,
                            device="cuda") for p in range(W)]
        dev.append((d_in, torch.from_numpy(x.splits).cuda(), d_out,
                    torch.empty((W, 2, W), dtype=torch.int64, device="cuda")))
    eng = a2av.A2av(W)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream() if two_streams else main
    side.wait_stream(main)
    torch.cuda.synchronize()
    eng.run(*dev[0], lw.row_bytes, stream=side)
    eng.run(*dev[1], w.row_bytes, stream=main)
    main.wait_stream(side)
    torch.cuda.synchronize()
    assert eng.status() == a2av.OK
    eng.close()
    o = oracle.default()
    for (d_in, _, d_out, d_so), x in zip(dev, parts):
        ref, ref_so = o.exchange(x.inputs, x.splits, x.row_bytes)
        assert np.array_equal(d_so.cpu().numpy(), ref_so), x.name
        for p in range(W):
            assert np.array_equal(d_out[p].cpu().numpy(), ref[p]), (x.name, p)
    l_so, k_so = dev[0][3].cpu().numpy(), dev[1][3].cpu().numpy()
    for p in range(W):  # peer p can cut the keys from rank r into bags
        lens = dev[0][2][p].cpu().numpy().view(np.int32)
        for r in range(W):
            o0, n0 = int(l_so[p][1][r]), int(l_so[p][0][r])
            assert int(lens[o0:o0 + n0].sum()) == int(k_so[p][0][r])
