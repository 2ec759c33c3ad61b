"""GPU parity of the fused combine (a2av_combine_items): every item's row
from the peers' dispatch-layout buffers back into item order, against the
oracle and as the inverse of the GPU's own fused dispatch -- byte for byte,
with sentinel rows past every output and guard bands around misaligned
buffers."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests._gpu import Guarded, SENTINEL, aligned_copy_kernel

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()


def _combine_checked(K, peers, S, keys, pos, rb, mis=None, expect=None, expect_copy=None):
    """Run the fused combine on host arrays; compare with the oracle's (and,
    with ``expect_copy``, that the library moved the rows with that kernel)."""
    W = len(peers)
    mis = mis or [0] * (2 * W)
    g_peer = [Guarded(peers[p].size, mis[p], host=peers[p]) for p in range(W)]
    m = [k.size for k in keys]
    g_out = [Guarded((m[r] + 2) * rb, mis[W + r], fill=SENTINEL) for r in range(W)]
    d_key = [torch.from_numpy(np.ascontiguousarray(k, np.int32)).cuda() for k in keys]
    d_pos = [torch.from_numpy(np.ascontiguousarray(x, np.int64)).cuda() for x in pos]
    d_S = torch.from_numpy(np.ascontiguousarray(S, np.int64)).cuda()
    with a2av.A2av(W) as eng:
        eng.combine_items([g.view for g in g_peer], d_S, d_key, d_pos, K,
                          [g.view for g in g_out], rb)
        st = eng.status()
        chain = eng.last_dispatch()
    ref = [np.full((m[r] + 2) * rb, SENTINEL, np.uint8) for r in range(W)]
    rc = oracle.default().combine_items(K, peers, S, keys, pos, ref, rb)
    assert st == rc, f"device status {st}, oracle {rc}"
    for r in range(W):
        got = g_out[r].view.cpu().numpy()
        assert np.array_equal(got, ref[r]), f"rank {r} differs from the oracle"
        assert g_out[r].guards_intact() and g_peer[r].guards_intact()
        assert np.array_equal(g_peer[r].view.cpu().numpy(), peers[r]), "peers were modified"
    if expect is not None:
        for r in range(W):
            assert np.array_equal(g_out[r].view.cpu().numpy()[: m[r] * rb], expect[r])
    if expect_copy is not None:
        assert chain["copy_kernel"] == expect_copy, chain
    return st


@pytest.mark.parametrize("rb", [1, 8, 13, 64, 100, 256, 1040, 2048, 4096, 9216, 14336, 20480,
                                40000])
def test_inverse_of_the_gpu_dispatch(rb):
    """combine_items(dispatch(x)) on the GPU puts every item's source row back."""
    rng = np.random.default_rng(rb)
    W, K, n, m = 4, 3, 300, 2500
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, n, m).astype(np.int32) for _ in range(W)]
    key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.from_numpy(x).cuda() for x in src]
    d_key = [torch.from_numpy(x).cuda() for x in key]
    S = np.zeros((W, W), np.int64)
    for r in range(W):
        S[r] = np.bincount(key[r] // K, minlength=W)
    d_out = [torch.empty(int(S[:, p].sum()) * rb, dtype=torch.uint8, device="cuda")
             for p in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    isp = torch.empty((W, W), dtype=torch.int64, device="cuda")
    d_pos = [torch.empty(m, dtype=torch.int64, device="cuda") for _ in range(W)]
    back = [torch.full((m * rb,), 0xEE, dtype=torch.uint8, device="cuda") for _ in range(W)]
    with a2av.A2av(W) as eng:
        eng.dispatch(d_rows, d_src, d_key, K, d_out, so, d_pos, rb, in_splits=isp)
        eng.combine_items(d_out, isp, d_key, d_pos, K, back, rb)  # same stream, no sync
        assert eng.status() == a2av.OK
    for r in range(W):
        want = rows[r].reshape(-1, rb)[src[r]].reshape(-1)
        assert np.array_equal(back[r].cpu().numpy(), want), r


@pytest.mark.parametrize("hidden", [7168, 512])
def test_full_size_moe_round_trip(hidden):
    """The MoE workload at full size (W=8, 8192 tokens a rank, top-2), in the
    launch configuration the benchmark times: combine_items(dispatch(x))
    gives every item its token's row back (14 KiB rows: the gather; 1 KiB
    rows: the warp copy at eight vectors per lane)."""
    w = wl.cfg3(0, hidden=hidden)
    K, rows, src, key = wl.dispatch_items(w)
    W, rb = w.W, w.row_bytes
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.from_numpy(x).cuda() for x in src]
    d_key = [torch.from_numpy(x).cuda() for x in key]
    d_out = [torch.empty(int(w.splits[:, p].sum()) * rb, dtype=torch.uint8, device="cuda")
             for p in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    isp = torch.empty((W, W), dtype=torch.int64, device="cuda")
    d_pos = [torch.empty(x.size, dtype=torch.int64, device="cuda") for x in key]
    back = [torch.full((x.size * rb,), 0xEE, dtype=torch.uint8, device="cuda") for x in key]
    with a2av.A2av(W) as eng:
        eng.dispatch(d_rows, d_src, d_key, K, d_out, so, d_pos, rb, in_splits=isp)
        eng.combine_items(d_out, isp, d_key, d_pos, K, back, rb)
        assert eng.status() == a2av.OK
    assert np.array_equal(isp.cpu().numpy(), w.splits), "split matrix differs from the workload's"
    for r in range(W):
        want = torch.index_select(d_rows[r].view(-1, rb), 0, d_src[r].long())
        assert torch.equal(back[r].view(-1, rb), want), f"rank {r}: rows not restored"


@pytest.mark.parametrize("rb", [3, 16, 64, 2048, 14336])
@pytest.mark.parametrize("aligned", [True, False])
def test_against_the_oracle(rb, aligned):
    """Peers hold rows of their own (an expert's output), not the dispatch's."""
    rng = np.random.default_rng(rb * 2 + aligned)
    w = wl.cfg3(1, tokens=512, hidden=max(rb // 2, 1)) if rb % 2 == 0 else None
    if w is not None and w.row_bytes == rb:
        K, rows, src, key = wl.dispatch_items(w)
    else:
        W, K = 3, 4
        rows = [rng.integers(0, 256, 50 * rb, dtype=np.uint8) for _ in range(W)]
        src = [rng.integers(0, 50, 700).astype(np.int32) for _ in range(W)]
        key = [rng.integers(0, W * K, 700).astype(np.int32) for _ in range(W)]
    outs, so, pos, S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    peers = [rng.integers(0, 256, b.size, dtype=np.uint8) for b in outs]
    W = len(peers)
    mis = None if aligned else [int(rng.integers(1, 16)) for _ in range(2 * W)]
    assert _combine_checked(K, peers, S, key, pos, rb, mis) == a2av.OK


@pytest.mark.parametrize("case", ["key", "negative_key", "pos_outside_group", "pos_too_large",
                                  "negative_split", "null_peer"])
def test_errors_write_nothing(case):
    W, K, rb = 2, 2, 16
    S = np.array([[2, 1], [0, 2]], np.int64)
    peers = [np.arange(2 * rb, dtype=np.uint8), np.arange(3 * rb, dtype=np.uint8)]
    key = [np.array([0, 2, 1], np.int32), np.array([3, 2], np.int32)]
    pos = [np.array([0, 2, 1], np.int64), np.array([1, 0], np.int64)]
    want = {"key": a2av.ERR_BAD_INDEX, "negative_key": a2av.ERR_BAD_INDEX,
            "pos_outside_group": a2av.ERR_BAD_INDEX, "pos_too_large": a2av.ERR_BAD_INDEX,
            "negative_split": a2av.ERR_BAD_SPLITS, "null_peer": a2av.ERR_BAD_SPLITS}[case]
    if case == "key":
        key[1] = np.array([4, 2], np.int32)
    elif case == "negative_key":
        key[0] = np.array([0, -1, 1], np.int32)
    elif case == "pos_outside_group":
        pos[0] = np.array([0, 1, 2], np.int64)
    elif case == "pos_too_large":
        pos[1] = np.array([2, 0], np.int64)
    elif case == "negative_split":
        S = np.array([[2, 1], [-1, 2]], np.int64)
    if case == "null_peer":  # peer 1 has no buffer but receives rows
        d_S = torch.from_numpy(S).cuda()
        outs = [torch.full((5 * rb,), SENTINEL, dtype=torch.uint8, device="cuda") for _ in range(W)]
        with a2av.A2av(W) as eng:
            eng.combine_items([torch.from_numpy(peers[0]).cuda(), None], d_S,
                              [torch.from_numpy(k).cuda() for k in key],
                              [torch.from_numpy(x).cuda() for x in pos], K, outs, rb)
            assert eng.status() == want
        assert all(bool((o == SENTINEL).all()) for o in outs)
        return
    assert _combine_checked(K, peers, S, key, pos, rb) == want


def test_decode_size_and_host_checks():
    w = wl.cfg3(2, tokens=128)  # 14 KiB rows, few items per CTA
    K, rows, src, key = wl.dispatch_items(w)
    outs, so, pos, S = oracle.default().dispatch_exchange(K, rows, src, key, w.row_bytes)
    expect = [r.reshape(-1, w.row_bytes)[s].reshape(-1) for r, s in zip(rows, src)]
    assert _combine_checked(K, outs, S, key, pos, w.row_bytes, expect=expect) == a2av.OK
    with a2av.A2av(2) as eng:
        rc = a2av.a2av_combine_items(eng.handle, 1, [0, 0], 0, [0, 0], [0, 0], [0, 0], [0, 0], 8,
                                     0, 0)
        assert rc == a2av.ERR_INVALID_ARG
        ws = torch.empty(64, dtype=torch.uint8, device="cuda")
        S2 = torch.zeros((2, 2), dtype=torch.int64, device="cuda")
        rc = a2av.a2av_combine_items(eng.handle, 1, [0, 0], S2.data_ptr(), [0, 0], [0, 0], [0, 0],
                                     [0, 0], 8, ws.data_ptr(), ws.numel())
        assert rc == a2av.ERR_INVALID_ARG  # workspace too small


# The combine's copy by row size (many items: the check kernel, then the
# cp.async.bulk gather: lanes issuing their own rows up to 2 KiB, one-row
# rings above) and its one-kernel path (at most 4096 items: row slots for
# aligned rows, registers otherwise).
@pytest.mark.parametrize("rb,m", [(64, 20011), (512, 9001), (1024, 6007), (2048, 6007),
                                  (4096, 3001), (14336, 1801), (32768, 1801)])
def test_aligned_copy_shapes(rb, m):
    """(more than 4096 items in all: past the one-kernel path)"""
    rng = np.random.default_rng(rb + m + 1)
    W, K = 4, 3
    counts = [m, m - 17, m // 3, 1]
    key = [rng.integers(0, W * K, c).astype(np.int32) for c in counts]
    rows = [rng.integers(0, 256, 50 * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, 50, c).astype(np.int32) for c in counts]
    outs, so, pos, S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    peers = [rng.integers(0, 256, b.size, dtype=np.uint8) for b in outs]
    assert _combine_checked(K, peers, S, key, pos, rb,
                            expect_copy=aligned_copy_kernel(rb, combine=True)) == a2av.OK


@pytest.mark.parametrize("rb", [1, 8, 16, 64, 1024, 14336, 40000])
@pytest.mark.parametrize("aligned", [True, False])
def test_one_kernel_path(rb, aligned):
    rng = np.random.default_rng(rb * 5 + aligned)
    for W, K, total in ((8, 8, 2048), (3, 5, 40), (32, 2, 4096), (1, 1, 900)):
        if rb * total > (64 << 20):
            total = (64 << 20) // rb
        share = rng.dirichlet(np.ones(W)) * total
        m = [int(x) for x in share]
        m[0] += total - sum(m)
        rows = [rng.integers(0, 256, 30 * rb, dtype=np.uint8) for _ in range(W)]
        src = [rng.integers(0, 30, m[r]).astype(np.int32) for r in range(W)]
        key = [rng.integers(0, W * K, m[r]).astype(np.int32) for r in range(W)]
        outs, so, pos, S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
        peers = [rng.integers(0, 256, b.size, dtype=np.uint8) for b in outs]
        mis = None if aligned else [int(rng.integers(1, 16)) for _ in range(2 * W)]
        assert _combine_checked(K, peers, S, key, pos, rb, mis,
                                expect_copy="combine_tiny_kernel") == a2av.OK


# The one-launch combine of rows under 64 bytes (check, grid barrier, copy):
# rows of 4, 8 and 16 bytes loaded all at once when aligned, other sizes and
# misaligned buffers one row at a time; ragged ranks and an empty one, 32
# ranks, and the embedding size.
@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("rb", [1, 4, 8, 13, 16, 24, 48])
@pytest.mark.parametrize("W,K,counts", [
    (4, 3, [5000, 17, 1, 0]),
    (32, 2, [300 + 11 * r for r in range(32)]),
    (2, 13, [640_000, 638_590]),
])
def test_order_kernel_path(W, K, counts, rb, aligned):
    rng = np.random.default_rng(rb * 3 + W + aligned)
    key = [np.minimum(rng.geometric(0.08, c) - 1, W * K - 1).astype(np.int32) for c in counts]
    rows = [rng.integers(0, 256, 40 * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, 40, c).astype(np.int32) for c in counts]
    outs, so, pos, S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    peers = [rng.integers(0, 256, b.size, dtype=np.uint8) for b in outs]
    mis = None if aligned else [int(rng.integers(1, 16)) for _ in range(2 * W)]
    assert _combine_checked(K, peers, S, key, pos, rb, mis,
                            expect_copy="combine_order_kernel") == a2av.OK


@pytest.mark.parametrize("order", ["0", "2"])
@pytest.mark.parametrize("rb", [8, 13, 64, 1024, 14336])
@pytest.mark.parametrize("case", ["key", "pos_outside_group", "pos_too_large", "negative_split"])
def test_large_errors_write_nothing(case, rb, order, monkeypatch):
    """The combine's checks past the one-kernel size (3000 items a rank): with
    order "2", rows under 64 bytes by the one-launch combine, aligned rows of
    64 B .. 2 KiB by the gather that checks before it copies (a grid barrier
    between) and longer ones by the check kernel; with order "0", all by the
    check kernel.  Nothing is written."""
    monkeypatch.setenv("A2AV_DISPATCH_ORDER", order)
    rng = np.random.default_rng(rb + len(case))
    W, K, m = 2, 3, 3000
    key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
    rows = [rng.integers(0, 256, 40 * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, 40, m).astype(np.int32) for _ in range(W)]
    outs, so, pos, S = oracle.default().dispatch_exchange(K, rows, src, key, rb)
    peers = [rng.integers(0, 256, b.size, dtype=np.uint8) for b in outs]
    pos = [p.copy() for p in pos]
    S = S.copy()
    want = a2av.ERR_BAD_INDEX
    if case == "key":
        key[1][2999] = W * K
    elif case == "pos_outside_group":
        i = 1234
        p = key[0][i] // K
        lo = int(S[0, :p].sum())
        pos[0][i] = lo + int(S[0, p]) if p + 1 < W else lo - 1
    elif case == "pos_too_large":
        pos[1][17] = m
    elif case == "negative_split":
        S[1, 0] = -1
        want = a2av.ERR_BAD_SPLITS
    assert _combine_checked(K, peers, S, key, pos, rb) == want
