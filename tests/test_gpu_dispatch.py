"""GPU parity of the fused dispatch (a2av_dispatch) against the CPU oracle:
grouping unsorted items by key on the device, gathering their rows into the
exchange's outputs, positions and split matrix -- byte for byte."""
import numpy as np
import pytest
import torch

import workloads as wl
from tests._gpu import aligned_copy_kernel, dispatch_checked

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()
    a2av.load()


@pytest.mark.parametrize("tokens", [128, 1024, 8192])
def test_moe_top2_dispatch(tokens):
    w = wl.cfg3(0, tokens=tokens)
    K, rows, src, key = wl.dispatch_items(w)
    ref, *_ = dispatch_checked(K, rows, src, key, w.row_bytes)
    for p in range(w.W):  # and it equals the exchange of the pre-grouped rows
        assert ref[p].size == int(w.splits[:, p].sum()) * w.row_bytes


@pytest.mark.parametrize("hidden", [256, 512, 768, 1024])
@pytest.mark.parametrize("tokens", [2048, 8192])
def test_moe_top2_short_rows(tokens, hidden):
    """512 B .. 2 KiB MoE rows (the register copy of 512-byte pieces, the
    gather's multi-row stages): a token's two items are consecutive, so the
    token's row is loaded once and stored to both destinations."""
    w = wl.cfg3(1, tokens=tokens, hidden=hidden)
    K, rows, src, key = wl.dispatch_items(w)
    dispatch_checked(K, rows, src, key, w.row_bytes, expect_copy=aligned_copy_kernel(w.row_bytes))


@pytest.mark.parametrize("rb", [512, 1024, 1536, 2048])
def test_runs_of_one_source_row(rb):
    """Items that share a source row in runs of 1 to 8 (top-k routing of up
    to eight experts, ragged at batch edges), keys in any order: every
    destination of a run gets the row."""
    rng = np.random.default_rng(rb)
    W, K, n = 4, 5, 300
    rows, src, key = [], [], []
    for r in range(W):
        rows.append(rng.integers(0, 256, n * rb, dtype=np.uint8))
        runs = rng.integers(1, 9, 1500)
        s = np.repeat(rng.integers(0, n, runs.size), runs)[: 6000 - 37 * r]
        src.append(s.astype(np.int32))
        key.append(rng.integers(0, W * K, s.size).astype(np.int32))
    dispatch_checked(K, rows, src, key, rb, expect_copy=aligned_copy_kernel(rb))


def test_moe_dedup_dispatch():
    w = wl.cfg3(3, tokens=2048, hidden=512, dedup=True)
    K, rows, src, key = wl.dispatch_items(w)
    assert K == 1
    ref, *_ = dispatch_checked(K, rows, src, key, w.row_bytes)
    for p in range(w.W):
        assert ref[p].size == int(w.splits[:, p].sum()) * w.row_bytes


def test_embedding_key_dispatch():
    w = wl.cfg5(0)
    K, rows, src, key = wl.dispatch_items(w)
    dispatch_checked(K, rows, src, key, w.row_bytes)


@pytest.mark.parametrize("rb", [1, 3, 8, 13, 64, 100, 256, 1040])
def test_random_dispatch(rb):
    rng = np.random.default_rng(rb)
    for W, K in ((1, 1), (2, 5), (3, 32), (8, 8), (32, 32), (5, 200)):
        n = [int(rng.integers(0, 300)) for _ in range(W)]
        m = [int(rng.integers(0, 3000)) if n[r] else 0 for r in range(W)]
        rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
        src = [rng.integers(0, max(n[r], 1), m[r]).astype(np.int32) for r in range(W)]
        if rng.random() < 0.5:  # skewed keys: most items on a few keys
            key = [np.minimum(rng.geometric(0.2, m[r]) - 1, W * K - 1).astype(np.int32)
                   for r in range(W)]
        else:
            key = [rng.integers(0, W * K, m[r]).astype(np.int32) for r in range(W)]
        mis = [int(rng.integers(0, 16)) for _ in range(W)]
        dispatch_checked(K, rows, src, key, rb, rows_mis=mis, out_mis=mis[::-1])


@pytest.mark.parametrize("rb", [64, 80, 256, 1040, 4096, 8176, 8192, 65536 + 16])
def test_aligned_row_sizes(rb):
    """16-byte aligned buffers and rows across the warp copy's flat vector runs
    (64 B .. 64 KiB), the switch to the cp.async.bulk gather (8 KiB .. 32 KiB)
    and rows too long for either (span copy); item counts leave ragged tails of
    32-item batches."""
    rng = np.random.default_rng(rb)
    W, K = 4, 3
    n = [int(rng.integers(1, 40)) for _ in range(W)]
    m = [int(rng.integers(0, 300)) for _ in range(W)]
    rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
    src = [rng.integers(0, n[r], m[r]).astype(np.int32) for r in range(W)]
    key = [rng.integers(0, W * K, m[r]).astype(np.int32) for r in range(W)]
    dispatch_checked(K, rows, src, key, rb)


@pytest.mark.parametrize("order", ["0", "2"])
@pytest.mark.parametrize("rb", [2048, 9216, 20480])
def test_few_items_past_the_one_kernel_size(rb, order, monkeypatch):
    """More keys than the one-kernel-per-rank count takes (W*K > 256) and
    more items than the one-kernel path takes, but only a few thousand:
    without the order kernel, the count kernel, the scan kernel (400 keys:
    more than one block thread a key), then the gather in batches of 8
    items; with it, the order kernel, then the gather."""
    monkeypatch.setenv("A2AV_DISPATCH_ORDER", order)
    rng = np.random.default_rng(rb + 5)
    W, K, n, m = 2, 200, 64, 3000
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, n, m).astype(np.int32) for _ in range(W)]
    key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
    dispatch_checked(K, rows, src, key, rb, expect_copy=aligned_copy_kernel(rb),
                     expect_kernels=3 if order == "0" else 2)


def test_dispatch_without_items():
    rows = [np.arange(64, dtype=np.uint8)] * 3
    empty = [np.zeros(0, np.int32)] * 3
    dispatch_checked(2, rows, empty, empty, 16)


@pytest.mark.parametrize("W,K", [(2, 100), (4, 100)])
def test_dispatch_without_items_many_keys(W, K):
    """Past the one-kernel key count (W*K > 256) an empty batch still goes
    through the counting kernels: 200 keys with the count kernel's own scan,
    400 with the scan kernel; both write zero splits and offsets."""
    rows = [np.arange(64, dtype=np.uint8)] * W
    empty = [np.zeros(0, np.int32)] * W
    dispatch_checked(K, rows, empty, empty, 16)


@pytest.mark.parametrize("rb", [16, 64])
@pytest.mark.parametrize("W,K,m,kernels", [
    (2, 128, 65536, 2),   # 32 groups of 2048 items over 256 keys: the count kernel scans
    (2, 128, 65537, 3),   # 33 groups: the scan kernel
    (8, 32, 65536, 2),    # the same limit with eight ranks
    (8, 32, 65537, 3),
])
def test_group_scan_either_side_of_the_fused_limit(W, K, m, kernels, rb, monkeypatch):
    """The count kernel's last block per rank scans the group counts when a
    thread's share of one key is at most 32 groups (256 keys: one thread a
    key); one group more and the scan kernel runs (the order kernel off)."""
    monkeypatch.setenv("A2AV_DISPATCH_ORDER", "0")
    rng = np.random.default_rng(m + rb)
    n = 500
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    counts = [m] + [int(rng.integers(2049, m + 1)) for _ in range(W - 2)] + [0]
    src = [rng.integers(0, n, c).astype(np.int32) for c in counts]
    key = [np.minimum(rng.geometric(0.05, c) - 1, W * K - 1).astype(np.int32) for c in counts]
    dispatch_checked(K, rows, src, key, rb, expect_kernels=kernels,
                     expect_copy="dispatch_place_copy_kernel" if rb < 64 else
                     aligned_copy_kernel(rb))


@pytest.mark.parametrize("rb", [8, 64])
@pytest.mark.parametrize("W,K,m,kernels", [(2, 13, 589_824, 2), (2, 13, 640_000, 3),
                                           (2, 200, 640_000, 3)])
def test_embedding_size_batches(W, K, m, kernels, rb, monkeypatch):
    """Batches of the embedding-key size (640 K items a rank), the order
    kernel off: the count kernel's last block scans up to 288 groups of 2048
    items over 26 keys (9 block threads a key, 32 groups each); past that, or
    with 400 keys (more than one block thread a key), the scan kernel runs."""
    monkeypatch.setenv("A2AV_DISPATCH_ORDER", "0")
    rng = np.random.default_rng(K + rb + m)
    n = 4000
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, n, m - 1000 * r).astype(np.int32) for r in range(W)]
    key = [rng.integers(0, W * K, m - 1000 * r).astype(np.int32) for r in range(W)]
    dispatch_checked(K, rows, src, key, rb, expect_kernels=kernels,
                     expect_copy="dispatch_place_copy_kernel" if rb < 64 else
                     aligned_copy_kernel(rb))


# The one-launch order kernel (all items in the grid's registers): rows under
# 64 bytes copied by it (4, 8 and 16-byte rows loaded all at once when
# aligned, other sizes and misaligned buffers one row at a time), longer rows
# by the copy kernel that follows; ragged ranks, an empty rank, 32 ranks, the
# largest key count, and the embedding and MoE sizes.
ORDER_CASES = [
    ("ragged", 4, 3, [5000, 17, 1, 0]),
    ("moe", 8, 32, [16384] * 8),
    ("ranks32", 32, 2, [2100 + 7 * r for r in range(32)]),
    ("keys1024", 2, 512, [8000, 7000]),
    ("embedding", 2, 13, [640_000, 638_590]),
]


@pytest.mark.parametrize("mis", [False, True])
@pytest.mark.parametrize("rb", [1, 4, 8, 13, 16, 24, 64, 1024, 2048, 14336])
@pytest.mark.parametrize("case", [c[0] for c in ORDER_CASES])
def test_order_kernel_path(case, rb, mis, monkeypatch):
    monkeypatch.setenv("A2AV_DISPATCH_ORDER", "2")  # (every row size)
    _, W, K, counts = next(c for c in ORDER_CASES if c[0] == case)
    total = sum(counts)
    if total * rb > (256 << 20):
        pytest.skip("more than 256 MiB of rows")
    rng = np.random.default_rng(rb * 7 + W + mis)
    n = [int(rng.integers(1, 3000)) for _ in range(W)]
    rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
    src = [rng.integers(0, n[r], counts[r]).astype(np.int32) for r in range(W)]
    key = [np.minimum(rng.geometric(0.08, counts[r]) - 1, W * K - 1).astype(np.int32)
           for r in range(W)]
    mis_r = [int(rng.integers(1, 16)) for _ in range(W)] if mis else None
    if rb < 64:
        copy, kernels = "dispatch_order_kernel", 1
    else:
        copy, kernels = aligned_copy_kernel(rb) if not mis else "dispatch_copy_kernel", 2
    dispatch_checked(K, rows, src, key, rb, rows_mis=mis_r, out_mis=mis_r[::-1] if mis else None,
                     expect_copy=copy, expect_kernels=kernels)


@pytest.mark.parametrize("W,K,counts", [
    (2, 13, [1_300_000, 1_300_000]),   # more items than the grid's registers hold
    (2, 512, [40_000, 40_000]),        # 1024 keys over ~80 CTAs a rank: too many counts
])
def test_order_kernel_falls_back(W, K, counts):
    """Batches the order kernel does not take go through the count chain."""
    rng = np.random.default_rng(W * K)
    rb, n = 8, 1000
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, n, c).astype(np.int32) for c in counts]
    key = [rng.integers(0, W * K, c).astype(np.int32) for c in counts]
    dispatch_checked(K, rows, src, key, rb, expect_copy="dispatch_place_copy_kernel")


# Aligned rows by the copy kernels' shapes (the register warp copy up to 2
# KiB, in flat runs or by 512-byte pieces; the gather's one-row rings, items
# in strided order, above 2 KiB), with ragged last batches per rank.
@pytest.mark.parametrize("rb,m", [(64, 20011), (256, 20011), (272, 9001), (512, 9001),
                                  (1024, 6007), (1536, 6007), (2048, 6007), (3072, 3001),
                                  (4096, 3001), (4112, 3001), (8192, 1801), (14336, 1801),
                                  (16384, 1801), (32768, 1801)])
def test_aligned_copy_shapes(rb, m):
    """(more than 4096 items in all: past the one-kernel path)"""
    rng = np.random.default_rng(rb + m)
    W, K, n = 4, 3, 97
    rows = [rng.integers(0, 256, n * rb, dtype=np.uint8) for _ in range(W)]
    counts = [m, m - 17, m // 3, 1]
    src = [rng.integers(0, n, c).astype(np.int32) for c in counts]
    key = [rng.integers(0, W * K, c).astype(np.int32) for c in counts]
    dispatch_checked(K, rows, src, key, rb, expect_copy=aligned_copy_kernel(rb))


# The one-kernel path (at most 4096 items over all ranks): row slots through
# cp.async.bulk for aligned rows of 64 B .. 176 KiB, register copies for the
# rest (misaligned buffers, short rows, rows too long for the slots); one
# item per block when there are fewer items than SMs; 4096 items exactly,
# and 4097 (past it).
@pytest.mark.parametrize("rb", [1, 8, 13, 16, 64, 80, 1024, 14336, 40000, 200000])
@pytest.mark.parametrize("mis", [False, True])
def test_one_kernel_path(rb, mis):
    rng = np.random.default_rng(rb * 3 + mis)
    for W, K, total in ((8, 8, 2048), (3, 5, 50), (32, 2, 4096), (1, 1, 700), (5, 40, 1500)):
        if rb * total > (64 << 20):
            total = (64 << 20) // rb
        share = rng.dirichlet(np.ones(W)) * total
        m = [int(x) for x in share]
        m[0] += total - sum(m)
        n = [int(rng.integers(1, 60)) for _ in range(W)]
        rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
        src = [rng.integers(0, n[r], m[r]).astype(np.int32) for r in range(W)]
        key = [np.minimum(rng.geometric(0.1, m[r]) - 1, W * K - 1).astype(np.int32)
               for r in range(W)]
        mis_r = [int(rng.integers(1, 16)) for _ in range(W)] if mis else None
        dispatch_checked(K, rows, src, key, rb, rows_mis=mis_r,
                         out_mis=mis_r[::-1] if mis else None,
                         expect_copy="dispatch_tiny_kernel", expect_kernels=1)
    # one past the one-kernel size
    W, K = 2, 3
    rows = [rng.integers(0, 256, 40 * rb, dtype=np.uint8) for _ in range(W)]
    src = [rng.integers(0, 40, c).astype(np.int32) for c in (2049, 2048)]
    key = [rng.integers(0, W * K, c).astype(np.int32) for c in (2049, 2048)]
    with a2av.A2av(W) as eng:
        dispatch_checked(K, rows, src, key, rb, engine=eng)
        assert eng.last_dispatch()["copy_kernel"] != "dispatch_tiny_kernel"


def test_dispatch_then_combine_restores_key_order():
    w = wl.cfg3(7, tokens=512, hidden=256)
    K, rows, src, key = wl.dispatch_items(w)
    W, rb = w.W, w.row_bytes
    eng = a2av.A2av(W)
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    d_src = [torch.from_numpy(s).cuda() for s in src]
    d_key = [torch.from_numpy(k).cuda() for k in key]
    d_pos = [torch.empty(k.size, dtype=torch.int64, device="cuda") for k in key]
    out = [torch.empty(int(w.splits[:, p].sum()) * rb, dtype=torch.uint8, device="cuda")
           for p in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    back = [torch.empty(k.size * rb, dtype=torch.uint8, device="cuda") for k in key]
    cso = torch.empty_like(so)
    eng.dispatch(d_rows, d_src, d_key, K, out, so, d_pos, rb)
    eng.combine(out, so, back, cso, rb)
    assert eng.status() == a2av.OK
    eng.close()
    for r in range(W):
        # item i's row comes back at its sorted position
        got = back[r].view(-1, rb)[d_pos[r]].cpu().numpy()
        want = rows[r].reshape(-1, rb)[src[r]]
        assert np.array_equal(got, want)


@pytest.mark.parametrize("case", ["key", "negative_key", "src", "capacity", "null_out"])
def test_dispatch_errors_write_nothing(case):
    W, K, rb = 2, 2, 4
    rows = [torch.arange(12, dtype=torch.uint8, device="cuda"),
            torch.arange(8, dtype=torch.uint8, device="cuda")]
    src = [torch.tensor([0, 2, 1], dtype=torch.int32, device="cuda"),
           torch.tensor([1, 0], dtype=torch.int32, device="cuda")]
    key = [torch.tensor([0, 3, 1], dtype=torch.int32, device="cuda"),
           torch.tensor([2, 2], dtype=torch.int32, device="cuda")]
    cap = 0
    outs = [torch.full((16,), 0xEE, dtype=torch.uint8, device="cuda") for _ in range(W)]
    if case == "key":
        key[1][1] = 4
    elif case == "negative_key":
        key[0][1] = -1
    elif case == "src":
        src[1][0] = 2
    elif case == "capacity":
        cap = 2
    elif case == "null_out":
        outs[1] = torch.empty(0, dtype=torch.uint8, device="cuda")
    pos = [torch.full((3,), -1, dtype=torch.int64, device="cuda"),
           torch.full((2,), -1, dtype=torch.int64, device="cuda")]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    isp = torch.full((W, W), -7, dtype=torch.int64, device="cuda")
    eng = a2av.A2av(W, 0, cap)
    eng.dispatch(rows, src, key, K, outs, so, pos, rb, in_splits=isp)
    st = eng.status()
    eng.close()
    want = a2av.ERR_BAD_INDEX if case in ("key", "negative_key", "src") else a2av.ERR_BAD_SPLITS
    assert st == want
    torch.cuda.synchronize()
    assert all(bool((o == 0xEE).all()) for o in outs if o.numel())
    assert bool((so == -7).all()) and bool((isp == -7).all())
    assert all(bool((p == -1).all()) for p in pos)


@pytest.mark.parametrize("order", ["0", "2"])
@pytest.mark.parametrize("rb", [4, 64, 1024, 2048])
@pytest.mark.parametrize("case", ["key", "src", "capacity", "null_out"])
def test_large_dispatch_errors_write_nothing(case, rb, order, monkeypatch):
    """The same checks past the one-kernel size (3000 items per rank), by the
    order kernel (order "2": it copies rows under 64 bytes itself) and by the
    count chain (order "0": short rows by the place-and-copy kernel); longer
    rows by the warp copy kernel or the cp.async.bulk gather."""
    monkeypatch.setenv("A2AV_DISPATCH_ORDER", order)
    W, K, m, n = 2, 3, 3000, 500
    rng = np.random.default_rng(rb)
    rows = [torch.from_numpy(rng.integers(0, 256, n * rb, dtype=np.uint8)).cuda()
            for _ in range(W)]
    src = [torch.from_numpy(rng.integers(0, n, m).astype(np.int32)).cuda() for _ in range(W)]
    key = [torch.from_numpy(rng.integers(0, W * K, m).astype(np.int32)).cuda() for _ in range(W)]
    cap = 0
    outs = [torch.full((W * m * rb,), 0xEE, dtype=torch.uint8, device="cuda") for _ in range(W)]
    if case == "key":
        key[1][2999] = W * K
    elif case == "src":
        src[0][1234] = n
    elif case == "capacity":
        cap = m // 2
    elif case == "null_out":
        outs[1] = torch.empty(0, dtype=torch.uint8, device="cuda")
    pos = [torch.full((m,), -1, dtype=torch.int64, device="cuda") for _ in range(W)]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    isp = torch.full((W, W), -7, dtype=torch.int64, device="cuda")
    eng = a2av.A2av(W, 0, cap)
    eng.dispatch(rows, src, key, K, outs, so, pos, rb, in_splits=isp)
    st = eng.status()
    eng.close()
    want = a2av.ERR_BAD_INDEX if case in ("key", "src") else a2av.ERR_BAD_SPLITS
    assert st == want
    torch.cuda.synchronize()
    assert all(bool((o == 0xEE).all()) for o in outs if o.numel())
    assert bool((so == -7).all()) and bool((isp == -7).all())
    assert all(bool((p == -1).all()) for p in pos)


def test_dispatch_host_rejections():
    rc, h = a2av.a2av_create(4)
    assert rc == a2av.OK
    z = [0] * 4
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    so = torch.empty((4, 2, 4), dtype=torch.int64, device="cuda")
    args = dict(rows_ptrs=z, rows_per_rank=z, src_row_ptrs=z, key_ptrs=z, items_per_rank=z,
                out_ptrs=z, out_splits_offsets_dev=so.data_ptr(), sorted_pos_ptrs=z,
                in_splits_dev=0, row_bytes=8, workspace=ws.data_ptr(), workspace_bytes=ws.numel())
    assert a2av.a2av_dispatch(h, 2, **args) == a2av.OK  # nothing to do is fine
    assert a2av.a2av_dispatch(h, 0, **args) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_dispatch(h, 257, **args) == a2av.ERR_UNSUPPORTED  # 4 x 257 keys
    assert a2av.a2av_dispatch(h, 2, **{**args, "workspace_bytes": 64}) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_dispatch(h, 2, **{**args, "workspace": ws.data_ptr() + 8}) \
        == a2av.ERR_INVALID_ARG
    assert a2av.a2av_dispatch(h, 2, **{**args, "items_per_rank": [-1, 0, 0, 0]}) \
        == a2av.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert a2av.a2av_status(h)[1] == a2av.OK
    a2av.a2av_destroy(h)
    assert a2av.a2av_dispatch_workspace_bytes(4, 257, 10) == -1
    assert a2av.a2av_dispatch_workspace_bytes(4, 8, 1000) > 0


@pytest.mark.parametrize("rb", [8, 16, 1040])
def test_small_dispatch_path(rb):
    # every rank at most 2048 items and at most 256 keys: the fused
    # count/scan/rank kernel; W=32 with 8 keys per peer is its widest case
    rng = np.random.default_rng(100 + rb)
    for W, K in ((32, 8), (8, 32), (4, 1), (1, 256)):
        n = [int(rng.integers(1, 200)) for _ in range(W)]
        m = [int(rng.integers(0, 2049)) for _ in range(W)]
        m[0] = 2048
        rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
        src = [rng.integers(0, n[r], m[r]).astype(np.int32) for r in range(W)]
        key = [np.minimum(rng.geometric(0.05, m[r]) - 1, W * K - 1).astype(np.int32)
               for r in range(W)]
        dispatch_checked(K, rows, src, key, rb)


@pytest.mark.parametrize("rb", [20480, 40000, 16384 + 16])
def test_dispatch_large_rows(rb):
    # 16..32 KiB rows use the gather's 4 x 32 KiB ring; 40000 B rows (over
    # 32 KiB) the warp path; 16400 B the large ring's lower edge
    rng = np.random.default_rng(rb)
    W, K = 4, 3
    n = [int(rng.integers(1, 40)) for _ in range(W)]
    m = [int(rng.integers(0, 120)) for _ in range(W)]
    rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
    src = [rng.integers(0, n[r], m[r]).astype(np.int32) for r in range(W)]
    key = [rng.integers(0, W * K, m[r]).astype(np.int32) for r in range(W)]
    dispatch_checked(K, rows, src, key, rb)
