"""a2av_run_multi: several independent exchanges in one launch, each checked
byte for byte against the oracle's exchange of the same inputs (the result
must equal that of one a2av_run per exchange), with sentinel rows past every
output's received rows left untouched."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")

SENTINEL = 0xEE
SLACK = 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()


def _device(w):
    W, S, rb = w.W, w.splits, w.row_bytes
    d_in = [torch.from_numpy(b).cuda() for b in w.inputs]
    d_out = [torch.full(((int(S[:, p].sum()) + SLACK) * rb,), SENTINEL, dtype=torch.uint8,
                        device="cuda") for p in range(W)]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    return d_in, torch.from_numpy(np.ascontiguousarray(S)).cuda(), d_out, so


def _check(w, dev, valid=True):
    d_in, _, d_out, so = dev
    if not valid:
        assert np.all(so.cpu().numpy() == -7)
        assert all(bool((t == SENTINEL).all()) for t in d_out)
        return
    ref, ref_so = oracle.default().exchange(w.inputs, w.splits, w.row_bytes)
    assert np.array_equal(so.cpu().numpy(), ref_so)
    for p in range(w.W):
        got = d_out[p].cpu().numpy()
        assert np.array_equal(got[: ref[p].size], ref[p]), p
        assert np.all(got[ref[p].size:] == SENTINEL), p
    for r in range(w.W):  # inputs untouched
        assert np.array_equal(d_in[r].cpu().numpy(), w.inputs[r])


def _run_multi(ws, path=a2av.PATH_AUTO, devs=None):
    devs = devs or [_device(w) for w in ws]
    eng = a2av.A2av(ws[0].W, path=path)
    eng.run_multi([(*d, w.row_bytes) for d, w in zip(devs, ws)])
    st = eng.status()
    launch = eng.last_launch()
    eng.close()
    return devs, st, launch


def _scales(w, nbytes, seed):
    """Per-row side data with the same splits (e.g. MoE token scales)."""
    rng = np.random.default_rng(seed)
    ins = [rng.integers(0, 256, int(w.splits[r].sum()) * nbytes, dtype=np.uint8)
           for r in range(w.W)]
    return wl.Workload("scales", w.W, nbytes, w.splits, ins, {})


def test_keyed_jagged_lengths_and_keys_in_one_launch():
    w = wl.cfg5(1, batch=2048)
    ws = [wl.cfg5_lengths(w), w]
    devs, st, launch = _run_multi(ws)
    assert st == a2av.OK and launch["path"] == a2av.PATH_STAGED
    for x, d in zip(ws, devs):
        _check(x, d)


def test_moe_tokens_and_scales_in_one_launch():
    w = wl.cfg3(2, tokens=1024, hidden=512)
    ws = [w, _scales(w, 32, 5)]
    devs, st, launch = _run_multi(ws)
    assert st == a2av.OK and launch["path"] == a2av.PATH_BULK
    for x, d in zip(ws, devs):
        _check(x, d)


@pytest.mark.parametrize("path", [a2av.PATH_AUTO, a2av.PATH_STAGED, a2av.PATH_VECTOR])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_four_mixed_exchanges(path, seed):
    modes = ["uniform", "skew", "sparse", "empty", "one", "diag"]
    rbs = [1, 13, 16, 1024, 7, 48]
    ws = [wl.random_case(100 * seed + k, 5, rbs[(seed + k) % 6], max_rows=300,
                         mode=modes[(seed + 2 * k) % 6]) for k in range(4)]
    devs, st, launch = _run_multi(ws, path)
    assert st == a2av.OK
    if path != a2av.PATH_AUTO:
        assert launch["path"] == path
    for x, d in zip(ws, devs):
        _check(x, d)


@pytest.mark.parametrize("W", [1, 32])
def test_extreme_world_sizes(W):
    ws = [wl.random_case(70 + W, W, rb, max_rows=40, mode=mode)
          for rb, mode in ((24, "uniform"), (5, "sparse"), (64, "skew"))]
    devs, st, _ = _run_multi(ws)
    assert st == a2av.OK
    for x, d in zip(ws, devs):
        _check(x, d)


def test_lopsided_sizes_each_get_a_cta():
    big = wl.cfg2(1 << 24, seed=3)  # 16 MiB per rank
    tiny = wl.random_case(9, 4, 16, mode="one")
    devs, st, _ = _run_multi([big, tiny, tiny])
    assert st == a2av.OK
    for x, d in zip([big, tiny, tiny], devs):
        _check(x, d)


def test_one_exchange_equals_run():
    w = wl.cfg4(4, rows=1 << 14)
    devs, st, _ = _run_multi([w])
    assert st == a2av.OK
    _check(w, devs[0])


def test_invalid_exchange_writes_nothing_of_its_own():
    good = wl.random_case(11, 4, 13, max_rows=200)
    bad = wl.random_case(12, 4, 16, max_rows=200)
    dev_bad = _device(bad)
    dev_bad[1][1, 2] = -1  # a negative split
    devs, st, _ = _run_multi([good, bad], devs=[_device(good), dev_bad])
    assert st == a2av.ERR_BAD_SPLITS
    _check(good, devs[0])
    _check(bad, devs[1], valid=False)


def test_host_rejections():
    w = wl.random_case(1, 2, 8)
    eng = a2av.A2av(2)
    d = _device(w)
    with pytest.raises(ValueError):
        eng.run_multi([])
    with pytest.raises(ValueError):
        eng.run_multi([(*d, 8)] * (a2av.MAX_EXCHANGES + 1))
    assert a2av.a2av_run_multi(eng.handle, []) == a2av.ERR_INVALID_ARG
    ptrs = [t.data_ptr() for t in d[0]], d[1].data_ptr(), [t.data_ptr() for t in d[2]]
    five = [(ptrs[0], ptrs[1], ptrs[2], d[3].data_ptr(), 8)] * 5
    assert a2av.a2av_run_multi(eng.handle, five) == a2av.ERR_UNSUPPORTED
    zero_rb = [(ptrs[0], ptrs[1], ptrs[2], d[3].data_ptr(), 0)]
    assert a2av.a2av_run_multi(eng.handle, zero_rb) == a2av.ERR_INVALID_ARG
    eng.close()


def test_pinned_host_buffers_zero_copy():
    """Pinned host inputs and outputs: the binding selects the vector engine,
    which reaches host memory with plain loads and stores."""
    ws = [wl.random_case(90, 3, 24, max_rows=100), wl.random_case(91, 3, 7, max_rows=100)]
    bufs = []
    for w in ws:
        ins = [torch.from_numpy(b).pin_memory() for b in w.inputs]
        outs = [torch.full(((int(w.splits[:, p].sum()) + SLACK) * w.row_bytes,), SENTINEL,
                           dtype=torch.uint8).pin_memory() for p in range(w.W)]
        so = torch.full((w.W, 2, w.W), -7, dtype=torch.int64, device="cuda")
        bufs.append((ins, torch.from_numpy(w.splits).cuda(), outs, so))
    eng = a2av.A2av(3)
    eng.run_multi([(*b, w.row_bytes) for b, w in zip(bufs, ws)])
    assert eng.status() == a2av.OK
    assert eng.last_launch()["path"] == a2av.PATH_VECTOR
    eng.close()
    for w, (ins, _, outs, so) in zip(ws, bufs):
        ref, ref_so = oracle.default().exchange(w.inputs, w.splits, w.row_bytes)
        assert np.array_equal(so.cpu().numpy(), ref_so)
        for p in range(w.W):
            got = outs[p].numpy()
            assert np.array_equal(got[: ref[p].size], ref[p])
            assert np.all(got[ref[p].size:] == SENTINEL)
