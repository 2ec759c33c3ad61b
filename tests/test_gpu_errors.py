"""Error behaviour on the GPU: invalid splits write nothing and set the status.

Every case here is an input the kernel itself checks before it touches any
buffer (the split matrix is validated in every CTA before the first copy), or
an argument the host rejects before launching; none can fault the GPU.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()


def _setup(S, rb, out_rows=None):
    W = S.shape[0]
    ins = [torch.full((max(int(S[r].clip(min=0).sum()), 1) * rb,), r + 1, dtype=torch.uint8,
                      device="cuda") for r in range(W)]
    out_rows = out_rows or [max(int(S[:, p].clip(min=0).sum()), 1) for p in range(W)]
    outs = [torch.full((n * rb,), 0xEE, dtype=torch.uint8, device="cuda") for n in out_rows]
    so = torch.full((W, 2, W), -7, dtype=torch.int64, device="cuda")
    return ins, outs, so


def _untouched(outs, so):
    torch.cuda.synchronize()
    return all(bool((o == 0xEE).all()) for o in outs) and bool((so == -7).all())


S0 = np.array([[1, 2, 0], [0, 1, 1], [2, 0, 3]], dtype=np.int64)


@pytest.mark.parametrize("path", [a2av.PATH_AUTO, a2av.PATH_VECTOR, a2av.PATH_STAGED])
@pytest.mark.parametrize("case", ["negative", "in_cap", "out_cap", "limit", "null_in", "null_out"])
def test_bad_splits_write_nothing(case, path):
    rb = 16
    S = S0.copy()
    in_cap = out_cap = 0
    if case == "negative":
        S[1, 2] = -1
    elif case == "in_cap":
        in_cap = int(S.sum(axis=1).max()) - 1
    elif case == "out_cap":
        out_cap = int(S.sum(axis=0).max()) - 1
    elif case == "limit":
        S[0, 1] = (1 << 62) // (3 * rb) + 1
    ins, outs, so = _setup(np.minimum(S, 10), rb)
    if case == "null_in":
        ins[1] = None
    if case == "null_out":
        outs[2] = torch.empty(0, dtype=torch.uint8, device="cuda")
    eng = a2av.A2av(3, in_cap, out_cap, path=path)
    eng.run(ins, torch.from_numpy(S).cuda(), outs, so, rb)
    assert eng.status() == a2av.ERR_BAD_SPLITS
    assert eng.status() == a2av.OK, "reading the status clears it"
    eng.close()
    assert _untouched([o for o in outs if o.numel()], so)


def test_capacity_exactly_met_is_valid():
    rb = 8
    eng = a2av.A2av(3, int(S0.sum(axis=1).max()), int(S0.sum(axis=0).max()))
    ins, outs, so = _setup(S0, rb)
    eng.run(ins, torch.from_numpy(S0).cuda(), outs, so, rb)
    assert eng.status() == a2av.OK
    eng.close()


def test_status_keeps_first_error_until_read():
    rb = 4
    eng = a2av.A2av(3)
    bad = S0.copy()
    bad[0, 0] = -5
    ins, outs, so = _setup(S0, rb)
    eng.run(ins, torch.from_numpy(bad).cuda(), outs, so, rb)
    eng.run(ins, torch.from_numpy(S0).cuda(), outs, so, rb)  # valid run afterwards
    assert eng.status() == a2av.ERR_BAD_SPLITS
    eng.run(ins, torch.from_numpy(S0).cuda(), outs, so, rb)
    assert eng.status() == a2av.OK
    eng.close()


def test_host_rejections_launch_nothing():
    rc, h = a2av.a2av_create(3)
    assert rc == a2av.OK
    S = torch.from_numpy(S0).cuda()
    ins, outs, so = _setup(S0, 4)
    ip = [t.data_ptr() for t in ins]
    op = [t.data_ptr() for t in outs]
    assert a2av.a2av_run(h, ip, S.data_ptr(), op, so.data_ptr(), 0) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run(h, ip, 0, op, so.data_ptr(), 4) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run(h, ip, S.data_ptr(), op, 0, 4) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run(h, ip, S.data_ptr() + 4, op, so.data_ptr(), 4) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run(None, ip, S.data_ptr(), op, so.data_ptr(), 4) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_set_path(h, 7) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_set_path(h, 4) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_set_grid(h, 33) == a2av.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert _untouched(outs, so)
    assert a2av.a2av_status(h)[1] == a2av.OK
    assert a2av.a2av_destroy(h) == a2av.OK
    assert a2av.a2av_create(0)[0] == a2av.ERR_INVALID_ARG
    assert a2av.a2av_create(33)[0] == a2av.ERR_UNSUPPORTED
    assert a2av.a2av_create(4, -1)[0] == a2av.ERR_INVALID_ARG


def test_binding_rejects_bad_tensors():
    eng = a2av.A2av(2)
    S = torch.zeros((2, 2), dtype=torch.int64, device="cuda")
    so = torch.zeros((2, 2, 2), dtype=torch.int64, device="cuda")
    x = [torch.zeros(4, dtype=torch.uint8, device="cuda")] * 2
    with pytest.raises(ValueError):
        eng.run(x, S.to(torch.int32), x, so, 1)
    with pytest.raises(ValueError):
        eng.run(x, S, x, so[:, :1], 1)
    with pytest.raises(ValueError):
        eng.run(x[:1], S, x, so, 1)
    with pytest.raises(ValueError):
        eng.run([torch.zeros(4, dtype=torch.uint8)] * 2, S, x, so, 1)
    with pytest.raises(a2av.A2avError):
        eng.run(x, S, x, so, 0)
    eng.close()


def test_combine_with_bad_splits_writes_nothing():
    rb = 8
    dso = np.zeros((3, 2, 3), dtype=np.int64)
    dso[:, 0, :] = S0.T
    dso[1, 0, 2] = -3
    ins, outs, so = _setup(S0.T.copy(), rb)
    eng = a2av.A2av(3)
    eng.combine(ins, torch.from_numpy(dso).cuda(), outs, so, rb)
    assert eng.status() == a2av.ERR_BAD_SPLITS
    eng.close()
    assert _untouched(outs, so)
