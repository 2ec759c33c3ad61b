"""Parity at the benchmark's full size and launch configuration.

Config 2 at 4 GiB per rank (W=4, 14336-byte rows; 16 GiB in, 16 GiB out on
the device), run exactly as bench.py times it (default engine and grid).
Every peer's whole output is compared with the oracle's (computed one peer
at a time to bound host memory), rows sampled across each output are checked
one by one against the oracle's per-row source, and out_splits_offsets is
compared in full.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")

P = 1 << 32  # bytes per rank, the top of the payload sweep


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    free, _ = torch.cuda.mem_get_info()
    if free < 40 << 30:
        pytest.skip("needs about 33 GiB of free device memory")
    a2av.build()


def test_cfg2_4GiB_per_rank_bit_exact():
    rb = wl.CFG2_ROW_BYTES
    nbytes = (P // rb) * rb
    h_in = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=True) for _ in range(4)]
    w = wl.cfg2(P, seed=0, buffers=[t.numpy() for t in h_in])
    S = w.splits
    d_in = [t.cuda() for t in h_in]
    d_out = [torch.full((int(S[:, p].sum()) * rb,), 0xEE, dtype=torch.uint8, device="cuda")
             for p in range(4)]
    so = torch.full((4, 2, 4), -7, dtype=torch.int64, device="cuda")
    with a2av.A2av(4) as eng:  # bench.py's configuration: AUTO engine, default grid
        eng.run(d_in, torch.from_numpy(S).cuda(), d_out, so, rb)
        assert eng.status() == a2av.OK
        assert eng.last_launch()["path"] == a2av.PATH_BULK
    torch.cuda.synchronize()
    o = oracle.default()
    inputs = [t.numpy() for t in h_in]
    full_so = np.empty((4, 2, 4), np.int64)
    rng = np.random.default_rng(0)
    for p in range(4):
        want = np.empty(int(S[:, p].sum()) * rb, np.uint8)
        assert o.dest(inputs, S, p, want, full_so[p], rb) == 0
        got = d_out[p].cpu().numpy()
        assert np.array_equal(got, want), f"peer {p}: 4 GiB output differs from the oracle"
        rows = got.reshape(-1, rb)
        for k in np.concatenate([[0, rows.shape[0] - 1], rng.integers(0, rows.shape[0], 500)]):
            r, i = o.row_source(S, p, int(k))
            assert np.array_equal(rows[k], inputs[r][i * rb:(i + 1) * rb]), (p, k)
        del want, got, rows
    assert np.array_equal(so.cpu().numpy(), full_so)
