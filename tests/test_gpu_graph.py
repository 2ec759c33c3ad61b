"""The exchange captured once in a CUDA graph and replayed with new splits.

The splits live on the device and the library never reads them on the host,
so a captured a2av_run stays valid when the split matrix changes: the caller
writes new row counts into the same device buffer and replays the graph.
Each replay is checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

a2av = pytest.importorskip("variable_size_all_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    a2av.build()


@pytest.mark.parametrize("path", [a2av.PATH_AUTO, a2av.PATH_STAGED, a2av.PATH_VECTOR])
@pytest.mark.parametrize("rb", [16, 13])
def test_graph_replay_with_new_splits(path, rb):
    W, cap_rows = 4, 3000
    rng = np.random.default_rng(rb + path)
    inputs = [rng.integers(0, 256, cap_rows * rb, dtype=np.uint8) for _ in range(W)]
    d_in = [torch.from_numpy(b).cuda() for b in inputs]
    d_out = [torch.full((W * cap_rows * rb,), 0xEE, dtype=torch.uint8, device="cuda")
             for _ in range(W)]
    S = torch.zeros((W, W), dtype=torch.int64, device="cuda")
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    eng = a2av.A2av(W, in_capacity_rows=cap_rows, out_capacity_rows=W * cap_rows, path=path)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eng.run(d_in, S, d_out, so, rb, stream=s)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        eng.run(d_in, S, d_out, so, rb, stream=s)
    for trial in range(4):
        splits = np.stack([rng.multinomial(int(rng.integers(0, cap_rows + 1)),
                                           rng.dirichlet([0.3] * W)) for _ in range(W)])
        S.copy_(torch.from_numpy(splits.astype(np.int64)))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert eng.status() == a2av.OK
        used = [b[: int(splits[r].sum()) * rb] for r, b in enumerate(inputs)]
        ref, ref_so = oracle.default().exchange(used, splits, rb)
        assert np.array_equal(so.cpu().numpy(), ref_so)
        for p in range(W):
            assert np.array_equal(d_out[p][: ref[p].size].cpu().numpy(), ref[p]), (trial, p)
    # invalid splits written into the captured buffer are still caught on the device
    S.fill_(-1)
    graph.replay()
    torch.cuda.synchronize()
    assert eng.status() == a2av.ERR_BAD_SPLITS
    eng.close()


def test_graph_replay_multi_with_new_splits():
    """Two exchanges of one a2av_run_multi launch, captured once: new split
    values for both are written between replays."""
    W, cap_rows = 3, 2000
    rng = np.random.default_rng(42)
    rbs = [4, 8]
    inputs = [[rng.integers(0, 256, cap_rows * rb, dtype=np.uint8) for _ in range(W)]
              for rb in rbs]
    d_in = [[torch.from_numpy(b).cuda() for b in x] for x in inputs]
    d_out = [[torch.full((W * cap_rows * rb,), 0xEE, dtype=torch.uint8, device="cuda")
              for _ in range(W)] for rb in rbs]
    S = [torch.zeros((W, W), dtype=torch.int64, device="cuda") for _ in rbs]
    so = [torch.empty((W, 2, W), dtype=torch.int64, device="cuda") for _ in rbs]
    eng = a2av.A2av(W, in_capacity_rows=cap_rows, out_capacity_rows=W * cap_rows)
    ex = [(d_in[k], S[k], d_out[k], so[k], rbs[k]) for k in range(2)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eng.run_multi(ex, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        eng.run_multi(ex, stream=s)
    for trial in range(3):
        splits = [np.stack([rng.multinomial(int(rng.integers(0, cap_rows + 1)),
                                            rng.dirichlet([0.5] * W)) for _ in range(W)])
                  for _ in rbs]
        for k in range(2):
            S[k].copy_(torch.from_numpy(splits[k].astype(np.int64)))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert eng.status() == a2av.OK
        for k, rb in enumerate(rbs):
            used = [b[: int(splits[k][r].sum()) * rb] for r, b in enumerate(inputs[k])]
            ref, ref_so = oracle.default().exchange(used, splits[k], rb)
            assert np.array_equal(so[k].cpu().numpy(), ref_so)
            for p in range(W):
                got = d_out[k][p][: ref[p].size].cpu().numpy()
                assert np.array_equal(got, ref[p]), (trial, k, p)
    eng.close()


@pytest.mark.parametrize("rb,tokens", [(8, 3000), (14336 // 8, 256), (64, 3000)])
def test_graph_replay_dispatch_with_new_keys(rb, tokens):
    """The fused dispatch (a workspace memset and its kernels) captured
    once; new keys and source rows are written into the same device buffers
    between replays.  Covers the one-launch cooperative order kernel with its
    grid barrier (8-byte rows) and the count chain with the register copies
    (1792-byte and 64-byte rows)."""
    W, K = 4, 3
    rng = np.random.default_rng(rb)
    n_rows = tokens
    rows = [rng.integers(0, 256, n_rows * rb, dtype=np.uint8) for _ in range(W)]
    d_rows = [torch.from_numpy(r).cuda() for r in rows]
    m = 2 * tokens
    d_src = [torch.zeros(m, dtype=torch.int32, device="cuda") for _ in range(W)]
    d_key = [torch.zeros(m, dtype=torch.int32, device="cuda") for _ in range(W)]
    d_pos = [torch.empty(m, dtype=torch.int64, device="cuda") for _ in range(W)]
    d_out = [torch.full((W * m * rb,), 0xEE, dtype=torch.uint8, device="cuda") for _ in range(W)]
    so = torch.empty((W, 2, W), dtype=torch.int64, device="cuda")
    eng = a2av.A2av(W)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        eng.dispatch(d_rows, d_src, d_key, K, d_out, so, d_pos, rb, stream=s)  # allocates the workspace
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        eng.dispatch(d_rows, d_src, d_key, K, d_out, so, d_pos, rb, stream=s)
    for trial in range(3):
        src = [rng.integers(0, n_rows, m).astype(np.int32) for _ in range(W)]
        key = [rng.integers(0, W * K, m).astype(np.int32) for _ in range(W)]
        for r in range(W):
            d_src[r].copy_(torch.from_numpy(src[r]))
            d_key[r].copy_(torch.from_numpy(key[r]))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert eng.status() == a2av.OK
        ref, ref_so, ref_pos, _ = oracle.default().dispatch_exchange(K, rows, src, key, rb)
        assert np.array_equal(so.cpu().numpy(), ref_so)
        for p in range(W):
            assert np.array_equal(d_out[p][: ref[p].size].cpu().numpy(), ref[p]), (trial, p)
        for r in range(W):
            assert np.array_equal(d_pos[r].cpu().numpy(), ref_pos[r]), (trial, r)
    eng.close()
