"""The seeded input generators: determinism, shapes and the stated distributions."""
import numpy as np
import pytest

import workloads as wl


def _same(a, b):
    assert a.W == b.W and a.row_bytes == b.row_bytes
    assert np.array_equal(a.splits, b.splits)
    for x, y in zip(a.inputs, b.inputs):
        assert np.array_equal(x, y)


def _shape_ok(w):
    assert w.splits.shape == (w.W, w.W) and w.splits.dtype == np.int64
    assert np.all(w.splits >= 0)
    for r in range(w.W):
        assert w.inputs[r].dtype == np.uint8
        assert w.inputs[r].size == int(w.splits[r].sum()) * w.row_bytes


def test_cfg1_shape_and_determinism():
    a, b = wl.cfg1(0), wl.cfg1(0)
    _same(a, b)
    _shape_ok(a)
    assert a.W == 4 and a.row_bytes == 256
    assert np.all(a.splits.sum(axis=1) == 4096)
    v = a.inputs[0].view(np.uint16)
    f = (v.astype(np.uint32) << 16).view(np.float32)
    assert abs(float(f.mean())) < 0.02 and abs(float(f.std()) - 1) < 0.02
    assert not np.array_equal(wl.cfg1(1).inputs[0], a.inputs[0])


def test_cfg2_rows_and_prefix_consistency():
    w = wl.cfg2(1 << 20)
    _shape_ok(w)
    assert w.row_bytes == 14336 and np.all(w.splits.sum(axis=1) == (1 << 20) // 14336)
    big = wl.cfg2(1 << 22)
    for r in range(4):  # a smaller payload is a prefix of a larger one (same seed)
        assert np.array_equal(big.inputs[r][: w.inputs[r].size], w.inputs[r])
    # the page's fourteen payloads: 0.5 MiB .. 4 GiB in powers of two
    assert wl.CFG2_SWEEP_BYTES == [1 << k for k in range(19, 33)]


def test_random_bits_independent_of_threads(monkeypatch):
    a = np.empty(9 << 20, np.uint8)
    wl.random_bits(a, (3, 4))
    monkeypatch.setattr(wl, "_threads", lambda: 1)
    b = np.empty(9 << 20, np.uint8)
    wl.random_bits(b, (3, 4))
    assert np.array_equal(a, b)
    hist = np.bincount(a, minlength=256)
    assert hist.min() > 0.9 * a.size / 256


def test_cfg3_top2_dispatch_small():
    w = wl.cfg3(seed=1, tokens=512, hidden=64)
    _shape_ok(w)
    assert w.W == 8 and w.row_bytes == 128
    assert np.all(w.splits.sum(axis=1) == 2 * 512)
    for r, (tok, exp) in enumerate(w.meta["routes"]):
        pairs = tok * 64 + exp
        assert np.unique(pairs).size == pairs.size  # two distinct experts per token
        assert np.array_equal(np.bincount(exp // 8, minlength=8), w.splits[r])
        assert np.all(np.diff(exp // 8) >= 0)  # ordered by destination rank
    # Zipf(1.2) popularity: the most popular expert is routed to far more than the least
    counts = np.bincount(np.concatenate([e for _, e in w.meta["routes"]]), minlength=64)
    assert counts.max() > 8 * max(counts.min(), 1)


def test_cfg3_dedup_one_row_per_token_and_rank():
    full = wl.cfg3(seed=1, tokens=512, hidden=64)
    w = wl.cfg3(seed=1, tokens=512, hidden=64, dedup=True)
    _shape_ok(w)
    for r in range(8):
        assert np.array_equal(w.meta["choices"][r], full.meta["choices"][r])  # same routing
        dests = w.meta["choices"][r] // 8
        for p in range(8):  # tokens with at least one expert on rank p
            assert w.splits[r, p] == int(np.any(dests == p, axis=1).sum())
        tok, exp = w.meta["routes"][r]
        dest = exp // 8
        assert np.all(np.diff(dest * 512 + tok) > 0)  # (destination, token), no repeats
        rows = w.meta["token_rows"][r].reshape(512, -1)
        assert np.array_equal(w.inputs[r].reshape(-1, 128), rows[tok])
    assert w.splits.sum() < full.splits.sum()  # some tokens had both experts on one rank


def test_cfg5_lengths_go_with_the_keys():
    w = wl.cfg5(seed=2, batch=128)
    lw = wl.cfg5_lengths(w)
    _shape_ok(lw)
    assert lw.row_bytes == 4 and np.all(lw.splits == 13 * 128)
    for r in range(2):
        L = lw.inputs[r].view(np.int32)
        assert L[:13 * 128].sum() == w.splits[r, 0] and L[13 * 128:].sum() == w.splits[r, 1]
    with pytest.raises(ValueError):
        wl.cfg5_lengths(wl.cfg1(0))


def test_cfg4_skew():
    w = wl.cfg4(seed=3, rows=1 << 12)
    _shape_ok(w)
    assert w.row_bytes == 13 and np.all(w.splits.sum(axis=1) == 1 << 12)
    assert (w.splits == 0).sum() > 0  # Dirichlet(0.1): many empty chunks
    assert np.all(w.splits.max(axis=1) > (1 << 12) // 8)  # one peer dominates


def test_cfg5_embedding_keys_small():
    w = wl.cfg5(seed=0, batch=256)
    _shape_ok(w)
    assert w.W == 2 and w.row_bytes == 8
    for r in range(2):
        keys = w.inputs[r].view(np.int64)
        assert keys.min() >= 0 and keys.max() < 10 ** 7
        L = w.meta["lengths"][r]
        assert L.max() <= 20 and abs(L.mean() - 3) < 0.2
        assert w.splits[r, 0] == L[0::2].sum() and w.splits[r, 1] == L[1::2].sum()


@pytest.mark.parametrize("mode", ["uniform", "skew", "sparse", "empty", "diag", "one"])
def test_random_case_modes(mode):
    w = wl.random_case(5, 6, 7, mode=mode)
    _shape_ok(w)
    _same(w, wl.random_case(5, 6, 7, mode=mode))
