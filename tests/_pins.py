"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with what the definition of all_to_all_vdev and
plain mathematics fix:

* an independently written *scatter* formulation (each source row finds its
  peer and its destination row) on every split matrix with entries in
  {0, 1, 2} for W <= 3, with rows tagged by (rank, row);
* closed forms: W = 1 is the identity; uniform splits are a numpy transpose of
  a (W, W, s, row_bytes) array; diagonal splits keep every buffer in place; a
  permutation matrix permutes whole buffers;
* invariants: out_splits = transpose(in_splits) (numpy), offsets = exclusive
  scan (numpy cumsum), received rows sum to sent rows, the multiset of rows
  is conserved, every output row comes from the chunk the definition names;
* the round trip: exchanging the outputs with the transposed splits gives
  back the inputs;
* the validity rule and "no writes on invalid splits".

The same functions run in-process against the real oracle
(``test_oracle_pins.py``) and in a subprocess against copies of the oracle
with planted mistakes (``test_oracle_mutants.py``), where at least one of them
must fail.  Run as ``python -m tests._pins LIB`` to check one library and print
the first failing pin.
"""
from __future__ import annotations

import itertools
import sys

import numpy as np

SENTINEL = 0xEE


# ----------------------------------------------------------------- helpers --
def tagged_inputs(S, rb):
    """Row i of rank r carries a tag unique to (r, i) within the case."""
    S = np.asarray(S)
    W = S.shape[0]
    bufs = []
    for r in range(W):
        n = int(S[r].sum())
        b = np.empty((n, rb), dtype=np.uint8)
        for i in range(n):
            if rb == 1:
                b[i, 0] = (r * 64 + i) & 0xFF
            else:
                b[i, 0] = r
                b[i, 1] = i & 0xFF
                for j in range(2, rb):
                    b[i, j] = (r * 13 + i * 7 + j * 3 + (i >> 8)) & 0xFF
        bufs.append(b.reshape(-1))
    return bufs


def scatter_reference(inputs, S, rb):
    """all_to_all_vdev written as a scatter: every source row finds its peer.

    Source row i of rank r belongs to the first peer p whose chunk in rank r's
    input (chunks back to back in peer order) contains row i; it goes to peer
    p's output after all rows that lower ranks send to p, at position
    i - (first row of that chunk).
    """
    W = len(inputs)
    S = [[int(x) for x in row] for row in np.asarray(S)]
    received = [sum(S[r][p] for r in range(W)) for p in range(W)]
    outs = [np.full(received[p] * rb, SENTINEL, dtype=np.uint8) for p in range(W)]
    for r in range(W):
        rows = sum(S[r])
        for i in range(rows):
            first = 0
            for p in range(W):
                if first <= i < first + S[r][p]:
                    break
                first += S[r][p]
            below = sum(S[q][p] for q in range(r))
            k = below + (i - first)
            outs[p][k * rb:(k + 1) * rb] = inputs[r][i * rb:(i + 1) * rb]
    so = np.zeros((W, 2, W), dtype=np.int64)
    for p in range(W):
        for r in range(W):
            so[p, 0, r] = S[r][p]
            so[p, 1, r] = sum(S[q][p] for q in range(r))
    return outs, so


def run_fresh(o, inputs, S, rb, in_cap=0, out_cap=0, out_rows=None):
    """Run the oracle into sentinel-filled outputs; returns (rc, outs, so)."""
    W = len(inputs)
    S = np.asarray(S, dtype=np.int64)
    if out_rows is None:
        out_rows = [int(S[:, p].sum()) for p in range(W)]
    outs = [np.full(max(n, 0) * rb, SENTINEL, dtype=np.uint8) for n in out_rows]
    so = np.full((W, 2, W), -7, dtype=np.int64)
    rc = o.run(inputs, S, outs, so, rb, in_cap, out_cap)
    return rc, outs, so


def _eq(a, b, what):
    assert a.shape == b.shape and np.array_equal(a, b), what


# -------------------------------------------------------------------- pins --
def pin_identity_w1(o):
    for rb in (1, 5, 16):
        for n in (0, 1, 7):
            inp = [np.arange(n * rb, dtype=np.uint8) * 3]
            rc, outs, so = run_fresh(o, inp, [[n]], rb)
            assert rc == 0
            _eq(outs[0], inp[0], "W=1 must be the identity")
            _eq(so, np.array([[[n], [0]]]), "W=1 splits/offsets")


def pin_uniform_transpose(o):
    rng = np.random.default_rng(11)
    for W, s, rb in ((2, 3, 4), (3, 2, 7), (4, 5, 16), (5, 1, 1)):
        x = rng.integers(0, 256, size=(W, W, s, rb), dtype=np.uint8)  # [r][p][row][byte]
        inp = [x[r].reshape(-1).copy() for r in range(W)]
        rc, outs, so = run_fresh(o, inp, np.full((W, W), s), rb)
        assert rc == 0
        y = x.transpose(1, 0, 2, 3)  # [p][r][row][byte]
        for p in range(W):
            _eq(outs[p], y[p].reshape(-1), f"uniform splits: peer {p} != transpose")


def pin_diagonal_and_permutation(o):
    rng = np.random.default_rng(12)
    W, rb = 4, 6
    n = [3, 0, 5, 2]
    inp = [rng.integers(0, 256, size=n[r] * rb, dtype=np.uint8) for r in range(W)]
    rc, outs, _ = run_fresh(o, inp, np.diag(n), rb)
    assert rc == 0
    for p in range(W):
        _eq(outs[p], inp[p], "diagonal splits must keep buffers in place")
    perm = [2, 0, 3, 1]
    S = np.zeros((W, W), dtype=np.int64)
    for r in range(W):
        S[r, perm[r]] = n[r]
    rc, outs, _ = run_fresh(o, inp, S, rb)
    assert rc == 0
    for r in range(W):
        _eq(outs[perm[r]], inp[r], "permutation splits must permute buffers")


def pin_errors(o):
    W, rb = 3, 4
    S = np.array([[1, 2, 0], [0, 1, 1], [2, 0, 3]], dtype=np.int64)
    inp = [np.full(int(S[r].sum()) * rb, r + 1, dtype=np.uint8) for r in range(W)]
    rows_in = S.sum(axis=1)
    rows_out = S.sum(axis=0)
    # exactly at capacity is valid
    rc, _, _ = run_fresh(o, inp, S, rb, int(rows_in.max()), int(rows_out.max()))
    assert rc == 0, "splits exactly at capacity must be accepted"
    bad = [
        ("input capacity", S, int(rows_in.max()) - 1, 0),
        ("output capacity", S, 0, int(rows_out.max()) - 1),
    ]
    neg = S.copy()
    neg[1, 2] = -1
    bad.append(("negative split", neg, 0, 0))
    for what, SS, ic, oc in bad:
        rc, outs, so = run_fresh(o, inp, SS, rb, ic, oc,
                                 out_rows=[max(int(SS[:, p].sum()), 0) for p in range(W)])
        assert rc == -4, f"{what} must be rejected"
        for b in outs:
            assert np.all(b == SENTINEL), f"{what}: outputs written on rejected splits"
        assert np.all(so == -7), f"{what}: out_splits_offsets written on rejected splits"
    # a null input with rows to send, a null output with rows to receive
    assert o.check(S, rb, inputs=[inp[0], None, inp[2]]) == -4
    assert o.check(S, rb, outputs=[np.zeros(1, np.uint8), None, np.zeros(1, np.uint8)]) == -4
    z = S.copy()
    z[1] = 0
    assert o.check(z, rb, inputs=[inp[0], None, inp[2]]) == 0, "null input with no rows is valid"
    # 64-bit byte-offset limit: S <= 2^62 / (W * row_bytes)
    for W2, rb2 in ((4, 1), (2, 3), (8, 13)):
        lim = (1 << 62) // (W2 * rb2)
        T = np.zeros((W2, W2), dtype=np.int64)
        T[0, 1] = lim
        assert o.check(T, rb2) == 0, "a split at the 64-bit limit is valid"
        T[0, 1] = lim + 1
        assert o.check(T, rb2) == -4, "a split past the 64-bit limit must be rejected"
    assert o.check(S, 0) == -1, "row_bytes = 0 is an invalid argument"


def pin_bruteforce_tiny(o):
    """Every split matrix with entries in {0,1,2}, W <= 3, against the scatter form."""
    cases = []
    for W in (1, 2):
        for rb in (1, 3, 16):
            cases += [(W, rb, v) for v in itertools.product(range(3), repeat=W * W)]
    for v in itertools.product(range(3), repeat=9):
        cases.append((3, 3, v))
    for v in list(itertools.product(range(3), repeat=9))[::37]:
        cases += [(3, 1, v), (3, 16, v)]
    for W, rb, v in cases:
        S = np.array(v, dtype=np.int64).reshape(W, W)
        inp = tagged_inputs(S, rb)
        rc, outs, so = run_fresh(o, inp, S, rb)
        assert rc == 0
        ref_outs, ref_so = scatter_reference(inp, S, rb)
        for p in range(W):
            _eq(outs[p], ref_outs[p], f"W={W} rb={rb} S={S.tolist()} peer {p}")
        _eq(so, ref_so, f"W={W} rb={rb} S={S.tolist()} out_splits_offsets")


def pin_invariants_random(o):
    rng = np.random.default_rng(13)
    for trial in range(60):
        W = int(rng.integers(1, 33))
        rb = int(rng.choice([1, 2, 3, 8, 13, 16, 24]))
        mode = trial % 3
        if mode == 0:
            S = rng.integers(0, 9, size=(W, W))
        elif mode == 1:
            S = rng.integers(0, 9, size=(W, W)) * (rng.random((W, W)) < 0.3)
        else:
            S = np.stack([rng.multinomial(int(rng.integers(0, 40)), rng.dirichlet([0.1] * W))
                          for _ in range(W)])
        S = S.astype(np.int64)
        # rows tagged with (rank, row) in the first 5 bytes when they fit
        inp = []
        for r in range(W):
            n = int(S[r].sum())
            b = rng.integers(0, 256, size=(n, rb), dtype=np.uint8)
            if rb >= 5:
                b[:, 0] = r
                b[:, 1:5] = np.arange(n, dtype=np.uint32).view(np.uint8).reshape(n, 4)
            inp.append(b.reshape(-1))
        rc, outs, so = run_fresh(o, inp, S, rb)
        assert rc == 0
        _eq(so[:, 0, :], S.T, "out_splits must be the transpose of in_splits")
        excl = np.concatenate([np.zeros((W, 1), np.int64), np.cumsum(S.T, axis=1)[:, :-1]], axis=1)
        _eq(so[:, 1, :], excl, "offsets must be the exclusive scan of out_splits")
        assert sum(b.size for b in outs) == sum(b.size for b in inp), "bytes conserved"
        all_in = np.concatenate([b.reshape(-1, rb) for b in inp] + [np.zeros((0, rb), np.uint8)])
        all_out = np.concatenate([b.reshape(-1, rb) for b in outs] + [np.zeros((0, rb), np.uint8)])
        key_in = np.sort(all_in.view(np.dtype((np.void, rb))).reshape(-1))
        key_out = np.sort(all_out.view(np.dtype((np.void, rb))).reshape(-1))
        assert np.array_equal(key_in, key_out), "multiset of rows must be conserved"
        if rb >= 5:
            in_first = np.concatenate([np.zeros((W, 1), np.int64), np.cumsum(S, axis=1)[:, :-1]],
                                      axis=1)  # in_off[r][p]
            for p in range(W):
                rows = outs[p].reshape(-1, rb)
                src = rows[:, 0].astype(np.int64)
                idx = rows[:, 1:5].copy().view(np.uint32).reshape(-1).astype(np.int64)
                assert np.all(np.diff(src) >= 0), "sources must arrive in rank order"
                for r in range(W):
                    got = idx[src == r]
                    want = in_first[r, p] + np.arange(S[r, p])
                    _eq(got, want, f"peer {p} must receive rank {r}'s chunk rows in order")


def pin_round_trip(o):
    rng = np.random.default_rng(14)
    for W, rb in ((2, 8), (3, 13), (8, 1), (5, 16)):
        S = rng.integers(0, 6, size=(W, W)).astype(np.int64)
        inp = [rng.integers(0, 256, size=int(S[r].sum()) * rb, dtype=np.uint8) for r in range(W)]
        rc, outs, _ = run_fresh(o, inp, S, rb)
        assert rc == 0
        rc, back, _ = run_fresh(o, outs, S.T.copy(), rb)
        assert rc == 0
        for r in range(W):
            _eq(back[r], inp[r], "exchanging back with transposed splits must restore inputs")


def pin_dest_and_row_source(o):
    rng = np.random.default_rng(15)
    for W, rb in ((3, 5), (6, 8), (1, 2)):
        S = rng.integers(0, 5, size=(W, W)).astype(np.int64)
        inp = tagged_inputs(S, rb)
        ref_outs, ref_so = scatter_reference(inp, S, rb)
        for p in range(W):
            out_p = np.full(int(S[:, p].sum()) * rb, SENTINEL, np.uint8)
            so_p = np.zeros((2, W), np.int64)
            assert o.dest(inp, S, p, out_p, so_p, rb) == 0
            _eq(out_p, ref_outs[p], "dest() must match the scatter form")
            _eq(so_p, ref_so[p], "dest() offsets must match")
            for k in range(int(S[:, p].sum())):
                r, i = o.row_source(S, p, k)
                _eq(ref_outs[p][k * rb:(k + 1) * rb], inp[r][i * rb:(i + 1) * rb],
                    "row_source must name the row the scatter form put there")
            assert o.row_source(S, p, int(S[:, p].sum())) is None


def pin_combine_round_trip(o):
    """The reverse exchange undoes the exchange: rows come home in their
    original places, and its offsets are the original splits and their
    row-wise exclusive scan (numpy cumsum)."""
    rng = np.random.default_rng(16)
    for W, rb in ((1, 3), (2, 8), (3, 13), (5, 1), (8, 16)):
        S = rng.integers(0, 6, size=(W, W)).astype(np.int64)
        S[rng.random((W, W)) < 0.3] = 0
        inp = tagged_inputs(S, rb)
        rc, mid, dso = run_fresh(o, inp, S, rb)
        assert rc == 0
        outs = [np.full(b.size, SENTINEL, np.uint8) for b in inp]
        so = np.full((W, 2, W), -7, np.int64)
        assert o.combine(mid, dso, outs, so, rb) == 0
        for r in range(W):
            _eq(outs[r], inp[r], "combine must return every row to its original place")
        _eq(so[:, 0, :], S, "combine's splits must be the original splits")
        excl = np.concatenate([np.zeros((W, 1), np.int64), np.cumsum(S, axis=1)[:, :-1]], axis=1)
        _eq(so[:, 1, :], excl, "combine's offsets must be the row-wise exclusive scan")
        # uniform splits: the reverse exchange is the inverse transpose
        x = rng.integers(0, 256, size=(W, W, 2, rb), dtype=np.uint8)  # [p][r][row][byte]
        back = [np.full(W * 2 * rb, SENTINEL, np.uint8) for _ in range(W)]
        uso = np.zeros((W, 2, W), np.int64)
        uso[:, 0, :] = 2
        assert o.combine([x[p].reshape(-1).copy() for p in range(W)], uso, back,
                         np.zeros((W, 2, W), np.int64), rb) == 0
        for r in range(W):
            _eq(back[r], x.transpose(1, 0, 2, 3)[r].reshape(-1), "uniform combine = transpose")


def _dispatch_reference(K, rows, src, key, rb):
    """Fused dispatch written out: sort each rank's items with Python's stable
    sort on (key, item), gather their rows, then the scatter formulation."""
    W = len(rows)
    sorted_rows, pos, S = [], [], np.zeros((W, W), np.int64)
    for r in range(W):
        order = sorted(range(len(key[r])), key=lambda i: (int(key[r][i]), i))
        inv = np.empty(len(order), np.int64)
        for k, i in enumerate(order):
            inv[i] = k
            S[r, int(key[r][i]) // K] += 1
        buf = [rows[r][int(src[r][i]) * rb:(int(src[r][i]) + 1) * rb] for i in order]
        sorted_rows.append(np.concatenate(buf) if buf else np.zeros(0, np.uint8))
        pos.append(inv)
    outs, so = scatter_reference(sorted_rows, S, rb)
    return outs, so, pos, S


def pin_dispatch_small(o):
    rng = np.random.default_rng(17)
    for trial in range(300):
        W = int(rng.integers(1, 4))
        K = int(rng.integers(1, 4))
        rb = int(rng.choice([1, 3, 8]))
        n = [int(rng.integers(0, 5)) for _ in range(W)]
        m = [int(rng.integers(0, 7)) for _ in range(W)]
        rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
        src = [rng.integers(0, max(n[r], 1), m[r]).astype(np.int32) if n[r] else
               np.zeros(0, np.int32) for r in range(W)]
        m = [s.size for s in src]
        key = [rng.integers(0, W * K, m[r]).astype(np.int32) for r in range(W)]
        ref_outs, ref_so, ref_pos, ref_S = _dispatch_reference(K, rows, src, key, rb)
        outs = [np.full(b.size, SENTINEL, np.uint8) for b in ref_outs]
        so = np.full((W, 2, W), -7, np.int64)
        pos = [np.full(mm, -1, np.int64) for mm in m]
        isp = np.full((W, W), -1, np.int64)
        assert o.dispatch(K, rows, src, key, outs, so, pos, rb, isp) == 0
        for p in range(W):
            _eq(outs[p], ref_outs[p], f"dispatch peer {p} (W={W} K={K})")
        _eq(so, ref_so, "dispatch out_splits_offsets")
        _eq(isp, ref_S, "dispatch in_splits")
        for r in range(W):
            _eq(pos[r], ref_pos[r], "dispatch sorted positions")


def pin_dispatch_matches_generators(o):
    import workloads as wl
    for w in (wl.cfg3(2, tokens=96, hidden=4), wl.cfg3(2, tokens=96, hidden=4, dedup=True),
              wl.cfg5(3, batch=64)):
        K, rows, src, key = wl.dispatch_items(w)
        outs, so, pos, S = o.dispatch_exchange(K, rows, src, key, w.row_bytes)
        _eq(S, w.splits, f"{w.name}: dispatch splits must equal the generator's")
        ref, ref_so = o.exchange(w.inputs, w.splits, w.row_bytes)
        for p in range(w.W):
            _eq(outs[p], ref[p], f"{w.name}: dispatch must equal the exchange of the "
                                 "generator's pre-grouped rows")
        _eq(so, ref_so, f"{w.name}: offsets")
        for r in range(w.W):
            order = np.argsort(key[r], kind="stable")  # numpy's stable sort as the pin
            inv = np.empty(order.size, np.int64)
            inv[order] = np.arange(order.size)
            _eq(pos[r], inv, f"{w.name}: positions = inverse stable argsort")


def pin_kjt_lengths_cut_the_keys(o):
    """A keyed-jagged batch exchanged as two a2avs, the bag lengths and the
    keys: what peer p receives from rank r must be exactly rank r's bags of
    the features p owns, the lengths cutting the keys into those bags."""
    import workloads as wl
    w = wl.cfg5(4, features=5, batch=7, W=2)
    lw = wl.cfg5_lengths(w)
    keys, kso = o.exchange(w.inputs, w.splits, w.row_bytes)
    lens, lso = o.exchange(lw.inputs, lw.splits, lw.row_bytes)
    F = w.meta["features"]
    for p in range(w.W):
        owned = [f for f in range(F) if f % w.W == p]
        got_len = lens[p].view(np.int32)
        got_key = keys[p].view(np.int64)
        for r in range(w.W):
            L = w.meta["lengths"][r]
            starts = np.concatenate([[0], np.cumsum(L.sum(axis=1))])
            want_keys = np.concatenate([w.meta["kjt_keys"][r][starts[f]:starts[f + 1]]
                                        for f in owned])
            l0 = int(lso[p][1][r])
            rl = got_len[l0:l0 + int(lso[p][0][r])]
            _eq(rl, L[owned].reshape(-1).astype(np.int32), f"bag lengths {r} -> {p}")
            k0 = int(kso[p][1][r])
            rk = got_key[k0:k0 + int(kso[p][0][r])]
            assert int(rl.sum()) == rk.size, "the lengths must count the keys received"
            _eq(rk, want_keys, f"keys {r} -> {p}")


def _random_items(rng, W, K, rb):
    n = [int(rng.integers(1, 12)) for _ in range(W)]
    rows = [rng.integers(0, 256, n[r] * rb, dtype=np.uint8) for r in range(W)]
    m = [int(rng.integers(0, 25)) for _ in range(W)]
    src = [rng.integers(0, n[r], m[r]).astype(np.int32) for r in range(W)]
    key = [rng.integers(0, W * K, m[r]).astype(np.int32) for r in range(W)]
    return rows, src, key


def pin_combine_items_round_trip(o):
    """combine_items(dispatch(x)) puts every item's source row back in item
    order: item (r, i) gets rows[r][src[r][i]] (numpy fancy indexing)."""
    rng = np.random.default_rng(17)
    cases = 0
    for W, K, rb in ((1, 1, 3), (2, 3, 1), (3, 2, 16), (4, 5, 7), (5, 1, 24)):
        for _ in range(20):
            rows, src, key = _random_items(rng, W, K, rb)
            outs, so, pos, S = o.dispatch_exchange(K, rows, src, key, rb)
            back = o.combine_items_exchange(K, outs, S, key, pos, rb)
            for r in range(W):
                want = rows[r].reshape(-1, rb)[src[r]].reshape(-1)
                _eq(back[r], want, f"combine_items(dispatch(x)) (W={W} K={K} rb={rb})")
            cases += 1
    assert cases == 100


def pin_combine_items_is_combine_then_gather(o):
    """The same result as the plain reverse exchange (rows back in key order)
    followed by a gather by sorted position: a different formulation."""
    import workloads as wl
    w = wl.cfg3(4, tokens=64, hidden=8)
    K, rows, src, key = wl.dispatch_items(w)
    rb = w.row_bytes
    outs, so, pos, S = o.dispatch_exchange(K, rows, src, key, rb)
    # the experts write something of their own into the dispatch layout
    rng = np.random.default_rng(3)
    expert = [rng.integers(0, 256, b.size, dtype=np.uint8) for b in outs]
    back, _ = o.exchange_back(expert, so, rb)
    got = o.combine_items_exchange(K, expert, S, key, pos, rb)
    for r in range(w.W):
        want = back[r].reshape(-1, rb)[pos[r]].reshape(-1)
        _eq(got[r], want, "combine_items = combine + gather by sorted position")


def pin_combine_items_errors(o):
    W, K, rb = 2, 2, 4
    S = np.array([[2, 1], [0, 2]], np.int64)
    expert = [np.arange(8, dtype=np.uint8), np.arange(12, dtype=np.uint8)]
    good_key = [np.array([0, 2, 1], np.int32), np.array([3, 2], np.int32)]
    good_pos = [np.array([0, 2, 1], np.int64), np.array([1, 0], np.int64)]
    assert o.combine_items_exchange(K, expert, S, good_key, good_pos, rb)[0].size == 12
    for what, key, pos, s, code in (
            ("key too large", [good_key[0], np.array([4, 2], np.int32)], good_pos, S, -6),
            ("negative key", [np.array([0, -1, 1], np.int32), good_key[1]], good_pos, S, -6),
            ("position outside its group", good_key, [np.array([0, 1, 2], np.int64), good_pos[1]],
             S, -6),
            ("position past the rank", good_key, [good_pos[0], np.array([2, 0], np.int64)], S, -6),
            ("negative split", good_key, good_pos, np.array([[2, 1], [-1, 2]], np.int64), -4)):
        outs = [np.full(12, SENTINEL, np.uint8), np.full(8, SENTINEL, np.uint8)]
        rc = o.combine_items(K, expert, s, key, pos, outs, rb)
        assert rc == code, f"{what}: status {rc}, expected {code}"
        assert all(np.all(b == SENTINEL) for b in outs), what


def pin_dispatch_errors(o):
    rows = [np.arange(12, dtype=np.uint8), np.arange(8, dtype=np.uint8)]
    good_src = [np.array([0, 2, 1], np.int32), np.array([1, 0], np.int32)]
    good_key = [np.array([0, 3, 1], np.int32), np.array([2, 2], np.int32)]
    for what, src, key, cap, code in (
            ("key too large", good_src, [good_key[0], np.array([2, 4], np.int32)], 0, -6),
            ("negative key", good_src, [np.array([0, -1, 1], np.int32), good_key[1]], 0, -6),
            ("source row too large", [good_src[0], np.array([1, 2], np.int32)], good_key, 0, -6),
            ("output capacity", good_src, good_key, 2, -4)):
        outs = [np.full(16, SENTINEL, np.uint8), np.full(16, SENTINEL, np.uint8)]
        so = np.full((2, 2, 2), -7, np.int64)
        pos = [np.full(3, -1, np.int64), np.full(2, -1, np.int64)]
        isp = np.full((2, 2), -1, np.int64)
        rc = o.dispatch(2, rows, src, key, outs, so, pos, 4, isp, out_capacity_rows=cap)
        assert rc == code, f"{what}: status {rc}, expected {code}"
        assert all(np.all(b == SENTINEL) for b in outs) and np.all(so == -7), what
        assert all(np.all(p == -1) for p in pos) and np.all(isp == -1), what


PINS = [pin_identity_w1, pin_errors, pin_diagonal_and_permutation, pin_uniform_transpose,
        pin_round_trip, pin_combine_round_trip, pin_dispatch_errors, pin_dispatch_small,
        pin_dispatch_matches_generators, pin_kjt_lengths_cut_the_keys, pin_combine_items_errors,
        pin_combine_items_is_combine_then_gather, pin_combine_items_round_trip,
        pin_dest_and_row_source,
        pin_invariants_random,
        pin_bruteforce_tiny]


def main(argv):
    sys.path.insert(0, __file__.rsplit("/tests/", 1)[0])
    import oracle

    o = oracle.Oracle(argv[1] if len(argv) > 1 else None)
    for pin in PINS:
        try:
            pin(o)
        except AssertionError as e:
            print(f"FAILED {pin.__name__}: {e}")
            return 1
    print("ALL PINS PASS")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv))
