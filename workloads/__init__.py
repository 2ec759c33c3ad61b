"""Seeded synthetic inputs for the variable-size all-to-all (a2av).

This module only *draws inputs*: per-rank input buffers and the W x W matrix of
device splits ``S[r][p]`` (rows that source rank ``r`` sends to peer ``p``).  It
holds none of the exchange's own arithmetic -- no offsets, no transposes, no
copies -- so that the oracle and the CUDA path, which both consume these
inputs, share nothing else.

The five workloads follow the shapes of the pages' subject:

* ``cfg1``  -- W=4, 4096 rows of 128 bf16 (256 B) per rank, uniform
  multinomial splits.  Small enough that the CPU oracle runs in well under a
  second.
* ``cfg2``  -- W=4 payload sweep: ``floor(P / 14336)`` rows of 7168 bf16 per
  rank for per-rank payloads P from 1 MiB to 4 GiB, uniform random bits.  This
  is the sweep of "[a2av] Improve tuning for 4 GPUs" (pytorch PR 154580,
  "Before"/"After" tables: MiB, us, BusBw).
* ``cfg3``  -- W=8 MoE token dispatch: 8192 tokens/rank, hidden 7168 bf16,
  top-2 routing over 64 experts (8 per rank) with Zipf(1.2) expert popularity
  shuffled per seed (the "MoE related region" remark of the same PR).
* ``cfg4``  -- W=8 skew/alignment stress: 2^20 rows of 13 bytes per rank,
  splits ~ Multinomial(2^20, Dirichlet(0.1)).
* ``cfg5``  -- W=2 sparse embedding-key exchange (torchrec PR 2570,
  "EmbeddingKey alltoall"): 26 features x 8192 bags, bag lengths
  min(Poisson(3), 20), int64 keys uniform in [0, 10^7), feature f owned by
  rank f mod 2.

Large buffers are filled in fixed 4 MiB pieces, each from its own
``SeedSequence(key + (piece,))``, on a thread pool: the bytes depend only on
the seed and the position, never on the thread count, and a shorter buffer is
a prefix of a longer one drawn under the same key.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "cfg1",
    "cfg2",
    "cfg2_splits",
    "cfg3",
    "cfg4",
    "cfg5",
    "cfg5_lengths",
    "random_case",
    "dispatch_items",
    "random_bits",
    "normal_bf16",
    "CFG2_ROW_BYTES",
    "CFG2_SWEEP_BYTES",
]

_PIECE = 4 << 20  # bytes per independently seeded piece

CFG2_ROW_BYTES = 7168 * 2
# per-rank payloads of the sweep: 0.5 MiB .. 4 GiB in powers of two, the
# fourteen rows of the "Before" and "After" tables of "[a2av] Improve tuning
# for 4 GPUs" (pytorch PR 154580)
CFG2_SWEEP_BYTES = [1 << k for k in range(19, 33)]


@dataclass
class Workload:
    """One a2av problem instance.

    ``splits[r, p]`` is the number of rows source rank ``r`` sends to peer
    ``p`` (int64, row-major by source rank).  ``inputs[r]`` is a flat uint8
    buffer holding exactly ``splits[r].sum() * row_bytes`` bytes, the chunks
    laid out back to back in peer order.
    """

    name: str
    W: int
    row_bytes: int
    splits: np.ndarray
    inputs: list
    meta: dict = field(default_factory=dict)

    @property
    def in_rows(self) -> np.ndarray:
        return self.splits.sum(axis=1)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _pieces(nbytes: int):
    return [(i, min(_PIECE, nbytes - i * _PIECE)) for i in range((nbytes + _PIECE - 1) // _PIECE)]


def random_bits(out: np.ndarray, key) -> np.ndarray:
    """Fill the uint8 array ``out`` with uniform random bits drawn under ``key``."""
    out = out.reshape(-1).view(np.uint8)
    key = tuple(int(k) for k in key)

    def fill(piece):
        i, n = piece
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(key + (i,))))
        words = g.bit_generator.random_raw((n + 7) // 8).view(np.uint8)
        out[i * _PIECE : i * _PIECE + n] = words[:n]

    ps = _pieces(out.nbytes)
    if len(ps) <= 2:
        for p in ps:
            fill(p)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, ps))
    return out


def normal_bf16(out_u16: np.ndarray, key) -> np.ndarray:
    """Fill the uint16 array ``out_u16`` with bf16 bit patterns of N(0,1) draws.

    Each float32 draw is rounded to bf16 with round-to-nearest-even on its bit
    pattern (the draws are finite, so no NaN handling is needed).
    """
    out = out_u16.reshape(-1)
    assert out.dtype == np.uint16
    key = tuple(int(k) for k in key)
    per = _PIECE // 2  # values per piece

    def fill(i):
        lo = i * per
        n = min(per, out.size - lo)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(key + (i,))))
        f = g.standard_normal(n, dtype=np.float32)
        b = f.view(np.uint32)
        b = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        out[lo : lo + n] = b.astype(np.uint16)

    count = (out.size + per - 1) // per
    if count <= 2:
        for i in range(count):
            fill(i)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(count)))
    return out


def _alloc(nbytes: int, buf=None) -> np.ndarray:
    if buf is None:
        return np.empty(nbytes, dtype=np.uint8)
    buf = buf.reshape(-1).view(np.uint8)
    if buf.nbytes < nbytes:
        raise ValueError(f"buffer of {buf.nbytes} B is smaller than the {nbytes} B needed")
    return buf[:nbytes]


def cfg1(seed: int = 0, rows: int = 4096, hidden: int = 128, W: int = 4) -> Workload:
    """W=4, 4096 rows of 128 bf16 per rank, splits ~ Multinomial(4096, 1/4 each)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 1]))
    splits = np.stack([rng.multinomial(rows, [1.0 / W] * W) for _ in range(W)]).astype(np.int64)
    rb = hidden * 2
    inputs = []
    for r in range(W):
        buf = np.empty(rows * hidden, dtype=np.uint16)
        normal_bf16(buf, (seed, 1, r))
        inputs.append(buf.view(np.uint8))
    return Workload("cfg1", W, rb, splits, inputs, {"rows_per_rank": rows, "dtype": "bf16"})


def cfg2_splits(per_rank_bytes: int, seed: int = 0, W: int = 4,
                row_bytes: int = CFG2_ROW_BYTES) -> np.ndarray:
    """The split matrix of ``cfg2`` alone: Multinomial(floor(P / row_bytes), 1/W each) per rank."""
    rows = per_rank_bytes // row_bytes
    rng = np.random.default_rng(np.random.SeedSequence([seed, 2, per_rank_bytes]))
    return np.stack([rng.multinomial(rows, [1.0 / W] * W) for _ in range(W)]).astype(np.int64)


def cfg2(per_rank_bytes: int, seed: int = 0, W: int = 4, row_bytes: int = CFG2_ROW_BYTES,
         buffers=None) -> Workload:
    """W=4 payload-sweep point: floor(P / row_bytes) rows per rank, uniform random bits.

    ``buffers`` optionally supplies W preallocated uint8 arrays (for example
    views of pinned host memory) to fill instead of allocating.
    """
    rows = per_rank_bytes // row_bytes
    splits = cfg2_splits(per_rank_bytes, seed, W, row_bytes)
    inputs = []
    for r in range(W):
        buf = _alloc(rows * row_bytes, None if buffers is None else buffers[r])
        random_bits(buf, (seed, 2, r))
        inputs.append(buf)
    return Workload("cfg2", W, row_bytes, splits, inputs,
                    {"per_rank_bytes": per_rank_bytes, "rows_per_rank": rows})


def cfg3(seed: int = 0, tokens: int = 8192, hidden: int = 7168, experts: int = 64,
         topk: int = 2, zipf_s: float = 1.2, W: int = 8, dedup: bool = False) -> Workload:
    """W=8 MoE token dispatch with top-2 routing over Zipf(1.2)-popular experts.

    Expert popularity rank k (1-based) has weight k^-s; the ids are shuffled
    per seed.  Each token draws ``topk`` distinct experts with probability
    proportional to those weights (Gumbel top-k, i.e. successive sampling
    without replacement).  One input row per (token, expert) pair, ordered by
    (destination rank, local expert, token), destination = expert // (experts/W).

    ``dedup``: one input row per distinct (token, destination rank) pair
    instead, ordered by (destination rank, token): a token whose experts sit
    on the same rank is sent there once.  The routing draws are the same.
    """
    per_rank = experts // W
    rng = np.random.default_rng(np.random.SeedSequence([seed, 3]))
    perm = rng.permutation(experts)
    weights = np.empty(experts)
    weights[perm] = np.arange(1, experts + 1, dtype=np.float64) ** (-zipf_s)
    logp = np.log(weights / weights.sum())
    rb = hidden * 2
    splits = np.zeros((W, W), dtype=np.int64)
    inputs, routes, token_rows, choices = [], [], [], []
    for r in range(W):
        scores = logp[None, :] + rng.gumbel(size=(tokens, experts))
        chosen = np.argsort(-scores, axis=1, kind="stable")[:, :topk]  # [tokens, topk]
        choices.append(chosen.astype(np.int64))
        tok = np.repeat(np.arange(tokens), topk)
        exp = chosen.reshape(-1)
        dest, local = exp // per_rank, exp % per_rank
        if dedup:
            # one (token, destination) pair per group; its first expert stands for it
            first = np.unique(tok * W + dest, return_index=True)[1]
            tok, exp, dest, local = tok[first], exp[first], dest[first], local[first] * 0
        order = np.lexsort((tok, local, dest))
        tok, exp, dest = tok[order], exp[order], dest[order]
        splits[r] = np.bincount(dest, minlength=W)
        x = np.empty((tokens, hidden), dtype=np.uint16)
        normal_bf16(x, (seed, 3, r))
        inputs.append(np.ascontiguousarray(x[tok]).view(np.uint8).reshape(-1))
        routes.append((tok.astype(np.int64), exp.astype(np.int64)))
        token_rows.append(x.view(np.uint8).reshape(-1))
    return Workload("cfg3", W, rb, splits, inputs,
                    {"tokens": tokens, "experts": experts, "topk": topk, "routes": routes,
                     "expert_weight": weights, "token_rows": token_rows, "choices": choices,
                     "dedup": dedup})


def cfg4(seed: int = 0, rows: int = 1 << 20, row_bytes: int = 13, alpha: float = 0.1,
         W: int = 8) -> Workload:
    """W=8, rows of 13 bytes, splits ~ Multinomial(rows, Dirichlet(alpha * 1_W)) per rank."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 4]))
    splits = np.zeros((W, W), dtype=np.int64)
    for r in range(W):
        pi = rng.dirichlet([alpha] * W)
        splits[r] = rng.multinomial(rows, pi / pi.sum())
    inputs = []
    for r in range(W):
        buf = np.empty(rows * row_bytes, dtype=np.uint8)
        random_bits(buf, (seed, 4, r))
        inputs.append(buf)
    return Workload("cfg4", W, row_bytes, splits, inputs, {"alpha": alpha, "rows_per_rank": rows})


def cfg5(seed: int = 0, features: int = 26, batch: int = 8192, lam: float = 3.0,
         max_len: int = 20, key_max: int = 10 ** 7, W: int = 2) -> Workload:
    """W=2 embedding-key exchange; feature f is owned by rank f mod W.

    Per rank: bag lengths L[f, b] = min(Poisson(lam), max_len); one int64 key
    per row (8 B), uniform in [0, key_max).  Input rows ordered by
    (owner rank, feature, bag, position).
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 5]))
    splits = np.zeros((W, W), dtype=np.int64)
    inputs, lengths, kjt = [], [], []
    for r in range(W):
        L = np.minimum(rng.poisson(lam, size=(features, batch)), max_len).astype(np.int64)
        per_feature = L.sum(axis=1)
        keys = rng.integers(0, key_max, size=int(per_feature.sum()), dtype=np.int64)
        kjt.append(keys)
        starts = np.concatenate([[0], np.cumsum(per_feature)])
        blocks = []
        for p in range(W):
            fs = [f for f in range(features) if f % W == p]
            splits[r, p] = per_feature[fs].sum()
            blocks += [keys[starts[f]:starts[f + 1]] for f in fs]
        inputs.append(np.concatenate(blocks).view(np.uint8))
        lengths.append(L)
    return Workload("cfg5", W, 8, splits, inputs,
                    {"features": features, "batch": batch, "lengths": lengths, "kjt_keys": kjt})


def cfg5_lengths(w: Workload) -> Workload:
    """The bag-length exchange that goes with a ``cfg5`` key exchange.

    A keyed-jagged batch sends, beside its keys, the length of every bag:
    per rank, one int32 row (4 B) per (feature, bag), ordered by (owner rank,
    feature, bag) like the keys, so S[r][p] = (features owned by p) x batch.
    Peer p can cut the keys it received from rank r into bags only with these
    lengths: their sum over the rows from r is the number of keys from r.
    """
    if w.name != "cfg5":
        raise ValueError("bag lengths go with a cfg5 workload")
    W, F, B = w.W, w.meta["features"], w.meta["batch"]
    owned = [[f for f in range(F) if f % W == p] for p in range(W)]
    splits = np.array([[len(owned[p]) * B for p in range(W)] for _ in range(W)], dtype=np.int64)
    inputs = [np.ascontiguousarray(np.concatenate([L[fs] for fs in owned]).astype(np.int32))
              .view(np.uint8).reshape(-1) for L in w.meta["lengths"]]
    return Workload("cfg5_lengths", W, 4, splits, inputs, {"features": F, "batch": B})


def dispatch_items(w: Workload):
    """Unsorted items for the fused dispatch of an MoE or embedding-key workload.

    Returns (K, rows, src_rows, keys): per rank, the source rows as bytes and,
    per item, its source row and its key (destination = key // K).
      cfg3: items (token t, choice k) in token-major order, source row t, key =
            the chosen expert (K = experts per rank); with ``dedup``, one
            item per distinct (token, destination) in token-major order, key
            = the destination (K = 1).
      cfg5: items = the keys in feature-major (feature, bag, position) order,
            each its own source row; key = (f mod W) * ceil(F / W) + f // W,
            so that keys order items by (owner, feature).
    Ordering each rank's items stably by key gives exactly ``w.inputs``.
    """
    W = w.W
    if w.name == "cfg3" and w.meta.get("dedup"):
        # one item per distinct (token, destination rank); key = destination
        rows, src, key = w.meta["token_rows"], [], []
        for ch in w.meta["choices"]:
            tokens, topk = ch.shape
            tok = np.repeat(np.arange(tokens), topk)
            dest = ch.reshape(-1) // (w.meta["experts"] // W)
            first = np.unique(tok * W + dest, return_index=True)[1]  # token-major order
            src.append(tok[first].astype(np.int32))
            key.append(dest[first].astype(np.int32))
        return 1, rows, src, key
    if w.name == "cfg3":
        K = w.meta["experts"] // W
        rows = w.meta["token_rows"]
        src, key = [], []
        for ch in w.meta["choices"]:
            tokens, topk = ch.shape
            src.append(np.repeat(np.arange(tokens, dtype=np.int32), topk))
            key.append(ch.reshape(-1).astype(np.int32))
        return K, rows, src, key
    if w.name == "cfg5":
        F = w.meta["features"]
        K = -(-F // W)
        rows, src, key = [], [], []
        for r in range(W):
            per_feature = w.meta["lengths"][r].sum(axis=1)
            f = np.repeat(np.arange(F), per_feature)
            rows.append(w.meta["kjt_keys"][r].view(np.uint8))
            src.append(np.arange(f.size, dtype=np.int32))
            key.append(((f % W) * K + f // W).astype(np.int32))
        return K, rows, src, key
    raise ValueError(f"{w.name} has no dispatch items")


def random_case(seed: int, W: int, row_bytes: int, max_rows: int = 64, mode: str = "uniform") -> Workload:
    """Random splits for property tests.

    ``mode``: ``uniform`` (entries uniform in [0, max_rows]), ``skew``
    (Dirichlet(0.1) shares of up to W*max_rows rows), ``sparse`` (uniform
    entries, each zeroed with probability 1/2), ``empty`` (all zero),
    ``diag`` (only self chunks), ``one`` (a single nonzero entry).
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 6, W, row_bytes]))
    if mode == "uniform":
        S = rng.integers(0, max_rows + 1, size=(W, W))
    elif mode == "skew":
        S = np.stack([rng.multinomial(int(rng.integers(0, W * max_rows + 1)),
                                      (lambda q: q / q.sum())(rng.dirichlet([0.1] * W)))
                      for _ in range(W)])
    elif mode == "sparse":
        S = rng.integers(0, max_rows + 1, size=(W, W)) * (rng.random((W, W)) < 0.5)
    elif mode == "empty":
        S = np.zeros((W, W))
    elif mode == "diag":
        S = np.diag(rng.integers(0, max_rows + 1, size=W))
    elif mode == "one":
        S = np.zeros((W, W))
        S[rng.integers(W), rng.integers(W)] = rng.integers(1, max_rows + 1)
    else:
        raise ValueError(mode)
    S = np.asarray(S, dtype=np.int64)
    inputs = []
    for r in range(W):
        buf = np.empty(int(S[r].sum()) * row_bytes, dtype=np.uint8)
        random_bits(buf, (seed, 6, W, row_bytes, r))
        inputs.append(buf)
    return Workload(f"random-{mode}", W, row_bytes, S, inputs, {"seed": seed})
