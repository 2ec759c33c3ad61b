"""CPU oracle for the variable-size all-to-all (a2av) -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The library's product path never calls it, and it shares
no code with the CUDA path: the arithmetic lives in ``a2av_oracle.c`` (plain C,
a triple loop of ``memcpy`` per row, sequential scans), compiled with gcc and
called through ctypes here.  See ``a2av_oracle.c`` for the definition it
implements and the passages it follows.

Every function here pins to the plain definition of all_to_all_vdev ("[a2av]
Improve tuning for 4 GPUs", pytorch PR 154580, section "Problem"); the tests
under ``tests/test_oracle_*.py`` check it against brute force, closed forms and
invariants.  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "a2av_oracle.c")
LIBRARY = os.path.join(HERE, "liba2av_oracle.so")

OK = 0
INVALID_ARG = -1
BAD_SPLITS = -4
BAD_INDEX = -6

_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)


def build(source: str = SOURCE, library: str = LIBRARY) -> str:
    """Compile the oracle with gcc into a shared library (no CUDA involved)."""
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", "-fPIC", "-shared",
           "-o", library, source]
    subprocess.run(cmd, check=True)
    return library


def _bind(lib):
    vpp = ctypes.POINTER(ctypes.c_void_p)
    lib.a2av_oracle.argtypes = [ctypes.c_int, vpp, _i64p, vpp, _i64p, ctypes.c_int64,
                                ctypes.c_int64, ctypes.c_int64]
    lib.a2av_oracle_dest.argtypes = [ctypes.c_int, ctypes.c_int, vpp, _i64p, ctypes.c_void_p,
                                     _i64p, ctypes.c_int64]
    lib.a2av_oracle_check.argtypes = [ctypes.c_int, _i64p, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, vpp, vpp]
    lib.a2av_oracle_row_source.argtypes = [ctypes.c_int, _i64p, ctypes.c_int, ctypes.c_int64,
                                           ctypes.POINTER(ctypes.c_int), _i64p]
    lib.a2av_oracle_combine.argtypes = [ctypes.c_int, vpp, _i64p, vpp, _i64p, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64]
    lib.a2av_oracle_dispatch.argtypes = [ctypes.c_int, ctypes.c_int, vpp, _i64p, vpp, vpp, _i64p,
                                         vpp, _i64p, vpp, _i64p, ctypes.c_int64, ctypes.c_int64]
    lib.a2av_oracle_combine_items.argtypes = [ctypes.c_int, ctypes.c_int, vpp, _i64p, vpp, vpp,
                                              _i64p, vpp, ctypes.c_int64]
    for f in (lib.a2av_oracle, lib.a2av_oracle_dest, lib.a2av_oracle_check,
              lib.a2av_oracle_row_source, lib.a2av_oracle_combine, lib.a2av_oracle_dispatch,
              lib.a2av_oracle_combine_items):
        f.restype = ctypes.c_int
    return lib


def load(library: str | None = None):
    """Load (building first if needed) the oracle library.

    With ``library`` given, load that file instead (used by the tests that
    plant mistakes in a copy of the oracle and check that the pins catch
    them)."""
    global _lib
    if library is not None:
        return _bind(ctypes.CDLL(library))
    with _lock:
        if _lib is None:
            if (not os.path.exists(LIBRARY)
                    or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
                build()
            _lib = _bind(ctypes.CDLL(LIBRARY))
    return _lib


def _ptrs(bufs):
    arr = (ctypes.c_void_p * len(bufs))()
    for k, b in enumerate(bufs):
        arr[k] = None if b is None else b.ctypes.data
    return arr


def _splits(S, W):
    S = np.ascontiguousarray(S, dtype=np.int64)
    if S.shape != (W, W):
        raise ValueError(f"splits must be [{W}][{W}], got {S.shape}")
    return S


class Oracle:
    """numpy-facing wrapper over the C oracle (one loaded library)."""

    def __init__(self, library: str | None = None):
        self.lib = load(library)

    def run(self, inputs, splits, outputs, out_splits_offsets, row_bytes,
            in_capacity_rows=0, out_capacity_rows=0) -> int:
        """The whole exchange into caller-provided numpy buffers; returns the status."""
        W = len(inputs)
        S = _splits(splits, W)
        assert out_splits_offsets.dtype == np.int64 and out_splits_offsets.size == 2 * W * W
        assert out_splits_offsets.flags.c_contiguous
        return self.lib.a2av_oracle(W, _ptrs(inputs), S.ctypes.data_as(_i64p), _ptrs(outputs),
                                    out_splits_offsets.ctypes.data_as(_i64p), int(row_bytes),
                                    int(in_capacity_rows), int(out_capacity_rows))

    def dest(self, inputs, splits, p, out_p, out_so_p, row_bytes) -> int:
        """Peer p's output alone (out_p / out_so_p may be None to skip)."""
        W = len(inputs)
        S = _splits(splits, W)
        so = None if out_so_p is None else out_so_p.ctypes.data_as(_i64p)
        buf = None if out_p is None else out_p.ctypes.data
        return self.lib.a2av_oracle_dest(W, int(p), _ptrs(inputs), S.ctypes.data_as(_i64p), buf,
                                         so, int(row_bytes))

    def check(self, splits, row_bytes, in_capacity_rows=0, out_capacity_rows=0,
              inputs=None, outputs=None) -> int:
        S = np.ascontiguousarray(splits, dtype=np.int64)
        W = S.shape[0]
        vi = None if inputs is None else _ptrs(inputs)
        vo = None if outputs is None else _ptrs(outputs)
        return self.lib.a2av_oracle_check(W, S.ctypes.data_as(_i64p), int(row_bytes),
                                          int(in_capacity_rows), int(out_capacity_rows), vi, vo)

    def row_source(self, splits, p, k):
        """(source rank, source row) of row k of peer p's output, or None."""
        S = np.ascontiguousarray(splits, dtype=np.int64)
        r = ctypes.c_int()
        i = ctypes.c_int64()
        rc = self.lib.a2av_oracle_row_source(S.shape[0], S.ctypes.data_as(_i64p), int(p), int(k),
                                             ctypes.byref(r), ctypes.byref(i))
        return None if rc != OK else (r.value, i.value)

    def combine(self, inputs, dispatch_so, outputs, out_splits_offsets, row_bytes,
                in_capacity_rows=0, out_capacity_rows=0) -> int:
        """The reverse exchange, splits read from a dispatch's [W][2][W] out_splits_offsets."""
        W = len(inputs)
        dso = np.ascontiguousarray(dispatch_so, dtype=np.int64)
        assert dso.size == 2 * W * W and out_splits_offsets.size == 2 * W * W
        assert out_splits_offsets.dtype == np.int64 and out_splits_offsets.flags.c_contiguous
        return self.lib.a2av_oracle_combine(W, _ptrs(inputs), dso.ctypes.data_as(_i64p),
                                            _ptrs(outputs), out_splits_offsets.ctypes.data_as(_i64p),
                                            int(row_bytes), int(in_capacity_rows),
                                            int(out_capacity_rows))

    def dispatch(self, K, rows, src_rows, keys, outputs, out_splits_offsets, sorted_pos,
                 row_bytes, in_splits=None, out_capacity_rows=0) -> int:
        """Fused dispatch preparation (see a2av_oracle.c); numpy arrays in and out."""
        W = len(rows)
        src = [np.ascontiguousarray(x, dtype=np.int32) for x in src_rows]
        key = [np.ascontiguousarray(x, dtype=np.int32) for x in keys]
        n_rows = (ctypes.c_int64 * W)(*[r.size // int(row_bytes) for r in rows])
        n_items = (ctypes.c_int64 * W)(*[k.size for k in key])
        assert all(p.dtype == np.int64 and p.size == k.size for p, k in zip(sorted_pos, key))
        isp = None if in_splits is None else in_splits.ctypes.data_as(_i64p)
        return self.lib.a2av_oracle_dispatch(
            W, int(K), _ptrs(rows), n_rows, _ptrs(src), _ptrs(key), n_items, _ptrs(outputs),
            out_splits_offsets.ctypes.data_as(_i64p), _ptrs(sorted_pos), isp, int(row_bytes),
            int(out_capacity_rows))

    def combine_items(self, K, expert, S, keys, sorted_pos, item_out, row_bytes) -> int:
        """The fused combine (see a2av_oracle.c): each item's row from the
        dispatch-layout buffers ``expert`` back into ``item_out`` in item order."""
        W = len(expert)
        S = _splits(S, W)
        key = [np.ascontiguousarray(x, dtype=np.int32) for x in keys]
        pos = [np.ascontiguousarray(x, dtype=np.int64) for x in sorted_pos]
        n_items = (ctypes.c_int64 * W)(*[k.size for k in key])
        return self.lib.a2av_oracle_combine_items(
            W, int(K), _ptrs(expert), S.ctypes.data_as(_i64p), _ptrs(key), _ptrs(pos), n_items,
            _ptrs(item_out), int(row_bytes))

    def combine_items_exchange(self, K, expert, S, keys, sorted_pos, row_bytes):
        """Return the item-order rows of a fused combine (raises if rejected)."""
        outs = [np.empty(np.asarray(k).size * row_bytes, np.uint8) for k in keys]
        rc = self.combine_items(K, expert, S, keys, sorted_pos, outs, row_bytes)
        if rc != OK:
            raise ValueError(f"oracle rejected the combine (status {rc})")
        return outs

    def dispatch_exchange(self, K, rows, src_rows, keys, row_bytes):
        """Return (outputs, out_splits_offsets, sorted_pos, S) of a fused dispatch."""
        W = len(rows)
        S = np.zeros((W, W), np.int64)
        for r in range(W):  # output sizes only
            for k in np.asarray(keys[r]).reshape(-1):
                S[r, int(k) // K] += 1
        outs = [np.empty(int(S[:, p].sum()) * row_bytes, np.uint8) for p in range(W)]
        so = np.empty((W, 2, W), np.int64)
        pos = [np.empty(np.asarray(k).size, np.int64) for k in keys]
        isp = np.empty((W, W), np.int64)
        rc = self.dispatch(K, rows, src_rows, keys, outs, so, pos, row_bytes, isp)
        if rc != OK:
            raise ValueError(f"oracle rejected the dispatch (status {rc})")
        return outs, so, pos, isp

    # ---- convenience: allocate outputs of exactly the received size -------
    def exchange(self, inputs, splits, row_bytes):
        """Return (outputs, out_splits_offsets[W][2][W]) for valid splits."""
        W = len(inputs)
        S = _splits(splits, W)
        outs = [np.empty(int(S[:, p].sum()) * row_bytes, dtype=np.uint8) for p in range(W)]
        so = np.empty((W, 2, W), dtype=np.int64)
        rc = self.run(inputs, S, outs, so, row_bytes)
        if rc != OK:
            raise ValueError(f"oracle rejected the splits (status {rc})")
        return outs, so

    def exchange_back(self, inputs, dispatch_so, row_bytes):
        """Return (outputs, out_splits_offsets) of the reverse exchange."""
        W = len(inputs)
        dso = np.ascontiguousarray(dispatch_so, dtype=np.int64).reshape(W, 2, W)
        outs = [np.empty(int(dso[:, 0, r].sum()) * row_bytes, dtype=np.uint8) for r in range(W)]
        so = np.empty((W, 2, W), dtype=np.int64)
        rc = self.combine(inputs, dso, outs, so, row_bytes)
        if rc != OK:
            raise ValueError(f"oracle rejected the splits (status {rc})")
        return outs, so


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
