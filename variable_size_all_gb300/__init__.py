"""Python binding of the GB300 variable-size all-to-all (``liba2av.so``).

The functions below carry the C ABI's names (``include/a2av.h``) and only
marshal arguments: every step of the exchange -- reading the device splits,
the scans, ``out_splits_offsets``, the copies -- runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams; nothing here falls back
to a CPU or PyTorch implementation, and every call raises if the compiled
library is missing.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIBRARY, build

__all__ = [
    "A2av", "A2avError", "load", "build",
    "a2av_create", "a2av_run", "a2av_combine", "a2av_status", "a2av_destroy", "a2av_set_path",
    "a2av_set_grid", "a2av_last_launch", "a2av_last_dispatch", "a2av_error_string", "a2av_version", "a2av_run_noalloc",
    "a2av_dispatch", "a2av_dispatch_workspace_bytes", "ERR_BAD_INDEX", "MAX_DISPATCH_KEYS",
    "a2av_run_multi", "A2avExchange", "MAX_EXCHANGES", "BoundCall", "a2av_combine_items",
    "COMBINE_WORKSPACE_BYTES",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_BAD_SPLITS", "ERR_TIMEOUT",
    "PATH_AUTO", "PATH_VECTOR", "PATH_BULK", "PATH_STAGED", "MAX_RANKS",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_BAD_SPLITS, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
ERR_BAD_INDEX = -6
MAX_DISPATCH_KEYS = 1024
PATH_AUTO, PATH_VECTOR, PATH_BULK, PATH_STAGED = 0, 1, 2, 3
MAX_RANKS = 32
MAX_EXCHANGES = 4
COMBINE_WORKSPACE_BYTES = 256 + 16 * 32 * 32

_lib = None


class A2avExchange(ctypes.Structure):
    """``a2av_exchange_t``: one exchange of an ``a2av_run_multi`` call."""
    _fields_ = [("in_ptrs", ctypes.POINTER(ctypes.c_void_p)),
                ("in_splits_dev", ctypes.c_void_p),
                ("out_ptrs", ctypes.POINTER(ctypes.c_void_p)),
                ("out_splits_offsets_dev", ctypes.c_void_p),
                ("row_bytes", ctypes.c_int64)]


class A2avError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {a2av_error_string(code)} ({code})")
        self.code = code


def load():
    """The loaded ``liba2av.so`` (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise ImportError(
            f"{LIBRARY} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIBRARY)
    vp, i64, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    pp = ctypes.POINTER(ctypes.c_void_p)
    lib.a2av_create.argtypes = [ci, i64, i64, pp]
    lib.a2av_run.argtypes = [vp, pp, vp, pp, vp, i64, vp]
    lib.a2av_combine.argtypes = [vp, pp, vp, pp, vp, i64, vp]
    lib.a2av_status.argtypes = [vp, vp, ctypes.POINTER(ci)]
    lib.a2av_destroy.argtypes = [vp]
    lib.a2av_set_path.argtypes = [vp, ci]
    lib.a2av_set_grid.argtypes = [vp, ci]
    lib.a2av_last_launch.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci),
                                     ctypes.POINTER(ci)]
    lib.a2av_run_noalloc.argtypes = [ci, i64, i64, pp, vp, pp, vp, i64, vp, ctypes.POINTER(ci)]
    lib.a2av_last_dispatch.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(ci),
                                       ctypes.POINTER(ctypes.c_char_p)]
    i64p = ctypes.POINTER(i64)
    lib.a2av_dispatch_workspace_bytes.argtypes = [ci, ci, i64]
    lib.a2av_dispatch_workspace_bytes.restype = i64
    lib.a2av_dispatch.argtypes = [vp, ci, pp, i64p, pp, pp, i64p, pp, vp, pp, vp, i64, vp, i64, vp]
    lib.a2av_dispatch.restype = ci
    lib.a2av_run_multi.argtypes = [vp, ci, ctypes.POINTER(A2avExchange), vp]
    lib.a2av_combine_items.argtypes = [vp, ci, pp, vp, pp, pp, i64p, pp, i64, vp, i64, vp]
    lib.a2av_combine_items.restype = ci
    lib.a2av_error_string.argtypes = [ci]
    lib.a2av_error_string.restype = ctypes.c_char_p
    lib.a2av_version.argtypes = []
    for f in ("a2av_create", "a2av_run", "a2av_combine", "a2av_status", "a2av_destroy", "a2av_set_path",
              "a2av_set_grid", "a2av_last_launch", "a2av_version", "a2av_run_noalloc",
              "a2av_run_multi"):
        getattr(lib, f).restype = ci
    _lib = lib
    return lib


# ------------------------------------------------ the C ABI, name for name --
def a2av_version() -> int:
    return load().a2av_version()


def a2av_error_string(code: int) -> str:
    return load().a2av_error_string(int(code)).decode()


def a2av_create(world_size: int, in_capacity_rows: int = 0, out_capacity_rows: int = 0):
    """Returns (status, handle); handle is None unless status is OK."""
    h = ctypes.c_void_p()
    rc = load().a2av_create(int(world_size), int(in_capacity_rows), int(out_capacity_rows),
                            ctypes.byref(h))
    return rc, (h if rc == OK else None)


def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * max(len(ptrs), 1))()
    for k, p in enumerate(ptrs):
        arr[k] = int(p) if p else None
    return arr


def a2av_run(handle, in_ptrs, in_splits_dev: int, out_ptrs, out_splits_offsets_dev: int,
             row_bytes: int, stream: int = 0) -> int:
    """Raw entry point: integer device addresses, integer cudaStream_t."""
    return load().a2av_run(handle, _ptr_array(in_ptrs), ctypes.c_void_p(int(in_splits_dev) or None),
                           _ptr_array(out_ptrs),
                           ctypes.c_void_p(int(out_splits_offsets_dev) or None), int(row_bytes),
                           ctypes.c_void_p(int(stream) or None))


def a2av_combine(handle, in_ptrs, dispatch_splits_offsets_dev: int, out_ptrs,
                 out_splits_offsets_dev: int, row_bytes: int, stream: int = 0) -> int:
    """Raw reverse exchange: integer device addresses, integer cudaStream_t."""
    return load().a2av_combine(handle, _ptr_array(in_ptrs),
                               ctypes.c_void_p(int(dispatch_splits_offsets_dev) or None),
                               _ptr_array(out_ptrs),
                               ctypes.c_void_p(int(out_splits_offsets_dev) or None),
                               int(row_bytes), ctypes.c_void_p(int(stream) or None))


def a2av_run_multi(handle, exchanges, stream: int = 0) -> int:
    """``exchanges``: a sequence of (in_ptrs, in_splits_dev, out_ptrs,
    out_splits_offsets_dev, row_bytes), each as for ``a2av_run``."""
    arr = (A2avExchange * max(len(exchanges), 1))()
    keep = []
    for k, (ins, sp, outs, so, rb) in enumerate(exchanges):
        ia, oa = _ptr_array(ins), _ptr_array(outs)
        keep += [ia, oa]
        arr[k] = A2avExchange(ctypes.cast(ia, ctypes.POINTER(ctypes.c_void_p)), int(sp) or None,
                              ctypes.cast(oa, ctypes.POINTER(ctypes.c_void_p)), int(so) or None,
                              int(rb))
    return load().a2av_run_multi(handle, len(exchanges), arr if exchanges else None,
                                 ctypes.c_void_p(int(stream) or None))


def a2av_combine_items(handle, keys_per_peer: int, peer_ptrs, in_splits_dev: int, key_ptrs,
                       sorted_pos_ptrs, items_per_rank, item_out_ptrs, row_bytes: int,
                       workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Raw fused combine: integer device addresses, host lists of counts."""
    return load().a2av_combine_items(
        handle, int(keys_per_peer), _ptr_array(peer_ptrs),
        ctypes.c_void_p(int(in_splits_dev) or None), _ptr_array(key_ptrs),
        _ptr_array(sorted_pos_ptrs), _i64_array(items_per_rank), _ptr_array(item_out_ptrs),
        int(row_bytes), ctypes.c_void_p(int(workspace) or None), int(workspace_bytes),
        ctypes.c_void_p(int(stream) or None))


def a2av_status(handle, stream: int = 0):
    """Returns (status, device_status)."""
    v = ctypes.c_int(0)
    rc = load().a2av_status(handle, ctypes.c_void_p(int(stream) or None), ctypes.byref(v))
    return rc, v.value


def a2av_destroy(handle) -> int:
    return load().a2av_destroy(handle)


def a2av_set_path(handle, path: int) -> int:
    return load().a2av_set_path(handle, int(path))


def a2av_set_grid(handle, ctas_per_sm: int) -> int:
    return load().a2av_set_grid(handle, int(ctas_per_sm))


def a2av_last_launch(handle):
    """Returns (status, path, grid, block) of the handle's last run."""
    p, g, b = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    rc = load().a2av_last_launch(handle, ctypes.byref(p), ctypes.byref(g), ctypes.byref(b))
    return rc, p.value, g.value, b.value


def a2av_last_dispatch(handle):
    """Returns (status, kernels, memsets, copy_kernel) of the handle's last
    a2av_dispatch or a2av_combine_items."""
    k, m, name = ctypes.c_int(), ctypes.c_int(), ctypes.c_char_p()
    rc = load().a2av_last_dispatch(handle, ctypes.byref(k), ctypes.byref(m), ctypes.byref(name))
    return rc, k.value, m.value, (name.value or b"").decode()


def a2av_run_noalloc(world_size: int, in_capacity_rows: int, out_capacity_rows: int, in_ptrs,
                     in_splits_dev: int, out_ptrs, out_splits_offsets_dev: int, row_bytes: int,
                     stream: int = 0, wait: bool = True):
    """The allocation-free entry point (no handle; see include/a2av.h).

    Returns (status, device_status); with ``wait`` False the call is
    asynchronous and device_status is None."""
    v = ctypes.c_int(0)
    rc = load().a2av_run_noalloc(int(world_size), int(in_capacity_rows), int(out_capacity_rows),
                                 _ptr_array(in_ptrs), ctypes.c_void_p(int(in_splits_dev) or None),
                                 _ptr_array(out_ptrs),
                                 ctypes.c_void_p(int(out_splits_offsets_dev) or None),
                                 int(row_bytes), ctypes.c_void_p(int(stream) or None),
                                 ctypes.byref(v) if wait else None)
    return rc, (v.value if wait else None)


def a2av_dispatch_workspace_bytes(world_size: int, keys_per_peer: int,
                                  max_items_per_rank: int) -> int:
    return load().a2av_dispatch_workspace_bytes(int(world_size), int(keys_per_peer),
                                                int(max_items_per_rank))


def _i64_array(values):
    return (ctypes.c_int64 * max(len(values), 1))(*[int(v) for v in values])


def a2av_dispatch(handle, keys_per_peer: int, rows_ptrs, rows_per_rank, src_row_ptrs, key_ptrs,
                  items_per_rank, out_ptrs, out_splits_offsets_dev: int, sorted_pos_ptrs,
                  in_splits_dev: int, row_bytes: int, workspace: int, workspace_bytes: int,
                  stream: int = 0) -> int:
    """Raw fused dispatch: integer device addresses, host lists of counts."""
    return load().a2av_dispatch(
        handle, int(keys_per_peer), _ptr_array(rows_ptrs), _i64_array(rows_per_rank),
        _ptr_array(src_row_ptrs), _ptr_array(key_ptrs), _i64_array(items_per_rank),
        _ptr_array(out_ptrs), ctypes.c_void_p(int(out_splits_offsets_dev) or None),
        _ptr_array(sorted_pos_ptrs), ctypes.c_void_p(int(in_splits_dev) or None),
        int(row_bytes), ctypes.c_void_p(int(workspace) or None), int(workspace_bytes),
        ctypes.c_void_p(int(stream) or None))


# --------------------------------------------------------- torch-facing --
class BoundCall:
    """One library call whose arguments were marshalled once (``A2av.bind_run``,
    ``bind_run_multi``, ``bind_dispatch``).  Calling it enqueues the same
    launch again -- on the stream given at bind time, or on ``stream`` -- with
    the same buffers: the tensors must stay alive and keep their storage, while
    the device data they hold (splits, keys, rows) may change between calls.
    It skips the per-call Python checks and pointer gathering, which cost more
    host time than a small exchange takes on the device."""

    def __init__(self, engine, fn, what, args, stream_index, keep):
        self._engine, self._fn, self._what = engine, fn, what
        self._args, self._si, self._keep = tuple(args), stream_index, keep

    def __call__(self, stream=None):
        args = self._args
        if stream is not None:
            args = list(args)
            args[self._si] = ctypes.c_void_p(A2av._stream(stream) or None)
        rc = self._fn(*args)
        if rc != OK:
            raise A2avError(rc, self._what)


class A2av:
    """One handle over ``world_size`` ranks; tensors in, tensors out.

    ``run(inputs, in_splits, outputs, out_splits_offsets, row_bytes)`` takes
    W CUDA tensors (any dtype, contiguous; ``None`` or empty for a rank
    without a buffer), the int64 [W, W] split matrix on the device, W output
    tensors and the int64 [W, 2, W] out_splits_offsets tensor, and enqueues
    the exchange on ``stream`` (default: torch's current stream).  Device
    detected errors are read with ``status()``.
    """

    def __init__(self, world_size: int, in_capacity_rows: int = 0, out_capacity_rows: int = 0,
                 path: int = PATH_AUTO, ctas_per_sm: int = 0):
        rc, h = a2av_create(world_size, in_capacity_rows, out_capacity_rows)
        if rc != OK:
            raise A2avError(rc, "a2av_create")
        self.handle, self.world_size, self._path = h, int(world_size), int(path)
        if path != PATH_AUTO:
            self._check(a2av_set_path(h, path), "a2av_set_path")
        if ctas_per_sm:
            self._check(a2av_set_grid(h, ctas_per_sm), "a2av_set_grid")

    @staticmethod
    def _check(rc, what):
        if rc != OK:
            raise A2avError(rc, what)

    @staticmethod
    def _stream(stream):
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        return int(getattr(stream, "cuda_stream", stream))

    def _buffers(self, tensors, what):
        """Pointer array for W buffers; True when one lives in pinned host memory."""
        W = self.world_size
        if len(tensors) != W:
            raise ValueError(f"{what}: expected {W} buffers, got {len(tensors)}")
        arr = (ctypes.c_void_p * W)()
        host = False
        for k, t in enumerate(tensors):
            if t is None or t.numel() == 0:
                continue
            if not t.is_contiguous():
                raise ValueError(f"{what}: buffers must be contiguous")
            if t.is_cuda:
                arr[k] = t.data_ptr()
            elif t.is_pinned():
                arr[k] = t.data_ptr()
                host = True
            else:
                raise ValueError(f"{what}: buffers must be CUDA tensors or pinned host tensors")
        return arr, host

    @staticmethod
    def _matrix(t, shape, name):
        import torch
        if (not isinstance(t, torch.Tensor) or t.dtype != torch.int64 or not t.is_cuda
                or tuple(t.shape) != shape or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA int64 tensor of shape {shape}")
        return ctypes.c_void_p(t.data_ptr())

    def _launch_args(self, inputs, splits, outputs, out_splits_offsets, row_bytes, stream,
                     split_shape):
        """The C call's arguments (stream last) and whether a buffer is host memory."""
        W = self.world_size
        sp = self._matrix(splits, split_shape, "splits")
        so = self._matrix(out_splits_offsets, (W, 2, W), "out_splits_offsets")
        ins, host_in = self._buffers(inputs, "inputs")
        outs, host_out = self._buffers(outputs, "outputs")
        st = ctypes.c_void_p(self._stream(stream) or None)
        return [self.handle, ins, sp, outs, so, int(row_bytes), st], host_in or host_out

    def _launch(self, fn, what, inputs, splits, outputs, out_splits_offsets, row_bytes, stream,
                split_shape):
        # (buffers in pinned host memory are routed to the vector engine by
        # the library itself)
        args, _ = self._launch_args(inputs, splits, outputs, out_splits_offsets, row_bytes,
                                    stream, split_shape)
        self._check(fn(*args), what)

    def bind_run(self, inputs, in_splits, outputs, out_splits_offsets, row_bytes: int,
                 stream=None) -> BoundCall:
        """``run`` marshalled once: returns a BoundCall that re-enqueues the
        exchange on these buffers."""
        W = self.world_size
        args, _ = self._launch_args(inputs, in_splits, outputs, out_splits_offsets, row_bytes,
                                    stream, (W, W))
        keep = (inputs, in_splits, outputs, out_splits_offsets)
        return BoundCall(self, load().a2av_run, "a2av_run", args, len(args) - 1, keep)

    def run(self, inputs, in_splits, outputs, out_splits_offsets, row_bytes: int, stream=None):
        W = self.world_size
        self._launch(load().a2av_run, "a2av_run", inputs, in_splits, outputs, out_splits_offsets,
                     row_bytes, stream, (W, W))

    def run_multi(self, exchanges, stream=None):
        """Several exchanges over the same ranks in one launch (see
        include/a2av.h, a2av_run_multi).  ``exchanges``: a sequence of
        (inputs, in_splits, outputs, out_splits_offsets, row_bytes), each as
        for ``run``."""
        args, _, _ = self._multi_args(exchanges, stream)
        self._check(load().a2av_run_multi(*args), "a2av_run_multi")

    def _multi_args(self, exchanges, stream):
        W = self.world_size
        if not 1 <= len(exchanges) <= MAX_EXCHANGES:
            raise ValueError(f"run_multi takes 1..{MAX_EXCHANGES} exchanges")
        arr = (A2avExchange * len(exchanges))()
        keep, host = [arr], False
        for k, (inputs, splits, outputs, so, rb) in enumerate(exchanges):
            sp = self._matrix(splits, (W, W), "splits")
            sop = self._matrix(so, (W, 2, W), "out_splits_offsets")
            ins, h_in = self._buffers(inputs, "inputs")
            outs, h_out = self._buffers(outputs, "outputs")
            host = host or h_in or h_out
            keep += [ins, outs]
            arr[k] = A2avExchange(ctypes.cast(ins, ctypes.POINTER(ctypes.c_void_p)), sp,
                                  ctypes.cast(outs, ctypes.POINTER(ctypes.c_void_p)), sop,
                                  int(rb))
        st = ctypes.c_void_p(self._stream(stream) or None)
        return [self.handle, len(exchanges), arr, st], host, keep

    def bind_run_multi(self, exchanges, stream=None) -> BoundCall:
        """``run_multi`` marshalled once."""
        args, _, keep = self._multi_args(exchanges, stream)
        return BoundCall(self, load().a2av_run_multi, "a2av_run_multi", args, 3,
                         keep + [exchanges])

    def combine(self, inputs, dispatch_splits_offsets, outputs, out_splits_offsets,
                row_bytes: int, stream=None):
        """The reverse exchange: send every received chunk back to its source
        rank; ``dispatch_splits_offsets`` is the [W, 2, W] tensor a previous
        ``run`` wrote."""
        W = self.world_size
        self._launch(load().a2av_combine, "a2av_combine", inputs, dispatch_splits_offsets,
                     outputs, out_splits_offsets, row_bytes, stream, (W, 2, W))

    def dispatch(self, rows, src_rows, keys, keys_per_peer: int, outputs, out_splits_offsets,
                 sorted_pos, row_bytes: int, in_splits=None, workspace=None, stream=None,
                 _bind=False):
        """Fused dispatch: group each rank's items by key on the device and
        exchange their rows (see include/a2av.h, a2av_dispatch).

        ``rows[r]``: rank r's source rows (uint8 CUDA tensor, a multiple of
        ``row_bytes``); ``src_rows[r]`` / ``keys[r]``: int32 CUDA tensors, one
        entry per item; ``sorted_pos[r]``: int64 CUDA tensor receiving each
        item's position in key order; ``in_splits``: optional int64 [W, W]
        receiving the split matrix.  ``workspace`` defaults to a buffer the
        object keeps (torch allocation, sized by the largest item count)."""
        import torch
        W = self.world_size
        for name, ts, dt in (("src_rows", src_rows, torch.int32), ("keys", keys, torch.int32),
                             ("sorted_pos", sorted_pos, torch.int64)):
            if len(ts) != W:
                raise ValueError(f"{name}: expected {W} tensors")
            for t in ts:
                if t is not None and t.numel() and (t.dtype != dt or not t.is_cuda
                                                    or not t.is_contiguous()):
                    raise ValueError(f"{name} must be contiguous CUDA {dt} tensors")
        if not (isinstance(out_splits_offsets, torch.Tensor) and out_splits_offsets.is_cuda
                and out_splits_offsets.dtype == torch.int64
                and tuple(out_splits_offsets.shape) == (W, 2, W)
                and out_splits_offsets.is_contiguous()):
            raise ValueError(f"out_splits_offsets must be a contiguous CUDA int64 [{W}, 2, {W}]")
        if in_splits is not None and (in_splits.dtype != torch.int64 or not in_splits.is_cuda
                                      or tuple(in_splits.shape) != (W, W)):
            raise ValueError(f"in_splits must be a CUDA int64 [{W}, {W}] tensor")
        items = [0 if t is None else t.numel() for t in keys]
        if any((0 if s is None else s.numel()) != m for s, m in zip(src_rows, items)):
            raise ValueError("src_rows and keys must have one entry per item")
        if any((0 if t is None else t.numel()) != m for t, m in zip(sorted_pos, items)):
            raise ValueError("sorted_pos must have one entry per item")
        need = a2av_dispatch_workspace_bytes(W, keys_per_peer, max(items))
        if need < 0:
            raise A2avError(ERR_UNSUPPORTED, "a2av_dispatch_workspace_bytes")
        if workspace is None:
            ws = getattr(self, "_workspace", None)
            if ws is None or ws.numel() < need:
                ws = torch.empty(need, dtype=torch.uint8, device="cuda")
                self._workspace = ws
            workspace = ws
        n_rows = [0 if t is None else t.numel() // int(row_bytes) for t in rows]
        ptr = lambda ts: [0 if t is None or t.numel() == 0 else t.data_ptr() for t in ts]
        rows_arr, host_rows = self._buffers(rows, "rows")
        outs_arr, host_outs = self._buffers(outputs, "outputs")
        if host_rows or host_outs:
            raise ValueError("a2av_dispatch takes device buffers only")
        args = [self.handle, int(keys_per_peer), _ptr_array(list(rows_arr)), _i64_array(n_rows),
                _ptr_array(ptr(src_rows)), _ptr_array(ptr(keys)), _i64_array(items),
                _ptr_array(list(outs_arr)), ctypes.c_void_p(out_splits_offsets.data_ptr()),
                _ptr_array(ptr(sorted_pos)),
                ctypes.c_void_p(None if in_splits is None else in_splits.data_ptr()),
                int(row_bytes), ctypes.c_void_p(workspace.data_ptr()), int(workspace.numel()),
                ctypes.c_void_p(self._stream(stream) or None)]
        if _bind:
            keep = (rows, src_rows, keys, outputs, out_splits_offsets, sorted_pos, in_splits,
                    workspace)
            return BoundCall(self, load().a2av_dispatch, "a2av_dispatch", args, 14, keep)
        self._check(load().a2av_dispatch(*args), "a2av_dispatch")

    def bind_dispatch(self, rows, src_rows, keys, keys_per_peer: int, outputs,
                      out_splits_offsets, sorted_pos, row_bytes: int, in_splits=None,
                      workspace=None, stream=None) -> BoundCall:
        """``dispatch`` marshalled once: the item counts are fixed at bind time
        (the keys and source rows themselves may change between calls)."""
        return self.dispatch(rows, src_rows, keys, keys_per_peer, outputs, out_splits_offsets,
                             sorted_pos, row_bytes, in_splits, workspace, stream, _bind=True)

    def bind_combine_items(self, peers, in_splits, keys, sorted_pos, keys_per_peer: int,
                           item_out, row_bytes: int, workspace=None, stream=None) -> BoundCall:
        """``combine_items`` marshalled once (see BoundCall)."""
        return self.combine_items(peers, in_splits, keys, sorted_pos, keys_per_peer, item_out,
                                  row_bytes, workspace, stream, _bind=True)

    def combine_items(self, peers, in_splits, keys, sorted_pos, keys_per_peer: int, item_out,
                      row_bytes: int, workspace=None, stream=None, _bind=False):
        """The fused combine (see include/a2av.h, a2av_combine_items): every
        item's row from the peers' dispatch-layout buffers back to row i of
        ``item_out[r]``.  ``in_splits``, ``keys`` and ``sorted_pos`` as a
        dispatch took or wrote them."""
        import torch
        W = self.world_size
        sp = self._matrix(in_splits, (W, W), "in_splits")
        for name, ts, dt in (("keys", keys, torch.int32), ("sorted_pos", sorted_pos, torch.int64)):
            if len(ts) != W:
                raise ValueError(f"{name}: expected {W} tensors")
            for t in ts:
                if t is not None and t.numel() and (t.dtype != dt or not t.is_cuda
                                                    or not t.is_contiguous()):
                    raise ValueError(f"{name} must be contiguous CUDA {dt} tensors")
        items = [0 if t is None else t.numel() for t in keys]
        if any((0 if t is None else t.numel()) != m for t, m in zip(sorted_pos, items)):
            raise ValueError("sorted_pos must have one entry per item")
        if any((0 if t is None else t.numel()) < m * int(row_bytes)
               for t, m in zip(item_out, items)):
            raise ValueError("item_out[r] must hold one row per item of rank r")
        if workspace is None:
            ws = getattr(self, "_combine_workspace", None)
            if ws is None:
                ws = torch.empty(COMBINE_WORKSPACE_BYTES, dtype=torch.uint8, device="cuda")
                self._combine_workspace = ws
            workspace = ws
        peer_arr, host_p = self._buffers(peers, "peers")
        out_arr, host_o = self._buffers(item_out, "item_out")
        if host_p or host_o:
            raise ValueError("a2av_combine_items takes device buffers only")
        ptr = lambda ts: [0 if t is None or t.numel() == 0 else t.data_ptr() for t in ts]
        args = [self.handle, int(keys_per_peer), _ptr_array(list(peer_arr)), sp,
                _ptr_array(ptr(keys)), _ptr_array(ptr(sorted_pos)), _i64_array(items),
                _ptr_array(list(out_arr)), int(row_bytes), ctypes.c_void_p(workspace.data_ptr()),
                int(workspace.numel()), ctypes.c_void_p(self._stream(stream) or None)]
        if _bind:
            keep = (peers, in_splits, keys, sorted_pos, item_out, workspace)
            return BoundCall(self, load().a2av_combine_items, "a2av_combine_items", args, 11, keep)
        self._check(load().a2av_combine_items(*args), "a2av_combine_items")

    def status(self, stream=None) -> int:
        rc, v = a2av_status(self.handle, self._stream(stream))
        self._check(rc, "a2av_status")
        return v

    def last_launch(self):
        rc, p, g, b = a2av_last_launch(self.handle)
        self._check(rc, "a2av_last_launch")
        return {"path": p, "grid": g, "block": b}

    def last_dispatch(self):
        """What the last ``dispatch`` or ``combine_items`` enqueued."""
        rc, k, m, name = a2av_last_dispatch(self.handle)
        self._check(rc, "a2av_last_dispatch")
        return {"kernels": k, "memsets": m, "copy_kernel": name}

    def close(self):
        if self.handle is not None:
            a2av_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
