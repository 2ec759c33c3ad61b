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
    "a2av_set_grid", "a2av_last_launch", "a2av_error_string", "a2av_version", "a2av_run_noalloc",
    "OK", "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_BAD_SPLITS", "ERR_TIMEOUT",
    "PATH_AUTO", "PATH_VECTOR", "PATH_BULK", "PATH_STAGED", "MAX_RANKS",
]

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_BAD_SPLITS, ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
PATH_AUTO, PATH_VECTOR, PATH_BULK, PATH_STAGED = 0, 1, 2, 3
MAX_RANKS = 32

_lib = None


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
    lib.a2av_error_string.argtypes = [ci]
    lib.a2av_error_string.restype = ctypes.c_char_p
    lib.a2av_version.argtypes = []
    for f in ("a2av_create", "a2av_run", "a2av_combine", "a2av_status", "a2av_destroy", "a2av_set_path",
              "a2av_set_grid", "a2av_last_launch", "a2av_version", "a2av_run_noalloc"):
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


# --------------------------------------------------------- torch-facing --
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
        self.handle, self.world_size = h, int(world_size)
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
        import torch
        if len(tensors) != self.world_size:
            raise ValueError(f"{what}: expected {self.world_size} buffers, got {len(tensors)}")
        ptrs = []
        for t in tensors:
            if t is None or t.numel() == 0:
                ptrs.append(0)
                continue
            if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{what}: buffers must be contiguous CUDA tensors")
            ptrs.append(t.data_ptr())
        return ptrs

    def run(self, inputs, in_splits, outputs, out_splits_offsets, row_bytes: int, stream=None):
        import torch
        W = self.world_size
        for t, shape, name in ((in_splits, (W, W), "in_splits"),
                               (out_splits_offsets, (W, 2, W), "out_splits_offsets")):
            if (not isinstance(t, torch.Tensor) or t.dtype != torch.int64 or not t.is_cuda
                    or tuple(t.shape) != shape or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA int64 tensor of shape {shape}")
        rc = a2av_run(self.handle, self._buffers(inputs, "inputs"), in_splits.data_ptr(),
                      self._buffers(outputs, "outputs"), out_splits_offsets.data_ptr(),
                      row_bytes, self._stream(stream))
        self._check(rc, "a2av_run")

    def combine(self, inputs, dispatch_splits_offsets, outputs, out_splits_offsets,
                row_bytes: int, stream=None):
        """The reverse exchange: send every received chunk back to its source
        rank; ``dispatch_splits_offsets`` is the [W, 2, W] tensor a previous
        ``run`` wrote."""
        import torch
        W = self.world_size
        for t, name in ((dispatch_splits_offsets, "dispatch_splits_offsets"),
                        (out_splits_offsets, "out_splits_offsets")):
            if (not isinstance(t, torch.Tensor) or t.dtype != torch.int64 or not t.is_cuda
                    or tuple(t.shape) != (W, 2, W) or not t.is_contiguous()):
                raise ValueError(f"{name} must be a contiguous CUDA int64 tensor of shape "
                                 f"{(W, 2, W)}")
        rc = a2av_combine(self.handle, self._buffers(inputs, "inputs"),
                          dispatch_splits_offsets.data_ptr(), self._buffers(outputs, "outputs"),
                          out_splits_offsets.data_ptr(), row_bytes, self._stream(stream))
        self._check(rc, "a2av_combine")

    def status(self, stream=None) -> int:
        rc, v = a2av_status(self.handle, self._stream(stream))
        self._check(rc, "a2av_status")
        return v

    def last_launch(self):
        rc, p, g, b = a2av_last_launch(self.handle)
        self._check(rc, "a2av_last_launch")
        return {"path": p, "grid": g, "block": b}

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
