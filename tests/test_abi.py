"""The C ABI without a GPU: the library builds, loads and exports every
symbol include/a2av.h declares; host-side argument checks answer before any
CUDA call."""
import ctypes
import os
import re

import pytest

import variable_size_all_gb300 as a2av

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    a2av.build()
    return a2av.load()


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(a2av_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for required in ("a2av_create", "a2av_run", "a2av_status", "a2av_destroy"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
        assert hasattr(a2av, name), f"{name} has no Python binding of the same name"


def test_host_checks_without_gpu(lib):
    assert a2av.a2av_version() >= 10000
    assert a2av.a2av_error_string(a2av.ERR_BAD_SPLITS).startswith("invalid split")
    assert a2av.a2av_error_string(12345) == "unknown status"
    for code in (a2av.ERR_INVALID_ARG, a2av.ERR_UNSUPPORTED, a2av.ERR_CUDA, a2av.ERR_BAD_SPLITS,
                 a2av.ERR_TIMEOUT, a2av.ERR_BAD_INDEX):
        assert a2av.a2av_error_string(code) != "unknown status", code
    assert "out of range" in a2av.a2av_error_string(a2av.ERR_BAD_INDEX)
    assert a2av.a2av_create(0)[0] == a2av.ERR_INVALID_ARG
    assert a2av.a2av_create(a2av.MAX_RANKS + 1)[0] == a2av.ERR_UNSUPPORTED
    assert a2av.a2av_create(2, -1, 0)[0] == a2av.ERR_INVALID_ARG
    assert lib.a2av_create(2, 0, 0, None) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run(None, [], 0, [], 0, 1) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_destroy(None) == a2av.OK
    assert a2av.a2av_set_path(None, 0) == a2av.ERR_INVALID_ARG
    assert a2av.a2av_last_launch(None)[0] == a2av.ERR_INVALID_ARG
    assert a2av.a2av_last_dispatch(None)[0] == a2av.ERR_INVALID_ARG
    assert a2av.a2av_run_multi(None, []) == a2av.ERR_INVALID_ARG
    assert lib.a2av_run_multi(None, 1, None, None) == a2av.ERR_INVALID_ARG


def test_create_without_device_is_a_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert a2av.a2av_create(4)[0] == a2av.ERR_CUDA


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(a2av, "_lib", None)
    monkeypatch.setattr(a2av, "LIBRARY", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        a2av.load()
