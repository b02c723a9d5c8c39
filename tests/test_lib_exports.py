"""The C-ABI library builds, loads and exports every entry point include/moe.h
declares (CPU only: no compute calls, no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT
from sparse_mixture_experts_54_b300 import _lib, build

HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("moe_create", "moe_route", "moe_forward", "moe_destroy", "moe_status", "moe_workspace_bytes"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(_lib.SIGNATURES), "binding and header disagree"
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in names:
        assert name in exported, f"{name} not exported (C linkage)"
        assert getattr(lib, name) is not None


def test_library_is_built_for_sm_103a(lib):
    # the fatbin holds a cubin for sm_103a; cuobjdump only lists the ELF names here
    out = subprocess.run(["/usr/local/cuda/bin/cuobjdump", "--list-elf", _lib.LIB_PATH], capture_output=True,
                         text=True)
    assert "sm_103a" in out.stdout


def test_calls_without_context_fail_cleanly(lib):
    assert _lib.moe_status(None) == _lib.MOE_ERR_INVALID
    assert _lib.moe_forward(None, 0, 0, 0, 0, 0, 0, 4, 0) == _lib.MOE_ERR_INVALID
    assert _lib.moe_route(None, 0, 0, 4, 0, 0, 0, 0, 0, 0) == _lib.MOE_ERR_INVALID
    assert _lib.moe_set_option(None, _lib.MOE_OPT_DECODE_MAX_T, 4) == _lib.MOE_ERR_INVALID
    assert _lib.moe_workspace_bytes(None, 10) == 0
    _lib.moe_destroy(None)
    assert _lib.moe_error_string(_lib.MOE_ERR_TIMEOUT) == "MOE_ERR_TIMEOUT"
    assert _lib.moe_error_string(12345) == "MOE_ERR_UNKNOWN"


def test_create_rejects_bad_shapes(lib):
    # rejected on argument checks, before any CUDA call
    assert not _lib.moe_create(0, 14336, 8, 2)
    assert not _lib.moe_create(4096, 14336, 8, 9)
    assert not _lib.moe_create(4100, 14336, 8, 2)      # d % 8 != 0
    assert not _lib.moe_create(4096, 14336, 64, 2)     # more than 32 experts


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load()


def test_binding_wraps_every_entry_point():
    # the Python binding has a same-named function for every declared entry point
    for name in declared_functions():
        assert callable(getattr(_lib, name, None)), f"_lib.{name} missing"
