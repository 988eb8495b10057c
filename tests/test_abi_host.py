"""The C ABI library loads, exports every function include/h2o.h declares,
and rejects bad arguments on the host before touching a device (CPU only:
none of these calls reaches a kernel)."""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import pytest

import h2o_heavy_hitter_decode_gb300 as h2o
from h2o_heavy_hitter_decode_gb300 import build as hbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    hbuild.build()
    return h2o.lib()


def test_header_declares_the_boundary():
    names = h2o.declared_functions()
    for n in ("h2o_cache_create", "h2o_prefill", "h2o_decode_step", "h2o_decode_steps", "h2o_cache_export",
              "h2o_cache_import", "h2o_cache_workspace_bytes", "h2o_get_error", "h2o_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", h2o.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = [n for n in h2o.declared_functions() if n not in exported]
    assert not missing, missing
    for n in h2o.declared_functions():
        getattr(L, n)  # resolvable through ctypes too


def test_build_targets_sm103a_only(L):
    """Every translation unit is compiled for sm_103a and nothing else (the
    device-side check of what actually loads is in test_gpu_arch.py)."""
    assert hbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert L.h2o_build_arch() == 1030


def test_status_strings(L):
    for s in range(7):
        assert L.h2o_status_str(s)
    assert L.h2o_status_str(0) == b"ok"


def test_bad_shapes_rejected_on_host(L):
    ws = C.c_void_p(256)  # never dereferenced: the shape check fails first
    h = C.c_void_p()
    assert L.h2o_cache_create(0, 1, 64, 1, 1, 0, ws, None, C.byref(h)) == 1
    assert L.h2o_cache_create(1, 1, 64, 0, 0, 0, ws, None, C.byref(h)) == 1
    assert L.h2o_cache_create(1, 1, 64, -1, 2, 0, ws, None, C.byref(h)) == 1
    assert L.h2o_cache_create(1, 1, 64, 1, 1, 7, ws, None, C.byref(h)) == 1
    assert L.h2o_cache_create(1, 1, 96, 1, 1, 0, ws, None, C.byref(h)) == 6  # d not 64/128
    assert L.h2o_cache_create(1, 1, 64, 1, 1, 0, None, None, C.byref(h)) == 1  # no workspace
    assert L.h2o_cache_create(1, 1, 64, 1, 1, 0, C.c_void_p(260), None, C.byref(h)) == 1  # misaligned
    assert L.h2o_cache_create(1, 1, 64, 1, 1, 0, ws, None, None) == 1
    assert L.h2o_cache_workspace_bytes(0, 1, 64, 1, 1, 0) == 0
    assert L.h2o_cache_workspace_bytes(1, 1, 80, 1, 1, 0) == 0


def test_null_handle_rejected(L):
    assert L.h2o_prefill(None, None, None, None, 4, None, None, None) == 1
    assert L.h2o_decode_step(None, None, None, None, None) == 1
    assert L.h2o_decode_steps(None, 1, None, None, None, None, None) == 1
    assert L.h2o_cache_export(None, None, None, None, None, None, None) == 1
    assert L.h2o_cache_import(None, None, None, None, None, 0, 0) == 1
    assert L.h2o_get_error(None) == 1
    assert L.h2o_set_stream(None, None) == 1
    assert L.h2o_cache_set_policy(None, 0, 0) == 1
    assert L.h2o_cache_get_policy(None, None, None) == 1
    assert L.h2o_cache_export_scales(None, None, None) == 1
    assert L.h2o_prefill_rows(None, 0, 1, None, None, None, 4, None, None, None) == 1
    assert L.h2o_cache_import_scales(None, None, None) == 1
    assert L.h2o_cache_destroy(None) == 0


def test_binding_refuses_without_library(tmp_path, monkeypatch):
    """The product path has no fallback: a missing library is an error."""
    monkeypatch.setattr(h2o, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(h2o, "_lib", None)
    with pytest.raises(ImportError):
        h2o.lib()


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "h2o_heavy_hitter_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt and "h2o_oracle" not in txt, f
