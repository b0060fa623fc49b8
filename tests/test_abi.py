"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
entry point include/dendrite.h declares (no compute calls here)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dendrite.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dendrite_[a-z_]+)\s*\(", src)))


def test_header_declares_the_pool_fork_append_attend_free_calls():
    names = declared_functions()
    for n in ("dendrite_pool_create", "dendrite_fork", "dendrite_append_kv",
              "dendrite_tree_attn_decode", "dendrite_free"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    import __graft_entry__ as g
    g.build()
    from copy_write_forked_gb300 import dendrite
    L = dendrite.lib()
    for n in declared_functions():
        assert hasattr(L, n), n
    assert b"sm_103a" in L.dendrite_version()
    out = subprocess.run(["nm", "-D", "--defined-only", dendrite._build.LIB_PATH], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (dendrite_[a-z_]+)", out.stdout))
    assert set(declared_functions()) <= exported


def test_library_is_built_for_sm_103a_only():
    from copy_write_forked_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_no_fallback_when_library_missing(monkeypatch, tmp_path):
    from copy_write_forked_gb300 import dendrite, _build
    monkeypatch.setattr(_build, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(dendrite, "_LIB", None)
    with pytest.raises(ImportError):
        dendrite.lib()


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "copy_write_forked_gb300")
    for dp, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cpp", ".h")):
                txt = open(os.path.join(dp, f)).read()
                assert "import oracle" not in txt and "from oracle" not in txt, f


def test_pool_calls_reject_null_pool_without_gpu():
    from copy_write_forked_gb300 import dendrite
    L = dendrite.lib()
    assert L.dendrite_sync(None, None) == -1
    assert L.dendrite_pool_destroy(None) == -1
    assert L.dendrite_free(None, None, 0, None) == -1


def test_pool_options_are_checked_before_any_device_call():
    """Out-of-range pool options fail with EINVAL before the pool touches a
    device (so this runs without a GPU)."""
    import ctypes
    from copy_write_forked_gb300 import dendrite
    L = dendrite.lib()
    h = ctypes.c_void_p()
    for field, bad in (("tc_sms", -2), ("device_planning", 2), ("fold_segments", -2), ("tc_min_rows", -2)):
        o = dendrite._Opts()
        setattr(o, field, bad)
        assert L.dendrite_pool_create(64, 16, 8, 128, 1, ctypes.byref(o), ctypes.byref(h)) == -1, field
    o = dendrite._Opts()
    o.reserved[0] = 1
    assert L.dendrite_pool_create(64, 16, 8, 128, 1, ctypes.byref(o), ctypes.byref(h)) == -1
