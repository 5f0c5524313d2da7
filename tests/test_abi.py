"""The C-ABI library builds, loads without a GPU and exports every entry
point include/dflash.h declares.  No compute calls (no GPU here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "dflash.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def so():
    from block_drafter_verify_gb300 import build
    return ctypes.CDLL(build.build())


def test_header_declares_the_four_path_calls():
    names = _declared()
    for n in ("dflash_lmhead_topk", "dflash_pair_score", "dflash_path_walk",
              "dflash_verify"):
        assert n in names


def test_every_declared_symbol_is_exported(so):
    missing = [n for n in _declared() if not hasattr(so, n)]
    assert not missing, missing


def test_binding_covers_the_header():
    import block_drafter_verify_gb300 as pkg
    assert set(pkg.EXPORTS) == set(_declared())
    for n in _declared():
        if n != "dflash_status_string":
            assert callable(getattr(pkg, n))


def test_host_only_calls(so):
    so.dflash_workspace_bytes.restype = ctypes.c_size_t
    so.dflash_workspace_bytes.argtypes = [ctypes.c_int] * 5
    assert so.dflash_workspace_bytes(0, 32, 8, 2048, 151936) > 0
    assert so.dflash_workspace_bytes(1, 32, 8, 0, 151936) > 0
    assert so.dflash_workspace_bytes(0, 1, 17, 64, 100) == 0   # K > 16
    assert so.dflash_workspace_bytes(0, 1, 4, 4, 100) == 0     # H < 8
    so.dflash_status_string.restype = ctypes.c_char_p
    assert so.dflash_status_string(0) == b"ok"
    assert so.dflash_status_string(1) == b"invalid argument"
    so.dflash_profile_stage.restype = ctypes.c_int
    so.dflash_profile_stage.argtypes = [ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_void_p]
    assert so.dflash_profile_stage(99, None, None) == 1
    assert so.dflash_profile_stage(0, None, None) == 0


def test_compiled_for_sm103a_only():
    from block_drafter_verify_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_binding_fails_loudly_without_library(tmp_path):
    import block_drafter_verify_gb300.binding as b
    with pytest.raises(RuntimeError):
        b.load(str(tmp_path / "missing.so"))
