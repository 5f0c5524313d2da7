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


def test_argument_checks_come_before_any_device_work(so):
    """Invalid arguments are refused on the host (DFLASH_ERR_INVALID_ARG)
    before the library looks for a device, so these run without a GPU."""
    vp, i32, f32, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                             ctypes.c_uint64, ctypes.c_size_t)
    fake = ctypes.c_void_p(0x100000)   # never dereferenced: checks fail first
    q = so.dflash_quantize_e4m3_rows
    q.restype, q.argtypes = i32, [vp, i32, i32, vp, vp, vp]
    assert q(None, 4, 32, fake, fake, None) == 1            # no input
    assert q(fake, 4, 24, fake, fake, None) == 1            # H % 16 != 0
    assert q(fake, 0, 32, fake, fake, None) == 1            # no rows
    d = so.dflash_draft_e4m3
    d.restype = i32
    d.argtypes = [vp] * 8 + [i32] * 5 + [f32, u64, u64] + [vp] * 8 + [sz, vp]
    args = [fake, None, fake, fake, fake, fake, fake, fake,   # conv_w NULL
            2, 4, 64, 1000, 32, 1.0, 1, 0] + [fake] * 8 + [1 << 30, None]
    assert d(*args) == 1
    args[1] = fake
    args[10] = 40                                             # H % 16 != 0
    assert d(*args) == 1
    so.dflash_workspace_bytes.restype = sz
    so.dflash_workspace_bytes.argtypes = [i32] * 5
    w2 = so.dflash_workspace_bytes(2, 32, 8, 2048, 151936)
    w3 = so.dflash_workspace_bytes(3, 32, 8, 2048, 151936)
    assert w3 >= w2 + 32 * 8 * 2048 + 32 * 8 * 4
    assert so.dflash_workspace_bytes(3, 1, 4, 8, 100) == 0   # H < 16
    v = so.dflash_path_viterbi
    v.restype, v.argtypes = i32, [vp, vp, i32, i32, vp, vp, vp, vp]
    assert v(fake, fake, 2, 17, fake, fake, fake, None) == 1  # K > 16
    r = so.dflash_top16_recall
    r.restype, r.argtypes = i32, [vp, vp, i32, i32, i32, vp, vp, vp]
    assert r(None, fake, 2, 4, 100, fake, fake, None) == 1
    c = so.dflash_commit
    c.restype, c.argtypes = i32, [vp, vp, i32, i32, vp, vp, vp, i32, vp, vp]
    assert c(fake, fake, 2, 4, fake, fake, fake, 0, fake, None) == 1  # cap 0


def test_noalloc_verify_refuses_bad_arguments_on_the_host(so):
    """dflash_verify_noalloc shares dflash_verify's host-side checks: a
    null pointer, T < 0, target logits not 16-byte aligned and K > 16 are
    refused before any device work (no GPU needed)."""
    vp, i32, f32, u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                         ctypes.c_uint64)
    fake = ctypes.c_void_p(0x100000)
    f = so.dflash_verify_noalloc
    f.restype = i32
    f.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp, vp]
    ok = [fake, fake, fake, fake, 2, 4, 100, 1.0, 1, 0, fake, fake, None]

    def call(**kw):
        a = list(ok)
        for k, v in kw.items():
            a[{"L": 0, "draft": 1, "topi": 2, "q": 3, "B": 4, "K": 5,
               "V": 6, "T": 7, "n": 10, "out": 11}[k]] = v
        return f(*a)
    assert call(L=None) == 1
    assert call(q=None) == 1
    assert call(out=None) == 1
    assert call(T=-1.0) == 1
    assert call(T=float("inf")) == 1
    assert call(L=ctypes.c_void_p(0x100004)) == 1     # not 16-byte aligned
    assert call(K=17) == 1
    assert call(K=0) == 1
    assert call(B=0) == 1
    assert call(V=0) == 1
    # the same checks in dflash_verify (its workspace present and large)
    g = so.dflash_verify
    g.restype = i32
    g.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, u64, u64, vp, vp, vp,
                  ctypes.c_size_t, vp]
    big = ctypes.c_void_p(0x200000)
    base = [fake, fake, fake, fake, 2, 4, 100, 1.0, 1, 0, fake, fake, big,
            1 << 30, None]
    for i, v in ((0, None), (7, -1.0), (0, ctypes.c_void_p(0x100004)),
                 (5, 17)):
        a = list(base)
        a[i] = v
        assert g(*a) == 1
    a = list(base)
    a[12] = ctypes.c_void_p(0x200010)                 # ws not 256-aligned
    assert g(*a) == 1
    a = list(base)
    a[13] = 16                                        # ws too small
    assert g(*a) == 1


def test_cycle_refuses_bad_arguments_on_the_host(so):
    """dflash_cycle checks the verify's arguments, then the draft's, before
    any launch: a null target, a misaligned or too small verify workspace,
    the 8-bit head with fp32 storage and a draft-side size error are all
    refused on the host (no GPU needed)."""
    vp, i32, f32, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                             ctypes.c_uint64, ctypes.c_size_t)
    fake = ctypes.c_void_p(0x100000)
    f = so.dflash_cycle
    f.restype = i32
    f.argtypes = ([vp] * 9 + [i32] * 6 + [f32, u64, u64] + [vp] * 9 +
                  [vp, sz, vp, sz, vp])
    names = ["h", "conv_w", "w_lm", "w_scale", "w_gate", "e_in", "e_out",
             "anchor", "L", "B", "K", "H", "V", "r", "dt", "T", "seed",
             "cycle", "topv", "topi", "lse", "scores", "slot", "draft", "q",
             "n", "out", "wsd", "wsd_bytes", "wsv", "wsv_bytes", "stream"]
    ok = dict(zip(names, [fake, fake, fake, None, fake, fake, fake, fake,
                          fake, 2, 4, 64, 1000, 32, 0, 1.0, 1, 0] +
                  [fake] * 9 + [fake, 1 << 30, fake, 1 << 30, None]))

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*[a[k] for k in names])
    assert call(L=None) == 1                               # no target
    assert call(n=None) == 1                               # no output
    assert call(wsv=None) == 1
    assert call(wsv=ctypes.c_void_p(0x100010)) == 1        # not 256-aligned
    assert call(wsv_bytes=16) == 1                         # too small
    assert call(w_scale=fake, dt=1) == 1                   # 8-bit, fp32
    assert call(H=60) == 1                                 # H % 8 != 0
    assert call(K=17) == 1
    assert call(T=-1.0) == 1
