"""C-ABI library checks that need no GPU: it builds, loads, exports every
entry point declared in include/jfa.h, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from jagged_flash_attention_gb300 import build, lib
    build.build()
    return lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "jfa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(jfa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert {"jfa_fwd", "jfa_bwd", "jfa_fwd_bq", "jfa_bwd_bq", "jfa_last_error"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_version(L):
    assert b"sm_103a" in L.jfa_version()


def _fwd(L, **kw):
    a = dict(q=16, k=16, v=16, off=16, B=2, H=2, D=128, max_len=10, bq=0, causal=0, scale=0.1,
             out=16, lse=16)
    a.update(kw)
    return L.jfa_fwd(a["q"], a["k"], a["v"], a["off"], a["B"], a["H"], a["D"], a["max_len"],
                     a["bq"], a["causal"], a["scale"], a["out"], a["lse"], 0)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(D=96), 2, "D must be 64 or 128"),
    (dict(bq=1), 1, "jfa_fwd_bq"),
    (dict(B=0), 1, "B must be"),
    (dict(H=0), 1, "H must be"),
    # work items hold the head in bits 16-30 of an int32
    (dict(H=32768), 1, "H must be in [1, 32767]"),
    (dict(scale=float("nan")), 1, "scale"),
    (dict(scale=-1.0), 1, "scale"),
    (dict(q=0), 1, "non-null"),
    (dict(k=24), 1, "16-byte aligned"),
    (dict(off=0), 1, "offsets"),
    (dict(out=8), 1, "out must be"),
    (dict(lse=0), 1, "lse must be"),
    (dict(max_len=-1), 1, "max_len"),
])
def test_host_argument_errors(L, kw, status, needle):
    assert _fwd(L, **kw) == status
    assert needle in L.jfa_last_error().decode()


def test_causal_broadcast_unsupported(L):
    st = L.jfa_fwd_bq(16, 16, 16, 16, 2, 2, 128, 10, 64, 1, 1, 0.1, 16, 16, 0)
    assert st == 2 and b"self-attention only" in L.jfa_last_error()
    st = L.jfa_bwd_bq(16, 16, 16, 16, 2, 2, 128, 10, 0, 1, 0, 0.1, 16, 16, 16, 16, 16, 16, 0)
    assert st == 1 and b"q_len" in L.jfa_last_error()


def test_bwd_argument_errors(L):
    st = L.jfa_bwd(16, 16, 16, 16, 2, 2, 128, 10, 0, 0, 0.1, 16, 16, 16, 0, 16, 16, 0)
    assert st == 1 and b"non-null" in L.jfa_last_error()
    st = L.jfa_bwd(16, 16, 16, 16, 2, 2, 64, 10, 0, 0, 0.1, 16, 16, 16, 16, 16, 40, 0)
    assert st == 1 and b"16-byte" in L.jfa_last_error()


def test_product_path_does_not_touch_oracle():
    """The package and the CUDA sources never reference the oracle."""
    pkg = os.path.join(ROOT, "jagged_flash_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in txt.lower(), f


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import jagged_flash_attention_gb300 as jfa
    monkeypatch.setattr(jfa, "_LIB", None)
    monkeypatch.setattr(jfa, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        jfa.lib()


def test_profile_read_arguments(L):
    L.jfa_profile_read.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    assert L.jfa_profile_read(None, None, 0) == 0
    assert L.jfa_profile_read(None, None, 3) == 1
    assert b"profile_read" in L.jfa_last_error()
    assert L.jfa_profile_read(None, None, -1) == 1


def test_launch_count_without_launches():
    import jagged_flash_attention_gb300 as jfa
    n0 = jfa.launch_count()
    assert n0 >= 0
    jfa.profile_enable(True)
    jfa.profile_enable(False)
    prof = jfa.profile_read()
    assert set(prof) == set(jfa.KERNEL_KINDS)
    assert jfa.launch_count() == n0
    jfa.profile_select(["bwd_kv", "fwd"])
    jfa.profile_select(None)
    with pytest.raises(ValueError):
        jfa.profile_select(["no_such_kernel"])


def test_worklist_argument_errors(L):
    """jfa_worklist rejects bad arguments on the host, before touching a GPU."""
    fn = L.jfa_worklist
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    assert fn(16, 4, 2, 100, 0, 0, 0, 4, 16, 100, 16, 0) == 1
    assert b"list must be" in L.jfa_last_error()
    assert fn(16, 4, 2, 100, 64, 1, 0, 2, 16, 100, 16, 0) == 1
    assert b"self-attention only" in L.jfa_last_error()
    assert fn(16, 4, 2, 100, 0, 0, 0, 3, 16, 100, 16, 0) == 1
    assert fn(16, 4, 2, 100, 64, 1, 1, 1, 16, 100, 16, 0) == 1
    assert fn(16, 4, 2, 100, 0, 0, 0, 0, 8, 100, 16, 0) == 1  # items not 16-byte aligned
    assert b"16-byte" in L.jfa_last_error()
    assert fn(16, 4, 32768, 100, 0, 0, 0, 0, 16, 100, 16, 0) == 1  # head beyond the item encoding
    assert b"32767" in L.jfa_last_error()


def _fwd_ex(L, **kw):
    a = dict(H=4, Hkv=2, q_len=0, bq=0, causal=0, wl=-1, wr=-1)
    a.update(kw)
    return L.jfa_fwd_ex(16, 16, 16, 16, 2, a["H"], a["Hkv"], 128, 10, a["q_len"], a["bq"],
                        a["causal"], a["wl"], a["wr"], 0.1, 16, 16, 0)


@pytest.mark.parametrize("kw,status,needle", [
    (dict(Hkv=3), 1, "H_kv must divide H"),
    (dict(Hkv=0), 1, "H_kv must divide H"),
    (dict(Hkv=8), 1, "H_kv must divide H"),
    (dict(wl=-2), 1, "window bounds"),
    (dict(wr=-3), 1, "window bounds"),
    (dict(causal=1, wr=5), 1, "right side by 0"),
    (dict(bq=1, q_len=64, wl=16), 2, "self-attention only"),
    (dict(bq=1, q_len=64, wr=0), 2, "self-attention only"),
])
def test_variant_argument_errors(L, kw, status, needle):
    """GQA / window arguments of jfa_fwd_ex and jfa_bwd_ex are checked on the
    host before anything touches a GPU."""
    import jagged_flash_attention_gb300  # noqa: F401  (sets the argument types)
    assert _fwd_ex(L, **kw) == status
    assert needle in L.jfa_last_error().decode()
    a = dict(H=4, Hkv=2, q_len=0, bq=0, causal=0, wl=-1, wr=-1)
    a.update(kw)
    st = L.jfa_bwd_ex(16, 16, 16, 16, 2, a["H"], a["Hkv"], 128, 10, a["q_len"], a["bq"],
                      a["causal"], a["wl"], a["wr"], 0.1, 16, 16, 16, 16, 16, 16, 0)
    assert st == status and needle in L.jfa_last_error().decode()


def test_sparse_argument_errors(L):
    """Block selection and the sparse forward reject bad arguments on the host."""
    import jagged_flash_attention_gb300 as jfa
    sel = lambda **kw: jfa.lib().jfa_block_select(
        16, 16, 16, 2, 4, kw.get("Hkv", 2), 128, kw.get("max_len", 1000), kw.get("q_len", 0),
        kw.get("bq", 0), kw.get("permille", 500), kw.get("blocks", 16), kw.get("counts", 16), 0)
    L.jfa_block_select.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 8 + [ctypes.c_void_p] * 3
    assert sel(permille=0) == 1 and b"permille" in L.jfa_last_error()
    assert sel(permille=1001) == 1 and b"permille" in L.jfa_last_error()
    assert sel(max_len=300000) == 1 and b"max_len must be <=" in L.jfa_last_error()
    assert sel(blocks=0) == 1 and b"blocks and counts" in L.jfa_last_error()
    assert sel(counts=18) == 1 and b"blocks and counts" in L.jfa_last_error()
    assert sel(Hkv=3) == 1 and b"H_kv must divide H" in L.jfa_last_error()
    assert sel(bq=1, q_len=0) == 1 and b"q_len" in L.jfa_last_error()
    L.jfa_fwd_sparse.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] * 7 + [ctypes.c_float]
                                 + [ctypes.c_void_p] * 5)
    st = L.jfa_fwd_sparse(16, 16, 16, 16, 2, 4, 2, 128, 1000, 0, 0, 0.1, 0, 16, 16, 16, 0)
    assert st == 1 and b"blocks and counts" in L.jfa_last_error()
    st = L.jfa_fwd_sparse(16, 16, 16, 16, 2, 4, 2, 96, 1000, 0, 0, 0.1, 16, 16, 16, 16, 0)
    assert st == 2 and b"D must be" in L.jfa_last_error()


def test_local_sparse_argument_errors(L):
    """The _ex forms of the block-sparse calls check the mask arguments like
    jfa_fwd_ex does, on the host."""
    L.jfa_block_select_ex.argtypes = ([ctypes.c_void_p] * 3 + [ctypes.c_int] * 11
                                      + [ctypes.c_void_p] * 3)
    L.jfa_fwd_sparse_ex.argtypes = ([ctypes.c_void_p] * 4 + [ctypes.c_int] * 10 + [ctypes.c_float]
                                    + [ctypes.c_void_p] * 5)

    def both(bq, q_len, causal, wl, wr):
        s1 = L.jfa_block_select_ex(16, 16, 16, 2, 4, 2, 128, 1000, q_len, bq, causal, wl, wr, 500,
                                   16, 16, 0)
        e1 = L.jfa_last_error().decode()
        s2 = L.jfa_fwd_sparse_ex(16, 16, 16, 16, 2, 4, 2, 128, 1000, q_len, bq, causal, wl, wr,
                                 0.1, 16, 16, 16, 16, 0)
        e2 = L.jfa_last_error().decode()
        return (s1, e1), (s2, e2)

    for (st, err) in both(0, 0, 1, -1, 4):
        assert st == 1 and "right side by 0" in err
    for (st, err) in both(0, 0, 0, -2, -1):
        assert st == 1 and "window bounds" in err
    for (st, err) in both(1, 64, 1, -1, -1):
        assert st == 2 and "self-attention only" in err
    for (st, err) in both(1, 64, 0, 32, -1):
        assert st == 2 and "self-attention only" in err
