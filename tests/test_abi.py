"""The C ABI: the library loads, exports what include/lizard.h declares, and rejects bad
arguments on the host before touching the GPU (no compute call here)."""
import ctypes
import os
import re

import pytest

from gated_linear_sliding_gb300 import _build
from gated_linear_sliding_gb300 import lizard as lz

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "lizard.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return lz.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lizard_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("lizard_attn_fwd", "lizard_attn_bwd", "lizard_decode_step"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(lz.EXPORTED) == sorted(declared_functions())


def test_status_strings_and_version(lib):
    for code in range(6):
        assert lz.status_string(code)
    assert "sm_103a" in lz.lizard_version()


def dims(**kw):
    base = dict(B=1, L=8192, Hq=32, Hkv=8, d=128, D=128, w=64, M=4, dtype=lz.LIZARD_BF16)
    base.update(kw)
    return lz.make_dims(base["B"], base["L"], base["Hq"], base["Hkv"], base["d"], base["D"],
                        base["w"], base["M"], base["dtype"], scale=kw.get("scale", 0.0),
                        chunk=kw.get("chunk", 0))


def test_workspace_constant_in_L(lib):
    """Sec. 2-A-1 (constant-memory state): the forward workspace holds per-segment
    boundary states whose count depends on B and Hkv only."""
    sizes = {L: lz.lizard_attn_fwd_workspace(dims(L=L)) for L in (64, 1000, 8192, 65536)}
    assert len(set(sizes.values())) == 1 and sizes[8192] > 0
    # backward: only the per-gate-element and per-query-row fp32 scratch grows with L
    b1 = lz.lizard_attn_bwd_workspace(dims(L=2048, B=8))
    b2 = lz.lizard_attn_bwd_workspace(dims(L=4096, B=8))
    assert b2 - b1 == 8 * 2048 * 8 * 128 * 4 + 2 * 8 * 2048 * 32 * 4


@pytest.mark.parametrize("bad", [dict(Hq=30), dict(D=127), dict(w=0), dict(M=-1), dict(M=65),
                                 dict(chunk=32), dict(dtype=7), dict(L=0), dict(B=0),
                                 dict(scale=-1.0)])
def test_invalid_dims_rejected(lib, bad):
    d = dims(**bad)
    assert lz.lizard_attn_fwd_workspace(d) == 0
    nul = [None] * 13
    st = lib.lizard_attn_fwd(ctypes.byref(d), *nul, 0, None)
    assert st == lz.LIZARD_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected(lib):
    d = dims(L=128)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first
    mis = ctypes.c_void_p(0x10004)
    args = [fake] * 6 + [fake] + [None] * 5 + [fake]
    st = lib.lizard_attn_fwd(ctypes.byref(d), None, *args[1:], 1 << 30, None)
    assert st == lz.LIZARD_ERR_INVALID_ARG
    args2 = list(args)
    args2[2] = mis
    st = lib.lizard_attn_fwd(ctypes.byref(d), *args2, 1 << 30, None)
    assert st == lz.LIZARD_ERR_INVALID_ARG
    # S_out without z_out
    args3 = list(args)
    args3[8] = fake
    st = lib.lizard_attn_fwd(ctypes.byref(d), *args3, 1 << 30, None)
    assert st == lz.LIZARD_ERR_INVALID_ARG


def test_unsupported_and_workspace_errors(lib):
    fake = ctypes.c_void_p(0x10000)
    d = dims(d=96, D=96)
    args = [fake] * 7 + [None] * 5 + [fake]
    assert lib.lizard_attn_fwd(ctypes.byref(d), *args, 1 << 30, None) == \
        lz.LIZARD_ERR_UNSUPPORTED
    d = dims(L=128)
    need = lz.lizard_attn_fwd_workspace(d)
    assert lib.lizard_attn_fwd(ctypes.byref(d), *args, need - 16, None) == \
        lz.LIZARD_ERR_WORKSPACE
    # decode: window beyond the staged maximum, and G beyond 8
    nul = [fake] * 12
    assert lib.lizard_decode_step(ctypes.byref(dims(w=300)), 0, *nul, 256, None) == \
        lz.LIZARD_ERR_UNSUPPORTED
    assert lib.lizard_decode_step(ctypes.byref(dims(Hq=32, Hkv=2)), 0, *nul, 256, None) == \
        lz.LIZARD_ERR_UNSUPPORTED
    assert lib.lizard_decode_step(ctypes.byref(dims()), -1, *nul, 256, None) == \
        lz.LIZARD_ERR_INVALID_ARG


def test_kernel_path_query(lib):
    assert lz.lizard_attn_fwd_kernel(dims(Hq=30)) == -1
    assert lz.lizard_attn_fwd_kernel(dims(dtype=lz.LIZARD_F32)) == 0
    assert lz.lizard_attn_fwd_kernel(dims(w=32)) == 0
    assert lz.lizard_attn_fwd_kernel(dims()) in (0, 1)  # 1 where the CUDA driver's TMA encoder exists


def test_varlen_offsets_validated_before_any_launch(lib):
    """lizard_attn_fwd_varlen refuses inconsistent offsets on the host; every tensor pointer
    here is null, so no call can reach a launch."""
    d = dims(L=10)
    d.B = 2
    nul = [None] * 13
    for cu in ([0, 4, 9], [1, 4, 10], [0, 6, 4, 10][:3], [0, 11, 10]):
        arr = (ctypes.c_int64 * len(cu))(*cu)
        st = lib.lizard_attn_fwd_varlen(ctypes.byref(d), arr, *nul, 1 << 30, None)
        assert st == lz.LIZARD_ERR_INVALID_ARG
    assert lib.lizard_attn_fwd_varlen(ctypes.byref(d), None, *nul, 1 << 30, None) == \
        lz.LIZARD_ERR_INVALID_ARG


def test_bwd_varlen_workspace_and_offsets(lib):
    """The packed backward's workspace grows with the longest sequence, covers the parameter
    gradient sums, and is 0 for inconsistent offsets (no device work involved)."""
    d = dims(L=3000)
    d.B = 3
    ok = (ctypes.c_int64 * 4)(0, 1000, 1000, 3000)
    short = (ctypes.c_int64 * 4)(0, 1000, 2000, 3000)
    bad = (ctypes.c_int64 * 4)(0, 1000, 999, 3000)
    lib.lizard_attn_bwd_varlen_workspace.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.lizard_attn_bwd_varlen_workspace.restype = ctypes.c_size_t
    w_ok = lib.lizard_attn_bwd_varlen_workspace(ctypes.byref(d), ok)
    w_short = lib.lizard_attn_bwd_varlen_workspace(ctypes.byref(d), short)
    one = dims(L=2000)
    assert w_ok > w_short > lz.lizard_attn_bwd_workspace(dims(L=1000))
    assert w_ok >= lz.lizard_attn_bwd_workspace(one) + 128 * 64 * 8 * 4
    assert lib.lizard_attn_bwd_varlen_workspace(ctypes.byref(d), bad) == 0
    nul = [None] * 16
    assert lib.lizard_attn_bwd_varlen(ctypes.byref(d), bad, *nul, 1 << 30, None) == \
        lz.LIZARD_ERR_INVALID_ARG
