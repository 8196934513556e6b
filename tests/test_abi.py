"""The C ABI: the library loads, exports what include/lizard.h declares, and rejects bad
arguments on the host before touching the GPU (no compute call here)."""
import ctypes
import json
import os
import re
import subprocess
import sys

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
                        chunk=kw.get("chunk", 0), decay=kw.get("decay", 0))


def test_dims_struct_layout(tmp_path):
    """The Python mirror of lizard_dims has the layout the C compiler gives the header's
    struct (size and every field offset)."""
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "lizard.h"\n'
                   'int main(void) { printf("%zu", sizeof(lizard_dims));\n' +
                   "".join(f'printf(" %zu", offsetof(lizard_dims, {n}));\n'
                           for n, _ in lz.lizard_dims._fields_) + "return 0; }\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.dirname(HEADER), "-o", str(exe), str(src)])
    got = [int(x) for x in subprocess.check_output([str(exe)], text=True).split()]
    want = [ctypes.sizeof(lz.lizard_dims)] + [getattr(lz.lizard_dims, n).offset
                                              for n, _ in lz.lizard_dims._fields_]
    assert got == want


@pytest.mark.parametrize("decay,elem", [(lz.LIZARD_DECAY_LAGGED, 2), (lz.LIZARD_DECAY_MASKED, 4)])
def test_reading_workspaces(lib, decay, elem):
    """The lagged reading adds one moved gate per gate element (dtype), the masked one an
    fp32 log gate product per element (and, in the backward, its gate term too)."""
    f1 = lz.lizard_attn_fwd_workspace(dims(L=2048, decay=decay))
    f2 = lz.lizard_attn_fwd_workspace(dims(L=4096, decay=decay))
    assert f2 - f1 == 2048 * 8 * 128 * elem
    assert f1 > lz.lizard_attn_fwd_workspace(dims(L=2048))
    b1 = lz.lizard_attn_bwd_workspace(dims(L=2048, B=8, decay=decay))
    b2 = lz.lizard_attn_bwd_workspace(dims(L=4096, B=8, decay=decay))
    per_gate = elem if decay == lz.LIZARD_DECAY_LAGGED else 2 * elem
    # masked: the key terms' suffix sums also keep one fp32 total per 64-row chunk
    chunks = 8 * (2048 // 64) * 8 * 128 * 4 if decay == lz.LIZARD_DECAY_MASKED else 0
    assert b2 - b1 == 8 * 2048 * 8 * 128 * (4 + per_gate) + 2 * 8 * 2048 * 32 * 4 + chunks
    # decode: the status word plus one value per (sequence, KV head, feature)
    assert lz.lizard_decode_workspace(dims(L=1, B=64, decay=decay)) == 256 + 64 * 8 * 128 * elem
    assert lz.lizard_decode_workspace(dims(L=1, B=64)) == 256


def test_tensor_core_path_by_reading(lib):
    """Both other readings keep the tensor-core forward on its shapes, and the SIMT walk on
    the others."""
    if lz.lizard_attn_fwd_kernel(dims()) != 1:
        pytest.skip("the CUDA driver's TMA encoder is not available here")
    for code in (lz.LIZARD_DECAY_LAGGED, lz.LIZARD_DECAY_MASKED):
        assert lz.lizard_attn_fwd_kernel(dims(decay=code)) == 1
        assert lz.lizard_attn_fwd_kernel(dims(decay=code, dtype=lz.LIZARD_F32)) == 0


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
                                 dict(scale=-1.0), dict(decay=3), dict(decay=-1)])
def test_invalid_dims_rejected(lib, bad):
    d = dims(**bad)
    assert lz.lizard_attn_fwd_workspace(d) == 0
    nul = [None] * 13
    st = lib.lizard_attn_fwd(ctypes.byref(d), *nul, 0, None)
    assert st == lz.LIZARD_ERR_INVALID_ARG


def _no_device_calls():
    """Run tests/_abi_calls.py with no visible CUDA device and return its status codes."""
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    script = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_abi_calls.py")
    r = subprocess.run([sys.executable, script], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_null_and_misaligned_pointers_rejected(lib):
    """Null, misaligned and unpaired pointers, unsupported sizes and a short workspace are
    refused on the host.  The calls that need non-null pointers get host buffers, in a child
    process that sees no CUDA device, so none of them can launch anything."""
    st = _no_device_calls()
    bad = lz.LIZARD_ERR_INVALID_ARG
    for case in ("fwd_null_q", "fwd_misaligned_v", "fwd_S_without_z", "fwd_misaligned_ws",
                 "noalloc_misaligned", "dec_neg_pos", "dec_misaligned", "fwd_bad_decay",
                 "dec_masked_no_gcache", "dec_masked_mis_gcache", "dec_lagged_no_gcache",
                 "dec_lagged_mis_gcache", "gfill_null", "gfill_mis", "gfill_bad_dims"):
        assert st[case] == bad, (case, st[case])
    assert st["dec_masked_small_ws"] == lz.LIZARD_ERR_WORKSPACE
    assert st["dec_lagged_small_ws"] == lz.LIZARD_ERR_WORKSPACE
    assert st["dec_delayed_no_gcache"] == lz.LIZARD_ERR_CUDA  # passes every check
    assert st["fwd_unsupported"] == lz.LIZARD_ERR_UNSUPPORTED
    assert st["fwd_small_ws"] == lz.LIZARD_ERR_WORKSPACE
    assert st["dec_w300"] == lz.LIZARD_ERR_UNSUPPORTED
    assert st["dec_G16"] == lz.LIZARD_ERR_UNSUPPORTED
    assert st["fwd_no_device"] == lz.LIZARD_ERR_CUDA
    assert st["proj_f32"] == lz.LIZARD_ERR_UNSUPPORTED
    assert st["proj_dm"] == lz.LIZARD_ERR_UNSUPPORTED
    assert st["proj_null"] == bad
    assert st["proj_bwd_mis"] == bad


def test_null_pointer_checks_in_process(lib):
    """With every tensor pointer null the forward, backward and decode entry points refuse the
    call before any device work."""
    d = dims(L=128)
    nul = [None] * 13
    assert lib.lizard_attn_fwd(ctypes.byref(d), *nul, 1 << 30, None) == lz.LIZARD_ERR_INVALID_ARG
    assert lib.lizard_attn_fwd_noalloc(ctypes.byref(d), *([None] * 13)) == \
        lz.LIZARD_ERR_INVALID_ARG
    assert lib.lizard_attn_bwd(ctypes.byref(d), *([None] * 16), 1 << 30, None) == \
        lz.LIZARD_ERR_INVALID_ARG
    assert lib.lizard_decode_step(ctypes.byref(d), 0, *([None] * 13), 256, None) == \
        lz.LIZARD_ERR_INVALID_ARG


def test_noalloc_scratch_query(lib):
    """The fixed array's use: 256 bytes plus one 66,560-byte boundary record per unit and
    record of the launch (tensor-core shape: at least one record)."""
    rec = (128 * 128 + 2 * 128) * 4
    small = lz.lizard_attn_fwd_noalloc_scratch(dims(L=64))
    assert (small - 256) % (8 * rec) == 0
    # the tensor-core path needs the CUDA driver's TMA encoder; without it the one-segment SIMT
    # launch uses no record
    tc = lz.lizard_attn_fwd_kernel(dims(L=64)) == 1
    assert small == 256 + 8 * rec if tc else small == 256
    if tc:
        assert lz.lizard_attn_fwd_noalloc_scratch(dims(B=64, L=64)) > 32 << 20
    f32 = lz.lizard_attn_fwd_noalloc_scratch(dims(B=37, L=4096, dtype=lz.LIZARD_F32))
    assert f32 > 32 << 20 and (f32 - 256) % (37 * 8 * rec) == 0
    assert lz.lizard_attn_fwd_noalloc_scratch(dims(Hq=30)) == 0


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


def test_fwd_varlen_workspace_query(lib):
    """The packed forward's workspace: one launch over all sequences needs a boundary record per
    (sequence x KV head, segment) plus the offsets, more than one sequence's workspace; where
    the tensor-core path is unavailable it is the sequence loop's workspace; 0 for
    inconsistent offsets (no device work involved)."""
    d = dims(L=3000)
    d.B = 3
    ok = (ctypes.c_int64 * 4)(0, 1000, 1000, 3000)
    bad = (ctypes.c_int64 * 4)(0, 1000, 999, 3000)
    lib.lizard_attn_fwd_varlen_workspace.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.lizard_attn_fwd_varlen_workspace.restype = ctypes.c_size_t
    w_ok = lib.lizard_attn_fwd_varlen_workspace(ctypes.byref(d), ok)
    loop = lz.lizard_attn_fwd_workspace(dims(L=3000))
    if lz.lizard_attn_fwd_kernel(dims(L=3000)) == 1:
        rec = (128 * 128 + 2 * 128) * 4
        assert w_ok >= 256 + 3 * 8 * rec + 4 * 8 and w_ok > loop
    else:
        assert w_ok == loop
    assert lib.lizard_attn_fwd_varlen_workspace(ctypes.byref(d), bad) == 0
