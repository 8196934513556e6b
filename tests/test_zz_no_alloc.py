"""lizard_attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin handed tensors by a framework that owns all device memory, or a
loop that must not risk cudaMalloc's device-wide synchronisation) pass only inputs and
outputs; the library keeps the scratch in a fixed device array.  The result must equal
that of lizard_attn_fwd with a caller-provided workspace, call after call, even though
every call reuses the same array.  This file is collected last on purpose.
"""
import ctypes

import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import assert_parity, to_dev, to_np

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


@pytest.mark.parametrize("wl,L", [(I.LLAMA3_8B_L8K, 2048), (I.TINY_F32, 300),
                                  (I.MISTRAL_7B_TRAIN.replace(B=2), 700)])
def test_noalloc_matches_workspace_entry_point(lz, wl, L):
    t = to_dev(I.make_inputs(wl, L=L), wl.dtype)
    B, Hq, Hkv, d, D = t["q"].shape[0], wl.Hq, wl.Hkv, wl.d, wl.D

    def outs():
        return dict(lse=torch.empty(B, L, Hq, device="cuda"),
                    S_out=torch.empty(B, Hkv, D, d, device="cuda"),
                    z_out=torch.empty(B, Hkv, D, device="cuda"))

    ref = outs()
    y_ref = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, **ref)
    torch.cuda.synchronize()
    for call in range(2):
        got = outs()
        y = lz.lizard_attn_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w,
                                       **got)
        torch.cuda.synchronize()
        assert_parity(to_np(y), to_np(y_ref), wl.dtype, f"y, call {call}")
        assert_parity(to_np(got["S_out"]), to_np(ref["S_out"]), wl.dtype, f"S, call {call}")
        assert_parity(to_np(got["lse"]), to_np(ref["lse"]), wl.dtype, f"lse, call {call}")


def test_noalloc_rejects_problems_beyond_its_scratch(lz):
    """fp32, 37 x 8 units cut into 2 segments: 2 * 296 * 66,560 bytes of boundary states,
    more than the 32 MiB array.  The size is checked before the pointers, so the call reports
    it with every pointer null; with null pointers no call of this test can launch."""
    lib = lz.load()
    dims = lz.make_dims(37, 4096, 32, 8, 128, 128, 64, 4, torch.float32)
    st = lib.lizard_attn_fwd_noalloc(ctypes.byref(dims), *([None] * 13))
    assert st == lz.LIZARD_ERR_WORKSPACE
    # a problem that fits is refused for its null pointers, again before any launch
    small = lz.make_dims(1, 256, 4, 2, 128, 128, 64, 4, torch.bfloat16)
    st = lib.lizard_attn_fwd_noalloc(ctypes.byref(small), *([None] * 13))
    assert st == lz.LIZARD_ERR_INVALID_ARG
