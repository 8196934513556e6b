"""lizard_attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin handed tensors by a framework that owns all device memory, or a
loop that must not risk cudaMalloc's device-wide synchronisation) pass only inputs and
outputs; the library keeps the scratch in a fixed device array.  It runs the same kernels
as lizard_attn_fwd with a caller-provided workspace, so the results must be bit-identical,
call after call, even though every call reuses the same array.  This file is collected last
on purpose.
"""
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lz():
    from gated_linear_sliding_gb300 import lizard

    lizard.load()
    return lizard


def _outs(wl, B, L):
    return dict(lse=torch.empty(B, L, wl.Hq, device="cuda"),
                S_out=torch.empty(B, wl.Hkv, wl.D, wl.d, device="cuda"),
                z_out=torch.empty(B, wl.Hkv, wl.D, device="cuda"))


def _run(lz, fn, t, wl, B, L):
    o = _outs(wl, B, L)
    y = fn(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, **o)
    return dict(y=y, **o)


# (workload, L, B); the middle workload of each pair differs in shape and is cut into several
# segments, so the array holds other boundary records when the first shape runs again
CASES = [
    (I.LLAMA3_8B_L8K, 2048, 1),
    (I.closed_gates(I.LLAMA3_8B_L8K), 3000, 1),   # hands steps to the exact tail walk
    (I.TINY_F32.replace(Hq=4, Hkv=2), 900, 2),
    (I.MISTRAL_7B_TRAIN, 700, 2),
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_noalloc_bit_identical_to_workspace_entry_point(lz, i):
    wl, L, B = CASES[i]
    other_wl, oL, oB = CASES[(i + 1) % len(CASES)]
    t = to_dev(I.make_inputs(wl, L=L, B=B), wl.dtype)
    o = to_dev(I.make_inputs(other_wl, L=oL, B=oB), other_wl.dtype)
    ref = _run(lz, lz.lizard_attn_fwd, t, wl, B, L)
    first = _run(lz, lz.lizard_attn_fwd_noalloc, t, wl, B, L)
    _run(lz, lz.lizard_attn_fwd_noalloc, o, other_wl, oB, oL)  # other contents in the array
    second = _run(lz, lz.lizard_attn_fwd_noalloc, t, wl, B, L)
    torch.cuda.synchronize()
    assert lz.lizard_read_noalloc_status() == lz.LIZARD_OK
    for got, call in ((first, "first"), (second, "second")):
        for n in ("y", "lse", "S_out", "z_out"):
            assert torch.equal(got[n], ref[n]), f"{n}, {call} call"


def test_noalloc_rejects_problems_beyond_its_scratch(lz):
    """64 x 8 units of the tensor-core shape need one 66,560-byte boundary record each: 34 MB,
    more than the 32 MiB array.  The call reports it before anything is launched and leaves y
    untouched."""
    wl = I.LLAMA3_8B_L8K
    B, L = 64, 64
    t = {n: torch.zeros(B, L, h, wl.d, dtype=torch.bfloat16, device="cuda")
         for n, h in (("q", wl.Hq), ("k", wl.Hkv), ("v", wl.Hkv))}
    t["g"] = torch.zeros(B, L, wl.Hkv, wl.D, dtype=torch.bfloat16, device="cuda")
    t["Wf"] = torch.zeros(wl.Hkv, wl.d, wl.D // 2, dtype=torch.bfloat16, device="cuda")
    t["sinks"] = torch.zeros(wl.Hq, wl.M, device="cuda")
    dims = lz.dims_of(t["q"], t["k"], t["g"], t["sinks"], wl.w)
    assert lz.lizard_attn_fwd_noalloc_scratch(dims) > 32 << 20
    y = torch.full_like(t["q"], 7.0)
    with pytest.raises(lz.LizardError) as e:
        lz.lizard_attn_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w, y=y)
    assert e.value.status == lz.LIZARD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())
    # the same heads at batch 4 fit
    small = lz.make_dims(4, L, wl.Hq, wl.Hkv, wl.d, wl.D, wl.w, wl.M, torch.bfloat16)
    assert 256 < lz.lizard_attn_fwd_noalloc_scratch(small) <= 32 << 20


def test_noalloc_device_status_is_readable(lz):
    """A bounded device-side wait that gives up records LIZARD_ERR_TIMEOUT in the array's status
    word (the self-test waits on a barrier nothing completes, then returns: no fault); the
    caller reads it with lizard_read_noalloc_status, reading clears it, and the next forward
    still matches lizard_attn_fwd bit for bit."""
    wl = I.LLAMA3_8B_L8K
    t = to_dev(I.make_inputs(wl, L=1024), wl.dtype)
    lz.lizard_attn_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w)
    assert lz.lizard_read_noalloc_status() == lz.LIZARD_OK
    lz.lizard_selftest_wait_timeout(None, 20_000_000)  # about 10 ms at 2 GHz
    assert lz.lizard_read_noalloc_status() == lz.LIZARD_ERR_TIMEOUT
    assert lz.lizard_read_noalloc_status() == lz.LIZARD_OK
    y = lz.lizard_attn_fwd_noalloc(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w)
    ref = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w)
    torch.cuda.synchronize()
    assert torch.equal(y, ref)
    assert lz.lizard_read_noalloc_status() == lz.LIZARD_OK
