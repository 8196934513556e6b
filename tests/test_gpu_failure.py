"""Failure detection without a GPU fault: a bounded device-side wait that can never
complete gives up, records a timeout status in the workspace, frees its TMEM and returns;
the host reads the status, the status clears, and the library keeps working."""
import pytest

from gated_linear_sliding_gb300 import inputs as I
from helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def test_bounded_wait_reports_timeout_and_context_survives():
    from gated_linear_sliding_gb300 import lizard as lz

    lz.load()
    ws = lz.new_workspace(256, "cuda")
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK
    lz.lizard_selftest_wait_timeout(ws, 20_000_000)  # ~10 ms at 2 GHz
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_ERR_TIMEOUT
    assert lz.lizard_read_device_status(ws) == lz.LIZARD_OK  # reading clears it
    # the context is intact: a forward on the tensor-core shapes still runs and matches
    wl = I.LLAMA3_8B_L8K
    t = to_dev(I.make_inputs(wl, L=256), wl.dtype)
    y1 = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w)
    y2 = lz.lizard_attn_fwd(t["q"], t["k"], t["v"], t["g"], t["Wf"], t["sinks"], wl.w)
    torch.cuda.synchronize()
    assert torch.isfinite(y1.float()).all() and torch.equal(y1, y2)
