"""Host-side logic of bench.py: algorithmic byte and flop counts of the workloads."""
import bench
from gated_linear_sliding_gb300 import inputs as I


def test_forward_bytes_llama_layer():
    # q 64 MiB + k, v, g 16 MiB each + y 64 MiB + Wf 128 KiB + sinks 512 B
    assert bench.fwd_algorithmic_bytes(I.LLAMA3_8B_L8K) == \
        2 * 67108864 + 3 * 16777216 + 131072 + 512


def test_forward_flops_llama_layer():
    # per query-head token dD + 2Dd + 2D + 4wd; per KV-head token dD + 3Dd + 2D
    wl = I.LLAMA3_8B_L8K
    fq = 128 * 128 + 2 * 128 * 128 + 2 * 128 + 4 * 64 * 128
    fk = 128 * 128 + 3 * 128 * 128 + 2 * 128
    assert bench.fwd_algorithmic_flops(wl) == 8192 * (32 * fq + 8 * fk)
    assert abs(bench.fwd_algorithmic_flops(wl) / 1e9 - 25.85) < 0.01


def test_decode_bytes_b64():
    b = bench.decode_algorithmic_bytes(I.DECODE_B64)
    assert 85e6 < b < 87e6


def test_peaks_file_or_fallback():
    hbm, tc, src = bench.load_peaks()
    assert hbm > 1000 and tc > 100 and src in ("measured", "fallback")
