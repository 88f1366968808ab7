"""Host-side helpers of bench.py that need no GPU: the hold before a timed region
and the byte accounting behind `roofline.achieved`."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_hold_covers_the_first_launches_and_is_capped():
    # Four times the host time of min(K, HOLD_LAUNCHES) calls plus 2 ms ...
    assert abs(bench.hold_time(10e-6, 20) - (2e-3 + 4 * 10e-6 * 20)) < 1e-12
    assert abs(bench.hold_time(10e-6, 20000) - (2e-3 + 4 * 10e-6 * bench.HOLD_LAUNCHES)) < 1e-12
    # ... never more than HOLD_MAX_S, however slow the host (a profiler, a busy box).
    assert bench.hold_time(1.0, 20000) == bench.HOLD_MAX_S
    # Monotone in both arguments.
    assert bench.hold_time(5e-6, 100) <= bench.hold_time(6e-6, 100) <= bench.hold_time(6e-6, 200)


def test_bytes_per_token_head_match_the_tensors():
    # k (K elements), g (fp32), beta, and the output row (chunk values).
    wl = workloads.CONFIGS["B2_T16384_H32_K128"]
    assert bench.bytes_per_token_head(wl, "bf16") == 128 * 2 + 4 + 2 + 64 * 2 == 390
    assert bench.bytes_per_token_head(wl, "f32") == 128 * 2 + 4 + 2 + 64 * 4 == 518
    f32k = wl.with_(k_dtype="f32")
    assert bench.bytes_per_token_head(f32k, "f32") == 128 * 4 + 4 + 2 + 64 * 4 == 774
    c128 = wl.with_(chunk=128)
    assert bench.bytes_per_token_head(c128, "bf16") == 128 * 2 + 4 + 2 + 128 * 2 == 518


def test_recorded_traffic_only_for_the_current_kernel_source():
    wl = workloads.CONFIGS["B2_T16384_H32_K128"]
    t = bench.recorded_traffic(wl, "bf16")
    # Either the committed capture matches this source (a DRAM byte count of the
    # right order: reads ~ 275 MB) or the lookup refuses it (None).
    assert t is None or 2.5e8 < t < 5e8
