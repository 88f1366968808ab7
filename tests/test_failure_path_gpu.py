"""The failure path of the kernels' pipeline waits, exercised without a GPU
fault: every mbarrier wait in the kernels is bounded by wall time and, when it
runs out, records GDR_ERR_TIMEOUT in a device status word and lets the kernel
return.  gdr_selftest_bounded_wait runs that same bounded wait (20 ms limit) on
a barrier phase nothing completes; the test checks that the host reads the
timeout, that reading resets it, and that the next real call works."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_reports_timeout_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda:0")
    assert gdr.device_status() == gdr.GDR_OK            # clean start
    assert gdr.selftest_bounded_wait() == gdr.GDR_OK
    assert gdr.device_status() == gdr.GDR_ERR_TIMEOUT   # the wait ran out and was recorded
    assert gdr.device_status() == gdr.GDR_OK            # reading resets it
    inp = workloads.make_inputs(workloads.CONFIGS["B1_T256_H8_K128"])
    out = gdr.kkt_solve(inp["k"].to(dev), inp["g"].to(dev), inp["beta"].to(dev))
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"])
    assert np.abs(out.double().cpu().numpy() - ref).max() <= 2e-3
