"""The fused call inside a CUDA graph: after one ordinary call on the device
(which sets up the library's per-device state), the call is captured into a
graph on a side stream, and every replay reproduces the direct call bit for
bit, including after the inputs are overwritten in place (the graph reads them
at replay time) and for a packed varlen batch.  A graph removes the per-call
launch cost that dominates small workloads."""
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _inputs(wl, dev):
    inp = workloads.make_inputs(wl)
    return {k: (None if v is None else v.to(dev)) for k, v in inp.items()}


@pytest.mark.parametrize("name,out_dtype", [("B2_T2000_H5_K128", torch.float32),
                                             ("varlen8_H16_K128", torch.bfloat16)])
def test_capture_and_replay_matches_direct_call(name, out_dtype):
    dev = _dev()
    wl = workloads.CONFIGS[name]
    x = _inputs(wl, dev)
    ref = gdr.kkt_solve(x["k"], x["g"], x["beta"], x["cu_seqlens"], output_dtype=out_dtype)
    torch.cuda.synchronize(dev)

    out = torch.empty_like(ref)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    with torch.cuda.graph(graph, stream=side):
        gdr.kkt_solve(x["k"], x["g"], x["beta"], x["cu_seqlens"], output_dtype=out_dtype, out=out)
    for _ in range(3):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize(dev)
        assert torch.equal(out, ref)
    assert gdr.device_status() == gdr.GDR_OK

    # New values in the same buffers: a replay computes on them.
    y = _inputs(wl.with_(seed=wl.seed + 100), dev)
    for key in ("k", "g", "beta"):
        x[key].copy_(y[key])
    ref2 = gdr.kkt_solve(y["k"], y["g"], y["beta"], y["cu_seqlens"], output_dtype=out_dtype)
    graph.replay()
    torch.cuda.synchronize(dev)
    assert torch.equal(out, ref2)
    assert not torch.equal(ref2, ref)
