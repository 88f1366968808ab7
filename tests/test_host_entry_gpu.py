"""gdr_kkt_solve_host (the fused call on host buffers, copies pipelined over two
streams) against the device call on the same inputs: equal bit for bit on
these inputs (every chunk's log-gate is within the factored gate's bound), for
fixed-length batches cut into many slices, partial chunks, 128-token chunks,
fp32 keys, page-locked and pageable host memory, and packed sequences, whose
output rows past the last sequence are left untouched."""
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _device_call(inp, dev, chunk, out_dtype):
    to = lambda t: None if t is None else t.to(dev)
    out = gdr.kkt_solve(to(inp["k"]), to(inp["g"]), to(inp["beta"]), to(inp["cu_seqlens"]), chunk_size=chunk,
                        output_dtype=out_dtype)
    torch.cuda.synchronize(dev)
    return out.cpu()


def _host_call(inp, dev, chunk, out_dtype, pinned, out=None):
    host = {k: (None if v is None else (v.pin_memory() if pinned else v.clone())) for k, v in inp.items()}
    with torch.cuda.device(dev):
        res = gdr.kkt_solve_host(host["k"], host["g"], host["beta"], host["cu_seqlens"], chunk_size=chunk,
                                 output_dtype=out_dtype, out=out)
        torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    return res


@pytest.mark.parametrize("wl,chunk,out_dtype,pinned", [
    (workloads.CONFIGS["B2_T2000_H5_K128"], 64, torch.float32, True),
    (workloads.CONFIGS["B2_T2000_H5_K128"], 64, torch.float32, False),
    (workloads.CONFIGS["B2_T2000_H5_K128"].with_(chunk=128, name="B2_T2000_H5_K128_C128"), 128, torch.bfloat16,
     True),
    (workloads.CONFIGS["B2_T2000_H5_K128"].with_(K=64, k_dtype="f32", name="B2_T2000_H5_K64_kf32"), 64,
     torch.bfloat16, True),
    (workloads.Workload("B3_T70000_H2_K128", 3, 70000, 2, 128, "bf16", seed=950), 64, torch.bfloat16, True),
    (workloads.CONFIGS["B2_T16384_H32_K128"], 64, torch.bfloat16, True),
])
def test_host_entry_equals_device_call(wl, chunk, out_dtype, pinned):
    dev = _dev()
    inp = workloads.make_inputs(wl)
    want = _device_call(inp, dev, chunk, out_dtype)
    got = _host_call(inp, dev, chunk, out_dtype, pinned)
    assert got.dtype == want.dtype and got.shape == want.shape
    assert torch.equal(got, want)


def test_host_entry_packed_sequences_leave_other_rows_untouched():
    dev = _dev()
    wl = workloads.CONFIGS["varlen8_H16_K128"]
    inp = workloads.make_inputs(wl)
    # Ten more token rows than the sequences cover.
    def pad(t):
        return torch.cat([t, torch.zeros((1, 10) + tuple(t.shape[2:]), dtype=t.dtype)], dim=1)
    inp = dict(inp, k=pad(inp["k"]), g=pad(inp["g"]), beta=pad(inp["beta"]))
    want = _device_call(inp, dev, 64, torch.float32)
    T = inp["k"].shape[1]
    real = int(inp["cu_seqlens"][-1])
    out = torch.full((1, T, wl.H, 64), 7.0, dtype=torch.float32).pin_memory()
    got = _host_call(inp, dev, 64, torch.float32, True, out=out)
    assert torch.equal(got[:, :real], want[:, :real])
    assert torch.all(got[:, real:] == 7.0)
