"""GPU check of gdr_kkt_solve_unfused_noalloc, the entry point for callers that
may not allocate device memory while they run (a serving runtime whose device
memory is planned up front, or code that cannot afford cudaMalloc's implicit
device synchronisation).  It runs the unfused chain through the library's fixed
device scratch, so it is compared, through the C ABI, with the existing entry
point gdr_kkt_solve_ex on the same inputs, on two calls in a row of different
sizes (the second call finds the first call's A in the shared scratch), and
each result is also compared with the fp64 oracle directly, within the same
tolerances as every other parity test.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it does not depend on them.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

F32_MAX_ABS, F32_MEAN_REL, BF16_MAX_ABS = 2e-3, 1e-5, 1.5e-2
CODES = {torch.float32: gdr.GDR_F32, torch.bfloat16: gdr.GDR_BF16, torch.float16: gdr.GDR_F16}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _both(wl, out_dtype, dev, stream):
    inp = workloads.make_inputs(wl)
    k, g, b = (None if inp[x] is None else inp[x].to(dev) for x in ("k", "g", "beta"))
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].to(dev)
    B = wl.B
    outs = []
    for fn in (gdr.kkt_solve_ex_raw, gdr.kkt_solve_unfused_noalloc_raw):
        out = torch.full((*k.shape[:3], 64), float("nan"), dtype=out_dtype, device=dev)
        rc = fn(k.data_ptr(), CODES[k.dtype], g.data_ptr(), b.data_ptr(), CODES[b.dtype],
                0 if cu is None else cu.data_ptr(), B, k.shape[1], wl.H, wl.K, 64, CODES[out_dtype],
                out.data_ptr(), stream)
        assert rc == gdr.GDR_OK, gdr.status_string(rc)
        outs.append(out)
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    rows = np.arange(wl.token_heads // wl.H)
    ref, got = (o.reshape(-1, wl.H, 64)[torch.from_numpy(rows).to(dev)].double().cpu().numpy() for o in outs)
    exact = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"]).reshape(-1, wl.H, 64)[rows]
    return ref, got, exact


def _within_tolerance(got, want, out_dtype, what):
    assert np.isfinite(got).all(), what
    d = np.abs(got - want)
    if out_dtype == torch.float32:
        assert d.max() <= F32_MAX_ABS and d.sum() / np.abs(want).sum() <= F32_MEAN_REL, (what, d.max())
    else:
        assert d.max() <= BF16_MAX_ABS, (what, d.max())


def test_noalloc_matches_the_existing_entry_point_on_two_calls_in_a_row():
    dev = _dev()
    stream = torch.cuda.current_stream(dev).cuda_stream
    lens = (1, 64, 0, 65, 130, 2, 200, 63)
    calls = [
        (workloads.CONFIGS["varlen8_H16_K128"], torch.float32),                       # varlen, 262144 token-heads at most
        (workloads.Workload("noalloc_small", 2, 300, 5, 128, "bf16", seed=601), torch.bfloat16),
        (workloads.Workload("noalloc_varlen", len(lens), sum(lens), 3, 256, "f32", seed=602,
                            varlen_lengths=lens), torch.float32),
    ]
    assert calls[0][0].token_heads <= 1 << 18
    for wl, out_dtype in calls:
        ref, got, exact = _both(wl, out_dtype, dev, stream)
        _within_tolerance(got, ref, out_dtype, wl.name + " vs gdr_kkt_solve_ex")
        _within_tolerance(got, exact, out_dtype, wl.name + " vs the oracle")
        # The chain runs the fused step's own arithmetic: the results agree exactly.
        assert np.array_equal(got, ref), (wl.name, np.abs(got - ref).max())


def test_noalloc_rejects_problems_beyond_its_scratch():
    dev = _dev()
    k = torch.zeros(1, 1 << 16, 5, 128, dtype=torch.bfloat16, device=dev)   # 327680 token-heads
    out = torch.zeros(1, 1 << 16, 5, 64, dtype=torch.float32, device=dev)
    rc = gdr.kkt_solve_unfused_noalloc_raw(k.data_ptr(), gdr.GDR_BF16, 0, 0, gdr.GDR_F32, 0, 1, 1 << 16, 5,
                                           128, 64, gdr.GDR_F32, out.data_ptr(), 0)
    assert rc == gdr.GDR_ERR_SCRATCH
    assert gdr.status_string(rc).startswith("problem too large")
