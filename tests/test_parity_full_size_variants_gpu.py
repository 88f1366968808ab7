"""GPU parity at the full (2, 16384, 32, K) size for every variant the benchmark
times at that size (the head dimensions, fp16 inputs and outputs, fp32 keys,
fp32 output and 128-token chunks; the default bf16 line is covered in
test_parity_gpu.py).  Each run goes through the same public call as the
benchmark, and every tile of the workload is compared with the fp64 oracle
element by element; every row is also checked for the properties that hold at
any size: finite values, unit diagonal, zero strictly-upper part.

Tolerances as everywhere: fp32 output max_abs <= 2e-3 and mean_rel <= 1e-5;
bf16 output max_abs <= 1.5e-2, every element |gpu - ref| <= 2^-8 |ref| + 1e-3,
and mean_rel at most twice that of the exact result rounded to bf16; fp16
output |gpu - ref| <= 2^-10 |ref| + 2e-5 for every element.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
BASE = workloads.CONFIGS["B2_T16384_H32_K128"]


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _check(got, ref, out_name, what):
    d = np.abs(got - ref)
    assert np.isfinite(got).all(), what
    mean_rel = float(d.sum() / np.abs(ref).sum())
    if out_name == "f32":
        assert d.max() <= 2e-3 and mean_rel <= 1e-5, (what, d.max(), mean_rel)
    elif out_name == "bf16":
        assert d.max() <= 1.5e-2, (what, d.max())
        excess = d - (np.abs(ref) * 2.0 ** -8 + 1e-3)
        assert excess.max() <= 0, (what, "element-wise bf16 bound", float(excess.max()))
        r = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        rnd = float(np.abs(r - ref).sum() / np.abs(ref).sum())
        assert mean_rel <= 2.0 * rnd, (what, "bf16 mean_rel", mean_rel, rnd)
    else:
        assert np.all(d <= np.abs(ref) * 2.0 ** -10 + 2e-5), (what, (d - np.abs(ref) * 2.0 ** -10).max())
    print(f"parity {what} {out_name}: max_abs={float(d.max()):.3e} mean_rel={mean_rel:.3e}")


@pytest.mark.parametrize("K,k_dtype,beta_dtype,chunk,out_name", [
    (128, "bf16", "bf16", 64, "f32"),
    (256, "bf16", "bf16", 64, "bf16"),
    (64, "bf16", "bf16", 64, "bf16"),
    (128, "f16", "f16", 64, "f16"),
    (128, "f32", "bf16", 64, "bf16"),
    (128, "f32", "bf16", 64, "f32"),
    (128, "bf16", "bf16", 128, "bf16"),
    (128, "bf16", "bf16", 128, "f32"),
])
def test_full_size_variant(K, k_dtype, beta_dtype, chunk, out_name):
    dev = _dev()
    wl = BASE.with_(K=K, k_dtype=k_dtype, beta_dtype=beta_dtype, chunk=chunk, out_dtype=out_name,
                    name=f"B2_T16384_H32_K{K}_k{k_dtype}_C{chunk}")
    inp = workloads.make_inputs(wl)
    out = gdr.kkt_solve(inp["k"].to(dev), inp["g"].to(dev), inp["beta"].to(dev), None,
                        chunk_size=chunk, output_dtype=OUT[out_name])
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    flat = out.view(-1, wl.H, chunk)
    # Every row: finite, unit diagonal, zeros above it (T is a multiple of the
    # chunk, so every chunk is full).
    assert torch.isfinite(flat).all()
    loc = torch.arange(wl.T, device=dev).remainder(chunk).repeat(wl.B)
    diag = flat.gather(2, loc.view(-1, 1, 1).expand(-1, wl.H, 1)).squeeze(-1)
    assert torch.all(diag == 1)
    upper = torch.arange(chunk, device=dev).view(1, 1, chunk) > loc.view(-1, 1, 1)
    assert torch.all(flat.masked_select(upper) == 0)
    # Every tile against the oracle.
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], chunk_size=chunk)
    got = out.double().cpu().numpy()
    del out, flat
    _check(got.reshape(-1, chunk), ref.reshape(-1, chunk), out_name, wl.name)
