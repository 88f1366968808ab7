"""GPU parity for the other input types and head sizes (the MindSpeed-Ops PR #135
page, "How was this patch tested": fp32/bf16/fp16 inputs): head dimension
K in {64, 192, 256}, fp16 keys, fp32 and fp16 beta, fp16 output.  Every case is
compared with the fp64 oracle element by element.

Tolerances: fp32 output as in the main parity tests (max_abs <= 2e-3,
mean_rel <= 1e-5); bf16 output max_abs <= 1.5e-2; fp16 output
|gpu - ref| <= 2^-10 |ref| + 2e-5 for every element (one fp16 rounding of an
fp32-accurate result is at most 2^-11 |ref| for normal values), which a
bf16-rounded result (2^-9) would fail.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

F32_MAX_ABS, F32_MEAN_REL, BF16_MAX_ABS = 2e-3, 1e-5, 1.5e-2
OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to(x, dev):
    return None if x is None else x.to(dev)


def _real_rows(wl):
    if wl.varlen_lengths is None:
        return np.arange(wl.B * wl.T)
    return np.arange(int(workloads.cu_seqlens_of(wl)[-1]))


def _parity(wl, out_name):
    dev = _dev()
    inp = workloads.make_inputs(wl)
    out = gdr.kkt_solve(_to(inp["k"], dev), _to(inp["g"], dev), _to(inp["beta"], dev),
                        _to(inp["cu_seqlens"], dev), output_dtype=OUT[out_name])
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"])
    rows = _real_rows(wl)
    got = out.double().cpu().numpy().reshape(-1, wl.H, 64)[rows]
    ref = ref.reshape(-1, wl.H, 64)[rows]
    assert np.isfinite(got).all()
    d = np.abs(got - ref)
    if out_name == "f32":
        mean_rel = d.sum() / np.abs(ref).sum()
        assert d.max() <= F32_MAX_ABS and mean_rel <= F32_MEAN_REL, (wl, d.max(), mean_rel)
    elif out_name == "bf16":
        assert d.max() <= BF16_MAX_ABS, (wl, d.max())
    else:
        assert np.all(d <= np.abs(ref) * 2.0 ** -10 + 2e-5), (wl, (d - np.abs(ref) * 2.0 ** -10).max())
    # Structure that holds exactly: unit diagonal, zero upper triangle.
    loc = np.concatenate([np.arange(e - s) % 64 for s, e in workloads._sequence_bounds(wl)])
    assert np.all(got[np.arange(len(rows)), :, loc] == 1.0)
    upper = np.arange(64)[None, :] > loc[:, None]
    assert np.all(got.transpose(0, 2, 1)[upper] == 0.0)
    return got, ref


VARLEN_LENS = (1, 64, 0, 65, 130, 2, 200, 63)


@pytest.mark.parametrize("K", [64, 192, 256])
@pytest.mark.parametrize("layout", ["fixed", "varlen"])
@pytest.mark.parametrize("out_name", ["f32", "bf16"])
def test_head_dims(K, layout, out_name):
    if layout == "fixed":
        wl = workloads.Workload(f"K{K}_fixed", 2, 300, 5, K, out_name, seed=100 + K)
    else:
        wl = workloads.Workload(f"K{K}_varlen", len(VARLEN_LENS), sum(VARLEN_LENS), 3, K, out_name,
                                seed=200 + K, varlen_lengths=VARLEN_LENS)
    _parity(wl, out_name)


@pytest.mark.parametrize("K", [64, 256])
def test_head_dims_many_pairs_per_cta(K):
    # Enough tiles that every CTA runs many pairs through the stage ring
    # (K = 256 takes two ring stages per pair).
    wl = workloads.Workload(f"K{K}_large", 2, 4096, 16, K, "f32", seed=300 + K)
    _parity(wl, "f32")


@pytest.mark.parametrize("name", ["B2_T2000_H5_K128", "varlen8_H16_K128"])
def test_fp16_keys(name):
    wl = workloads.CONFIGS[name].with_(k_dtype="f16")
    _parity(wl, "f32")


@pytest.mark.parametrize("beta_dtype", ["f32", "f16"])
@pytest.mark.parametrize("k_dtype", ["bf16", "f16"])
def test_beta_dtypes(beta_dtype, k_dtype):
    wl = workloads.CONFIGS["B2_T2000_H5_K128"].with_(beta_dtype=beta_dtype, k_dtype=k_dtype)
    _parity(wl, "f32")


@pytest.mark.parametrize("name", ["B2_T2000_H5_K128", "B1_T8192_H8_K128", "varlen8_H16_K128"])
def test_fp16_output(name):
    _parity(workloads.CONFIGS[name], "f16")


def test_fp16_all_inputs_fp16_output_large_k():
    wl = workloads.Workload("all_f16_K256", 1, 1000, 6, 256, "f16", seed=400, k_dtype="f16",
                            beta_dtype="f16")
    _parity(wl, "f16")


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("layout,out_name", [("fixed", "f32"), ("varlen", "f32"), ("fixed", "bf16")])
def test_fp32_keys(K, layout, out_name):
    # fp32 keys: for fp32 (and fp16) output the Gram is formed from tf32 parts
    # and remainders (the tf32 product of the parts plus bf16 cross products,
    # about 2^-18 relative per key product), so fp32 output still meets the
    # fp32 tolerance; bf16 output takes one tf32 product (see below).
    if layout == "fixed":
        wl = workloads.Workload(f"f32keys_K{K}", 2, 300, 5, K, out_name, seed=800 + K, k_dtype="f32")
    else:
        wl = workloads.Workload(f"f32keys_K{K}_varlen", len(VARLEN_LENS), sum(VARLEN_LENS), 3, K, out_name,
                                seed=810 + K, varlen_lengths=VARLEN_LENS, k_dtype="f32", beta_dtype="f32")
    _parity(wl, out_name)


def test_fp32_keys_many_pairs_per_cta():
    _parity(workloads.Workload("f32keys_large", 2, 4096, 16, 128, "f32", seed=820, k_dtype="f32"), "f32")


@pytest.mark.parametrize("K", [64, 128])
def test_fp32_keys_fp16_output(K):
    # fp16 output takes the split Gram too: one fp16 rounding of an fp32-accurate
    # result.
    wl = workloads.Workload(f"f32keys_K{K}_f16", 2, 300, 5, K, "f16", seed=830 + K, k_dtype="f32",
                            beta_dtype="f16")
    _parity(wl, "f16")


@pytest.mark.parametrize("K,layout", [(64, "fixed"), (128, "varlen"), (128, "large")])
def test_fp32_keys_bf16_output_one_tf32_product(K, layout):
    # bf16 output takes one tf32 product of the keys as given: each key element is
    # narrowed by at most 2^-10 of itself, far below the output's own rounding
    # (2^-9 |ref|).  Besides the bf16 tolerance every bf16 output meets, the mean
    # error must stay at that rounding's scale (a dropped K part or a wrong box
    # would put it orders of magnitude higher).
    if layout == "fixed":
        wl = workloads.Workload(f"f32keys_K{K}_bf16", 3, 1000, 4, K, "bf16", seed=840 + K, k_dtype="f32")
    elif layout == "varlen":
        wl = workloads.Workload(f"f32keys_K{K}_bf16_varlen", len(VARLEN_LENS), sum(VARLEN_LENS), 3, K, "bf16",
                                seed=850 + K, varlen_lengths=VARLEN_LENS, k_dtype="f32", beta_dtype="f32")
    else:
        wl = workloads.Workload(f"f32keys_K{K}_bf16_large", 2, 4096, 16, K, "bf16", seed=860 + K, k_dtype="f32")
    got, ref = _parity(wl, "bf16")
    mean_rel = np.abs(got - ref).sum() / np.abs(ref).sum()
    assert mean_rel <= 2.0 ** -8, (wl.name, mean_rel)
