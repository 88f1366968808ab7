"""GPU parity of the chunk-128 kernel (PyPTO page "GatedDeltaRule算子性能优化案例",
section 3.2: chunk_size 128, TileShape [128, 128]) against the fp64 oracle run
with chunk 128, element by element: (I + A)^{-1} of every 128-token chunk and
head, written as [B, T, H, 128].  The log-gate inputs restart their running
sum every 128 tokens, as a chunk-128 caller's would (the result only depends on
differences of g inside a chunk).

Tolerances as in the chunk-64 tests: fp32 output max_abs <= 2e-3 and
mean_rel <= 1e-5; bf16 max_abs <= 1.5e-2; fp16 |gpu - ref| <= 2^-10 |ref| + 2e-5.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

C = 128
OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to(x, dev):
    return None if x is None else x.to(dev)


def _parity(wl, out_name):
    dev = _dev()
    inp = workloads.make_inputs(wl)
    out = gdr.kkt_solve(_to(inp["k"], dev), _to(inp["g"], dev), _to(inp["beta"], dev),
                        _to(inp["cu_seqlens"], dev), chunk_size=C, output_dtype=OUT[out_name])
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    assert out.shape[-1] == C
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"], chunk_size=C)
    if wl.varlen_lengths is None:
        rows = np.arange(wl.B * wl.T)
    else:
        rows = np.arange(int(workloads.cu_seqlens_of(wl)[-1]))
    got = out.double().cpu().numpy().reshape(-1, wl.H, C)[rows]
    ref = ref.reshape(-1, wl.H, C)[rows]
    assert np.isfinite(got).all()
    d = np.abs(got - ref)
    if out_name == "f32":
        mean_rel = d.sum() / np.abs(ref).sum()
        assert d.max() <= 2e-3 and mean_rel <= 1e-5, (wl.name, d.max(), mean_rel)
    elif out_name == "bf16":
        assert d.max() <= 1.5e-2, (wl.name, d.max())
    else:
        assert np.all(d <= np.abs(ref) * 2.0 ** -10 + 2e-5), (wl.name, (d - np.abs(ref) * 2.0 ** -10).max())
    loc = np.concatenate([np.arange(e - s) % C for s, e in workloads._sequence_bounds(wl)])
    assert np.all(got[np.arange(len(rows)), :, loc] == 1.0)
    upper = np.arange(C)[None, :] > loc[:, None]
    assert np.all(got.transpose(0, 2, 1)[upper] == 0.0)


def _wl(name, B, T, H, K=128, out="f32", seed=700, **kw):
    return workloads.Workload(name, B, T, H, K, out, seed=seed, chunk=C, **kw)


@pytest.mark.parametrize("B,T,H", [(1, 128, 1), (1, 256, 8), (2, 2000, 5), (3, 1050, 3), (1, 64, 2),
                                   (2, 127, 4), (1, 129, 7)])
def test_shapes_fp32(B, T, H):
    # 2000 = 15*128 + 80 and 1050 = 8*128 + 26: a last chunk with a short second
    # half, and one with no second half.
    _parity(_wl(f"c128_{B}_{T}_{H}", B, T, H, seed=700 + T + H), "f32")


@pytest.mark.parametrize("out_name", ["bf16", "f16"])
def test_16_bit_outputs(out_name):
    _parity(_wl("c128_out16", 2, 2000, 5, out=out_name, seed=711), out_name)


def test_large_bf16():
    _parity(_wl("c128_large", 1, 8192, 8, out="bf16", seed=712), "bf16")


def test_head_dim_64_and_fp16_keys():
    _parity(_wl("c128_K64", 2, 1000, 4, K=64, seed=713), "f32")
    _parity(_wl("c128_f16", 2, 1000, 4, seed=714, k_dtype="f16", beta_dtype="f32"), "f32")


@pytest.mark.parametrize("use_g,use_beta", [(False, True), (True, False)])
def test_none_variants(use_g, use_beta):
    _parity(_wl("c128_none", 2, 700, 3, seed=715, use_g=use_g, use_beta=use_beta), "f32")


def test_varlen():
    lens = (1, 128, 0, 129, 64, 65, 300, 2, 255)
    _parity(_wl("c128_varlen", len(lens), sum(lens), 3, seed=716, varlen_lengths=lens), "f32")
    _parity(workloads.CONFIGS["varlen8_H16_K128"].with_(chunk=C, name="c4_c128"), "f32")


@pytest.mark.parametrize("out_name", ["bf16", "f16"])
def test_varlen_16_bit_outputs(out_name):
    # 16-bit output stores full chunks by TMA (four 64 x 64 boxes) and partial
    # chunks row by row: full chunks here sit between partial ones, in packed
    # sequences, so a box written past its chunk would show in a neighbour.
    lens = (128, 1, 256, 127, 129, 0, 384, 65)
    _parity(_wl("c128_varlen16", len(lens), sum(lens), 3, out=out_name, seed=717, varlen_lengths=lens),
            out_name)
