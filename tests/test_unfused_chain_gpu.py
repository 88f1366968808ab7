"""GPU checks of the unfused chain (MindSpeed-Ops PR #135 page, "What this PR
does": chunk_scaled_dot_kkt_fwd writes A [B, T, H, 64] to HBM and solve_tril
reads it; the fused call replaces the pair).

  * A from gdr_chunk_scaled_dot_kkt against the fp64 oracle's A, element by
    element (max_abs <= 2e-5: fp32 products of bf16 keys and fp32 gates), and
    exactly zero on and above the diagonal and past the chunk;
  * gdr_solve_tril of an arbitrary strictly lower A against the oracle's solve
    of the same A (fp32 tolerance of the main parity tests);
  * the chain of the two calls equals the fused call bit for bit, as the page's
    tests check the fused kernel against the unfused chain bit by bit ("How was
    this patch tested").
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

F32_MAX_ABS, F32_MEAN_REL = 2e-3, 1e-5
OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
VARLEN_LENS = (1, 64, 0, 65, 130, 2, 200, 63)


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to(x, dev):
    return None if x is None else x.to(dev)


def _rows(wl):
    if wl.varlen_lengths is None:
        return np.arange(wl.B * wl.T)
    return np.arange(int(workloads.cu_seqlens_of(wl)[-1]))


def _workload(name):
    if name == "varlen":
        return workloads.Workload("chain_varlen", len(VARLEN_LENS), sum(VARLEN_LENS), 3, 128, "f32",
                                  seed=501, varlen_lengths=VARLEN_LENS)
    if name == "K256":
        return workloads.Workload("chain_K256", 2, 300, 5, 256, "f32", seed=502)
    if name == "c2_nog":
        return workloads.CONFIGS["B2_T2000_H5_K128"].with_(use_g=False)
    return workloads.CONFIGS[name]


@pytest.mark.parametrize("name", ["B1_T256_H8_K128", "B2_T2000_H5_K128", "c2_nog", "varlen8_H16_K128", "varlen", "K256"])
def test_A_against_oracle(name):
    dev = _dev()
    wl = _workload(name)
    inp = workloads.make_inputs(wl)
    A = gdr.chunk_scaled_dot_kkt(_to(inp["k"], dev), _to(inp["g"], dev), _to(inp["beta"], dev),
                                 _to(inp["cu_seqlens"], dev))
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    ref = oracle.chunk_A_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"]).reshape(-1, wl.H, 64)
    rows = _rows(wl)
    got = A.double().cpu().numpy().reshape(-1, wl.H, 64)[rows]
    ref = ref[rows]
    d = np.abs(got - ref)
    assert d.max() <= 2e-5, d.max()
    loc = np.concatenate([np.arange(e - s) % 64 for s, e in workloads._sequence_bounds(wl)])
    upper = np.arange(64)[None, :] >= loc[:, None]            # on or above the diagonal
    assert np.all(got.transpose(0, 2, 1)[upper] == 0.0)


@pytest.mark.parametrize("layout", ["fixed", "varlen"])
@pytest.mark.parametrize("out_name", ["f32", "bf16", "f16"])
def test_solve_tril_of_given_A(layout, out_name):
    dev = _dev()
    rng = np.random.default_rng(503)
    if layout == "fixed":
        B, T, H, cu = 2, 300, 3, None
        bounds = [(b * T, (b + 1) * T) for b in range(B)]
        lead = (B, T)
    else:
        cu = np.concatenate([[0], np.cumsum(VARLEN_LENS)]).astype(np.int32)
        B, T, H = len(VARLEN_LENS), int(cu[-1]), 3
        bounds = [(int(cu[n]), int(cu[n + 1])) for n in range(B)]
        lead = (1, T)
    ntok = lead[0] * lead[1]
    A = np.zeros((ntok, H, 64), dtype=np.float32)
    for s, e in bounds:
        for c0 in range(s, e, 64):
            L = min(64, e - c0)
            for h in range(H):
                A[c0:c0 + L, h, :L] = np.tril(rng.standard_normal((L, L)).astype(np.float32) * 0.15, k=-1)
    At = torch.from_numpy(A).reshape(*lead, H, 64)
    cut = None if cu is None else torch.from_numpy(cu)
    X = gdr.solve_tril(At.to(dev), _to(cut, dev), output_dtype=OUT[out_name])
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    ref = oracle.solve_tril_ref(At.double(), cut).reshape(-1, H, 64)
    rows = np.concatenate([np.arange(s, e) for s, e in bounds])
    got = X.double().cpu().numpy().reshape(-1, H, 64)[rows]
    ref = ref[rows]
    d = np.abs(got - ref)
    if out_name == "f32":
        assert d.max() <= F32_MAX_ABS and d.sum() / np.abs(ref).sum() <= F32_MEAN_REL
    elif out_name == "bf16":
        assert d.max() <= 1.5e-2
    else:
        assert np.all(d <= np.abs(ref) * 2.0 ** -10 + 2e-5)


@pytest.mark.parametrize("name,out_name", [("B1_T256_H8_K128", "f32"), ("B2_T2000_H5_K128", "f32"), ("c2_nog", "f32"),
                                           ("B1_T8192_H8_K128", "bf16"), ("B1_T8192_H8_K128", "f32"), ("varlen8_H16_K128", "f32"),
                                           ("varlen", "bf16"), ("K256", "f16")])
def test_chain_equals_fused_bit_for_bit(name, out_name):
    dev = _dev()
    wl = _workload(name)
    inp = workloads.make_inputs(wl)
    k, g, b, cu = (_to(inp[x], dev) for x in ("k", "g", "beta", "cu_seqlens"))
    fused = gdr.kkt_solve(k, g, b, cu, output_dtype=OUT[out_name])
    A = gdr.chunk_scaled_dot_kkt(k, g, b, cu)
    chain = gdr.solve_tril(A, cu, output_dtype=OUT[out_name])
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    rows = torch.from_numpy(_rows(wl)).to(dev)
    f = fused.reshape(-1, wl.H, 64).index_select(0, rows)
    c = chain.reshape(-1, wl.H, 64).index_select(0, rows)
    bits = torch.int32 if f.element_size() == 4 else torch.int16
    assert torch.equal(f.contiguous().view(bits), c.contiguous().view(bits)), \
        (f.double() - c.double()).abs().max().item()
