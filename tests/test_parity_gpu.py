"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances (fixed for the method): fp32 output max_abs <= 2e-3 and
mean_rel <= 1e-5; bf16 output max_abs <= 1.5e-2, with
max_abs = max |gpu - ref| and mean_rel = sum |gpu - ref| / sum |ref| over the
rows of real tokens.  bf16 output is held to two more bounds derived from its
rounding: every element |gpu - ref| <= 2^-8 |ref| + 1e-3 (one bf16 rounding,
2^-9 relative, plus the single tf32 pass of the merge), and mean_rel at most
twice the mean_rel of rounding the exact result itself to bf16 (a systematic
one-ulp error would be about four times it).  Every workload, the
(2, 16384, 32, 128) one included, is compared with the oracle element by element
on every row of a real token.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import gated_deltanet_chunked_gdr_gb300 as gdr  # noqa: E402
import oracle  # noqa: E402
import workloads  # noqa: E402

pytestmark = pytest.mark.gpu

F32_MAX_ABS, F32_MEAN_REL, BF16_MAX_ABS = 2e-3, 1e-5, 1.5e-2


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to(x, dev):
    return None if x is None else x.to(dev)


def _run(inp, out_dtype, dev, stream=None):
    out = gdr.kkt_solve(_to(inp["k"], dev), _to(inp["g"], dev), _to(inp["beta"], dev),
                        _to(inp["cu_seqlens"], dev), output_dtype=out_dtype, stream=stream)
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    return out


def _metrics(got, ref):
    d = np.abs(got - ref)
    return float(d.max()), float(d.sum() / np.abs(ref).sum())


def _rounding_mean_rel(ref):
    """mean_rel of the exact result rounded to bf16 (round-to-nearest-even)."""
    r = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    return float(np.abs(r - ref).sum() / np.abs(ref).sum())


def _check(got, ref, out_dtype, what=""):
    max_abs, mean_rel = _metrics(got, ref)
    assert np.isfinite(got).all(), what
    if out_dtype == torch.float32:
        assert max_abs <= F32_MAX_ABS and mean_rel <= F32_MEAN_REL, (what, max_abs, mean_rel)
    else:
        assert max_abs <= BF16_MAX_ABS, (what, max_abs, mean_rel)
        excess = np.abs(got - ref) - (np.abs(ref) * 2.0 ** -8 + 1e-3)
        assert excess.max() <= 0, (what, "element-wise bf16 bound", float(excess.max()))
        rnd = _rounding_mean_rel(ref)
        assert mean_rel <= 2.0 * rnd, (what, "bf16 mean_rel", mean_rel, rnd)
    print(f"parity {what} {out_dtype}: max_abs={max_abs:.3e} mean_rel={mean_rel:.3e}")
    return max_abs, mean_rel


def _real_rows(wl):
    if wl.varlen_lengths is None:
        return np.arange(wl.B * wl.T)
    cu = workloads.cu_seqlens_of(wl)
    return np.arange(int(cu[-1]))


def _full_parity(wl, out_dtype, dev):
    inp = workloads.make_inputs(wl)
    out = _run(inp, out_dtype, dev)
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"])
    got = out.double().cpu().numpy().reshape(-1, wl.H, 64)
    rows = _real_rows(wl)
    return _check(got[rows], ref.reshape(-1, wl.H, 64)[rows], out_dtype, wl.name), out


@pytest.mark.parametrize("name,out_dtype", [
    ("B1_T256_H8_K128", torch.float32), ("B2_T2000_H5_K128", torch.float32), ("B1_T8192_H8_K128", torch.bfloat16), ("B1_T8192_H8_K128", torch.float32),
    ("varlen8_H16_K128", torch.float32), ("B1_T256_H8_K128", torch.bfloat16), ("varlen8_H16_K128", torch.bfloat16)])
def test_workload_full_parity(name, out_dtype):
    _full_parity(workloads.CONFIGS[name], out_dtype, _dev())


@pytest.mark.parametrize("use_g,use_beta", [(False, True), (True, False), (False, False)])
def test_none_variants_partial_chunk_odd_heads(use_g, use_beta):
    wl = workloads.CONFIGS["B2_T2000_H5_K128"].with_(use_g=use_g, use_beta=use_beta)
    _full_parity(wl, torch.float32, _dev())


@pytest.mark.parametrize("B,T,H", [(1, 1, 1), (3, 63, 1), (2, 64, 2), (3, 65, 3), (1, 130, 7),
                                   (2, 191, 4), (1, 64 * 5 + 17, 1)])
def test_edge_shapes(B, T, H):
    wl = workloads.Workload(f"edge_{B}_{T}_{H}", B, T, H, 128, "f32", seed=50 + T + H)
    _full_parity(wl, torch.float32, _dev())


def test_varlen_edge_lengths_and_empty_sequence():
    lens = (1, 64, 0, 65, 128, 2, 63, 200, 0, 129)
    wl = workloads.Workload("varlen_edges", len(lens), sum(lens), 3, 128, "f32", seed=77,
                            varlen_lengths=lens)
    _full_parity(wl, torch.float32, _dev())


def test_varlen_equals_separate_runs():
    dev = _dev()
    wl = workloads.CONFIGS["varlen8_H16_K128"]
    inp = workloads.make_inputs(wl)
    packed = _run(inp, torch.float32, dev)
    cu = workloads.cu_seqlens_of(wl)
    for n in range(wl.B):
        s, e = int(cu[n]), int(cu[n + 1])
        one = {"k": inp["k"][:, s:e], "g": inp["g"][:, s:e], "beta": inp["beta"][:, s:e],
               "cu_seqlens": None}
        alone = _run(one, torch.float32, dev)
        assert torch.equal(packed[:, s:e], alone), n


def test_steep_gate_within_clamp():
    # log-gates falling by up to ~0.7 per token: differences down to about -44.
    dev = _dev()
    wl = workloads.CONFIGS["B1_T256_H8_K128"]
    inp = workloads.make_inputs(wl)
    rng = np.random.default_rng(9)
    a = -0.7 * rng.random((wl.B * wl.T, wl.H)).astype(np.float32)
    g = np.empty_like(a)
    for c0 in range(0, wl.T, 64):
        g[c0:c0 + 64] = np.cumsum(a[c0:c0 + 64], axis=0, dtype=np.float32)
    inp["g"] = torch.from_numpy(g).reshape(wl.B, wl.T, wl.H)
    out = _run(inp, torch.float32, dev)
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"])
    _check(out.double().cpu().numpy(), ref, torch.float32, "steep gate")


def _with_gate(wl, per_token, seed):
    inp = workloads.make_inputs(wl)
    rng = np.random.default_rng(seed)
    a = per_token(rng, (wl.B * wl.T, wl.H)).astype(np.float32)
    g = np.empty_like(a)
    for b in range(wl.B):
        for c0 in range(b * wl.T, (b + 1) * wl.T, 64):
            c1 = min(c0 + 64, (b + 1) * wl.T)
            g[c0:c1] = np.cumsum(a[c0:c1], axis=0, dtype=np.float32)
    inp["g"] = torch.from_numpy(g).reshape(wl.B, wl.T, wl.H)
    return inp


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gate_range_beyond_factorisation_guard(out_dtype):
    # Decays up to 3 per token: a chunk's log-gate spans ~95, beyond the range
    # where exp(g_i - g_j) is factored, so the direct clamped form runs.
    dev = _dev()
    wl = workloads.CONFIGS["B2_T2000_H5_K128"]
    inp = _with_gate(wl, lambda rng, sh: -3.0 * rng.random(sh), 31)
    out = _run(inp, out_dtype, dev)
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"])
    _check(out.double().cpu().numpy(), ref, out_dtype, "steep decay")


def test_non_monotone_gate():
    # Log-gates that rise and fall inside a chunk (|steps| <= 0.3).
    dev = _dev()
    wl = workloads.CONFIGS["B1_T256_H8_K128"]
    inp = _with_gate(wl, lambda rng, sh: rng.uniform(-0.3, 0.3, sh), 32)
    out = _run(inp, torch.float32, dev)
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"])
    _check(out.double().cpu().numpy(), ref, torch.float32, "non-monotone gate")


def test_bf16_output_against_fp32_output():
    # The bf16 path rounds its fp32 result to bf16 (its merge products take one
    # tf32 pass, the fp32 path three): it must agree with the fp32 output to
    # within bf16 rounding plus a tf32-level term, and the unit diagonal and
    # the zero upper triangle must be exact.
    dev = _dev()
    inp = workloads.make_inputs(workloads.CONFIGS["B2_T2000_H5_K128"])
    f32 = _run(inp, torch.float32, dev).double()
    bf = _run(inp, torch.bfloat16, dev).double()
    diff = (bf - f32).abs()
    assert torch.all(diff <= f32.abs() * 2.0 ** -8 + 1e-3)
    flat_f, flat_b = f32.view(-1, 5, 64), bf.view(-1, 5, 64)
    loc = torch.arange(2000, device=dev).remainder(64).repeat(2)
    cols = torch.arange(64, device=dev)
    upper = (cols.view(1, 1, 64) > loc.view(-1, 1, 1)).expand_as(flat_b)
    assert torch.all(flat_b[upper] == 0)
    diag = flat_b.gather(2, loc.view(-1, 1, 1).expand(-1, 5, 1))
    assert torch.all(diag == 1)


def test_deterministic_and_stream_aware():
    dev = _dev()
    inp = workloads.make_inputs(workloads.CONFIGS["varlen8_H16_K128"])
    a = _run(inp, torch.float32, dev)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        b = _run(inp, torch.float32, dev, stream=s.cuda_stream)
    assert torch.equal(a, b)


def test_no_writes_outside_real_rows_or_buffer():
    # Canary: the output view sits inside a larger buffer filled with a
    # sentinel; cu[B] < T leaves the tail rows unwritten.
    dev = _dev()
    lens = (70, 1, 130)
    T = sum(lens) + 37
    wl = workloads.Workload("canary", len(lens), T, 5, 128, "f32", seed=5)
    inp = workloads.make_inputs(wl.with_(varlen_lengths=lens + (37,), B=4))
    cu = torch.tensor([0, 70, 71, 201], dtype=torch.int32)
    pad = 4096
    buf = torch.full((pad + T * 5 * 64 + pad,), 7.25, dtype=torch.float32, device=dev)
    out = buf[pad:pad + T * 5 * 64].view(1, T, 5, 64)
    gdr.kkt_solve(inp["k"].to(dev), inp["g"].to(dev), inp["beta"].to(dev), cu.to(dev), out=out)
    torch.cuda.synchronize(dev)
    assert gdr.device_status() == gdr.GDR_OK
    assert torch.all(buf[:pad] == 7.25) and torch.all(buf[-pad:] == 7.25)
    assert torch.all(out[:, 201:] == 7.25)
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], cu)
    _check(out[:, :201].double().cpu().numpy(), ref[:, :201], torch.float32, "canary")


def test_golden_fixture_rows():
    import os
    dev = _dev()
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    inp = workloads.make_inputs(mg.WL)
    out = _run(inp, torch.float32, dev).double().cpu().numpy().reshape(-1, mg.WL.H, 64)
    got, want = [], []
    for line in open(os.path.join(here, "oracle_small.txt")):
        if line.startswith("#"):
            continue
        parts = line.split()
        r, h = int(parts[0]), int(parts[1])
        got.append(out[r, h])
        want.append(np.array([float(v) for v in parts[2:]]))
    _check(np.array(got), np.array(want), torch.float32, "golden")


def test_full_size_bf16_every_tile():
    # The benchmark's workload and launch: all 16384 (chunk, head) tiles against
    # the oracle element by element, plus the exact structure of every row.
    dev = _dev()
    wl = workloads.CONFIGS["B2_T16384_H32_K128"]
    inp = workloads.make_inputs(wl)
    out = _run(inp, torch.bfloat16, dev)
    flat = out.view(-1, wl.H, 64)
    assert torch.isfinite(flat).all()
    loc = torch.arange(wl.T, device=dev).remainder(64).repeat(wl.B)       # row within chunk
    cols = torch.arange(64, device=dev)
    diag = flat.gather(2, loc.view(-1, 1, 1).expand(-1, wl.H, 1)).squeeze(-1)
    assert torch.all(diag == 1)
    upper = cols.view(1, 1, 64) > loc.view(-1, 1, 1)
    assert torch.all(flat.masked_select(upper) == 0)
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"])
    got = out.double().cpu().numpy()
    _check(got.reshape(-1, 64), ref.reshape(-1, 64), torch.bfloat16, "B2_T16384_H32_K128 all tiles")
    # Per-tile view: the worst tile, so a fault confined to one CTA, pair slot or
    # warpgroup would show even if the average stayed small.
    per_tile = np.abs(got - ref).reshape(wl.B, wl.T // 64, 64, wl.H, 64).max(axis=(2, 4))
    assert per_tile.max() <= BF16_MAX_ABS


def _sampled_parity_and_invariants(wl, out_dtype, count):
    dev = _dev()
    inp = workloads.make_inputs(wl)
    out = _run(inp, out_dtype, dev)
    flat = out.view(-1, wl.H, 64)
    rows = torch.from_numpy(_real_rows(wl)).to(dev)
    real = flat.index_select(0, rows)
    assert torch.isfinite(real).all()
    loc = torch.from_numpy(np.concatenate([np.arange(e - s) % 64 for s, e in workloads._sequence_bounds(wl)])).to(dev)
    diag = real.gather(2, loc.view(-1, 1, 1).expand(-1, wl.H, 1)).squeeze(-1)
    assert torch.all(diag == 1)
    upper = torch.arange(64, device=dev).view(1, 1, 64) > loc.view(-1, 1, 1)
    assert torch.all(real.masked_select(upper) == 0)
    tiles = workloads.sample_tiles(wl, count)
    refs = oracle.kkt_solve_ref_tiles(inp["k"], inp["g"], inp["beta"], tiles)
    got = np.concatenate([flat[r0:r0 + L, h].double().cpu().numpy() for (_, _, h, r0, L) in tiles])
    _check(got, np.concatenate(refs), out_dtype, wl.name)


def test_long_walks_many_pairs_per_cta():
    # 2^21 tokens of one head: every CTA walks over a hundred pairs, and the
    # chunk index crosses NT many times per warpgroup stride.
    wl = workloads.Workload("B1_T2097152_H1_K128", 1, 1 << 21, 1, 128, "f32", seed=901)
    _sampled_parity_and_invariants(wl, torch.float32, 512)


def test_thousands_of_packed_sequences():
    # 4000 packed sequences of 0..300 tokens (many empty, many shorter than a
    # chunk): the schedule steps over sequence boundaries at almost every pair.
    rng = np.random.default_rng(902)
    lens = tuple(int(x) for x in np.where(rng.random(4000) < 0.15, 0, rng.integers(1, 301, size=4000)))
    wl = workloads.Workload("varlen4000_H3_K128", len(lens), sum(lens), 3, 128, "bf16", seed=903,
                            varlen_lengths=lens)
    _sampled_parity_and_invariants(wl, torch.bfloat16, 1024)
