"""Pins of the CPU oracle against facts fixed by mathematics, not by the oracle.

The pages print no worked example, so the oracle is pinned by:
  * closed forms (a single coupled pair, L = 2 and L = 3 chains, collinear keys
    giving the delta-rule product form, the finite Neumann series),
  * special cases (beta = 0, mutually orthogonal keys -> identity),
  * brute force (Gaussian elimination with partial pivoting, written here),
  * invariants (residual, unit diagonal, zero upper triangle, zero columns past
    a partial chunk, shift invariance of g, chunk independence, varlen packing
    equal to separate sequences, g/beta = None equal to 0/1).
Each case is chosen so that a plausible slip in the oracle (beta on the wrong
index, a flipped gate sign, exp2 for exp, a transposed result, (I - A) for
(I + A), a dropped term of the dot product, chunks not restarting at sequence
starts) fails at least one test.
"""
import math

import numpy as np
import pytest

import oracle
import workloads

C = 64


def _gauss_inverse(M):
    """Dense inverse by Gauss-Jordan elimination with partial pivoting."""
    n = M.shape[0]
    aug = np.concatenate([M.astype(np.float64), np.eye(n)], axis=1)
    for col in range(n):
        piv = col + int(np.argmax(np.abs(aug[col:, col])))
        if piv != col:
            aug[[col, piv]] = aug[[piv, col]]
        aug[col] /= aug[col, col]
        for r in range(n):
            if r != col and aug[r, col] != 0.0:
                aug[r] -= aug[r, col] * aug[col]
    return aug[:, n:]


def _rand_chunk(rng, L, K, gate_scale=0.1):
    k = rng.standard_normal((L, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    g = np.cumsum(-gate_scale * rng.random(L))
    return k, g, beta


def _A_of(k, g, beta):
    """A written out from the definition (used with the brute-force and
    Neumann pins; the definition itself is pinned by the closed forms)."""
    L = k.shape[0]
    A = np.zeros((L, L))
    for i in range(L):
        for j in range(i):
            A[i, j] = beta[i] * float(k[i] @ k[j]) * math.exp(g[i] - g[j])
    return A


@pytest.mark.parametrize("L", [1, 2, 3, 17, 63, 64])
def test_structure_and_residual(L):
    rng = np.random.default_rng(100 + L)
    k, g, beta = _rand_chunk(rng, L, 128)
    X = oracle.kkt_solve_ref_chunk(k, g, beta)
    assert X.shape == (L, C)
    assert np.all(X[:, L:] == 0.0)                       # columns past the chunk
    Xl = X[:, :L]
    assert np.all(np.diag(Xl) == 1.0)                    # unit diagonal, exactly
    assert np.all(Xl[np.triu_indices(L, 1)] == 0.0)      # strictly upper exactly 0
    A = _A_of(k, g, beta)
    R = (np.eye(L) + A) @ Xl - np.eye(L)
    assert np.max(np.abs(R)) <= 1e-10


@pytest.mark.parametrize("L", [5, 32, 64])
def test_brute_force_gauss_jordan(L):
    rng = np.random.default_rng(7 * L)
    k, g, beta = _rand_chunk(rng, L, 128, gate_scale=0.3)
    X = oracle.kkt_solve_ref_chunk(k, g, beta)[:, :L]
    ref = _gauss_inverse(np.eye(L) + _A_of(k, g, beta))
    assert np.max(np.abs(X - ref)) <= 1e-12


def test_neumann_series_closed_form():
    # A is nilpotent (strictly lower), so (I + A)^{-1} = sum_{n<L} (-A)^n exactly.
    rng = np.random.default_rng(11)
    L = 64
    k, g, beta = _rand_chunk(rng, L, 128)
    A = _A_of(k, g, beta)
    S, P = np.eye(L), np.eye(L)
    for _ in range(1, L):
        P = P @ (-A)
        S = S + P
    X = oracle.kkt_solve_ref_chunk(k, g, beta)[:, :L]
    assert np.max(np.abs(X - S)) <= 1e-13


def test_single_coupled_pair_hand_value():
    # Only rows i0 = 40 and j0 = 9 carry keys; u.v = 1*2 + 2*(-1) + 3*1 = 3.
    # beta_i0 = 0.5, g_i0 - g_j0 = -ln 2  ->  a = 0.5 * 3 * 0.5 = 0.75 and
    # X = I - 0.75 e_i0 e_j0^T.  beta_j0 = 0.25 differs, so beta on the wrong
    # index gives 0.375; a flipped gate sign gives 3.0; exp2 gives 0.929...
    L, K, i0, j0 = 64, 8, 40, 9
    k = np.zeros((L, K))
    k[i0, [0, 1, 7]] = [1.0, 2.0, 3.0]
    k[j0, [0, 1, 7]] = [2.0, -1.0, 1.0]
    beta = np.full(L, 0.9)
    beta[i0], beta[j0] = 0.5, 0.25
    g = np.zeros(L)
    g[j0] = 1.0
    g[i0] = 1.0 - math.log(2.0)
    X = oracle.kkt_solve_ref_chunk(k, g, beta)
    expect = np.eye(L)
    expect[i0, j0] = -0.75
    np.testing.assert_allclose(X[:, :L], expect, rtol=0, atol=1e-15)


def test_chain_L3_closed_form():
    # L = 3: X[1,0] = -a10, X[2,1] = -a21, X[2,0] = a21*a10 - a20.
    k = np.array([[1.0, 0.0, 0.0], [0.5, 0.5, 0.0], [0.25, -1.0, 2.0]])
    beta = np.array([0.7, 0.2, 0.6])
    g = np.array([0.0, -0.3, -0.5])
    s10 = 0.5
    s20 = 0.25
    s21 = 0.125 - 0.5
    a10 = beta[1] * s10 * math.exp(g[1] - g[0])
    a20 = beta[2] * s20 * math.exp(g[2] - g[0])
    a21 = beta[2] * s21 * math.exp(g[2] - g[1])
    X = oracle.kkt_solve_ref_chunk(k, g, beta)
    want = np.array([[1, 0, 0], [-a10, 1, 0], [a21 * a10 - a20, -a21, 1]])
    np.testing.assert_allclose(X[:, :3], want, rtol=0, atol=1e-15)
    assert np.all(X[:, 3:] == 0.0)


def test_beta_zero_gives_identity():
    rng = np.random.default_rng(3)
    k, g, _ = _rand_chunk(rng, 64, 128)
    X = oracle.kkt_solve_ref_chunk(k, g, np.zeros(64))
    assert np.array_equal(X, np.eye(64))


def test_orthogonal_keys_give_identity():
    rng = np.random.default_rng(4)
    L, K = 64, 128
    k = np.zeros((L, K))
    k[np.arange(L), np.arange(L)] = 1.0          # k_t = e_t: mutually orthogonal
    _, g, beta = _rand_chunk(rng, L, 4)
    X = oracle.kkt_solve_ref_chunk(k, g, beta)
    assert np.array_equal(X, np.eye(L))


def test_collinear_keys_delta_rule_product_form():
    # All keys equal one unit vector: A[i,j] = beta_i exp(g_i - g_j), and the
    # inverse has the delta-rule product form
    #   X[i,j] = -beta_i exp(g_i - g_j) prod_{m=j+1}^{i-1} (1 - beta_m),  i > j.
    rng = np.random.default_rng(5)
    L, K = 64, 16
    u = rng.standard_normal(K)
    u /= np.linalg.norm(u)
    k = np.tile(u, (L, 1))
    _, g, beta = _rand_chunk(rng, L, 4, gate_scale=0.2)
    X = oracle.kkt_solve_ref_chunk(k, g, beta)[:, :L]
    want = np.eye(L)
    for i in range(L):
        for j in range(i):
            want[i, j] = -beta[i] * math.exp(g[i] - g[j]) * np.prod(1.0 - beta[j + 1:i])
    assert np.max(np.abs(X - want)) <= 1e-13


def test_gate_shift_invariance_and_none_defaults():
    rng = np.random.default_rng(6)
    k, g, beta = _rand_chunk(rng, 50, 128)
    X = oracle.kkt_solve_ref_chunk(k, g, beta)
    Xs = oracle.kkt_solve_ref_chunk(k, g + 3.25, beta)
    assert np.max(np.abs(X - Xs)) <= 1e-14
    np.testing.assert_array_equal(oracle.kkt_solve_ref_chunk(k, None, beta),
                                  oracle.kkt_solve_ref_chunk(k, np.zeros(50), beta))
    np.testing.assert_array_equal(oracle.kkt_solve_ref_chunk(k, g, None),
                                  oracle.kkt_solve_ref_chunk(k, g, np.ones(50)))


def test_block_merge_reproduces_dense_inverse():
    # The GPU path's algorithm: invert the four 16x16 diagonal blocks, then
    # X_ij = -D_ii * sum_{m=j}^{i-1} A_im X_mj.  It must equal the oracle.
    rng = np.random.default_rng(8)
    k, g, beta = _rand_chunk(rng, 64, 128, gate_scale=0.2)
    A = _A_of(k, g, beta)
    blk = lambda M, i, j: M[16 * i:16 * i + 16, 16 * j:16 * j + 16]
    D = [np.linalg.inv(np.eye(16) + blk(A, i, i)) for i in range(4)]
    Xb = np.zeros((64, 64))
    for i in range(4):
        Xb[16 * i:16 * i + 16, 16 * i:16 * i + 16] = D[i]
    for d in range(1, 4):
        for j in range(4 - d):
            i = j + d
            acc = sum(blk(A, i, m) @ Xb[16 * m:16 * m + 16, 16 * j:16 * j + 16] for m in range(j, i))
            Xb[16 * i:16 * i + 16, 16 * j:16 * j + 16] = -D[i] @ acc
    X = oracle.kkt_solve_ref_chunk(k, g, beta)[:, :64]
    assert np.max(np.abs(X - Xb)) <= 1e-13


def test_chunks_restart_and_are_independent():
    # A sequence of 100 tokens has chunks [0,64) and [64,100); chunk 2's output
    # equals the oracle on rows 64..99 alone, and chunk 1 never sees chunk 2.
    rng = np.random.default_rng(9)
    T, H, K = 100, 2, 32
    k = rng.standard_normal((1, T, H, K))
    g = -0.05 * rng.random((1, T, H))
    beta = rng.random((1, T, H))
    out = oracle.kkt_solve_ref(k, g, beta, threads=1)
    for h in range(H):
        first = oracle.kkt_solve_ref_chunk(k[0, :64, h], g[0, :64, h], beta[0, :64, h])
        second = oracle.kkt_solve_ref_chunk(k[0, 64:, h], g[0, 64:, h], beta[0, 64:, h])
        np.testing.assert_array_equal(out[0, :64, h], first)
        np.testing.assert_array_equal(out[0, 64:, h], second)
    k2 = k.copy()
    k2[0, 70:, :, :] *= -3.0
    out2 = oracle.kkt_solve_ref(k2, g, beta, threads=1)
    np.testing.assert_array_equal(out[0, :64], out2[0, :64])


def test_varlen_equals_separate_sequences():
    rng = np.random.default_rng(10)
    lens = [70, 1, 64, 129]
    H, K = 3, 16
    T = sum(lens)
    k = rng.standard_normal((1, T, H, K))
    g = -0.1 * rng.random((1, T, H))
    beta = rng.random((1, T, H))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    packed = oracle.kkt_solve_ref(k, g, beta, cu_seqlens=cu, threads=2)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        alone = oracle.kkt_solve_ref(k[:, s:e], g[:, s:e], beta[:, s:e], threads=1)
        np.testing.assert_array_equal(packed[:, s:e], alone)


def test_fixed_length_batches_are_separate_sequences():
    rng = np.random.default_rng(12)
    B, T, H, K = 2, 80, 2, 16
    k = rng.standard_normal((B, T, H, K))
    g = -0.1 * rng.random((B, T, H))
    beta = rng.random((B, T, H))
    out = oracle.kkt_solve_ref(k, g, beta, threads=2)
    for b in range(B):
        alone = oracle.kkt_solve_ref(k[b:b + 1], g[b:b + 1], beta[b:b + 1], threads=1)
        np.testing.assert_array_equal(out[b:b + 1], alone)


def test_threads_do_not_change_results():
    wl = workloads.CONFIGS["B2_T2000_H5_K128"].with_(T=300)
    inp = workloads.make_inputs(wl)
    a = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], threads=1)
    b = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], threads=5)
    np.testing.assert_array_equal(a, b)


def test_tiles_api_matches_full_run():
    wl = workloads.CONFIGS["B2_T2000_H5_K128"].with_(T=150)
    inp = workloads.make_inputs(wl)
    full = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], threads=2).reshape(-1, wl.H, C)
    tiles = workloads.tile_list(wl)
    outs = oracle.kkt_solve_ref_tiles(inp["k"], inp["g"], inp["beta"], tiles, threads=2)
    for (n, c, h, r0, L), o in zip(tiles, outs):
        np.testing.assert_array_equal(full[r0:r0 + L, h], o)


def test_golden_fixture_reproduces():
    # tests/golden/oracle_small.txt was written by tests/golden/make_golden.py
    # (oracle only); this guards the oracle against silent changes.
    import os
    import importlib.util
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    inp = workloads.make_inputs(mg.WL)
    out = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], threads=1).reshape(-1, mg.WL.H, C)
    n = 0
    with open(os.path.join(here, "oracle_small.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            parts = line.split()
            r, h = int(parts[0]), int(parts[1])
            vals = np.array([float(v) for v in parts[2:]])
            assert np.max(np.abs(out[r, h] - vals)) <= 1e-12
            n += 1
    assert n > 0


# ---------------------------------------------------------------------------
# The two halves of the unfused chain (A alone, and the solve of a given A).

def test_chunk_A_hand_values():
    # L = 3, K = 2, C = 4.  Keys, beta and g chosen so that beta_i vs beta_j,
    # the gate sign and exp vs exp2 all give different numbers.
    k = np.array([[1.0, 0.0], [0.5, 0.5], [2.0, 1.0]])
    beta = np.array([0.3, 0.5, 0.25])
    g = np.array([0.0, -math.log(2.0), -math.log(4.0)])
    A = oracle.chunk_A_ref(k.reshape(1, 3, 1, 2), g.reshape(1, 3, 1), beta.reshape(1, 3, 1),
                           chunk_size=4)[0, :, 0, :]
    want = np.zeros((3, 4))
    want[1, 0] = 0.5 * 0.5 * 0.5          # beta_1 (k1.k0) e^{g1-g0}
    want[2, 0] = 0.25 * 2.0 * 0.25        # beta_2 (k2.k0) e^{g2-g0}
    want[2, 1] = 0.25 * 1.5 * 0.5         # beta_2 (k2.k1) e^{g2-g1}
    assert np.array_equal(A, want)


def test_solve_tril_equals_library_inverse_and_reads_only_strict_lower():
    rng = np.random.default_rng(91)
    L = 37
    A = np.tril(rng.standard_normal((L, L)) * 0.2, k=-1)
    noisy = A + np.triu(rng.standard_normal((L, L)))          # diagonal and upper: ignored
    full = np.zeros((1, L, 1, C))
    full[0, :, 0, :L] = noisy
    full[0, :, 0, L:] = 7.0
    X = oracle.solve_tril_ref(full, cu_seqlens=np.array([0, L], dtype=np.int32))[0, :, 0, :]
    assert np.abs(X[:, :L] - np.linalg.inv(np.eye(L) + A)).max() <= 1e-12
    assert np.all(X[:, L:] == 0.0)


def test_solve_tril_L3_closed_form():
    a10, a20, a21 = 0.7, -0.4, 1.3
    A = np.zeros((1, 3, 1, C))
    A[0, 1, 0, 0], A[0, 2, 0, 0], A[0, 2, 0, 1] = a10, a20, a21
    X = oracle.solve_tril_ref(A, cu_seqlens=np.array([0, 3], dtype=np.int32))[0, :, 0, :3]
    want = np.array([[1.0, 0.0, 0.0], [-a10, 1.0, 0.0], [a21 * a10 - a20, -a21, 1.0]])
    assert np.abs(X - want).max() <= 1e-15


@pytest.mark.parametrize("name", ["B1_T256_H8_K128", "B2_T2000_H5_K128", "varlen"])
def test_chain_of_halves_equals_fused_oracle(name):
    if name == "varlen":
        lens = (1, 64, 0, 65, 130, 2)
        wl = workloads.Workload("chain_varlen", len(lens), sum(lens), 3, 32, "f32", seed=93,
                                varlen_lengths=lens)
    else:
        wl = workloads.CONFIGS[name].with_(T=min(workloads.CONFIGS[name].T, 300))
    inp = workloads.make_inputs(wl)
    A = oracle.chunk_A_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"])
    X = oracle.solve_tril_ref(A, inp["cu_seqlens"])
    ref = oracle.kkt_solve_ref(inp["k"], inp["g"], inp["beta"], inp["cu_seqlens"])
    assert np.abs(X - ref).max() <= 1e-12
    # A is strictly lower inside each chunk and zero past the chunk's length.
    Af = A.reshape(-1, wl.H, C)
    for s, e in workloads._sequence_bounds(wl):
        for c0 in range(s, e, C):
            L = min(C, e - c0)
            blk = Af[c0:c0 + L]                              # [L, H, C]
            upper = np.arange(C)[None, :] >= np.arange(L)[:, None]
            assert np.all(blk.transpose(0, 2, 1)[upper] == 0.0)
