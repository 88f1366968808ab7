"""Property-based pins of the oracle (CPU): for random small problems drawn by
hypothesis (chunk length, head dimension, chunk size, gate and beta values,
with and without g and beta), every chunk's output equals the inverse of
I + A computed by numpy's dense LU solver (another algorithm than the oracle's
forward substitution), the diagonal is exactly 1, and everything above it and
past the chunk is exactly 0.  A itself is rebuilt here from its definition, so
this pins the inverse step and the chunking across shapes; the formula of A is
pinned by the hand values in test_oracle_pins.py."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402


def _A(k, g, beta):
    L = k.shape[0]
    A = np.zeros((L, L))
    for i in range(L):
        for j in range(i):
            b = 1.0 if beta is None else beta[i]
            gate = 1.0 if g is None else np.exp(g[i] - g[j])
            A[i, j] = b * float(k[i] @ k[j]) * gate
    return A


@settings(max_examples=60, deadline=None)
@given(T=st.integers(1, 140), K=st.sampled_from([64, 128]), C=st.sampled_from([64, 128]),
       H=st.integers(1, 3), use_g=st.booleans(), use_beta=st.booleans(),
       gate_scale=st.floats(0.0, 0.5), seed=st.integers(0, 2 ** 31 - 1))
def test_oracle_equals_dense_solve(T, K, C, H, use_g, use_beta, gate_scale, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    g = None
    if use_g:
        steps = -gate_scale * rng.random((1, T, H))
        g = np.zeros_like(steps)
        for c0 in range(0, T, C):                   # chunk-local cumulative log-gate
            g[:, c0:c0 + C] = np.cumsum(steps[:, c0:c0 + C], axis=1)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, H)))) if use_beta else None
    out = oracle.kkt_solve_ref(k, g, beta, chunk_size=C)
    assert out.shape == (1, T, H, C)
    for c0 in range(0, T, C):
        L = min(C, T - c0)
        for h in range(H):
            A = _A(k[0, c0:c0 + L, h], None if g is None else g[0, c0:c0 + L, h],
                   None if beta is None else beta[0, c0:c0 + L, h])
            X = np.linalg.solve(np.eye(L) + A, np.eye(L))
            got = out[0, c0:c0 + L, h]
            np.testing.assert_allclose(got[:, :L], X, rtol=0, atol=1e-10 * max(1.0, np.abs(X).max()))
            assert np.all(np.diag(got[:, :L]) == 1.0)
            assert np.all(got[:, :L][np.triu_indices(L, 1)] == 0.0)
            assert np.all(got[:, L:] == 0.0)
