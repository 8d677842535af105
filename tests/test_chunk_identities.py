"""Algebraic facts the tensor-core kernels rely on, checked on the CPU in fp64
(numpy; the oracle where the token recurrence is the reference).  None of this
runs the CUDA library.

* The chunk transition: over one chunk the state map is S1 = T S0 + (terms
  without S0) with T = e^{gamma_n} I - Kt^T W, Kt = diag(e^{gamma_n - gamma}) K,
  W = A diag(b e^gamma) K; checked against the token recurrence.
* The reverse scan's coefficient of dS1 is T^T, so the composed reverse
  transition of a segment is the transpose of the forward one (N = M^T): the
  backward reads the forward summary's M instead of running its own chain.
* Zero-padded rows (k = q = v = 0, b = 0, g = 0) of a partial chunk change
  nothing.
* The tensor-core reformulation: Ut = A R, P' Y = P Ut, K^T Y = Kt^T Ut.
* The backward's stacked product: with Ut = A R, dA = dUt R^T, X = A^T dA and
  dR = A^T dUt, X A^T = dR Ut^T; and dL = -strict_tril(A^T dA A^T) is the
  gradient through A = (I + L)^-1 for a strictly lower L.
"""
import numpy as np

import oracle


def chunk_inputs(seed, n=40, K=6, V=5):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, K))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((n, K))
    v = rng.standard_normal((n, V))
    g = -np.logaddexp(0.0, -(2.0 + rng.standard_normal(n)))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(n)))
    return q, k, v, g, b


def chunk_terms(k, g, b):
    n = len(g)
    gam = np.cumsum(g)
    L = np.tril(b[:, None] * (k @ k.T) * np.exp(gam[:, None] - gam[None, :]), -1)
    A = np.linalg.inv(np.eye(n) + L)
    W = A @ ((b * np.exp(gam))[:, None] * k)
    Kt = np.exp(gam[-1] - gam)[:, None] * k
    T = np.exp(gam[-1]) * np.eye(k.shape[1]) - Kt.T @ W
    return gam, A, W, Kt, T


def oracle_state(q, k, v, g, b, S0):
    x = dict(q=q[None, :, None], k=k[None, :, None], v=v[None, :, None], g=g[None, :, None],
             beta=b[None, :, None], scale=1.0, h0=S0[None, None])
    return oracle.fwd(**x)["final_state"][0, 0]


def test_chunk_transition_matches_the_token_recurrence():
    q, k, v, g, b = chunk_inputs(0)
    _, _, _, _, T = chunk_terms(k, g, b)
    rng = np.random.default_rng(1)
    S0 = rng.standard_normal((6, 5))
    # the state map is affine in S0: its linear part is T
    lin = oracle_state(q, k, v, g, b, S0) - oracle_state(q, k, v, g, b, np.zeros_like(S0))
    np.testing.assert_allclose(lin, T @ S0, rtol=0, atol=1e-12)


def test_reverse_coefficient_is_the_transpose_and_segments_compose_to_M_transposed():
    rng = np.random.default_rng(2)
    Ts, Rs = [], []
    for c in range(4):
        q, k, v, g, b = chunk_inputs(10 + c)
        gam, A, W, Kt, T = chunk_terms(k, g, b)
        Ts.append(T)
        # the reverse scan's dS1 coefficient: e^{gamma_n} dS1 - W^T (Kt dS1)
        Rs.append(np.exp(gam[-1]) * np.eye(6) - W.T @ Kt)
        np.testing.assert_allclose(Rs[-1], T.T, rtol=0, atol=1e-13)
    M = np.eye(6)
    for T in Ts:  # forward: S_end = T_4 T_3 T_2 T_1 S_start + ...
        M = T @ M
    dS = rng.standard_normal((6, 5))
    N_dS = dS.copy()
    for R in reversed(Rs):  # reverse: from the segment's end back to its start
        N_dS = R @ N_dS
    np.testing.assert_allclose(N_dS, M.T @ dS, rtol=0, atol=1e-12)


def test_zero_padded_rows_are_inert():
    q, k, v, g, b = chunk_inputs(3, n=37)
    rng = np.random.default_rng(4)
    S0 = rng.standard_normal((6, 5))
    scale = 0.4

    def chunk(q, k, v, g, b):
        gam, A, W, Kt, T = chunk_terms(k, g, b)
        U = A @ (b[:, None] * v)
        Ut = U - W @ S0
        P = scale * np.tril(q @ k.T) * np.exp(gam[:, None] - gam[None, :])
        O = scale * np.exp(gam)[:, None] * (q @ S0) + P @ Ut
        return O, np.exp(gam[-1]) * S0 + Kt.T @ Ut

    O, S1 = chunk(q, k, v, g, b)
    pad = lambda a: np.concatenate([a, np.zeros((64 - 37,) + a.shape[1:])])  # noqa: E731
    Op, S1p = chunk(pad(q), pad(k), pad(v), pad(g), pad(b))
    np.testing.assert_allclose(S1p, S1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(Op[:37], O, rtol=0, atol=1e-13)
    # and the unpadded chunk is the token recurrence
    x = dict(q=q[None, :, None], k=k[None, :, None], v=v[None, :, None], g=g[None, :, None],
             beta=b[None, :, None], scale=scale, h0=S0[None, None])
    ref = oracle.fwd(**x)
    np.testing.assert_allclose(O, ref["o"][0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S1, ref["final_state"][0, 0], rtol=0, atol=1e-12)


def test_backward_stacked_product_and_the_inverse_gradient():
    rng = np.random.default_rng(5)
    n, V = 12, 7
    L = np.tril(0.3 * rng.standard_normal((n, n)), -1)
    A = np.linalg.inv(np.eye(n) + L)
    R = rng.standard_normal((n, V))
    dUt = rng.standard_normal((n, V))
    Ut = A @ R
    dA = dUt @ R.T
    X = A.T @ dA
    dR = A.T @ dUt
    np.testing.assert_allclose(X @ A.T, dR @ Ut.T, rtol=0, atol=1e-12)
    # dL = -strict_tril(A^T dA A^T): the gradient of <dA, (I + L)^-1> over strictly lower L
    dL = -np.tril(A.T @ dA @ A.T, -1)
    f = lambda LL: float(np.sum(dA * np.linalg.inv(np.eye(n) + LL)))  # noqa: E731
    h = 1e-6
    for (i, j) in [(3, 1), (11, 0), (7, 6), (5, 2)]:
        E = np.zeros((n, n))
        E[i, j] = h
        fd = (f(L + E) - f(L - E)) / (2 * h)
        assert abs(fd - dL[i, j]) <= 1e-6 * max(1.0, abs(dL[i, j]))


def test_tensor_core_reformulation():
    """Ut = A R with R = diag(b)(V - diag(e^gamma) K S0) is U - W S0; with
    Y = diag(e^{gamma_n - gamma}) Ut and P' = scale diag(e^{gamma - gamma_n})
    (Q K^T o tril_incl), P' Y = P Ut and K^T Y = Kt^T Ut."""
    q, k, v, g, b = chunk_inputs(6, n=50)
    gam, A, W, Kt, T = chunk_terms(k, g, b)
    rng = np.random.default_rng(7)
    S0 = rng.standard_normal((6, 5))
    scale = 0.41
    U = A @ (b[:, None] * v)
    Ut = U - W @ S0
    R = b[:, None] * (v - np.exp(gam)[:, None] * (k @ S0))
    np.testing.assert_allclose(A @ R, Ut, rtol=0, atol=1e-12)
    Y = np.exp(gam[-1] - gam)[:, None] * Ut
    P = scale * np.tril(q @ k.T) * np.exp(gam[:, None] - gam[None, :])
    Pp = scale * np.exp(gam - gam[-1])[:, None] * np.tril(q @ k.T)
    np.testing.assert_allclose(Pp @ Y, P @ Ut, rtol=0, atol=1e-12)
    np.testing.assert_allclose(k.T @ Y, Kt.T @ Ut, rtol=0, atol=1e-12)
