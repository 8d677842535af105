"""Why the tensor-core path splits every computed operand into two bf16 terms.

A numpy model of the chunk algebra the tensor-core kernels evaluate (not their
code): per 64-token chunk, with gamma the chunk-local cumulative log-gate,
    R  = diag(b) (V - diag(e^gamma) K S0),     Ut = A R,
    Y  = diag(e^{gamma_n - gamma}) Ut,
    O  = scale diag(e^gamma) Q S0 + P Ut,      P = scale (Q K^T o D o tril_incl),
    S1 = e^{gamma_n} S0 + K^T Y,
with the products taken as the MMAs take them: bf16 operands, fp32
accumulation.  q, k, v enter as the bf16 values they are.  The computed
operands (S0, R, A, Ut, Y, P) are either rounded to bf16 once, or split as
x = hi + lo (hi = bf16(x), lo = bf16(x - hi)) with three products
hi*hi + lo*hi + hi*lo.  Both are compared with the same algebra in fp64.

The model shows what the design relies on.  With single bf16 operands the
max error settles at 1-2e-2 of the RMS for the state and 2-3e-2 for o, already
after a few chunks: at or beyond the 2e-2 parity bound.  With the split it is
about 2e-5 for the state and 4-8e-5 for o, at 8, 48 and 128 chunks alike.
Everything here runs on the CPU and involves neither the oracle nor the CUDA
library.
"""
import numpy as np


def bf16(x):
    """Round fp32 values to the nearest bf16 (ties to even), returned as fp32."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def mm(a, b, split):
    """a @ b as the tensor cores take it: bf16 operands, fp32 accumulation.
    split == "none": each operand rounded to bf16 once; otherwise each enters
    as hi + lo with three products (for an exact bf16 input lo is zero)."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    if split == "none":
        return (bf16(a).astype(np.float64) @ bf16(b).astype(np.float64)).astype(np.float32)
    ah = bf16(a)
    al = bf16(a - ah)
    bh = bf16(b)
    bl = bf16(b - bh)
    f = lambda x, y: x.astype(np.float64) @ y.astype(np.float64)  # noqa: E731
    return (f(ah, bh) + f(al, bh) + f(ah, bl)).astype(np.float32)


def run(n_chunks, split, seed=0, K=64, V=64, C=64):
    rng = np.random.default_rng(seed)
    T = n_chunks * C
    q = rng.standard_normal((T, K)); q /= np.linalg.norm(q, axis=1, keepdims=True)
    k = rng.standard_normal((T, K)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, V))
    q, k, v = bf16(q).astype(np.float64), bf16(k).astype(np.float64), bf16(v).astype(np.float64)
    g = -np.logaddexp(0.0, -(4.0 + 1.5 * rng.standard_normal(T)))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    scale = K ** -0.5
    S64 = np.zeros((K, V))
    S32 = np.zeros((K, V), np.float32)
    worst_o = 0.0
    for c in range(n_chunks):
        sl = slice(c * C, (c + 1) * C)
        Q, Kc, Vc, bc = q[sl], k[sl], v[sl], b[sl]
        gam = np.cumsum(g[sl])
        D = np.exp(gam[:, None] - gam[None, :])
        L = np.tril(bc[:, None] * (Kc @ Kc.T) * D, -1)
        A = np.linalg.inv(np.eye(C) + L)
        P = scale * D * np.tril(Q @ Kc.T)
        eg, en = np.exp(gam), np.exp(gam[-1])
        # fp64 reference of the same algebra
        R = bc[:, None] * (Vc - eg[:, None] * (Kc @ S64))
        Y = np.exp(gam[-1] - gam)[:, None] * (A @ R)
        O64 = scale * eg[:, None] * (Q @ S64) + P @ (A @ R)
        S64 = en * S64 + Kc.T @ Y
        # the model: S0, R, A, Ut, Y, P computed; q, k, v exact bf16
        KS = mm(Kc, S32, split)
        R32 = (bc[:, None] * (Vc - eg[:, None] * KS)).astype(np.float32)
        Ut = mm(A.astype(np.float32), R32, split)
        Y32 = (np.exp(gam[-1] - gam)[:, None] * Ut).astype(np.float32)
        O32 = scale * eg[:, None] * mm(Q, S32, split) + mm(P.astype(np.float32), Ut, split)
        S32 = (en * S32 + mm(Kc.T, Y32, split)).astype(np.float32)
        worst_o = max(worst_o, float(np.max(np.abs(O32 - O64)) / np.sqrt(np.mean(O64 ** 2))))
    err_s = float(np.max(np.abs(S32 - S64)) / np.sqrt(np.mean(S64 ** 2)))
    return err_s, worst_o


def test_split_operands_keep_the_state_accurate_over_a_long_sequence():
    single_s, single_o = run(48, "none")
    split_s, split_o = run(48, "split")
    assert split_s < 1e-3 and split_o < 1e-3
    # single bf16 operands lose two to three orders of magnitude against the split
    assert single_s > 20 * split_s
    assert single_o > 10 * split_o


def test_bf16_rounding_model():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -3.14159265, 1e-20], np.float32)
    r = bf16(x)
    assert r[0] == 1.0 and r[1] == 1.0  # a tie rounds to even
    assert r[2] == np.float32(1.0 + 2 ** -7)
    assert abs(r[3] - x[3]) <= 2 ** -8 * abs(x[3])
    hi = bf16(x)
    lo = bf16(x - hi)
    assert np.all(np.abs((hi.astype(np.float64) + lo) - x) <= 2 ** -16 * np.abs(x) + 1e-45)
