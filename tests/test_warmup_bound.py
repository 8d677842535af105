"""The bound behind warm-up starts, checked on the CPU with the fp64 oracle.

A warm-up start approximates a segment's start state by running the
recurrence over the W chunks before it from a zero state (FlashQLA pages:
page 1 "balanced solution", page 3 "sliding-window warmup").  The library
takes it for a v-head only where it can bound the error: the difference
E = S_warm - S_true obeys E <- a_t (I - b_t k_t k_t^T) E (the write terms
cancel), and ||I - b k k^T||_2 = max(1, |1 - b |k|^2|), so

    ||E(segment start)||_F <= prod_t a_t max(1, |1 - b_t |k_t|^2|) * ||S_true(window start)||_F

over the window's tokens.  These tests run the oracle from the true window
start and from zero and check that inequality, and that the error does shrink
with the factor (the gate's threshold is 1e-6)."""
import numpy as np
import pytest

import oracle


def draw(seed, T, K=8, V=6, Hv=2, strong=False):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, T, 1, K))
    k = rng.standard_normal((1, T, 1, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    if strong:  # keys a little longer than unit: |1 - b |k|^2| can exceed 1
        k *= 1.0 + 0.5 * rng.random((1, T, 1, 1))
    v = rng.standard_normal((1, T, Hv, V))
    g = -np.logaddexp(0.0, -(4.0 + 1.5 * rng.standard_normal((1, T, Hv))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, Hv))))
    h0 = rng.standard_normal((1, Hv, K, V))
    return dict(q=q, k=k, v=v, g=g, beta=b, h0=h0, scale=K ** -0.5)


def factor(x, t0, t1, h):
    kk = np.sum(x["k"][0, t0:t1, 0] ** 2, axis=-1)
    b = x["beta"][0, t0:t1, h]
    a = np.exp(x["g"][0, t0:t1, h])
    return float(np.prod(a * np.maximum(1.0, np.abs(1.0 - b * kk))))


@pytest.mark.parametrize("seed,strong", [(0, False), (1, False), (2, True), (3, True)])
@pytest.mark.parametrize("C,W", [(4, 2), (16, 3), (64, 1)])
def test_warm_start_error_within_the_gate_bound(seed, strong, C, W):
    T = C * (W + 3)
    x = draw(seed, T, strong=strong)
    h = oracle.fwd(**x, chunk=C, want_h=True)["h"][0]  # states before each chunk
    for s in range(W, T // C):  # segment starting at chunk s, window chunks [s - W, s)
        t0, t1 = (s - W) * C, s * C
        part = {kk: (vv[:, t0:t1] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in x.items()}
        part["h0"] = None
        warm = oracle.fwd(**part)["final_state"][0]
        for hv in range(2):
            err = np.linalg.norm(warm[hv] - h[s, hv])
            bound = factor(x, t0, t1, hv) * np.linalg.norm(h[s - W, hv])
            assert err <= bound * (1 + 1e-9) + 1e-12, (s, hv, err, bound)


def test_error_vanishes_with_the_factor():
    # strong decay: the bound falls below the 1e-6 gate within a few chunks and
    # the warm start meets the true state to that accuracy
    C, W = 16, 4
    x = draw(5, C * 8)
    x["g"][:] = -0.5
    h = oracle.fwd(**x, chunk=C, want_h=True)["h"][0]
    s = 6
    t0, t1 = (s - W) * C, s * C
    part = {kk: (vv[:, t0:t1] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in x.items()}
    part["h0"] = None
    warm = oracle.fwd(**part)["final_state"][0]
    for hv in range(2):
        f = factor(x, t0, t1, hv)
        assert f < 1e-6
        rel = np.linalg.norm(warm[hv] - h[s, hv]) / np.linalg.norm(h[s - W, hv])
        assert rel <= f


def test_no_decay_never_passes_the_gate():
    # g = 0 heads: every factor is at least 1, so their segments keep the exact split
    x = draw(7, 64)
    x["g"][:] = 0.0
    assert factor(x, 0, 64, 0) >= 1.0 and factor(x, 0, 64, 1) >= 1.0
