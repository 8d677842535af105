"""Randomised pins of the fp64 oracle over shapes the fixed pins do not reach:
random lengths (varlen with empty sequences), head groupings, head sizes,
chunk sizes and context-parallel segmentations.  Each example compares the
token recurrence with the independent chunked/WY form (o, final_state and the
states before every chunk), checks A against its definition ((I + L) A = I with
L built here from k, g, beta by the strictly-lower-triangle formula), and
checks that two halves of a sequence, the second started from the first's
final state, give the whole.  Skipped where hypothesis is not installed."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

import oracle  # noqa: E402


def _draw_inputs(seed, lens, Hq, G, K, V, h0):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    Hv = Hq * G
    q = rng.standard_normal((1, T, Hq, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((1, T, Hq, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, Hv, V))
    g = -np.logaddexp(0.0, -(2.0 + 1.5 * rng.standard_normal((1, T, Hv))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((1, T, Hv))))
    hh = 0.1 * rng.standard_normal((len(lens), Hv, K, V)) if h0 else None
    cu = np.cumsum([0] + list(lens)).astype(np.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=hh, scale=K ** -0.5), cu


def _rel(a, b):
    den = max(float(np.max(np.abs(b))) if np.size(b) else 0.0, 1e-300)
    return float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) / den if np.size(b) else 0.0


shapes = st.fixed_dictionaries({
    "seed": st.integers(0, 2 ** 31 - 1),
    "lens": st.lists(st.integers(0, 70), min_size=1, max_size=4).filter(lambda l: sum(l) > 0),
    "Hq": st.integers(1, 2),
    "G": st.integers(1, 3),
    "K": st.integers(1, 8),
    "V": st.integers(1, 8),
    "C": st.sampled_from([1, 2, 4, 8, 16, 64]),
    "seg": st.integers(0, 5),
    "h0": st.booleans(),
})


@settings(max_examples=40, deadline=None)
@given(shapes)
def test_chunked_form_equals_token_recurrence(s):
    x, cu = _draw_inputs(s["seed"], s["lens"], s["Hq"], s["G"], s["K"], s["V"], s["h0"])
    tok = oracle.fwd(**x, cu_seqlens=cu, chunk=s["C"], want_h=True, nthreads=1)
    ch = oracle.chunked_fwd(**x, cu_seqlens=cu, chunk=s["C"], seg_chunks=s["seg"], nthreads=1)
    assert _rel(ch["o"], tok["o"]) <= 1e-10
    assert _rel(ch["final_state"], tok["final_state"]) <= 1e-10
    assert _rel(ch["h"], tok["h"]) <= 1e-10


@settings(max_examples=30, deadline=None)
@given(shapes)
def test_A_inverts_unit_lower_triangular_L(s):
    x, cu = _draw_inputs(s["seed"], s["lens"], s["Hq"], s["G"], s["K"], s["V"], False)
    C = s["C"]
    A = oracle.A_matrix(x["k"], x["g"], x["beta"], cu_seqlens=cu, chunk=C, nthreads=1)
    G = s["G"]
    worst = 0.0
    for n in range(len(cu) - 1):
        for c0 in range(cu[n], cu[n + 1], C):
            m = min(C, cu[n + 1] - c0)
            for h in range(s["Hq"] * G):
                kk = x["k"][0, c0:c0 + m, h // G]
                gam = np.cumsum(x["g"][0, c0:c0 + m, h])
                b = x["beta"][0, c0:c0 + m, h]
                L = np.tril(b[:, None] * (kk @ kk.T) * np.exp(gam[:, None] - gam[None, :]), -1)
                Ac = A[0, c0:c0 + m, h, :m]
                worst = max(worst, float(np.max(np.abs((np.eye(m) + L) @ Ac - np.eye(m)))))
                # rows past the chunk's length and columns past it stay zero
                assert not np.any(A[0, c0:c0 + m, h, m:])
    assert worst <= 1e-10


@settings(max_examples=30, deadline=None)
@given(shapes, st.integers(1, 69))
def test_state_continuation_over_a_cut(s, cut):
    lens = [max(2, sum(s["lens"]))]
    cut = 1 + cut % (lens[0] - 1)
    x, cu = _draw_inputs(s["seed"], lens, s["Hq"], s["G"], s["K"], s["V"], True)
    whole = oracle.fwd(**x, nthreads=1)
    part = lambda a, sl: a[:, sl] if a.ndim >= 3 else a  # noqa: E731
    first = {kk: (part(vv, slice(0, cut)) if isinstance(vv, np.ndarray) and kk != "h0" else vv) for kk, vv in x.items()}
    one = oracle.fwd(**first, nthreads=1)
    second = {kk: (part(vv, slice(cut, None)) if isinstance(vv, np.ndarray) and kk != "h0" else vv)
              for kk, vv in x.items()}
    second["h0"] = one["final_state"]
    two = oracle.fwd(**second, nthreads=1)
    assert _rel(np.concatenate([one["o"], two["o"]], axis=1), whole["o"]) <= 1e-12
    assert _rel(two["final_state"], whole["final_state"]) <= 1e-12
