"""Pins for the fp64 CPU oracle: each check compares the oracle with something
other than itself -- a closed form, an exact invariant, a textbook special case,
an independent chunked form, or central finite differences.

Readings (FlashQLA pages give no worked example and no formula; the recurrence
is the problem statement of the low-level forward):
* beta = 0 writes nothing, so the state only decays: S_T = exp(sum g) h0.
* With beta = 1 and a unit key the delta rule stores v exactly: S_t^T k_t = v_t.
* With orthonormal keys and h0 = 0 the delta correction vanishes and the layer
  is beta-weighted gated linear attention.
* A single token has the analytic state a (I - b k k^T) h0 + b k v^T.
"""
import os
import tempfile

import numpy as np
import pytest

import oracle


def _logsig(x):
    return -np.logaddexp(0.0, -x)


def rnd(seed, B=1, T=40, Hq=1, Hv=2, K=6, V=5, h0=True, Nseq=None):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, T, Hq, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, Hq, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, V))
    g = _logsig(4.0 + 1.5 * rng.standard_normal((B, T, Hv)))
    # make some gates strong so decay matters inside a few tokens
    g[..., -1] = _logsig(0.5 * rng.standard_normal((B, T)))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv))))
    N = Nseq if Nseq is not None else B
    hh = 0.1 * rng.standard_normal((N, Hv, K, V)) if h0 else None
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=hh, scale=K ** -0.5)


def relerr(a, b):
    a = np.asarray(a); b = np.asarray(b)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


# --------------------------------------------------------------------------
# checks (each returns an error figure; the pins assert it is tiny, the
# planted-mistake test asserts that some check becomes large)
# --------------------------------------------------------------------------

def check_beta_zero():
    x = rnd(1, B=2, T=70, Hq=1, Hv=2, K=5, V=3)
    x["beta"][:] = 0.0
    out = oracle.fwd(**x)
    G = x["g"].cumsum(axis=1)  # cumulative log-decay from the sequence start
    e1 = relerr(out["final_state"], np.exp(G[:, -1])[:, :, None, None] * x["h0"])
    hq = np.repeat(x["q"], 2, axis=2)  # both v-heads read qk-head 0
    o_ref = x["scale"] * np.exp(G)[..., None] * np.einsum("bthk,bhkv->bthv", hq, x["h0"])
    return max(e1, relerr(out["o"], o_ref))


def check_delta_memorisation():
    x = rnd(2, B=1, T=50, Hq=1, Hv=2, K=6, V=4)
    x["beta"][:] = 1.0
    x["q"] = x["k"].copy()
    x["scale"] = 1.0
    out = oracle.fwd(**x)
    return relerr(out["o"], x["v"])


def check_single_token():
    x = rnd(3, B=3, T=1, Hq=1, Hv=2, K=4, V=3)
    out = oracle.fwd(**x)
    err = 0.0
    for b in range(3):
        for h in range(2):
            a = np.exp(x["g"][b, 0, h]); be = x["beta"][b, 0, h]
            kk = x["k"][b, 0, 0]; vv = x["v"][b, 0, h]; qq = x["q"][b, 0, 0]
            S1 = a * (np.eye(4) - be * np.outer(kk, kk)) @ x["h0"][b, h] + be * np.outer(kk, vv)
            err = max(err, relerr(out["final_state"][b, h], S1))
            err = max(err, relerr(out["o"][b, 0, h], x["scale"] * S1.T @ qq))
    return err


def check_linear_attention(zero_gate):
    rng = np.random.default_rng(4)
    T = K = 8
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    x = rnd(5, B=1, T=T, Hq=1, Hv=2, K=K, V=3, h0=False)
    x["k"][0, :, 0, :] = Q.T  # rows are orthonormal keys
    if zero_gate:
        x["g"][:] = 0.0
    out = oracle.fwd(**x)
    G = x["g"][0].cumsum(axis=0)  # [T, Hv]
    ref = np.zeros((T, 2, 3))
    for h in range(2):
        for t in range(T):
            for s in range(t + 1):
                w = np.exp(G[t, h] - G[s, h]) * x["beta"][0, s, h] * (x["q"][0, t, 0] @ x["k"][0, s, 0])
                ref[t, h] += x["scale"] * w * x["v"][0, s, h]
    return relerr(out["o"][0], ref)


def check_matrix_form():
    x = rnd(6, B=1, T=9, Hq=1, Hv=2, K=3, V=2)
    x["g"][..., 0] = 0.0  # one head with an exact unit gate
    out = oracle.fwd(**x)
    err = 0.0
    for h in range(2):
        S = x["h0"][0, h].copy()
        for t in range(9):
            a = np.exp(x["g"][0, t, h]); be = x["beta"][0, t, h]
            kk = x["k"][0, t, 0]; vv = x["v"][0, t, h]
            S = a * (np.eye(3) - be * np.outer(kk, kk)) @ S + be * np.outer(kk, vv)
            err = max(err, relerr(out["o"][0, t, h], x["scale"] * S.T @ x["q"][0, t, 0]))
        err = max(err, relerr(out["final_state"][0, h], S))
    return err


def check_gqa_repeat():
    x = rnd(7, B=1, T=30, Hq=2, Hv=4, K=5, V=3)
    out = oracle.fwd(**x)
    xr = dict(x)
    xr["q"] = np.repeat(x["q"], 2, axis=2)  # v-head h reads qk-head h // 2
    xr["k"] = np.repeat(x["k"], 2, axis=2)
    outr = oracle.fwd(**xr)
    e = max(relerr(out["o"], outr["o"]), relerr(out["final_state"], outr["final_state"]))
    rng = np.random.default_rng(8)
    do = rng.standard_normal(x["v"].shape)
    gr = oracle.bwd(**x, do=do)
    grr = oracle.bwd(**xr, do=do)
    e = max(e, relerr(gr["dq"], grr["dq"].reshape(1, 30, 2, 2, 5).sum(axis=3)))
    e = max(e, relerr(gr["dk"], grr["dk"].reshape(1, 30, 2, 2, 5).sum(axis=3)))
    for key in ("dv", "dbeta", "dg", "dh0"):
        e = max(e, relerr(gr[key], grr[key]))
    return e


def check_chunked(C, seg, varlen=False):
    if varlen:
        lens = [37, 0, 64, 1, 70]
        x = rnd(9, B=1, T=sum(lens), Hq=2, Hv=4, K=6, V=5, Nseq=len(lens))
        cu = np.cumsum([0] + lens).astype(np.int32)
    else:
        x = rnd(9, B=2, T=150, Hq=2, Hv=4, K=6, V=5)
        cu = None
    tok = oracle.fwd(**x, cu_seqlens=cu, chunk=C, want_h=True)
    ch = oracle.chunked_fwd(**x, cu_seqlens=cu, chunk=C, seg_chunks=seg)
    return max(relerr(ch["o"], tok["o"]), relerr(ch["final_state"], tok["final_state"]),
               relerr(ch["h"], tok["h"]))


def check_A_forms():
    x = rnd(10, B=1, T=150, Hq=2, Hv=4, K=6, V=5)
    A1 = oracle.A_matrix(x["k"], x["g"], x["beta"])
    A2 = oracle.chunked_fwd(**x)["A"]
    e = relerr(A1, A2)
    # a two-token chunk: A = [[1, 0], [-b_1 exp(g_1) (k_1 . k_0), 1]]
    y = rnd(11, B=1, T=2, Hq=1, Hv=1, K=4, V=2)
    A = oracle.A_matrix(y["k"], y["g"], y["beta"])[0, :, 0, :2]
    a10 = -y["beta"][0, 1, 0] * np.exp(y["g"][0, 1, 0]) * (y["k"][0, 1, 0] @ y["k"][0, 0, 0])
    e = max(e, relerr(A, np.array([[1.0, 0.0], [a10, 1.0]])))
    # every single-token chunk has A = I (the strict triangle is empty)
    A1t = oracle.A_matrix(x["k"], x["g"], x["beta"], chunk=1)
    e = max(e, relerr(A1t[..., 0], np.ones_like(A1t[..., 0])))
    return e


def check_h_prefix():
    x = rnd(12, B=1, T=150, Hq=1, Hv=2, K=4, V=3)
    C = 16
    h = oracle.fwd(**x, chunk=C, want_h=True)["h"]
    err = 0.0
    for i in range(h.shape[1]):
        if i == 0:
            ref = x["h0"][0]
        else:
            xi = {kk: (vv[:, : i * C] if isinstance(vv, np.ndarray) and vv.ndim >= 3 and kk != "h0"
                       else vv) for kk, vv in x.items()}
            ref = oracle.fwd(**xi)["final_state"][0]
        err = max(err, relerr(h[0, i], ref))
    return err


def _objective(x, cu, Ro, Rs):
    out = oracle.fwd(**x, cu_seqlens=cu, nthreads=1)
    return float(np.sum(Ro * out["o"]) + np.sum(Rs * out["final_state"]))


def check_grad_fd():
    lens = [9, 11]
    cu = np.array([0, 9, 20], dtype=np.int32)
    x = rnd(13, B=1, T=20, Hq=1, Hv=2, K=4, V=3, Nseq=2)
    rng = np.random.default_rng(14)
    Ro = rng.standard_normal(x["v"].shape)
    Rs = rng.standard_normal(x["h0"].shape)
    an = oracle.bwd(**x, do=Ro, dht=Rs, cu_seqlens=cu, checkpoint=4, nthreads=1)
    eps = 1e-6
    err = 0.0
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("g", "dg"), ("beta", "dbeta"),
                        ("h0", "dh0")):
        base = x[name]
        fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = base[idx]
            base[idx] = old + eps
            jp = _objective(x, cu, Ro, Rs)
            base[idx] = old - eps
            jm = _objective(x, cu, Ro, Rs)
            base[idx] = old
            fd[idx] = (jp - jm) / (2 * eps)
        err = max(err, relerr(an[gname], fd))
    return err


# --------------------------------------------------------------------------
# the pins
# --------------------------------------------------------------------------

def test_beta_zero_is_pure_decay():
    assert check_beta_zero() < 1e-13


def test_delta_rule_memorises_with_unit_key_and_beta_one():
    assert check_delta_memorisation() < 1e-12


def test_single_token_analytic_state():
    assert check_single_token() < 1e-13


@pytest.mark.parametrize("zero_gate", [False, True])
def test_orthonormal_keys_reduce_to_gated_linear_attention(zero_gate):
    assert check_linear_attention(zero_gate) < 1e-12


def test_matrix_transition_form_brute_force():
    assert check_matrix_form() < 1e-12


def test_gqa_equals_materialised_repeat_fwd_and_bwd():
    assert check_gqa_repeat() < 1e-12


@pytest.mark.parametrize("C,seg", [(1, 0), (4, 0), (4, 3), (16, 0), (16, 1), (16, 2), (64, 0),
                                   (64, 1), (64, 2)])
def test_chunked_form_matches_token_recurrence(C, seg):
    assert check_chunked(C, seg) < 1e-10


@pytest.mark.parametrize("C,seg", [(16, 0), (16, 2), (64, 1)])
def test_chunked_form_matches_token_recurrence_varlen(C, seg):
    assert check_chunked(C, seg, varlen=True) < 1e-10


def test_A_two_forms_and_closed_forms():
    assert check_A_forms() < 1e-12


def test_A_is_inverse_of_unit_lower_triangular():
    # residual of (I + L) A = I with L from its definition, on a 64-token chunk
    x = rnd(15, B=1, T=64, Hq=1, Hv=1, K=8, V=2)
    A = oracle.A_matrix(x["k"], x["g"], x["beta"])[0, :, 0, :]
    gam = x["g"][0, :, 0].cumsum()
    kk = x["k"][0, :, 0, :]
    L = np.tril(x["beta"][0, :, 0][:, None] * (kk @ kk.T) * np.exp(gam[:, None] - gam[None, :]), -1)
    assert np.max(np.abs((np.eye(64) + L) @ A - np.eye(64))) < 1e-12
    assert np.all(np.triu(A, 1) == 0.0) and np.all(np.diag(A) == 1.0)


def test_h_is_the_state_before_each_chunk():
    assert check_h_prefix() < 1e-13


def test_state_continuation():
    x = rnd(16, B=2, T=90, Hq=1, Hv=2, K=5, V=4)
    full = oracle.fwd(**x)
    x1 = {k: (v[:, :50] if isinstance(v, np.ndarray) and k in ("q", "k", "v", "g", "beta") else v)
          for k, v in x.items()}
    x2 = {k: (v[:, 50:] if isinstance(v, np.ndarray) and k in ("q", "k", "v", "g", "beta") else v)
          for k, v in x.items()}
    p1 = oracle.fwd(**x1)
    x2["h0"] = p1["final_state"]
    p2 = oracle.fwd(**x2)
    assert relerr(np.concatenate([p1["o"], p2["o"]], axis=1), full["o"]) < 1e-13
    assert relerr(p2["final_state"], full["final_state"]) < 1e-13


def test_varlen_equals_separate_sequences():
    lens = [5, 0, 64, 65, 3]
    x = rnd(17, B=1, T=sum(lens), Hq=1, Hv=2, K=4, V=3, Nseq=len(lens))
    cu = np.cumsum([0] + lens).astype(np.int32)
    packed = oracle.fwd(**x, cu_seqlens=cu)
    rng = np.random.default_rng(18)
    do = rng.standard_normal(x["v"].shape)
    dht = rng.standard_normal(x["h0"].shape)
    gp = oracle.bwd(**x, do=do, dht=dht, cu_seqlens=cu)
    for n in range(len(lens)):
        a, b = cu[n], cu[n + 1]
        xs = {k: (v[:, a:b] if k in ("q", "k", "v", "g", "beta") else v) for k, v in x.items()}
        xs["h0"] = x["h0"][n:n + 1]
        one = oracle.fwd(**xs)
        assert relerr(packed["final_state"][n], one["final_state"][0]) < 1e-14
        if b > a:
            assert relerr(packed["o"][:, a:b], one["o"]) < 1e-14
        go = oracle.bwd(**xs, do=do[:, a:b], dht=dht[n:n + 1])
        assert relerr(gp["dh0"][n], go["dh0"][0]) < 1e-13
        for key in ("dq", "dk", "dv", "dbeta", "dg"):
            if b > a:
                assert relerr(gp[key][:, a:b], go[key]) < 1e-13


def test_gradients_match_central_finite_differences():
    assert check_grad_fd() < 1e-6


def test_bwd_checkpoint_interval_does_not_change_gradients():
    x = rnd(19, B=1, T=45, Hq=1, Hv=2, K=4, V=3)
    do = np.random.default_rng(20).standard_normal(x["v"].shape)
    a = oracle.bwd(**x, do=do, checkpoint=64)
    b = oracle.bwd(**x, do=do, checkpoint=7)
    for key in a:
        assert relerr(a[key], b[key]) < 1e-13


# --------------------------------------------------------------------------
# planted mistakes must be caught by at least one of the checks above
# --------------------------------------------------------------------------

_CHECKS = {
    "beta_zero": (check_beta_zero, 1e-13),
    "memorise": (check_delta_memorisation, 1e-12),
    "single": (check_single_token, 1e-13),
    "linattn": (lambda: check_linear_attention(False), 1e-12),
    "matrix": (check_matrix_form, 1e-12),
    "gqa": (check_gqa_repeat, 1e-12),
    "A": (check_A_forms, 1e-12),
    "chunked": (lambda: check_chunked(16, 2), 1e-10),
    "fd": (check_grad_fd, 1e-6),
}


@pytest.mark.parametrize("mutation", [1, 2, 3, 4, 5, 6])
def test_planted_mistake_is_caught(mutation):
    with tempfile.TemporaryDirectory() as d:
        path = oracle.build_variant(mutation, d)
        oracle.use_library(path)
        try:
            failed = []
            for name, (fn, tol) in _CHECKS.items():
                try:
                    if not fn() < tol:
                        failed.append(name)
                except Exception:
                    failed.append(name)
            assert failed, f"mutation {mutation} slipped through every pin"
        finally:
            oracle.use_library(None)
