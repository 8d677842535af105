"""GPU parity under strongly decaying gates, against the fp64 oracle.

The gate of the method is an exponential decay a_t = e^{g_t} (FlashQLA pages:
page 1 "balanced solution", page 3 "technical principles"), and nothing bounds
how fast it may decay.  Here g = logsigmoid(N(-4, 1.5)) (about -4 per token)
and one v-head has g = -3 in every token, so a full 64-token chunk's
log-decay reaches -192 and below: any factorisation of the pairwise decay
e^{gamma_r - gamma_s} into a row factor e^{gamma_r - gamma_n} and a column
factor e^{gamma_n - gamma_s} leaves fp32 there (e^88 overflows).  One v-head
keeps g = 0 so that decaying and non-decaying heads share qk-heads.  Forward
and backward on both paths, with and without a context-parallel split,
fixed-length and packed sequences, at the tolerances of the other parity tests.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_chunked_delta_gb300 import inputs
from parity import TOL, err, gpu_bwd, gpu_fwd, oracle_A, oracle_bwd, oracle_fwd, to_dev

pytestmark = pytest.mark.gpu

PATHS = ["simt", "tc"]


@pytest.fixture(scope="module")
def gdr():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_deltanet_chunked_delta_gb300 as m
    m.load(build_if_missing=True)
    return m


def _path(gdr, name):
    if name == "simt":
        return gdr.GDR_PATH_SIMT
    if not gdr.tc_available():
        pytest.skip("the library has no tensor-core path")
    return gdr.GDR_PATH_TC


def _spec(name, bwd=False, **kw):
    return inputs.small(Hq=2, Hv=4, K=128, V=128, zero_frac=0.25, gate_mu=-4.0, const_heads=1,
                        const_g=-3.0, bwd=bwd, name=name, **kw)


def _min_chunk_logdecay(x):
    """The most negative sum of g over a whole 64-token chunk (the test's regime check)."""
    g = x["g"].double()
    cu = x["cu_seqlens"]
    seqs = [g[b] for b in range(g.shape[0])] if cu is None else \
        [g[0, int(cu[i]):int(cu[i + 1])] for i in range(len(cu) - 1)]
    best = 0.0
    for s in seqs:
        for c0 in range(0, s.shape[0] - 63, 64):
            best = min(best, float(s[c0:c0 + 64].sum(dim=0).min()))
    return best


CASES = [
    ("fixed", dict(B=2, T=200)),
    ("varlen", dict(lengths=(64, 1, 130, 65))),
]


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case,kw", CASES, ids=[c for c, _ in CASES])
@pytest.mark.parametrize("cp", [1, 3])
def test_fwd_strong_decay(gdr, path, case, kw, cp):
    spec = _spec(f"strong_{case}", **kw)
    x = inputs.make(spec, seed=5)
    assert _min_chunk_logdecay(x) < -150  # far past where e^{-gamma} leaves fp32
    d = to_dev(x)
    out = gpu_fwd(gdr, d, path=_path(gdr, path), cp_segments=cp, want_h=True)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_fwd(x, want_h=True)
    tol = TOL[spec.in_dtype]
    e = {"o": err(out["o"], ref["o"], "o"),
         "final_state": err(out["final_state"], ref["final_state"], "final_state"),
         "A": err(out["A"], oracle_A(x), "A"),
         "h": err(out["h"], ref["h"].reshape(out["h"].shape), "h")}
    assert all(np.isfinite(v) and v <= tol for v in e.values()), e


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case,kw", CASES, ids=[c for c, _ in CASES])
@pytest.mark.parametrize("cp", [1, 3])
def test_bwd_strong_decay(gdr, path, case, kw, cp):
    spec = _spec(f"strong_{case}", bwd=True, **kw)
    x = inputs.make(spec, seed=5)
    d = to_dev(x)
    p = _path(gdr, path)
    out = gpu_fwd(gdr, d, path=p, cp_segments=cp)
    gr = gpu_bwd(gdr, d, out["A"], path=p, cp_segments=cp)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_bwd(x)
    tol = TOL[spec.in_dtype]
    e = {key: err(gr[key], ref[key], key) for key in ("dq", "dk", "dv", "dbeta", "dg", "dh0")}
    assert all(np.isfinite(v) and v <= tol for v in e.values()), e


def test_strong_decay_long_segments(gdr):
    """A context-parallel split with warm-up starts allowed (segments of 32
    chunks and more): the decaying heads pass the warm-up gate at once, the
    g = 0 head keeps the exact split; forward and backward on the tensor-core
    path against the oracle."""
    p = _path(gdr, "tc")
    spec = _spec("strong_long", bwd=True, B=1, T=64 * 70 + 9)
    x = inputs.make(spec, seed=7)
    d = to_dev(x)
    out = gpu_fwd(gdr, d, path=p, cp_segments=2, cp_warmup=8)
    gr = gpu_bwd(gdr, d, out["A"], path=p, cp_segments=2, cp_warmup=8)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_fwd(x)
    rg = oracle_bwd(x)
    tol = TOL[spec.in_dtype]
    e = {"o": err(out["o"], ref["o"], "o"), "final_state": err(out["final_state"], ref["final_state"], "final_state")}
    e.update({key: err(gr[key], rg[key], key) for key in ("dq", "dk", "dv", "dbeta", "dg", "dh0")})
    assert all(np.isfinite(v) and v <= tol for v in e.values()), e
