"""Warm-up starts of context-parallel segments (on the tensor-core path by
default for segments of at least 32 chunks, forced here): a v-head whose gates bound the warm-up error below 1e-6
skips the exact summary and combine; a head with g = 0 (no decay) keeps the
exact split.  Both must match the oracle; the no-decay heads must match the
exact-only run bit for bit, and the decaying heads must differ from it (the
warm-up ran)."""
import pytest
import torch

from gated_deltanet_chunked_delta_gb300 import inputs
from parity import TOL, err, gpu_fwd, gpu_bwd, oracle_bwd, oracle_fwd, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdr():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_deltanet_chunked_delta_gb300 as gdr
    gdr.load(build_if_missing=True)
    if not gdr.tc_available():
        pytest.skip("no tensor-core path")
    return gdr


@pytest.mark.parametrize("lengths", [None, (2100, 64, 1700)])
def test_warmup_starts(gdr, lengths):
    if lengths is None:
        spec = inputs.small(B=2, T=2048, Hq=2, Hv=4, K=128, V=128, zero_frac=0.5, bwd=True, name="fixed")
    else:
        spec = inputs.small(lengths=lengths, Hq=2, Hv=4, K=128, V=128, zero_frac=0.5, bwd=True, name="varlen")
    x = inputs.make(spec, seed=11)
    d = to_dev(x)
    warm = gpu_fwd(gdr, d, cp_segments=4, cp_warmup=8)
    exact = gpu_fwd(gdr, d, cp_segments=4, cp_warmup=-1)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_fwd(x)
    tol = TOL[spec.in_dtype]
    for out in (warm, exact):
        assert err(out["o"], ref["o"]) <= tol
        assert err(out["final_state"], ref["final_state"]) <= tol
    zero = x["zero_heads"]
    decaying = [h for h in range(spec.Hv) if h not in zero]
    assert zero and decaying
    for key in ("o", "final_state"):
        w, e = warm[key].float(), exact[key].float()
        hd = 2 if key == "o" else 1
        assert torch.equal(w.index_select(hd, torch.tensor(zero, device=w.device)),
                           e.index_select(hd, torch.tensor(zero, device=w.device))), key
    dec = torch.tensor(decaying, device=warm["o"].device)
    assert (warm["o"].float().index_select(2, dec) - exact["o"].float().index_select(2, dec)).abs().max() > 0
    # the backward's state recompute takes the same starts
    gr = gpu_bwd(gdr, d, warm["A"], cp_segments=4, cp_warmup=8)
    torch.cuda.synchronize()
    gdr.check_status()
    rg = oracle_bwd(x)
    e = {key: err(gr[key], rg[key]) for key in ("dq", "dk", "dv", "dbeta", "dg", "dh0")}
    assert all(v <= tol for v in e.values()), e
