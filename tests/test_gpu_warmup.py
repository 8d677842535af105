"""Warm-up starts of context-parallel segments (on the tensor-core path by
default for segments of at least 32 chunks, forced here): a v-head whose gates bound the warm-up error below 1e-6
skips the exact summary and combine; a head with g = 0 (no decay) keeps the
exact split.  Both must match the oracle; the no-decay heads must match the
exact-only run bit for bit."""
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
        assert err(out["o"], ref["o"], "o") <= tol
        assert err(out["final_state"], ref["final_state"], "final_state") <= tol
    zero = x["zero_heads"]
    decaying = [h for h in range(spec.Hv) if h not in zero]
    assert zero and decaying
    for key in ("o", "final_state"):
        w, e = warm[key].float(), exact[key].float()
        hd = 2 if key == "o" else 1
        assert torch.equal(w.index_select(hd, torch.tensor(zero, device=w.device)),
                           e.index_select(hd, torch.tensor(zero, device=w.device))), key
    # (the decaying heads' warm-up starts differ from the exact ones by less than
    # the gate's bound, 1e-6 of the state, so their outputs may or may not
    # differ from the exact run's in the last bit; both match the oracle above)
    # the backward's state recompute takes the same starts
    gr = gpu_bwd(gdr, d, warm["A"], cp_segments=4, cp_warmup=8)
    torch.cuda.synchronize()
    gdr.check_status()
    rg = oracle_bwd(x)
    e = {key: err(gr[key], rg[key], key) for key in ("dq", "dk", "dv", "dbeta", "dg", "dh0")}
    assert all(v <= tol for v in e.values()), e


def test_warmup_start_is_taken(gdr):
    """A case where the warm-up start differs visibly from the exact one: every
    k_t is the same unit vector, so the state's other rows carry only the
    decayed h0, which a start from zero does not have.  Head 0 decays by
    e^{-15} over the 8-chunk window (below the gate's 1e-6: it takes warm-up
    starts), head 1 not at all (exact split).  The state before the first chunk
    of segment 1 must then be zero off row 0 for head 0 in the warm run and
    equal to the exact run for head 1; both runs match the oracle."""
    spec = inputs.small(B=1, T=64 * 40, Hq=1, Hv=2, K=128, V=128, zero_frac=0.0, name="warm_taken")
    x = inputs.make(spec, seed=3)
    k = torch.zeros_like(x["k"], dtype=torch.float32)
    k[..., 0] = 1.0
    x["k"] = k.to(x["k"].dtype)
    x["beta"] = torch.full_like(x["beta"], 0.5)
    x["g"] = torch.zeros_like(x["g"])
    x["g"][:, :, 0] = -15.0 / 512
    d = to_dev(x)
    warm = gpu_fwd(gdr, d, cp_segments=4, cp_warmup=8, want_h=True)
    exact = gpu_fwd(gdr, d, cp_segments=4, cp_warmup=-1, want_h=True)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_fwd(x, want_h=True)
    for out in (warm, exact):
        assert err(out["o"], ref["o"], "o") <= TOL["bf16"]
        assert err(out["h"], ref["h"].reshape(out["h"].shape), "h") <= TOL["bf16"]
    hw, he = warm["h"][10], exact["h"][10]  # before chunk 10, the first of segment 1
    assert torch.count_nonzero(hw[0, 1:]) == 0          # head 0 started from zero 8 chunks back
    assert torch.count_nonzero(he[0, 1:]) > 0           # the exact start carries the decayed h0
    assert torch.equal(hw[1], he[1])                    # head 1 took the exact split in both runs
