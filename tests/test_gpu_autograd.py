"""The high-level differentiable call: forward and gradients through
torch.autograd against the fp64 oracle (the same tolerances as the parity
tests), for equal-length and packed varlen inputs, with and without an
initial state and with the final state used in the loss or not."""
import pytest
import torch

from gated_deltanet_chunked_delta_gb300 import inputs
from parity import TOL, err, oracle_bwd, oracle_fwd, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdr():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_deltanet_chunked_delta_gb300 as gdr
    gdr.load(build_if_missing=True)
    return gdr


@pytest.mark.parametrize("spec", [
    inputs.small(B=2, T=150, Hq=2, Hv=4, K=128, V=128, bwd=True, name="bf16_tc"),
    inputs.small(lengths=(70, 1, 130), Hq=2, Hv=4, K=128, V=128, bwd=True, name="bf16_tc_varlen"),
    inputs.small(B=1, T=100, Hq=1, Hv=2, K=64, V=64, in_dtype="f32", bwd=True, name="f32_simt"),
], ids=lambda s: s.name)
@pytest.mark.parametrize("use_final", [True, False])
def test_autograd_matches_oracle(gdr, spec, use_final):
    x = inputs.make(spec, seed=5)
    d = to_dev(x)
    leaves = {key: d[key].detach().clone().requires_grad_(True) for key in ("q", "k", "v", "g", "beta", "h0")}
    o, fs = gdr.chunk_gated_delta_rule(leaves["q"], leaves["k"], leaves["v"], leaves["g"], leaves["beta"],
                                       scale=x["scale"], initial_state=leaves["h0"], output_final_state=True,
                                       cu_seqlens=d["cu_seqlens"])
    do = d["do"]
    dht = d["dht"] if use_final else None
    loss = (o.float() * do.float()).sum()
    if use_final:
        loss = loss + (fs * dht).sum()
    loss.backward()
    torch.cuda.synchronize()
    gdr.check_status()
    tol = TOL[spec.in_dtype]
    ref = oracle_fwd(x)
    assert err(o.detach(), ref["o"], "o") <= tol
    assert err(fs.detach(), ref["final_state"], "final_state") <= tol
    y = dict(x)
    y["dht"] = x["dht"] if use_final else None
    rg = oracle_bwd(y)
    got = {"dq": leaves["q"].grad, "dk": leaves["k"].grad, "dv": leaves["v"].grad, "dbeta": leaves["beta"].grad,
           "dg": leaves["g"].grad, "dh0": leaves["h0"].grad}
    e = {key: err(got[key], rg[key], key) for key in got}
    assert all(v <= tol for v in e.values()), e
