"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (automatic path and context-parallel plan).  The oracle checks
whole qk-head groups (every output of the selected heads over the whole
sequence) where a full check would take too long on the host: one group with a
unit-gate head and one group whose heads all decay, per workload, forward and
backward."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_chunked_delta_gb300 import inputs
from parity import TOL, err, select_heads, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def gdr():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_deltanet_chunked_delta_gb300 as m
    m.load(build_if_missing=True)
    return m


def _groups(x):
    """qk-heads to check: one whose group holds a g == 0 head, and one gated."""
    spec = x["spec"]
    G = spec.Hv // spec.Hq
    zero = set(x["zero_heads"])
    with_zero = [hq for hq in range(spec.Hq) if any(h in zero for h in range(hq * G, hq * G + G))]
    gated = [hq for hq in range(spec.Hq) if not any(h in zero for h in range(hq * G, hq * G + G))]
    out = []
    if with_zero:
        out.append(with_zero[0])
    if gated:
        out.append(gated[-1])
    return out


def _fwd_case(gdr, name, full_oracle=False):
    x = inputs.make(name, seed=0)
    spec = x["spec"]
    d = to_dev(x)
    o_dtype = torch.float32 if spec.out_dtype == "f32" else torch.bfloat16
    out = gdr.gdr_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], h0=d["h0"],
                      cu_seqlens=d["cu_seqlens"], cu_seqlens_host=x["cu_seqlens"], o_dtype=o_dtype)
    torch.cuda.synchronize()
    gdr.check_status()
    tol = TOL[spec.in_dtype]
    hqs = range(spec.Hq) if full_oracle else _groups(x)
    for hq in hqs:
        y, hv = select_heads(x, hq)
        ref = oracle.fwd(y["q"], y["k"], y["v"], y["g"], y["beta"], x["scale"], h0=y["h0"],
                         cu_seqlens=x["cu_seqlens"], vblock=16)
        A_ref = oracle.A_matrix(y["k"], y["g"], y["beta"], cu_seqlens=x["cu_seqlens"])
        e = {"o": err(out["o"][:, :, hv], ref["o"], f"o hq{hq}"),
             "final_state": err(out["final_state"][:, hv], ref["final_state"], f"final_state hq{hq}"),
             "A": err(out["A"][:, :, hv], A_ref, f"A hq{hq}")}
        assert all(v <= tol for v in e.values()), (name, hq, e)


def test_fwd_context_parallel_workload(gdr):
    _fwd_case(gdr, "fwd_bf16_T8192_hq4_hv8_d128", full_oracle=True)


def test_fwd_varlen_workload(gdr):
    _fwd_case(gdr, "fwd_bf16_varlen4_hq16_hv32_d128")


def test_fwd_long_context_workload(gdr):
    _fwd_case(gdr, "fwd_bf16_T262144_hq8_hv16_d128")


def test_bwd_workload(gdr):
    name = "bwd_bf16_B2_T16384_hq32_hv64_d128"
    x = inputs.make(name, seed=0)
    spec = x["spec"]
    d = to_dev(x)
    out = gdr.gdr_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], h0=d["h0"])
    gr = gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], out["A"], d["do"], dht=d["dht"],
                     scale=x["scale"], h0=d["h0"])
    torch.cuda.synchronize()
    gdr.check_status()
    tol = TOL[spec.in_dtype]
    groups = _groups(x)
    assert len(groups) == 2  # one group holding a g == 0 head, one whose heads all decay
    for hq in groups:
        y, hv = select_heads(x, hq)
        ref = oracle.bwd(y["q"], y["k"], y["v"], y["g"], y["beta"], x["scale"], y["do"], dht=y["dht"],
                         h0=y["h0"])
        e = {key: err(gr[key][:, :, hq:hq + 1], ref[key], f"{key} hq{hq}") for key in ("dq", "dk")}
        e.update({key: err(gr[key][:, :, hv], ref[key], f"{key} hq{hq}") for key in ("dv", "dbeta", "dg")})
        e["dh0"] = err(gr["dh0"][:, hv], ref["dh0"], f"dh0 hq{hq}")
        assert all(v <= tol for v in e.values()), (name, hq, e)
