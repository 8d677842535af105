"""GPU parity of the C ABI against the fp64 oracle at oracle-friendly sizes
(several chunks, ragged tails, varlen, grouped heads, forced context-parallel
segmentations, degenerate gates).  Bounds: max|x - ref| / rms(ref) <= 2e-3 for
fp32 inputs and <= 2e-2 for bf16 inputs, for every output and gradient."""
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


def _path(gdr, name, spec):
    if name == "simt":
        return gdr.GDR_PATH_SIMT
    if spec.in_dtype != "bf16" or spec.K != 128 or spec.V != 128:
        pytest.skip("tensor-core path covers bf16 with K = V = 128")
    if not gdr.tc_available(spec.K, spec.V):
        pytest.skip("the library has no tensor-core path")
    return gdr.GDR_PATH_TC


def _check_fwd(gdr, spec, path, cp=0, want_h=True, seed=0):
    x = inputs.make(spec, seed=seed)
    d = to_dev(x)
    out = gpu_fwd(gdr, d, path=path, cp_segments=cp, want_h=want_h,
                  o_dtype=torch.float32 if spec.out_dtype == "f32" else None)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_fwd(x, want_h=want_h)
    tol = TOL[spec.in_dtype]
    e = {"o": err(out["o"], ref["o"], "o"), "final_state": err(out["final_state"], ref["final_state"], "final_state"),
         "A": err(out["A"], oracle_A(x), "A")}
    if want_h:
        e["h"] = err(out["h"], ref["h"].reshape(out["h"].shape), "h")
    assert all(v <= tol for v in e.values()), e
    return out


def _check_bwd(gdr, spec, path, cp=0, seed=0):
    x = inputs.make(spec, seed=seed)
    d = to_dev(x)
    out = gpu_fwd(gdr, d, path=path, cp_segments=cp)
    gr = gpu_bwd(gdr, d, out["A"], path=path, cp_segments=cp)
    torch.cuda.synchronize()
    gdr.check_status()
    ref = oracle_bwd(x)
    tol = TOL[spec.in_dtype]
    e = {key: err(gr[key], ref[key], key) for key in ("dq", "dk", "dv", "dbeta", "dg", "dh0")}
    assert all(v <= tol for v in e.values()), e


def test_fwd_fp32_correctness_workload(gdr):
    spec = inputs.CONFIGS["fwd_f32_T256_hq2_hv4_d64"]
    _check_fwd(gdr, spec, gdr.GDR_PATH_AUTO)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 200])
def test_fwd_ragged_lengths(gdr, path, T):
    spec = inputs.small(B=2, T=T, Hq=2, Hv=4, K=128, V=128, in_dtype="bf16")
    _check_fwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("K,V", [(64, 64), (64, 128), (128, 64), (128, 128)])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_fwd_head_dims(gdr, K, V, dt):
    spec = inputs.small(B=1, T=150, Hq=1, Hv=2, K=K, V=V, in_dtype=dt)
    _check_fwd(gdr, spec, gdr.GDR_PATH_SIMT)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("Hq,Hv", [(4, 4), (2, 4), (1, 4)])
def test_fwd_grouped_heads(gdr, path, Hq, Hv):
    spec = inputs.small(B=1, T=130, Hq=Hq, Hv=Hv, K=128, V=128)
    _check_fwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("lengths", [(1, 64, 65, 3), (0, 130, 7), (200,), (64, 0)])
def test_fwd_varlen(gdr, path, lengths):
    spec = inputs.small(lengths=lengths, Hq=2, Hv=4, K=128, V=128)
    _check_fwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("path", PATHS)
def test_fwd_context_parallel_segmentations(gdr, path):
    spec = inputs.small(B=1, T=640 + 17, Hq=1, Hv=2, K=128, V=128, zero_frac=0.5)
    p = _path(gdr, path, spec)
    outs = [_check_fwd(gdr, spec, p, cp=cp, want_h=True) for cp in (1, 2, 3, 5, 11)]
    # each segmentation is exact up to rounding: all agree with each other
    for o in outs[1:]:
        assert err(o["o"], outs[0]["o"].double().cpu().numpy(), "o vs cp=1") <= 2e-2
    # and a repeated run is bit-identical
    again = _check_fwd(gdr, spec, p, cp=3, want_h=True)
    assert torch.equal(again["o"], outs[2]["o"]) and torch.equal(again["final_state"], outs[2]["final_state"])


@pytest.mark.parametrize("path", PATHS)
def test_fwd_varlen_context_parallel(gdr, path):
    spec = inputs.small(lengths=(700, 1, 129, 0, 300), Hq=2, Hv=4, K=128, V=128)
    p = _path(gdr, path, spec)
    for cp in (1, 4):
        _check_fwd(gdr, spec, p, cp=cp)


@pytest.mark.parametrize("path", PATHS)
def test_fwd_beta_zero_is_pure_decay(gdr, path):
    spec = inputs.small(B=1, T=100, Hq=1, Hv=2, K=128, V=128)
    p = _path(gdr, path, spec)
    x = inputs.make(spec)
    x["beta"].zero_()
    d = to_dev(x)
    out = gpu_fwd(gdr, d, path=p)
    G = x["g"].double().cumsum(dim=1)
    q = x["q"].double().repeat_interleave(2, dim=2)
    o_ref = x["scale"] * torch.exp(G)[..., None] * torch.einsum("bthk,bhkv->bthv", q, x["h0"].double())
    assert err(out["o"], o_ref.numpy(), "o") <= TOL["bf16"]
    fs_ref = torch.exp(G[:, -1])[:, :, None, None] * x["h0"].double()
    assert err(out["final_state"], fs_ref.numpy(), "final_state") <= 1e-5


@pytest.mark.parametrize("path", PATHS)
def test_fwd_all_gates_one(gdr, path):
    spec = inputs.small(B=1, T=190, Hq=2, Hv=4, K=128, V=128, zero_frac=1.0)
    _check_fwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("path", PATHS)
def test_bwd_bf16(gdr, path):
    spec = inputs.small(B=2, T=200, Hq=2, Hv=4, K=128, V=128, bwd=True)
    _check_bwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("K,V", [(64, 64), (128, 64), (64, 128)])
def test_bwd_fp32_head_dims(gdr, K, V):
    spec = inputs.small(B=1, T=130, Hq=1, Hv=2, K=K, V=V, in_dtype="f32", bwd=True)
    _check_bwd(gdr, spec, gdr.GDR_PATH_SIMT)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("lengths", [(1, 64, 65, 3), (0, 150)])
def test_bwd_varlen(gdr, path, lengths):
    spec = inputs.small(lengths=lengths, Hq=2, Hv=4, K=128, V=128, bwd=True)
    _check_bwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("Hq,Hv", [(4, 4), (1, 4)])
def test_bwd_grouped_heads(gdr, path, Hq, Hv):
    # G = 1 (no qk-head sum) and G = 4 (the last of four v-heads adds the group)
    spec = inputs.small(B=1, T=130, Hq=Hq, Hv=Hv, K=128, V=128, bwd=True)
    _check_bwd(gdr, spec, _path(gdr, path, spec))


@pytest.mark.parametrize("path", PATHS)
def test_bwd_context_parallel_and_no_initial_state(gdr, path):
    spec = inputs.small(B=1, T=700, Hq=1, Hv=4, K=128, V=128, h0=False, bwd=True)
    p = _path(gdr, path, spec)
    for cp in (1, 4):
        _check_bwd(gdr, spec, p, cp=cp)


def test_debug_checks_clean_run(gdr):
    spec = inputs.small(B=1, T=100, Hq=1, Hv=2, K=64, V=64)
    x = inputs.make(spec)
    d = to_dev(x)
    gpu_fwd(gdr, d, path=gdr.GDR_PATH_SIMT, debug_checks=1)
    gdr.check_status()


def test_bounded_waits_report_timeout_and_leave_the_context_usable(gdr):
    """Every device-side wait of the tensor-core kernels is a bounded poll.  With
    a cap of one poll the waits run out: the kernels raise their abort flag,
    drain their own copies and MMAs, free tensor memory and return; the host
    reads GDR_ERR_TIMEOUT, and the next call on the same context is correct."""
    if not gdr.tc_available():
        pytest.skip("the library has no tensor-core path")
    spec = inputs.small(B=1, T=64 * 40, Hq=1, Hv=2, K=128, V=128, bwd=True)
    x = inputs.make(spec)
    d = to_dev(x)
    out = gpu_fwd(gdr, d, path=gdr.GDR_PATH_TC, cp_segments=4, timeout_spins=1)
    gpu_bwd(gdr, d, out["A"], path=gdr.GDR_PATH_TC, cp_segments=4, timeout_spins=1)
    with pytest.raises(gdr.GdrError) as info:
        gdr.check_status()
    assert info.value.code == 7
    gdr.check_status()  # the status word was cleared
    _check_fwd(gdr, spec, gdr.GDR_PATH_TC, cp=4)
    _check_bwd(gdr, spec, gdr.GDR_PATH_TC, cp=4)


@pytest.mark.slow
def test_bwd_qk_group_summed_in_place(gdr):
    """152 chunks x one qk-head of G = 4 v-heads: every CTA of the backward's
    chunk kernel takes whole qk-head groups and sums dq, dk over the group in
    place (the path the large workloads take; the small cases above take the
    separate head-order sum)."""
    spec = inputs.small(B=1, T=64 * 152, Hq=1, Hv=4, K=128, V=128, bwd=True)
    _check_bwd(gdr, spec, _path(gdr, "tc", spec))


# Head sizes beyond 128 (the CUDA-core path: K up to 192, V up to 256), forward
# and backward, fp32 and bf16 inputs, with a context-parallel split and packed
# sequences among the cases.
WIDE = [(128, 256), (64, 256), (192, 192), (192, 64), (192, 256), (64, 192)]


@pytest.mark.parametrize("K,V", WIDE)
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_wide_head_dims(gdr, K, V, dt):
    spec = inputs.small(B=1, T=150, Hq=1, Hv=2, K=K, V=V, in_dtype=dt, bwd=True)
    _check_fwd(gdr, spec, gdr.GDR_PATH_AUTO)
    _check_bwd(gdr, spec, gdr.GDR_PATH_AUTO)


@pytest.mark.parametrize("K,V", [(128, 256), (192, 192)])
def test_wide_head_dims_split_and_varlen(gdr, K, V):
    spec = inputs.small(B=1, T=64 * 9 + 5, Hq=1, Hv=2, K=K, V=V, bwd=True, name="wide_cp")
    _check_fwd(gdr, spec, gdr.GDR_PATH_AUTO, cp=3)
    _check_bwd(gdr, spec, gdr.GDR_PATH_AUTO, cp=3)
    spec = inputs.small(lengths=(64, 1, 130, 65), Hq=1, Hv=2, K=K, V=V, bwd=True, name="wide_varlen")
    _check_fwd(gdr, spec, gdr.GDR_PATH_AUTO)
    _check_bwd(gdr, spec, gdr.GDR_PATH_AUTO)
