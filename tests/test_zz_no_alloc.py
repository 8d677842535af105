"""gdr_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers (a plugin inside a host program that owns all device memory and
hands out no allocator, or a path where cudaMalloc's possible device
synchronisation is not allowed) call gdr_fwd_noalloc, which runs the same
forward as gdr_fwd on a fixed workspace compiled into the library.  This test
calls it through the C ABI twice in a row and compares every output with
gdr_fwd's, and checks that an oversized problem is refused before launch.
It sits in its own file, collected last, so that a stopped-at-first-failure
run has already run every other test.
"""
import ctypes

import pytest
import torch

from gated_deltanet_chunked_delta_gb300 import inputs
from parity import TOL, err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import gated_deltanet_chunked_delta_gb300 as gdr
    lb = gdr.load(build_if_missing=True)
    from gated_deltanet_chunked_delta_gb300 import binding as B
    P, vp = ctypes.POINTER, ctypes.c_void_p
    lb.gdr_fwd_noalloc.argtypes = [P(B.gdr_shape), B.gdr_buf, B.gdr_buf, B.gdr_buf, vp, vp, ctypes.c_float, vp,
                                   B.gdr_buf, vp, vp, vp, P(B.gdr_opts), vp]
    lb.gdr_fwd_noalloc.restype = ctypes.c_int
    return lb


def _call_noalloc(lib, d, scale, out, cp=0):
    import gated_deltanet_chunked_delta_gb300 as gdr
    from gated_deltanet_chunked_delta_gb300 import binding as B
    prob = gdr.Problem(d["q"], d["v"], d["cu_seqlens"])
    opts = gdr.make_opts(cp)
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.gdr_fwd_noalloc(ctypes.byref(prob.shape), B._buf(d["q"]), B._buf(d["k"]), B._buf(d["v"]),
                             d["g"].data_ptr(), d["beta"].data_ptr(), float(scale),
                             None if d["h0"] is None else d["h0"].data_ptr(), B._buf(out["o"]),
                             out["final_state"].data_ptr(), out["A"].data_ptr(), None, ctypes.byref(opts), stream)
    return rc


# (spec, cp_segments): one plain case per path, a forced context-parallel
# split (its summaries, composed transitions and start states live in the
# shared array too), and the bf16 context-parallel workload of 8192 tokens x 8
# v-heads, whose tensor-core plan fits the array although the CUDA-core plan
# of the same sizes would not.
CASES = [
    (inputs.small(B=1, T=300, Hq=2, Hv=4, K=128, V=128, name="bf16_tc"), 0),
    (inputs.small(B=2, T=130, Hq=1, Hv=2, K=64, V=64, in_dtype="f32", name="f32_simt"), 0),
    (inputs.small(B=1, T=64 * 20 + 5, Hq=1, Hv=2, K=128, V=128, name="bf16_tc_cp3"), 3),
    (inputs.CONFIGS["fwd_bf16_T8192_hq4_hv8_d128"], 0),
]


@pytest.mark.parametrize("spec,cp", CASES, ids=[s.name for s, _ in CASES])
def test_noalloc_matches_gdr_fwd_on_two_calls(lib, spec, cp):
    """Same kernels, same plan: the outputs must equal gdr_fwd's bit for bit,
    on two calls in a row (the second runs on what the first left in the array)."""
    import gated_deltanet_chunked_delta_gb300 as gdr
    x = inputs.make(spec, seed=3)
    d = to_dev(x)
    ref = gdr.gdr_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], x["scale"], h0=d["h0"], cp_segments=cp)
    torch.cuda.synchronize()
    tol = TOL[spec.in_dtype]
    for _ in range(2):
        out = {key: torch.full_like(ref[key], float("nan")) for key in ("o", "final_state", "A")}
        rc = _call_noalloc(lib, d, x["scale"], out, cp)
        assert rc == 0, lib.gdr_last_error().decode()
        torch.cuda.synchronize()
        gdr.check_status()
        for key in ("o", "final_state", "A"):
            assert torch.equal(out[key], ref[key]), key
            assert err(out[key], ref[key].double().cpu().numpy(), key) <= tol, key


def test_noalloc_rejects_oversized_problem(lib):
    # a workspace far beyond the fixed array: rejected before any launch
    spec = inputs.small(B=1, T=64, Hq=1, Hv=1, K=128, V=128)
    x = inputs.make(spec)
    d = to_dev(x)
    import gated_deltanet_chunked_delta_gb300 as gdr
    from gated_deltanet_chunked_delta_gb300 import binding as B
    big = B.gdr_shape(1, 1 << 22, 1, 64, 128, 128, 0, None, None)
    opts = gdr.make_opts()
    o = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    rc = lib.gdr_fwd_noalloc(ctypes.byref(big), B._buf(d["q"]), B._buf(d["k"]), B._buf(d["v"]),
                             d["g"].data_ptr(), d["beta"].data_ptr(), 0.1, None, B._buf(o), None, None, None,
                             ctypes.byref(opts), None)
    assert rc == 5
    assert "workspace" in lib.gdr_last_error().decode()


def test_noalloc_argument_errors_match_gdr_fwd(lib):
    """Invalid arguments get the codes gdr_fwd returns: a null shape is an
    argument error, a forced tensor-core path with fp32 inputs a dtype error."""
    import gated_deltanet_chunked_delta_gb300 as gdr
    from gated_deltanet_chunked_delta_gb300 import binding as B
    spec = inputs.small(B=1, T=64, Hq=1, Hv=1, K=128, V=128, in_dtype="f32")
    x = inputs.make(spec)
    d = to_dev(x)
    o = torch.empty_like(d["v"])
    args = (B._buf(d["q"]), B._buf(d["k"]), B._buf(d["v"]), d["g"].data_ptr(), d["beta"].data_ptr(), 0.1, None,
            B._buf(o), None, None, None)
    assert lib.gdr_fwd_noalloc(None, *args, ctypes.byref(gdr.make_opts()), None) == 1
    prob = gdr.Problem(d["q"], d["v"], None)
    rc = lib.gdr_fwd_noalloc(ctypes.byref(prob.shape), *args, ctypes.byref(gdr.make_opts(0, gdr.GDR_PATH_TC)),
                             None)
    assert rc == 3, lib.gdr_last_error().decode()
