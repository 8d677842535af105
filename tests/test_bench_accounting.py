"""The benchmark's algorithmic work figures, checked against sums written out
here from the workloads' shapes: a step's flops are the method's dense
contractions (forward 83.3k and backward 245.8k multiply-adds per token-head at
K = V = 128, C = 64, G = 2), its bytes the step's inputs read once and outputs
written once.  The forward-only workloads return o and final_state, so A counts
neither as written work nor as bytes there."""
import pytest

import bench
from gated_deltanet_chunked_delta_gb300 import inputs


PEAKS = {"bf16_tflops": 1000.0, "hbm_gbs": 1000.0, "sm_max_mhz": 2000.0, "source": "test"}


def _step(name, mode):
    spec = inputs.resolve(name)
    nch = spec.tokens // 64 * spec.Hv if spec.lengths is None else None
    if nch is None:
        nch = sum((n + 63) // 64 for n in spec.lengths) * spec.Hv
    per_kernel = {"tc_scan": [1.0], "tc_chunk": [0.5]}
    if mode != "fwd":
        per_kernel["tc_bwd_chunk"] = [2.0]
    return spec, bench.rooflines(spec, mode, per_kernel, PEAKS, nch, 4.0)


def test_long_forward_counts_o_and_final_state_only():
    spec, (roof, frac, step, kernels) = _step("fwd_bf16_T262144_hq8_hv16_d128", "fwd")
    T, Hq, Hv, d = 262144, 8, 16, 128
    q_k = 2 * T * Hq * d * 2          # q and k, bf16
    v = T * Hv * d * 2                # v, bf16
    g_b = 2 * T * Hv * 4              # g and beta, fp32
    o = T * Hv * d * 4                # o, fp32 on this workload
    fs = Hv * d * d * 4               # final_state (h0 absent)
    assert step["bytes"] == q_k + v + g_b + o + fs
    assert step["bytes"] == pytest.approx(4.33e9, rel=2e-3)  # the workload's published-shape figure
    assert step["flops"] == pytest.approx(T * Hv * 2 * 83.3e3, rel=1e-3)
    assert roof["kernel"] == "tc_scan"


def test_forward_chunk_kernel_writes_A_only_before_a_backward():
    spec = inputs.resolve("fwd_bf16_T262144_hq8_hv16_d128")
    n = spec.tokens // 64 * spec.Hv
    A = spec.tokens * spec.Hv * 64 * 4
    _, with_A = bench.kernel_work("tc_chunk", spec, 2, 4, n, with_A=True)
    _, without = bench.kernel_work("tc_chunk", spec, 2, 4, n, with_A=False)
    assert with_A - without == A
    # the backward's pass from A reads it whatever the forward wrote
    _, from_A = bench.kernel_work("tc_chunk_from_A", spec, 2, 4, n, with_A=False)
    assert from_A == with_A


def test_fwd_bwd_step_counts_A_written_and_read():
    spec, (roof, frac, step, kernels) = _step("bwd_bf16_B2_T16384_hq32_hv64_d128", "both")
    T, Hq, Hv, d = 2 * 16384, 32, 64, 128
    q_k, v, g_b = 2 * T * Hq * d * 2, T * Hv * d * 2, 2 * T * Hv * 4
    A = T * Hv * 64 * 4
    st = 2 * Hv * d * d * 4
    fwd = q_k + v + g_b + st + T * Hv * d * 2 + st + A          # h0 in; o, final_state, A out
    bwd = (q_k + 2 * v + g_b + A + 2 * st) + (q_k + v + g_b + st)  # q, k, v, do, g, beta, A, h0, dht in; grads out
    assert step["bytes"] == fwd + bwd
    assert step["flops"] == pytest.approx(T * Hv * 2 * (83.3e3 + 245.8e3), rel=1e-3)
    assert roof["kernel"] == "tc_bwd_chunk"


def test_overhead_kernel_is_named_beside_the_dominant_one():
    spec = inputs.resolve("fwd_bf16_T262144_hq8_hv16_d128")
    n = spec.tokens // 64 * spec.Hv
    per_kernel = {"tc_cp_summary": [3.0], "tc_scan": [1.0], "tc_chunk": [0.5]}
    roof, _, _, _ = bench.rooflines(spec, "fwd", per_kernel, PEAKS, n, 4.0)
    assert roof["kernel"] == "tc_scan" and roof["longest_kernel"] == "tc_cp_summary"
