"""The oracle regression fixture (tests/golden): the seeded generator still
draws the stored inputs, and the oracle built on this machine still returns the
stored outputs.  The pages print no worked example, so the fixture is the
oracle's own output (written by tests/golden/make_golden.py, which calls only
oracle/); what pins the oracle to the method is tests/test_oracle_pins.py."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
import make_golden  # noqa: E402


def test_generator_draws_the_stored_inputs():
    stored, scale = make_golden.load()
    xin, s = make_golden.draw()
    assert s == scale
    for n in make_golden.INPUTS:
        np.testing.assert_array_equal(xin[n], stored[n], err_msg=n)


def test_oracle_reproduces_the_stored_outputs():
    stored, scale = make_golden.load()
    xin = {n: stored[n] for n in make_golden.INPUTS}
    out = make_golden.compute(xin, scale)
    for n in make_golden.OUTPUTS:
        ref = stored[n]
        # fp64, same algorithm; only the summation order of a different
        # compiler or machine may differ
        tol = 1e-12 * max(1.0, float(np.abs(ref).max()))
        assert np.abs(out[n] - ref).max() <= tol, n


def test_fixture_is_consistent():
    """Checks on the stored values that need no oracle: shapes, the v-head with
    g = 0, and the final state of a decay-free head against the sum that
    defines it when its keys and values are replayed."""
    st, scale = make_golden.load()
    assert st["o"].shape == (1, 20, 2, 4) and st["final_state"].shape == (1, 2, 4, 4)
    assert st["dq"].shape == st["q"].shape and st["dv"].shape == st["v"].shape
    zero = [h for h in range(2) if np.all(st["g"][0, :, h] == 0.0)]
    assert len(zero) == 1
    # replay the defining recurrence for the g = 0 head and compare its final
    # state and outputs: S_t = (I - b k k^T) S_{t-1} + b k v^T, o_t = scale S_t^T q_t
    h = zero[0]
    S = st["h0"][0, h].copy()
    for t in range(20):
        kt, vt, bt, qt = st["k"][0, t, 0], st["v"][0, t, h], st["beta"][0, t, h], st["q"][0, t, 0]
        S = S - bt * np.outer(kt, kt @ S) + bt * np.outer(kt, vt)
        np.testing.assert_allclose(scale * S.T @ qt, st["o"][0, t, h], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, st["final_state"][0, h], rtol=0, atol=1e-12)
