"""Writes the oracle regression fixture ``oracle_T20_hq1_hv2_k4_v4.txt``.

The FlashQLA pages print no worked example of the gated delta rule (no input
with its output), so no fixture here holds the pages' own numbers.  This one is
a frozen copy of what the fp64 oracle (``oracle/``) returns for one small
seeded problem: inputs drawn by the package's seeded generator, outputs from
``oracle.fwd`` and ``oracle.bwd`` only.  ``tests/test_golden.py`` checks that
the generator still draws these inputs and that the oracle, built on whatever
machine runs the tests, still returns these outputs; the oracle's correctness
itself rests on the pins in ``tests/test_oracle_pins.py``.

What it computes (FlashQLA pages, page 1 "usage and requirements", the
forward's ``o`` and ``final_state`` and the backward's ``dq, dk, dv, db, dg,
dh0``): S_t = e^{g_t}(I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T,
o_t = scale S_t^T q_t, and the reverse mode of that map.

Run from the repository root: ``python tests/golden/make_golden.py``.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

NAME = "oracle_T20_hq1_hv2_k4_v4.txt"
SEED = 7
INPUTS = ("q", "k", "v", "g", "beta", "h0", "do", "dht")
OUTPUTS = ("o", "final_state", "dq", "dk", "dv", "dbeta", "dg", "dh0")


def spec():
    from gated_deltanet_chunked_delta_gb300 import inputs
    # 20 tokens, one qk-head shared by two v-heads (one of them with g = 0),
    # K = V = 4, fp32 inputs, initial state and dht drawn
    return inputs.small(B=1, T=20, Hq=1, Hv=2, K=4, V=4, in_dtype="f32", zero_frac=0.5, h0=True, bwd=True,
                        name="golden")


def draw():
    from gated_deltanet_chunked_delta_gb300 import inputs
    x = inputs.make(spec(), seed=SEED)
    return {n: x[n].double().numpy() for n in INPUTS}, float(x["scale"])


def compute(xin, scale):
    import oracle
    f = oracle.fwd(xin["q"], xin["k"], xin["v"], xin["g"], xin["beta"], scale, h0=xin["h0"])
    b = oracle.bwd(xin["q"], xin["k"], xin["v"], xin["g"], xin["beta"], scale, xin["do"], dht=xin["dht"],
                   h0=xin["h0"])
    return {"o": f["o"], "final_state": f["final_state"], **b}


def dump(path, xin, scale, out):
    with open(path, "w") as fh:
        fh.write("# Oracle regression fixture, written by tests/golden/make_golden.py (oracle/ only).\n")
        fh.write("# Not the pages' numbers: the FlashQLA pages print no worked example.\n")
        fh.write(f"# inputs: gated_deltanet_chunked_delta_gb300.inputs.small(B=1, T=20, Hq=1, Hv=2, K=4, V=4,\n")
        fh.write(f"#   in_dtype='f32', zero_frac=0.5, h0=True, bwd=True), seed {SEED}; scale = K^-1/2\n")
        fh.write(f"scale {scale!r}\n")
        for n in INPUTS + OUTPUTS:
            a = (xin if n in xin else out)[n]
            fh.write(f"{n} {' '.join(str(d) for d in a.shape)}\n")
            fh.write(" ".join(repr(float(t)) for t in a.ravel()) + "\n")


def load(path=os.path.join(HERE, NAME)):
    arrays, scale = {}, None
    with open(path) as fh:
        lines = [ln.rstrip("\n") for ln in fh if not ln.startswith("#")]
    i = 0
    while i < len(lines):
        head = lines[i].split()
        if head[0] == "scale":
            scale = float(head[1])
            i += 1
            continue
        shape = tuple(int(d) for d in head[1:])
        arrays[head[0]] = np.array([float(t) for t in lines[i + 1].split()], dtype=np.float64).reshape(shape)
        i += 2
    return arrays, scale


def main():
    xin, scale = draw()
    dump(os.path.join(HERE, NAME), xin, scale, compute(xin, scale))


if __name__ == "__main__":
    main()
