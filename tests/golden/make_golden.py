"""Writes tests/golden/tiny_f32_b1_t64_n2_k8_v8.json: inputs and fp64 oracle outputs.

The M²RNN study notes print no worked numeric example of the recurrence, so the
only stored expectation is the oracle's own output on the tiny fp32 workload
(B=1, T=64, N=2, K=V=8), frozen so that an accidental change to the oracle's
arithmetic shows up as a diff.  Inputs are stored too, so the fixture does not
depend on a torch random-number stream.  This script calls only the oracle and
the seeded input generator.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from matrix_state_nonlinear_gb300.inputs import WORKLOADS, all_f64, make_inputs  # noqa: E402
from oracle import m2rnn_forward_inputs  # noqa: E402

NAME = "tiny_f32_b1_t64_n2_k8_v8"


def main():
    wl = WORKLOADS[NAME]
    inp = all_f64(make_inputs(wl, "cpu", seed=0))
    y, HT = m2rnn_forward_inputs(inp)
    doc = {
        "workload": NAME,
        "shape": {"B": wl.B, "T": wl.T, "N": wl.N, "K": wl.K, "V": wl.V},
        "source": "fp64 oracle of Eq. (10)-(13)/(17) of the M2RNN notes; written by "
                  "tests/golden/make_golden.py (oracle only)",
        "inputs": {k: (None if v is None else v.ravel().tolist()) for k, v in inp.items()},
        "y": y.ravel().tolist(),
        "H_T": HT.ravel().tolist(),
    }
    with open(os.path.join(HERE, NAME + ".json"), "w") as fh:
        json.dump(doc, fh, indent=0)


if __name__ == "__main__":
    main()
