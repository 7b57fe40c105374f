"""The oracle still reproduces its committed tiny fixture (tests/golden/oracle_tiny.json,
written by tests/golden/make_golden.py from the oracle alone; GQA 2:1, causal with
S_q < S_k, so the bottom-right mask and the group sum are both exercised)."""
import json
import os

import numpy as np

import oracle

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_tiny.json")


def test_oracle_matches_tiny_fixture():
    g = json.load(open(GOLD))
    arr = {k: np.array(g[k]) for k in ("Q", "K", "V", "dO")}
    O, LSE = oracle.ref_fwd(arr["Q"], arr["K"], arr["V"], g["scale"], g["causal"])
    dQ, dK, dV, D = oracle.ref_bwd(arr["dO"], arr["Q"], arr["K"], arr["V"], O, LSE, g["scale"], g["causal"])
    for name, got in (("O", O), ("LSE", LSE), ("D", D), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        np.testing.assert_allclose(got, np.array(g[name]), rtol=1e-12, atol=1e-13, err_msg=name)
