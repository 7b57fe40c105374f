"""Writes tests/golden/oracle_tiny.json from the fp64 oracle only (no CUDA path).

A small regression fixture: if the oracle's arithmetic is ever changed, the
change must show up here and be justified (the pages print no worked example
with values, so the fixture's values are the oracle's, pinned by the tests in
test_oracle_pins.py).  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402


def case():
    rng = np.random.default_rng(2024)
    B, H, H_kv, S_q, S_k, d = 1, 2, 1, 3, 4, 4
    Q = np.round(rng.standard_normal((B, H, S_q, d)), 3)
    K = np.round(rng.standard_normal((B, H_kv, S_k, d)), 3)
    V = np.round(rng.standard_normal((B, H_kv, S_k, d)), 3)
    dO = np.round(rng.standard_normal((B, H, S_q, d)), 3)
    return dict(B=B, H=H, H_kv=H_kv, S_q=S_q, S_k=S_k, d=d, scale=0.5, causal=True,
                Q=Q, K=K, V=V, dO=dO)


def main():
    c = case()
    O, LSE = oracle.ref_fwd(c["Q"], c["K"], c["V"], c["scale"], c["causal"])
    dQ, dK, dV, D = oracle.ref_bwd(c["dO"], c["Q"], c["K"], c["V"], O, LSE, c["scale"], c["causal"])
    out = {k: (v.tolist() if isinstance(v, np.ndarray) else v) for k, v in c.items()}
    out.update(O=O.tolist(), LSE=LSE.tolist(), D=D.tolist(), dQ=dQ.tolist(), dK=dK.tolist(), dV=dV.tolist())
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
